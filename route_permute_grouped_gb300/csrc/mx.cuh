// MXFP8 (microscaling FP8) device helpers: quantisation of 32-element blocks
// and the tile-ready layout of the block scales read by the block-scaled
// tcgen05 MMA.
//
// Format (OCP Microscaling Formats v1.0, MXFP8 with E4M3 elements; the report
// names the recipe: captions page, Table 11 and Fig. 30): a block of 32
// consecutive elements along a GEMM operand's K shares one E8M0 scale
// X = 2^s, s = floor(log2 max|v|) - 8 clamped to [-127, 127] (-127 for an
// all-zero block), stored as the byte s + 127; each element is v / X rounded to
// E4M3 to nearest, ties to even, saturating at +-448.
//
// Scale layout in TMEM (as the block-scaled MMA with scale_vec::1X reads it,
// M = 128): the scale of A row m is byte `id` of the 32-bit cell (lane m,
// column sfa + m / 32); the scale of B row n is byte `id` of the cell
// (lane 32 q + n % 32, column sfb + n / 32) for the lane quarter q of every
// output row, i.e. B's scales are replicated in the four lane quarters. `id`
// selects the K=32 step inside a 128-element k block. tcgen05.cp 32x128b
// .warpx4 writes exactly that from 512 contiguous bytes: byte 16 r + 4 c + s
// of a scale block is the scale of row 32 c + r of a 128-row block, K step s.
// A 128-row operand block and a k block of 128 elements therefore own one
// 512-byte scale block; a 192-row B tile owns two (rows 128.. in the second,
// the unused half zero).
#pragma once
#include "common.cuh"

namespace moe {

constexpr int kMxBlock = 32;     // elements per scale
constexpr int kMxKB = 128;       // elements (bytes) per k block of an FP8 stage
constexpr int kMxSfBytes = 512;  // scale block of 128 rows x one k block

// FP8 expert GEMM tiles: gate/up tiles of 96 gate + 96 up columns, down tiles
// of 192 columns (two 192-column accumulators and the scale columns fit the
// 512 TMEM columns)
constexpr int kMxTileF1 = 96;
constexpr int kMxTileN2 = 192;
constexpr int kMxBN = 192;  // UMMA N of both

// byte offset of the scale of row `row` (0..127 of its block), K step s
__host__ __device__ __forceinline__ int mx_sf_pos(int row, int s) {
  return 16 * (row & 31) + 4 * ((row >> 5) & 3) + s;
}

// E8M0 scale byte of a block with maximum magnitude amax (finite, >= 0):
// floor(log2 amax) - 8 + 127 is the fp32 biased exponent minus 8; subnormal
// and zero maxima give s = -127 (byte 0).
__device__ __forceinline__ uint32_t mx_scale_byte(float amax) {
  const int e = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu);
  return static_cast<uint32_t>(e > 8 ? e - 8 : 0);
}

// two fp32 -> two E4M3 bytes (round to nearest even, saturating): lo in the
// low byte
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// E4M3 codes of 8 elements of a block whose scale byte is sb (w[0] holds
// elements 0..3, low byte first)
__device__ __forceinline__ void mx_codes8(const float (&v)[8], uint32_t sb, uint32_t (&w)[2]) {
  const float inv = __uint_as_float((254u - sb) << 23);  // 1 / X, as in mx_quant32
#pragma unroll
  for (int j = 0; j < 2; ++j)
    w[j] = cvt_e4m3x2(v[4 * j] * inv, v[4 * j + 1] * inv) | (cvt_e4m3x2(v[4 * j + 2] * inv, v[4 * j + 3] * inv) << 16);
}

// Quantise one 32-element block: codes in w[0..7] (byte j of the block at
// byte j of w), returns the scale byte.
__device__ __forceinline__ uint32_t mx_quant32(const float (&v)[32], uint32_t (&w)[8]) {
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(v[j]));
  const uint32_t sb = mx_scale_byte(amax);
  // 1 / X = 2^(127 - sb) as an fp32 bit pattern (sb in [0, 246]: exponent
  // field 254 - sb in [8, 254], a normal power of two); v / X is exact
  const float inv = __uint_as_float((254u - sb) << 23);
#pragma unroll
  for (int j = 0; j < 8; ++j)
    w[j] = cvt_e4m3x2(v[4 * j] * inv, v[4 * j + 1] * inv) | (cvt_e4m3x2(v[4 * j + 2] * inv, v[4 * j + 3] * inv) << 16);
  return sb;
}

// Tiles of `rows` rows before each expert: s_pt[e] = sum over e' < e of
// ceil(count_e' / rows), from the row offsets s_off[0..E] (E <= 256). Run by
// one whole warp: lane l sums experts 8 l .. 8 l + 7, then a warp scan;
// s_pt[E] is the total.
__device__ __forceinline__ void tile_prefix_warp(const int* s_off, int* s_pt, int E, int lane, int rows) {
  int t[8], sum = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int e = 8 * lane + j;
    t[j] = e < E ? (s_off[e + 1] - s_off[e] + rows - 1) / rows : 0;
    sum += t[j];
  }
  int incl = sum;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += v;
  }
  int run = incl - sum;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int e = 8 * lane + j;
    if (e <= E) s_pt[e] = run;
    run += t[j];
  }
}

// First 256-row CTA-pair tile of each expert in the grouped GEMMs' schedule
__device__ __forceinline__ void pair_tile_prefix_warp(const int* s_off, int* s_pt, int E, int lane) {
  tile_prefix_warp(s_off, s_pt, E, lane, 256);
}

// expert e with s_off[e] <= row < s_off[e + 1] (binary search over E experts)
__device__ __forceinline__ int expert_of_row(const int* s_off, int E, int row) {
  int lo = 0, hi = E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_off[mid] <= row) lo = mid; else hi = mid;
  }
  return lo;
}

// Byte offset of the scale of row `rel` (relative to its expert's first row)
// and 32-element block `b` (of nkb k blocks of 128) in the activations'
// tile-ready scale blocks: block 2 P + h, P = pt_first + rel / 256 (the
// row's CTA-pair tile), h = (rel / 128) % 2 (its CTA of the pair).
__device__ __forceinline__ size_t mx_act_sf_offset(int pt_first, int rel, int b, int nkb) {
  const int blk = 2 * (pt_first + rel / 256) + ((rel / 128) & 1);
  return (static_cast<size_t>(blk) * nkb + b / 4) * kMxSfBytes + mx_sf_pos(rel % 128, b & 3);
}

}  // namespace moe

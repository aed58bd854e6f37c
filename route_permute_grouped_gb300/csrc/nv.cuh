// NVFP4 device helpers: quantisation of 16-element blocks and the tile-ready
// layout of the block scales read by the block-scaled tcgen05 MMA
// (kind::mxf4nvf4, scale_vec::4X).
//
// Format (NVIDIA's NVFP4; the report lists the precision: summary page,
// "Modeling" and "Key Terms"): E2M1 elements (magnitudes 0, 0.5, 1, 1.5, 2,
// 3, 4, 6), a positive E4M3 scale per 16 consecutive elements along K, and
// an fp32 tensor scale g = amax(tensor) / (6 * 448) (1 for a zero tensor).
// Encoding in fp32, each operation rounded to nearest even:
//   s_b = E4M3(fp32(amax_b / 6) / g), t = fp32(s_b * g), q = E2M1(v / t)
// (q = 0 where t == 0); E4M3 and E2M1 round to nearest even and saturate.
// Codes are packed two per byte, element 2j in the low nibble.
//
// Scale layout in TMEM (measured: scale_vec::4X, M = 128): the scales of one
// K=64 MMA step (four 16-element blocks) are the four bytes of one 32-bit
// cell, at the same (lane, column) places as the E8M0 scales of the MXFP8
// MMA (A row m: lane m, column sfa + m / 32; B row n: lane 32 q + n % 32 of
// every lane quarter q, column sfb + n / 32). A k block of 256 elements has
// four steps, so its 128-row scale block is 4 x 512 bytes: byte
// 512 s + 16 r + 4 c + j = scale of row 32 c + r, 16-element block 4 s + j.
#pragma once
#include <cuda_fp4.h>

#include "common.cuh"
#include "mx.cuh"

namespace moe {

constexpr int kNvBlock = 16;        // elements per scale
constexpr int kNvKB = 256;          // elements per k block (128 bytes of codes per row)
constexpr int kNvSfBytes = 2048;    // scale block of 128 rows x one k block (4 steps x 512 bytes)
constexpr int kNvTileN = 192;       // B rows per tile (two 192-column accumulators)
constexpr float kNvScaleDen = 6.0f * 448.0f;

// byte offset of the scale of row `row` (0..127 of its block), 16-element
// block `blk` (0..15) of the k block
__host__ __device__ __forceinline__ int nv_sf_pos(int row, int blk) {
  return 512 * (blk >> 2) + 16 * (row & 31) + 4 * ((row >> 5) & 3) + (blk & 3);
}

__device__ __forceinline__ float nv_tensor_scale(float amax) {
  const float g = __fdiv_rn(amax, kNvScaleDen);
  return g == 0.0f ? 1.0f : g;
}

// E4M3 byte of a non-negative fp32 (round to nearest even, saturating) and its
// value
__device__ __forceinline__ uint32_t e4m3_byte(float s) { return cvt_e4m3x2(s, 0.0f) & 0xFFu; }
__device__ __forceinline__ float e4m3_value(uint32_t c) {
  const uint32_t e = (c >> 3) & 15u, m = c & 7u;
  // subnormal: m 2^-9; normal: (8 + m) 2^(e - 10)
  return e == 0 ? static_cast<float>(m) * 0.001953125f
                : __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// Quantise one 16-element block with tensor scale g: codes in w[0..1] (byte j
// of the block's 8 bytes at byte j of w), returns the scale byte.
__device__ __forceinline__ uint32_t nv_quant16(const float (&v)[16], float g, uint32_t (&w)[2]) {
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(v[j]));
  const uint32_t sb = e4m3_byte(__fdiv_rn(__fdiv_rn(amax, 6.0f), g));
  const float t = __fmul_rn(e4m3_value(sb), g);
  uint32_t b[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float lo = t > 0.0f ? __fdiv_rn(v[2 * j], t) : 0.0f;
    const float hi = t > 0.0f ? __fdiv_rn(v[2 * j + 1], t) : 0.0f;
    b[j] = static_cast<uint32_t>(__nv_cvt_float2_to_fp4x2(make_float2(lo, hi), __NV_E2M1, cudaRoundNearest));
  }
  w[0] = b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24);
  w[1] = b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24);
  return sb;
}

}  // namespace moe

// MXFP8 quantisers: row-major blocks of a bf16 matrix, and the expert weights
// transposed to K-major E4M3 with their scales in the tile-ready layout of the
// FP8 expert GEMMs (see mx.cuh for the format and the scale layout).
#include "host_util.h"
#include "mx.cuh"

namespace moe {

// q[M, K] codes and s[M, K/32] scales of x[M, K] (row-major, blocks along K).
// Thread = one block of 32 elements: four 16-byte loads, two 16-byte stores.
__global__ void __launch_bounds__(256) mx_quantize_rows_kernel(const __nv_bfloat16* __restrict__ x, long long M,
                                                               int K, uint8_t* __restrict__ q,
                                                               uint8_t* __restrict__ s) {
  const int nb = K / kMxBlock;
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= M * nb) return;
  const long long row = i / nb;
  const int b = static_cast<int>(i - row * nb);
  const uint4* src = reinterpret_cast<const uint4*>(x + row * K + b * kMxBlock);
  float v[32];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const uint4 w = __ldg(src + u);
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[8 * u + 2 * j] = bf16_lo(ww[j]);
      v[8 * u + 2 * j + 1] = bf16_hi(ww[j]);
    }
  }
  uint32_t c[8];
  s[i] = static_cast<uint8_t>(mx_quant32(v, c));
  uint4* dst = reinterpret_cast<uint4*>(q + row * K + b * kMxBlock);
  dst[0] = make_uint4(c[0], c[1], c[2], c[3]);
  dst[1] = make_uint4(c[4], c[5], c[6], c[7]);
}

// Weight W[E][K][N] bf16 (K rows, N contiguous) -> codes Wq (expert e at
// wq + e * wq_estride, row n of K contiguous codes) and the scale of
// (e, n, 32-element K block kb32) in expert e's tile-ready scale blocks
// (sf + e * sf_estride): tile n / tile_n, k block kb32 / 4, B row of the tile
// b = n % tile_n + row_off (row_off: 0 for W1 and W2, tile_n for W3, whose
// rows follow W1's in a gate/up tile); every (tile, k block) owns two 512-byte
// blocks (B rows 0..127, 128..255). Block = one (e, 128-element k block, 64
// columns): the 128 x 64 bf16 tile is staged in shared memory with 16-byte
// loads (whole 128-byte rows), thread = one (column, 32-element block) (a warp:
// 32 consecutive columns of one block) quantises from shared memory into a
// staged 64 x 128-byte code tile, which leaves in whole 128-byte lines. N is a
// multiple of 8, K of 128.
constexpr int kMxWqCols = 64;
__global__ void __launch_bounds__(256) mx_quantize_weight_kernel(const __nv_bfloat16* __restrict__ w, int E, int K,
                                                                 int N, uint8_t* __restrict__ wq, size_t wq_estride,
                                                                 uint8_t* __restrict__ sf, size_t sf_estride,
                                                                 int tile_n, int row_off) {
  __shared__ __align__(16) __nv_bfloat16 tile[kMxKB][kMxWqCols + 8];  // 144-byte rows
  __shared__ __align__(16) uint8_t codes[kMxWqCols][kMxKB + 16];      // 144-byte rows
  const int nkb = K / kMxKB;
  const int nnb = (N + kMxWqCols - 1) / kMxWqCols;
  long long bid = blockIdx.x;
  const int kb = static_cast<int>(bid % nkb);
  bid /= nkb;
  const int nb = static_cast<int>(bid % nnb);
  const int e = static_cast<int>(bid / nnb);
  if (e >= E) return;
  const int n0 = nb * kMxWqCols;
  const int ncols = min(kMxWqCols, N - n0);
  const __nv_bfloat16* src = w + (static_cast<size_t>(e) * K + static_cast<size_t>(kb) * kMxKB) * N + n0;
  const int t = threadIdx.x;
  {
    // 128 rows x 8 chunks of 16 bytes: thread t takes chunk t % 8 of rows t / 8 + 32 i
    const int c = t & 7;
    if (8 * c < ncols) {
      uint4 v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        v[i] = __ldg(reinterpret_cast<const uint4*>(src + static_cast<size_t>((t >> 3) + 32 * i) * N) + c);
#pragma unroll
      for (int i = 0; i < 4; ++i) *reinterpret_cast<uint4*>(&tile[(t >> 3) + 32 * i][8 * c]) = v[i];
    }
  }
  __syncthreads();
  const int col = t & 63, blk = t >> 6;  // column of the tile, 32-element block of the k block
  if (col < ncols) {
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __bfloat162float(tile[32 * blk + j][col]);
    uint32_t c[8];
    const uint32_t sb = mx_quant32(v, c);
    uint4* d = reinterpret_cast<uint4*>(&codes[col][32 * blk]);
    d[0] = make_uint4(c[0], c[1], c[2], c[3]);
    d[1] = make_uint4(c[4], c[5], c[6], c[7]);
    const int n = n0 + col;
    const int kb32 = 4 * kb + blk;
    const int tl = n / tile_n;
    const int b = n % tile_n + row_off;  // B row of the tile
    const size_t sblk = static_cast<size_t>(tl) * (K / kMxKB) + kb32 / 4;
    sf[e * sf_estride + sblk * 2 * kMxSfBytes + (b >> 7) * kMxSfBytes + mx_sf_pos(b & 127, kb32 & 3)] =
        static_cast<uint8_t>(sb);
  }
  __syncthreads();
  // 64 code rows of 128 bytes: thread t stores 16-byte pieces t % 8 of rows t / 8 and t / 8 + 32
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int r = (t >> 3) + 32 * i;
    if (r < ncols)
      reinterpret_cast<uint4*>(wq + e * wq_estride + static_cast<size_t>(n0 + r) * K +
                               static_cast<size_t>(kb) * kMxKB)[t & 7] =
          *reinterpret_cast<const uint4*>(&codes[r][16 * (t & 7)]);
  }
}

static unsigned mx_weight_blocks(int E, int K, int N) {
  return static_cast<unsigned>(static_cast<long long>(E) * (K / kMxKB) * ((N + kMxWqCols - 1) / kMxWqCols));
}

cudaError_t launch_mx_quantize_rows(const __nv_bfloat16* x, long long M, int K, uint8_t* q, uint8_t* s,
                                    cudaStream_t st) {
  const long long n = M * (K / kMxBlock);
  if (n == 0) return cudaSuccess;
  mx_quantize_rows_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, st>>>(x, M, K, q, s);
  return cudaGetLastError();
}

// W1/W3 [E, H, F] -> w13q [E][2][F][H] (W1 then W3 per expert) and sf13; W2
// [E, F, H] -> w2q [E][H][F] and sf2. The scale buffers are zeroed first (the
// unused half of each tile's second scale block stays zero).
cudaError_t launch_mx_quantize_weights(const moe_config& c, const __nv_bfloat16* W1, const __nv_bfloat16* W3,
                                       const __nv_bfloat16* W2, uint8_t* w13q, uint8_t* sf13, uint8_t* w2q,
                                       uint8_t* sf2, cudaStream_t st) {
  const int E = c.E, H = c.H, F = c.F;
  const int nt1 = mx_ntiles1(c), nt2 = mx_ntiles2(c);
  cudaError_t err = cudaMemsetAsync(sf13, 0, mx_sf13_bytes(c), st);
  if (err != cudaSuccess) return err;
  err = cudaMemsetAsync(sf2, 0, mx_sf2_bytes(c), st);
  if (err != cudaSuccess) return err;
  // W1 and W3 of expert e land in w13q[e][0] and w13q[e][1]
  const size_t sf13_e = static_cast<size_t>(nt1) * (H / kMxKB) * 2 * kMxSfBytes;
  for (int which = 0; which < 2; ++which) {
    mx_quantize_weight_kernel<<<mx_weight_blocks(E, H, F), 256, 0, st>>>(
        which == 0 ? W1 : W3, E, H, F, w13q + static_cast<size_t>(which) * F * H, 2ull * F * H, sf13, sf13_e,
        kMxTileF1, which * kMxTileF1);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  const size_t sf2_e = static_cast<size_t>(nt2) * (F / kMxKB) * 2 * kMxSfBytes;
  mx_quantize_weight_kernel<<<mx_weight_blocks(E, F, H), 256, 0, st>>>(
      W2, E, F, H, w2q, static_cast<size_t>(H) * F, sf2, sf2_e, kMxTileN2, 0);
  return cudaGetLastError();
}

// 32 bf16 (64 contiguous bytes, 16-byte aligned) to fp32
__device__ __forceinline__ void ld_bf16x32(const __nv_bfloat16* p, float (&v)[32]) {
  const uint4* src = reinterpret_cast<const uint4*>(p);
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const uint4 w = __ldg(src + u);
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[8 * u + 2 * j] = bf16_lo(ww[j]);
      v[8 * u + 2 * j + 1] = bf16_hi(ww[j]);
    }
  }
}
__device__ __forceinline__ void st_codes32(uint8_t* dst, const uint32_t (&c)[8]) {
  uint4* d = reinterpret_cast<uint4*>(dst);
  d[0] = make_uint4(c[0], c[1], c[2], c[3]);
  d[1] = make_uint4(c[4], c[5], c[6], c[7]);
}
// Weight rows with K contiguous (row n of expert e at w + e * w_estride +
// n * ldw) -> codes at wq + e * wq_estride + n * ldq + 128 kb_off + 32 kb32
// and the scale of (n, kb32) in expert e's tile-ready blocks (sf +
// e * sf_estride): tile n / tile_n, k block kb_off + kb32 / 4 of nkb_row per
// tile, B row n % tile_n. Thread = one (e, n, kb32), kb32 fastest: four
// 16-byte loads, two 16-byte stores.
__global__ void __launch_bounds__(256) mx_quantize_weight_rows_kernel(
    const __nv_bfloat16* __restrict__ w, int E, int N, int K, size_t w_estride, int ldw, uint8_t* __restrict__ wq,
    size_t wq_estride, int ldq, int kb_off, int nkb_row, uint8_t* __restrict__ sf, size_t sf_estride, int tile_n) {
  const int nkb32 = K / kMxBlock;
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= static_cast<long long>(E) * N * nkb32) return;
  const int kb32 = static_cast<int>(i % nkb32);
  const long long r = i / nkb32;
  const int n = static_cast<int>(r % N);
  const int e = static_cast<int>(r / N);
  float v[32];
  ld_bf16x32(w + e * w_estride + static_cast<size_t>(n) * ldw + kb32 * kMxBlock, v);
  uint32_t c[8];
  const uint32_t sb = mx_quant32(v, c);
  st_codes32(wq + e * wq_estride + static_cast<size_t>(n) * ldq + kb_off * kMxKB + kb32 * kMxBlock, c);
  const int b = n % tile_n;
  const size_t blk = static_cast<size_t>(n / tile_n) * nkb_row + kb_off + kb32 / 4;
  sf[e * sf_estride + blk * 2 * kMxSfBytes + (b >> 7) * kMxSfBytes + mx_sf_pos(b & 127, kb32 & 3)] =
      static_cast<uint8_t>(sb);
}

// The transposed MXFP8 operand of a weight-gradient GEMM, whose K runs over
// each expert's tokens: rows of X [R, C] bf16 (row stride ldx) grouped by
// expert (offsets[0..E]) -> XT [C][ldk] E4M3 codes, column p of XT = padded token position p (expert
// e's rows at P_e .. P_e + count_e - 1, zeros up to P_{e+1}; P_e = 128 * sum
// over e' < e of ceil(count_e' / 128), so every 128-position k block lies in
// one expert), blocks of 32 positions along a row of XT sharing one E8M0
// scale. Scales in the tile-ready layout of an MXFP8 operand with tile_rows
// rows per tile (128: an A operand, 192: a B operand): the scale of (row c,
// block g) at byte ((c / tile_rows * kbt + g / 4) * nblk + (c % tile_rows) /
// 128) * 512 + pos((c % tile_rows) % 128, g % 4), nblk = ceil(tile_rows / 128),
// kbt = k blocks of the padded axis. Block (x, y) = positions 32 x .. 32 x + 31
// and columns 256 y ..: the 32 x 256 bf16 tile is staged in shared memory with
// 16-byte loads (one 512-byte row per warp load), then thread t quantises
// column t from it (one 32-byte store). Block (0, 0) also writes P[0..E].
__global__ void __launch_bounds__(256) mx_quantize_tokens_kernel(const __nv_bfloat16* __restrict__ X, int C, int ldx,
                                                                 int E, const int32_t* __restrict__ offsets,
                                                                 uint8_t* __restrict__ XT, size_t ldk,
                                                                 uint8_t* __restrict__ sf, int tile_rows, int kbt,
                                                                 int32_t* __restrict__ pad_off) {
  __shared__ int s_off[kMaxGroups + 1];
  __shared__ int s_kb[kMaxGroups + 1];  // 128-position k blocks before each expert
  __shared__ __align__(16) __nv_bfloat16 s_x[32][256];
  const int tid = threadIdx.x;
  for (int i = tid; i <= E; i += blockDim.x) s_off[i] = offsets[i];
  __syncthreads();
  if (tid < 32) tile_prefix_warp(s_off, s_kb, E, tid, kMxKB);
  __syncthreads();
  if (blockIdx.x == 0 && blockIdx.y == 0)
    for (int i = tid; i <= E; i += blockDim.x) pad_off[i] = kMxKB * s_kb[i];
  const int g = blockIdx.x;  // 32-position block
  const int pos = kMxBlock * g;
  if (pos >= kMxKB * s_kb[E]) return;  // uniform over the block
  const int e = expert_of_row(s_kb, E, pos / kMxKB);
  const int j0 = pos - kMxKB * s_kb[e];
  const int cnt = s_off[e + 1] - s_off[e];
  const int c0 = 256 * blockIdx.y;
  // stage: warp w loads rows w, w + 8, w + 16, w + 24; lane l columns 8 l ..
  const int w = tid >> 5, l = tid & 31;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = w + 8 * i;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (j0 + r < cnt && c0 + 8 * l < C)
      v = __ldg(reinterpret_cast<const uint4*>(X + static_cast<size_t>(s_off[e] + j0 + r) * ldx + c0 + 8 * l));
    *reinterpret_cast<uint4*>(&s_x[r][8 * l]) = v;
  }
  __syncthreads();
  const int c = c0 + tid;
  if (c >= C) return;
  float v[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __bfloat162float(s_x[i][tid]);
  uint32_t q[8];
  const uint32_t sb = mx_quant32(v, q);
  st_codes32(XT + static_cast<size_t>(c) * ldk + pos, q);
  const int b = c % tile_rows;
  const int nblk = (tile_rows + 127) / 128;
  sf[((static_cast<size_t>(c / tile_rows) * kbt + g / 4) * nblk + (b >> 7)) * kMxSfBytes + mx_sf_pos(b & 127, g & 3)] =
      static_cast<uint8_t>(sb);
}

cudaError_t launch_mx_quantize_tokens(const __nv_bfloat16* X, int R, int C, int ldx, int E, const int32_t* offsets,
                                      uint8_t* XT, uint8_t* sf, int tile_rows, int32_t* pad_off, cudaStream_t st) {
  const int kbt = mx_wg_kbt(R, E);
  cudaError_t err = cudaMemsetAsync(sf, 0, mx_tok_sf_bytes(C, tile_rows, kbt), st);
  if (err != cudaSuccess) return err;
  const dim3 grid(static_cast<unsigned>(kbt * (kMxKB / kMxBlock)), static_cast<unsigned>((C + 255) / 256));
  mx_quantize_tokens_kernel<<<grid, 256, 0, st>>>(X, C, ldx, E, offsets, XT, static_cast<size_t>(kbt) * kMxKB, sf,
                                                   tile_rows, kbt, pad_off);
  return cudaGetLastError();
}

// Weights of the two data-gradient GEMMs: W2 [E, F, H] quantised along H
// (B rows = F, tiles of 192) -> w2h [E][F][H], sf2h; W1 | W3 [E, H, F]
// quantised along F into one K = 2F operand (B rows = H, tiles of 192; W1 in
// k blocks 0 .. F/128 - 1, W3 after it) -> w13f [E][H][2F], sf13f.
cudaError_t launch_mx_quantize_bwd_weights(const moe_config& c, const __nv_bfloat16* W1, const __nv_bfloat16* W3,
                                           const __nv_bfloat16* W2, uint8_t* w2h, uint8_t* sf2h, uint8_t* w13f,
                                           uint8_t* sf13f, cudaStream_t st) {
  const int E = c.E, H = c.H, F = c.F;
  cudaError_t err = cudaMemsetAsync(sf2h, 0, mx_sf2h_bytes(c), st);
  if (err != cudaSuccess) return err;
  err = cudaMemsetAsync(sf13f, 0, mx_sf13f_bytes(c), st);
  if (err != cudaSuccess) return err;
  const long long n2 = static_cast<long long>(E) * F * (H / kMxBlock);
  const int nkb2 = H / kMxKB;
  mx_quantize_weight_rows_kernel<<<static_cast<unsigned>((n2 + 255) / 256), 256, 0, st>>>(
      W2, E, F, H, static_cast<size_t>(F) * H, H, w2h, static_cast<size_t>(F) * H, H, 0, nkb2, sf2h,
      mx_sf2h_bytes(c) / E, kMxTileN2);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const long long n13 = static_cast<long long>(E) * H * (F / kMxBlock);
  const int nkb13 = 2 * F / kMxKB;
  for (int which = 0; which < 2; ++which) {
    mx_quantize_weight_rows_kernel<<<static_cast<unsigned>((n13 + 255) / 256), 256, 0, st>>>(
        which == 0 ? W1 : W3, E, H, F, static_cast<size_t>(H) * F, F, w13f, 2ull * H * F, 2 * F,
        which * (F / kMxKB), nkb13, sf13f, mx_sf13f_bytes(c) / E, kMxTileN2);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
}

}  // namespace moe

// NVFP4 quantisers (see nv.cuh for the format and the scale layout): tensor
// maxima, row-major blocks of a bf16 matrix, expert weights transposed to
// K-major codes with tile-ready scales, and the grouped rows of an expert
// GEMM's activations with tile-ready scales per 256-row pair tile.
#include "host_util.h"
#include "nv.cuh"

namespace moe {

// out[grp] = bits of max |x| over group grp's n_per elements (non-negative
// fp32 values order like their bit patterns); 8 elements per 16-byte load
__global__ void __launch_bounds__(256) nv_amax_kernel(const __nv_bfloat16* __restrict__ x, long long n_per,
                                                      unsigned* __restrict__ out) {
  const uint4* base = reinterpret_cast<const uint4*>(x + static_cast<size_t>(blockIdx.y) * n_per);
  const long long nv = n_per / 8;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  float m = 0.0f;
  // four independent 16-byte loads in flight per thread
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < nv; i += 4 * stride) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = i + u * stride < nv ? __ldg(base + i + u * stride) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) m = fmaxf(m, fmaxf(fabsf(bf16_lo(w[j])), fabsf(bf16_hi(w[j]))));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) atomicMax(out + blockIdx.y, __float_as_uint(m));
}

// g[i] = tensor scale of the maximum whose bits g[i] holds
__global__ void nv_scale_from_amax_kernel(float* g, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) g[i] = nv_tensor_scale(g[i]);
}

__device__ __forceinline__ void load_bf16x16(const __nv_bfloat16* src, float (&v)[16]) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const uint4 w = __ldg(s + u);
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[8 * u + 2 * j] = bf16_lo(ww[j]);
      v[8 * u + 2 * j + 1] = bf16_hi(ww[j]);
    }
  }
}

// x [M, K] -> q [M, K/2] (two codes per byte), s [M, K/16] E4M3 bytes, with
// the tensor scale *g; thread = one 16-element block
__global__ void __launch_bounds__(256) nv_quantize_rows_kernel(const __nv_bfloat16* __restrict__ x, long long M,
                                                               int K, const float* __restrict__ g,
                                                               uint8_t* __restrict__ q, uint8_t* __restrict__ s) {
  const int nb = K / kNvBlock;
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= M * nb) return;
  const long long row = i / nb;
  const int b = static_cast<int>(i - row * nb);
  float v[16];
  load_bf16x16(x + row * K + b * kNvBlock, v);
  uint32_t w[2];
  s[i] = static_cast<uint8_t>(nv_quant16(v, *g, w));
  *reinterpret_cast<uint2*>(q + row * (K / 2) + b * (kNvBlock / 2)) = make_uint2(w[0], w[1]);
}

// Weights W[E][K][N] -> codes wq[E][N][K/2] (K-major) and the scale of
// (e, n, block kb16) in the tile-ready blocks sf[e][n / 192][kb16 / 16][2][2048]
// (B row b = n % 192 of the tile: block b / 128, row b % 128), tensor scale
// g[e]; thread = one (e, n, kb16): 16 strided loads, coalesced over n.
// Columns [split, N) come from a second weight w_hi (row stride N - split):
// the gate/up weights W1 | W3 quantised as one tensor per expert. With
// gate_up set, the scales follow the gate/up GEMM's tiles instead: tile t
// holds W1 columns 96 t .. as B rows 0..95 and W3 columns 96 t .. as B rows
// 96..191 (ceil(split / 96) tiles).
__global__ void __launch_bounds__(256) nv_quantize_weight_kernel(const __nv_bfloat16* __restrict__ w,
                                                                 const __nv_bfloat16* __restrict__ w_hi, int split,
                                                                 int gate_up, int E, int K, int N,
                                                                 const float* __restrict__ g,
                                                                 uint8_t* __restrict__ wq, uint8_t* __restrict__ sf) {
  const int nkb16 = K / kNvBlock;
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= static_cast<long long>(E) * nkb16 * N) return;
  const int n = static_cast<int>(i % N);
  const long long r = i / N;
  const int kb16 = static_cast<int>(r % nkb16);
  const int e = static_cast<int>(r / nkb16);
  const bool hi = n >= split;
  const int ld = hi ? N - split : split;
  const __nv_bfloat16* src = (hi ? w_hi : w) + (static_cast<size_t>(e) * K + static_cast<size_t>(kb16) * kNvBlock) * ld +
                             (hi ? n - split : n);
  float v[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = __bfloat162float(src[static_cast<size_t>(j) * ld]);
  uint32_t c[2];
  const uint32_t sb = nv_quant16(v, g[e], c);
  *reinterpret_cast<uint2*>(wq + (static_cast<size_t>(e) * N + n) * (K / 2) + static_cast<size_t>(kb16) * 8) =
      make_uint2(c[0], c[1]);
  int ntiles, tile, b;
  if (gate_up) {
    const int f = hi ? n - split : n;
    ntiles = (split + kMxTileF1 - 1) / kMxTileF1;
    tile = f / kMxTileF1;
    b = f % kMxTileF1 + (hi ? kMxTileF1 : 0);
  } else {
    ntiles = (N + kNvTileN - 1) / kNvTileN;
    tile = n / kNvTileN;
    b = n % kNvTileN;
  }
  const size_t blk = (static_cast<size_t>(e) * ntiles + tile) * (K / kNvKB) + kb16 / 16;
  sf[blk * 2 * kNvSfBytes + (b >> 7) * kNvSfBytes + nv_sf_pos(b & 127, kb16 & 15)] = static_cast<uint8_t>(sb);
}

// Grouped rows of x [R, K] (expert e's rows offsets[e]..offsets[e+1]) ->
// codes xq [R, K/2] and scale blocks 2 P + h per k block, P = the expert's
// first 256-row pair tile + rel / 256, h = (rel / 128) % 2 (rel = row -
// offsets[e]); thread = one 16-element block. Scales of rows past an expert's
// count are left as they are (zeroed by the caller).
__global__ void __launch_bounds__(256) nv_quantize_grouped_kernel(const __nv_bfloat16* __restrict__ x, int R, int K,
                                                                  int E, const int32_t* __restrict__ offsets,
                                                                  const float* __restrict__ g,
                                                                  uint8_t* __restrict__ xq,
                                                                  uint8_t* __restrict__ sf) {
  __shared__ int s_off[kMaxGroups + 1];
  __shared__ int s_pt[kMaxGroups + 1];  // first pair tile of each expert
  for (int i = threadIdx.x; i <= E; i += blockDim.x) s_off[i] = offsets[i];
  __syncthreads();
  if (threadIdx.x < 32) pair_tile_prefix_warp(s_off, s_pt, E, threadIdx.x);
  __syncthreads();
  const int nb = K / kNvBlock;
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= static_cast<long long>(R) * nb) return;
  const int row = static_cast<int>(i / nb);
  const int b = static_cast<int>(i - static_cast<long long>(row) * nb);
  const int lo = expert_of_row(s_off, E, row);
  const int rel = row - s_off[lo];
  float v[16];
  load_bf16x16(x + static_cast<size_t>(row) * K + b * kNvBlock, v);
  uint32_t c[2];
  const uint32_t sb = nv_quant16(v, *g, c);
  *reinterpret_cast<uint2*>(xq + static_cast<size_t>(row) * (K / 2) + b * 8) = make_uint2(c[0], c[1]);
  const int blk = 2 * (s_pt[lo] + rel / (2 * kBM)) + ((rel / kBM) & 1);
  sf[(static_cast<size_t>(blk) * (K / kNvKB) + b / 16) * kNvSfBytes + nv_sf_pos(rel % kBM, b & 15)] =
      static_cast<uint8_t>(sb);
}

cudaError_t launch_nv_amax(const __nv_bfloat16* x, long long n_per, int groups, float* out_bits, cudaStream_t st,
                           const __nv_bfloat16* x2) {
  cudaError_t e = cudaMemsetAsync(out_bits, 0, sizeof(float) * groups, st);
  if (e != cudaSuccess) return e;
  if (x2 != nullptr) {
    // the maxima cover a second tensor of the same shape too
    long long b2 = (n_per / 8 + 255) / 256;
    if (b2 > 8 * num_sms()) b2 = 8 * num_sms();
    if (b2 < 1) b2 = 1;
    nv_amax_kernel<<<dim3(static_cast<unsigned>(b2), groups), 256, 0, st>>>(x2, n_per,
                                                                            reinterpret_cast<unsigned*>(out_bits));
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  long long blocks = (n_per / 8 + 255) / 256;
  if (blocks > 8 * num_sms()) blocks = 8 * num_sms();
  if (blocks < 1) blocks = 1;
  nv_amax_kernel<<<dim3(static_cast<unsigned>(blocks), groups), 256, 0, st>>>(x, n_per,
                                                                              reinterpret_cast<unsigned*>(out_bits));
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  nv_scale_from_amax_kernel<<<(groups + 255) / 256, 256, 0, st>>>(out_bits, groups);
  return cudaGetLastError();
}

cudaError_t launch_nv_quantize_rows(const __nv_bfloat16* x, long long M, int K, const float* g, uint8_t* q,
                                    uint8_t* s, cudaStream_t st) {
  const long long n = M * (K / kNvBlock);
  if (n == 0) return cudaSuccess;
  nv_quantize_rows_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, st>>>(x, M, K, g, q, s);
  return cudaGetLastError();
}

cudaError_t launch_nv_quantize_weights(const __nv_bfloat16* w, int E, int K, int N, const float* g, uint8_t* wq,
                                       uint8_t* sf, cudaStream_t st, const __nv_bfloat16* w_hi, int split) {
  const bool gate_up = w_hi != nullptr;
  cudaError_t e = cudaMemsetAsync(sf, 0, gate_up ? nv_weight_sf_bytes_gu(E, K, split) : nv_weight_sf_bytes(E, K, N), st);
  if (e != cudaSuccess) return e;
  const long long n = static_cast<long long>(E) * (K / kNvBlock) * N;
  nv_quantize_weight_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, st>>>(
      w, w_hi, gate_up ? split : N, gate_up ? 1 : 0, E, K, N, g, wq, sf);
  return cudaGetLastError();
}

cudaError_t launch_nv_scale_from_amax(float* g, int n, cudaStream_t st) {
  nv_scale_from_amax_kernel<<<(n + 255) / 256, 256, 0, st>>>(g, n);
  return cudaGetLastError();
}

cudaError_t launch_nv_quantize_grouped(const __nv_bfloat16* x, int R, int K, int E, const int32_t* offsets,
                                       const float* g, uint8_t* xq, uint8_t* sf, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(sf, 0, nv_act_sf_bytes(R, E, K), st);
  if (e != cudaSuccess) return e;
  const long long n = static_cast<long long>(R) * (K / kNvBlock);
  if (n == 0) return cudaSuccess;
  nv_quantize_grouped_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, st>>>(x, R, K, E, offsets, g, xq, sf);
  return cudaGetLastError();
}

}  // namespace moe

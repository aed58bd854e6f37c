// NVFP4 quantisers (see nv.cuh for the format and the scale layout): tensor
// maxima, row-major blocks of a bf16 matrix, expert weights (transposed, or
// row-wise for the data gradients) to K-major codes with tile-ready scales,
// and the grouped rows of an expert GEMM's activations with tile-ready scales
// per 256-row pair tile; and the SwiGLU backward of the NVFP4 training step.
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
// offsets[e]); thread = one 16-element block (grid-stride, so that each block
// forms the experts' tile prefix once for many). Scales of rows past an
// expert's count are left as they are (zeroed by the caller).
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
  const float gs = *g;
  const long long n = static_cast<long long>(R) * nb;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int row = static_cast<int>(i / nb);
    const int b = static_cast<int>(i - static_cast<long long>(row) * nb);
    const int lo = expert_of_row(s_off, E, row);
    const int rel = row - s_off[lo];
    float v[16];
    load_bf16x16(x + static_cast<size_t>(row) * K + b * kNvBlock, v);
    uint32_t c[2];
    const uint32_t sb = nv_quant16(v, gs, c);
    *reinterpret_cast<uint2*>(xq + static_cast<size_t>(row) * (K / 2) + b * 8) = make_uint2(c[0], c[1]);
    const int blk = 2 * (s_pt[lo] + rel / (2 * kBM)) + ((rel / kBM) & 1);
    sf[(static_cast<size_t>(blk) * (K / kNvKB) + b / 16) * kNvSfBytes + nv_sf_pos(rel % kBM, b & 15)] =
        static_cast<uint8_t>(sb);
  }
}

// Weights stored row-major W[E][N][K] (row n of expert e holds the K
// elements of one GEMM output column; columns [split, K) come from a second
// weight w_hi [E][N][K - split]) -> codes wq[E][N][K/2] and the scales in the
// tile-ready layout of nv_quantize_weight_kernel (B row b = n % 192 of tile
// n / 192), tensor scale g[e]; thread = one (e, n, kb16): two 16-byte loads,
// consecutive threads on consecutive blocks of a row. The data gradients read
// their weights this way: W2_e [F, H] along H, [W1_e | W3_e] [H, 2F] along 2F.
__global__ void __launch_bounds__(256) nv_quantize_weight_rows_kernel(const __nv_bfloat16* __restrict__ w,
                                                                      const __nv_bfloat16* __restrict__ w_hi,
                                                                      int split, int E, int K, int N,
                                                                      const float* __restrict__ g,
                                                                      uint8_t* __restrict__ wq,
                                                                      uint8_t* __restrict__ sf) {
  const int nkb16 = K / kNvBlock;
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= static_cast<long long>(E) * N * nkb16) return;
  const int kb16 = static_cast<int>(i % nkb16);
  const long long r = i / nkb16;
  const int n = static_cast<int>(r % N);
  const int e = static_cast<int>(r / N);
  const int k0 = kb16 * kNvBlock;
  const bool hi = k0 >= split;
  const int ld = hi ? K - split : split;
  const __nv_bfloat16* src =
      (hi ? w_hi : w) + (static_cast<size_t>(e) * N + n) * static_cast<size_t>(ld) + (hi ? k0 - split : k0);
  float v[16];
  load_bf16x16(src, v);
  uint32_t c[2];
  const uint32_t sb = nv_quant16(v, g[e], c);
  *reinterpret_cast<uint2*>(wq + (static_cast<size_t>(e) * N + n) * (K / 2) + static_cast<size_t>(kb16) * 8) =
      make_uint2(c[0], c[1]);
  const int ntiles = (N + kNvTileN - 1) / kNvTileN;
  const int tile = n / kNvTileN, b = n % kNvTileN;
  const size_t blk = (static_cast<size_t>(e) * ntiles + tile) * (K / kNvKB) + kb16 / 16;
  sf[blk * 2 * kNvSfBytes + (b >> 7) * kNvSfBytes + nv_sf_pos(b & 127, kb16 & 15)] = static_cast<uint8_t>(sb);
}

// SwiGLU backward of the NVFP4 training step; thread = 8 columns f.. of row r
// (rows below *n_rows, the routed rows): da fp32 [R, F] and the saved bf16
// pre-activations h13 [R, 2F] (h1 | h3) give dh1 = da h3 SiLU'(h1) and
// dh3 = da SiLU(h1), stored bf16 to dh13 [R, 2F] (h1's columns then h3's), and
// the largest magnitude of the stored values into *amax_bits. Grid-stride
// (blockDim 256): one atomic per block.
__global__ void __launch_bounds__(256) nv_swiglu_bwd_kernel(const float* __restrict__ da,
                                                            const __nv_bfloat16* __restrict__ h13, int R, int F,
                                                            const int32_t* __restrict__ n_rows,
                                                            __nv_bfloat16* __restrict__ dh13,
                                                            unsigned* __restrict__ amax_bits) {
  const int nv = F / 8;
  const int rows = min(R, max(__ldg(n_rows), 0));
  const long long n = static_cast<long long>(rows) * nv;
  float m = 0.0f;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long r = i / nv;
    const int c = static_cast<int>(i - r * nv) * 8;
    const float4* dp = reinterpret_cast<const float4*>(da + r * F + c);
    const float4 d0 = __ldg(dp), d1 = __ldg(dp + 1);
    const float d[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
    const __nv_bfloat16* hr = h13 + r * 2 * F;
    const uint4 v1 = __ldg(reinterpret_cast<const uint4*>(hr + c));
    const uint4 v3 = __ldg(reinterpret_cast<const uint4*>(hr + F + c));
    const uint32_t a1[4] = {v1.x, v1.y, v1.z, v1.w};
    const uint32_t a3[4] = {v3.x, v3.y, v3.z, v3.w};
    uint32_t o1[4], o3[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float d1v[2], d3v[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const float x1 = u ? bf16_hi(a1[q]) : bf16_lo(a1[q]);
        const float x3 = u ? bf16_hi(a3[q]) : bf16_lo(a3[q]);
        const float s = 1.0f / (1.0f + __expf(-x1));
        d1v[u] = d[2 * q + u] * x3 * (s * (1.0f + x1 * (1.0f - s)));
        d3v[u] = d[2 * q + u] * x1 * s;
      }
      o1[q] = pack_bf16x2(d1v[0], d1v[1]);
      o3[q] = pack_bf16x2(d3v[0], d3v[1]);
      m = fmaxf(m, fmaxf(fmaxf(fabsf(bf16_lo(o1[q])), fabsf(bf16_hi(o1[q]))),
                         fmaxf(fabsf(bf16_lo(o3[q])), fabsf(bf16_hi(o3[q])))));
    }
    __nv_bfloat16* orow = dh13 + r * 2 * F;
    *reinterpret_cast<uint4*>(orow + c) = make_uint4(o1[0], o1[1], o1[2], o1[3]);
    *reinterpret_cast<uint4*>(orow + F + c) = make_uint4(o3[0], o3[1], o3[2], o3[3]);
  }
  // one atomic per block
  __shared__ float s_m[8];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) s_m[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < static_cast<int>(blockDim.x >> 5); ++w) m = fmaxf(m, s_m[w]);
    if (m > 0.0f) atomicMax(amax_bits, __float_as_uint(m));
  }
}

cudaError_t launch_nv_amax(const __nv_bfloat16* x, long long n_per, int groups, float* out_bits, cudaStream_t st,
                           const __nv_bfloat16* x2) {
  cudaError_t e = cudaMemsetAsync(out_bits, 0, sizeof(float) * groups, st);
  if (e != cudaSuccess) return e;
  // about eight 256-thread blocks per SM over all groups together (one wave;
  // each thread keeps four 16-byte loads in flight), at most one 16-byte load
  // per thread of a group
  long long blocks = (n_per / 8 + 255) / 256;
  const long long cap = (8ll * num_sms() + groups - 1) / groups;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  if (x2 != nullptr) {
    // the maxima cover a second tensor of the same shape too
    nv_amax_kernel<<<dim3(static_cast<unsigned>(blocks), groups), 256, 0, st>>>(x2, n_per,
                                                                                reinterpret_cast<unsigned*>(out_bits));
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  nv_amax_kernel<<<dim3(static_cast<unsigned>(blocks), groups), 256, 0, st>>>(x, n_per,
                                                                              reinterpret_cast<unsigned*>(out_bits));
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  nv_scale_from_amax_kernel<<<(groups + 255) / 256, 256, 0, st>>>(out_bits, groups);
  return cudaGetLastError();
}

cudaError_t launch_nv_quantize_weight_rows(const __nv_bfloat16* w, int E, int K, int N, const float* g, uint8_t* wq,
                                           uint8_t* sf, cudaStream_t st, const __nv_bfloat16* w_hi, int split) {
  cudaError_t e = cudaMemsetAsync(sf, 0, nv_weight_sf_bytes(E, K, N), st);
  if (e != cudaSuccess) return e;
  const long long n = static_cast<long long>(E) * N * (K / kNvBlock);
  nv_quantize_weight_rows_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, st>>>(
      w, w_hi, w_hi != nullptr ? split : K, E, K, N, g, wq, sf);
  return cudaGetLastError();
}

cudaError_t launch_nv_swiglu_bwd(const float* da, const __nv_bfloat16* h13, int R, int F, const int32_t* n_rows,
                                 __nv_bfloat16* dh13, float* g, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(g, 0, sizeof(float), st);
  if (e != cudaSuccess) return e;
  const long long n = static_cast<long long>(R) * (F / 8);
  if (n > 0) {
    long long blocks = (n + 255) / 256;
    if (blocks > 8 * num_sms()) blocks = 8 * num_sms();
    nv_swiglu_bwd_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(da, h13, R, F, n_rows, dh13,
                                                                        reinterpret_cast<unsigned*>(g));
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  nv_scale_from_amax_kernel<<<1, 32, 0, st>>>(g, 1);
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
  long long blocks = (n + 255) / 256;
  if (blocks > 8 * num_sms()) blocks = 8 * num_sms();
  nv_quantize_grouped_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(x, R, K, E, offsets, g, xq, sf);
  return cudaGetLastError();
}

}  // namespace moe

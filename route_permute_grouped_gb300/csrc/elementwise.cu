// Bandwidth-bound kernels of the path: combine (weighted gather-sum), its
// backward, the permute backward (unweighted gather-sum), the router's
// element-wise backward, the auxiliary-loss value and the split-K reduction.
// One warp per token, 16-byte vectors along H, fp32 arithmetic.
#include "host_util.h"
#include "mx.cuh"

namespace moe {

template <bool F32>
struct Vec8 {  // 8 consecutive elements of a bf16 or fp32 row
  __device__ __forceinline__ static void load(const void* base, size_t elem, float* f) {
    if constexpr (F32) {
      const float4* p = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(base) + elem);
      const float4 a = __ldg(p), b = __ldg(p + 1);
      f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
    } else {
      const uint4 w = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(base) + elem));
      f[0] = bf16_lo(w.x); f[1] = bf16_hi(w.x); f[2] = bf16_lo(w.y); f[3] = bf16_hi(w.y);
      f[4] = bf16_lo(w.z); f[5] = bf16_hi(w.z); f[6] = bf16_lo(w.w); f[7] = bf16_hi(w.w);
    }
  }
  __device__ __forceinline__ static void store(void* base, size_t elem, const float* f) {
    if constexpr (F32) {
      float4* p = reinterpret_cast<float4*>(reinterpret_cast<float*>(base) + elem);
      p[0] = make_float4(f[0], f[1], f[2], f[3]);
      p[1] = make_float4(f[4], f[5], f[6], f[7]);
    } else {
      uint4 w;
      w.x = pack_bf16x2(f[0], f[1]); w.y = pack_bf16x2(f[2], f[3]);
      w.z = pack_bf16x2(f[4], f[5]); w.w = pack_bf16x2(f[6], f[7]);
      *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(base) + elem) = w;
    }
  }
};

constexpr int kWarpsPerBlock = 8;

// y[t] = shared[t] + sum_i g[t,i] * y_perm[row[t,i]]  (fp32, slot order).
// With gate == nullptr the weights are 1 (permute backward) and `extra` (fp32,
// nullable) is added instead of `shared`; `add` (nullable, [T,H], the storage
// type of y_perm) is added last (the permute backward: the shared expert's
// input gradient).
template <bool YP32, bool SH32, bool OUT32>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    gather_sum_kernel(const void* __restrict__ y_perm, const int32_t* __restrict__ row_id_map,
                      const float* __restrict__ gate, const void* __restrict__ shared, void* __restrict__ y, int T,
                      int H, int k, const void* __restrict__ add = nullptr, DevStatus* st = nullptr) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kWarpsPerBlock + warp;
  if (t >= T) return;
  int my_r = 0;
  float my_g = 1.0f;
  if (lane < k) {
    my_r = row_id_map[static_cast<size_t>(t) * k + lane];
    if (gate != nullptr) my_g = gate[static_cast<size_t>(t) * k + lane];
    if (!row_valid(my_r, static_cast<long long>(T) * k, st, 21)) {
      my_r = 0;  // a dropped slot: row 0 read with weight 0
      my_g = 0.0f;
    }
  }
  // every lane takes all k (row, gate) pairs before the H loop, whose trip
  // count differs between lanes when H/8 is not a multiple of 32
  int rows[16];
  float gs[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    rows[i] = __shfl_sync(0xffffffffu, my_r, i < k ? i : 0);
    gs[i] = __shfl_sync(0xffffffffu, my_g, i < k ? i : 0);
  }
  const int nvec = H / 8;
  for (int v = lane; v < nvec; v += 32) {
    float acc[8];
    if (shared != nullptr) {
      Vec8<SH32>::load(shared, static_cast<size_t>(t) * H + v * 8, acc);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (i < k) {
        float f[8];
        Vec8<YP32>::load(y_perm, static_cast<size_t>(rows[i]) * H + v * 8, f);
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = fmaf(gs[i], f[j], acc[j]);
      }
    }
    if (add != nullptr) {
      float f[8];
      Vec8<YP32>::load(add, static_cast<size_t>(t) * H + v * 8, f);
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] += f[j];
    }
    Vec8<OUT32>::store(y, static_cast<size_t>(t) * H + v * 8, acc);
  }
}

// Combine backward: dy_perm[row[t,i]] = bf16(g[t,i] * dO[t]),
// dgate[t,i] = <dO[t], y_perm[row[t,i]]> (fp32). All k expert-output vectors
// of a position are loaded before any store is issued, so the loads of the k
// rows are in flight together. DG = false (memory-saving backward, no y_perm):
// dy_perm only; the gate gradient comes from the down-projection dgrad.
// MXQ (the MXFP8 training step): the bf16 dy_perm rows are also quantised
// (blocks of 32 along H, one block per four lanes) into codes mq [R, H] and
// scales in the activations' tile-ready layout (msf), the row's expert and
// its offset from topk_idx and offsets. AMAX (the NVFP4 training step): the
// largest magnitude of the stored dy_perm values, as fp32 bits, maximised
// into *amax_bits.
template <bool YP32, int KMAX, bool DG = true, bool MXQ = false, bool AMAX = false>
__global__ void __launch_bounds__(kWarpsPerBlock * 32, KMAX <= 8 ? 2 : 1)
    combine_bwd_kernel(const __nv_bfloat16* __restrict__ dO, const void* __restrict__ y_perm,
                       const int32_t* __restrict__ row_id_map, const float* __restrict__ gate,
                       __nv_bfloat16* __restrict__ dy_perm, float* __restrict__ dgate, int T, int H, int k,
                       uint8_t* __restrict__ mq = nullptr, uint8_t* __restrict__ msf = nullptr,
                       const int32_t* __restrict__ offsets = nullptr, const int32_t* __restrict__ topk_idx = nullptr,
                       int E = 0, DevStatus* st = nullptr, unsigned* __restrict__ amax_bits = nullptr) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kWarpsPerBlock + warp;
  __shared__ int s_off[MXQ ? kMaxGroups + 1 : 1];
  __shared__ int s_pt[MXQ ? kMaxGroups + 1 : 1];
  if constexpr (MXQ) {
    for (int i = threadIdx.x; i <= E; i += blockDim.x) s_off[i] = offsets[i];
    __syncthreads();
    if (warp == 0) pair_tile_prefix_warp(s_off, s_pt, E, lane);
    __syncthreads();
  }
  if (t >= T) return;
  int my_r = -1, my_e = 0;
  float my_g = 0.0f;
  if (lane < k) {
    my_r = row_id_map[static_cast<size_t>(t) * k + lane];
    if (!row_valid(my_r, static_cast<long long>(T) * k, st, 22)) my_r = -1;  // a dropped slot: no row
    my_g = gate[static_cast<size_t>(t) * k + lane];
    if (MXQ) my_e = topk_idx[static_cast<size_t>(t) * k + lane];
    if (MXQ && (my_e < 0 || my_e >= E)) my_r = -1;
  }
  float dot[KMAX];
  int rows[KMAX];
  float gs[KMAX];
#pragma unroll
  for (int i = 0; i < KMAX; ++i) {
    dot[i] = 0.0f;
    rows[i] = __shfl_sync(0xffffffffu, my_r, i < k ? i : 0);  // outside the divergent H loop
    gs[i] = __shfl_sync(0xffffffffu, my_g, i < k ? i : 0);
  }
  const int nvec = H / 8;
  float am = 0.0f;  // AMAX: largest |g dO| this warp stores
  for (int v = lane; v < nvec; v += 32) {
    float d[8];
    Vec8<false>::load(dO, static_cast<size_t>(t) * H + v * 8, d);
    float f[KMAX][8];
#pragma unroll
    for (int i = 0; i < KMAX; ++i)  // a dropped slot (row -1) loads row 0; its results are discarded
      if (DG && i < k) Vec8<YP32>::load(y_perm, static_cast<size_t>(rows[i] >= 0 ? rows[i] : 0) * H + v * 8, f[i]);
#pragma unroll
    for (int i = 0; i < KMAX; ++i) {
      if (i < k) {
        float o[8];
        float s = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (DG) s = fmaf(d[j], f[i][j], s);
          o[j] = gs[i] * d[j];
        }
        dot[i] += s;
        if (rows[i] >= 0) {
          Vec8<false>::store(dy_perm, static_cast<size_t>(rows[i]) * H + v * 8, o);
          if constexpr (AMAX) {
#pragma unroll
            for (int j = 0; j < 8; ++j) am = fmaxf(am, fabsf(o[j]));
          }
        }
      }
    }
  }
  if constexpr (AMAX) {
    // the maximum of the stored bf16 values is the bf16 rounding of the fp32
    // maximum (rounding is monotone)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
    am = __bfloat162float(__float2bfloat16_rn(am));
    if (lane == 0 && am > 0.0f) atomicMax(amax_bits, __float_as_uint(am));
  }
  if constexpr (MXQ) {
    // second pass: the MXFP8 rows of dy_perm, from the same products g dO
    // (the dO row is re-read from cache) rounded to bf16 as stored above; a
    // block of 32 spans four lanes
    const unsigned gmask = 0xFu << (lane & ~3);
    const int nkb = H / kMxKB;
#pragma unroll 1
    for (int i = 0; i < k; ++i) {
      const int r = __shfl_sync(0xffffffffu, my_r, i);
      const float gi = __shfl_sync(0xffffffffu, my_g, i);
      const int e = __shfl_sync(0xffffffffu, my_e, i);
      if (r < 0) continue;  // warp-uniform
      const size_t sf0 = mx_act_sf_offset(s_pt[e], r - s_off[e], 0, nkb);
#pragma unroll 4
      for (int v = lane; v < nvec; v += 32) {
        float d[8], o[8];
        Vec8<false>::load(dO, static_cast<size_t>(t) * H + v * 8, d);
        float amax = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          o[j] = __bfloat162float(__float2bfloat16_rn(gi * d[j]));
          amax = fmaxf(amax, fabsf(o[j]));
        }
        amax = fmaxf(amax, __shfl_xor_sync(gmask, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(gmask, amax, 2));
        const uint32_t sb = mx_scale_byte(amax);
        uint32_t w[2];
        mx_codes8(o, sb, w);
        *reinterpret_cast<uint2*>(mq + static_cast<size_t>(r) * H + v * 8) = make_uint2(w[0], w[1]);
        if ((lane & 3) == 0) {
          const int b = v / 4;
          msf[sf0 + (b / 4) * kMxSfBytes + (b & 3)] = static_cast<uint8_t>(sb);
        }
      }
    }
  }
  if (!DG) return;
#pragma unroll
  for (int i = 0; i < KMAX; ++i) {
    if (i < k) {
      float s = dot[i];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if (lane == 0) dgate[static_cast<size_t>(t) * k + i] = rows[i] >= 0 ? s : 0.0f;
    }
  }
}

// Router backward, element-wise part (one warp per token). Gate gradient ->
// logit gradient:
//   softmax: g = c q, q = softmax over the selected logits:
//            dL_sel = c q (dg - <q, dg>), 0 off the selection;
//   sigmoid: g = c s_sel / S: ds = (c / S)(dg - <dg, s_sel> / S),
//            dL_sel = ds s (1 - s);
//   aux (softmax): dL += p (dp - <p, dp>), dp_e = alpha E counts_e / (T k T).
// Output dL split into bf16 hi = bf16(dL) and lo = bf16(dL - hi), written as
// row t of dL_hl [T, 2 Ep]: hi at columns [0,E), lo at [Ep, Ep+E), zero padding.
// Memory-saving backward (dg_part != nullptr): the gate gradient of slot i is
// (sum over the n_part tile partials of its permuted row) / g, 0 where g = 0.
__device__ __forceinline__ float slot_dgate(const float* dgate, const float* dg_part, int n_part,
                                            const int32_t* row_id_map, const float* gate, size_t slot, long long R,
                                            DevStatus* st) {
  if (dg_part == nullptr) return dgate[slot];
  const int r = row_id_map[slot];
  if (!row_valid(r, R, st, 23)) return 0.0f;  // a dropped slot
  const float* pr = dg_part + static_cast<size_t>(r) * n_part;
  float s = 0.0f;
  for (int j = 0; j < n_part; ++j) s += pr[j];
  const float g = gate[slot];
  return g != 0.0f ? s / g : 0.0f;
}
// One warp per token; lane j holds experts j, j + 32, ... (NJ of them, NJ * 32
// >= Ep): every load of the token (its slots, the logits, the counts) is
// issued before any arithmetic, the softmax of the aux term is formed once in
// registers, and each lane writes its columns of hi and lo.
template <int NJ>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    router_bwd_kernel(const float* __restrict__ logits, const int32_t* __restrict__ topk_idx,
                      const float* __restrict__ gate, const float* __restrict__ dgate,
                      const float* __restrict__ dg_part, int n_part, const int32_t* __restrict__ row_id_map,
                      const int32_t* __restrict__ counts, int T, int E, int k, int score, float gate_scale,
                      float aux_coeff, int Ep, __nv_bfloat16* __restrict__ dL_hl, DevStatus* st) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kWarpsPerBlock + warp;
  if (t >= T) return;
  const bool aux = (score == MOE_SCORE_SOFTMAX) && aux_coeff != 0.0f;
  const float* Lrow = logits + static_cast<size_t>(t) * E;
  // loads; a slot whose expert index is out of range contributes nothing
  int my_e = -1;
  float g_or_L = 0.0f, dg = 0.0f;
  if (lane < k) {
    const size_t slot = static_cast<size_t>(t) * k + lane;
    my_e = topk_idx[slot];
    if (my_e < 0 || my_e >= E) {
      if (kBoundsCheck) set_status(st, MOE_ERR_DEVICE_INDEX, 24);
      my_e = -1;
    } else {
      dg = slot_dgate(dgate, dg_part, n_part, row_id_map, gate, slot, static_cast<long long>(T) * k, st);
      g_or_L = score == MOE_SCORE_SOFTMAX ? gate[slot] : Lrow[my_e];
    }
  }
  float v[NJ];
  float cnt[NJ];
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const int e = lane + 32 * j;
    v[j] = (aux && e < E) ? Lrow[e] : -INFINITY;
    cnt[j] = (aux && e < E) ? static_cast<float>(counts[e]) : 0.0f;
  }
  // the gate term of the selected slots
  float my_dl;
  if (score == MOE_SCORE_SOFTMAX) {
    const float q = (lane < k && my_e >= 0) ? g_or_L / gate_scale : 0.0f;
    float inner = q * dg;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) inner += __shfl_xor_sync(0xffffffffu, inner, o);
    my_dl = gate_scale * q * (dg - inner);
  } else {
    const float sg = (lane < k && my_e >= 0) ? 1.0f / (1.0f + __expf(-g_or_L)) : 0.0f;
    float S = sg, inner = dg * sg;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      S += __shfl_xor_sync(0xffffffffu, S, o);
      inner += __shfl_xor_sync(0xffffffffu, inner, o);
    }
    const float ds = (gate_scale / S) * (dg - inner / S);
    my_dl = ds * sg * (1.0f - sg);
  }
  // the aux term: p (dp - <p, dp>), dp_e = alpha E counts_e / (T k T)
  float d[NJ];
#pragma unroll
  for (int j = 0; j < NJ; ++j) d[j] = 0.0f;
  if (aux) {
    const float dp_scale = aux_coeff * static_cast<float>(E) / (static_cast<float>(T) * k * static_cast<float>(T));
    float mx = -INFINITY;
#pragma unroll
    for (int j = 0; j < NJ; ++j) mx = fmaxf(mx, v[j]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float sum = 0.0f, pdp = 0.0f;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      v[j] = __expf(v[j] - mx);  // 0 past E
      sum += v[j];
      pdp += v[j] * (dp_scale * cnt[j]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      sum += __shfl_xor_sync(0xffffffffu, sum, o);
      pdp += __shfl_xor_sync(0xffffffffu, pdp, o);
    }
    pdp /= sum;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const float p = v[j] / sum;
      d[j] = p * (dp_scale * cnt[j] - pdp);
    }
  }
  // scatter the selected slots' terms to their experts' lanes
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    if (i < k) {
      const int e = __shfl_sync(0xffffffffu, my_e, i);
      const float x = __shfl_sync(0xffffffffu, my_dl, i);
#pragma unroll
      for (int j = 0; j < NJ; ++j)
        if (e == lane + 32 * j) d[j] += x;
    }
  }
  __nv_bfloat16* out = dL_hl + static_cast<size_t>(t) * 2 * Ep;
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const int e = lane + 32 * j;
    if (e < Ep) {
      const float dd = e < E ? d[j] : 0.0f;
      const __nv_bfloat16 hi = __float2bfloat16_rn(dd);
      out[e] = hi;
      out[Ep + e] = __float2bfloat16_rn(dd - __bfloat162float(hi));
    }
  }
}

// aux loss value: alpha * E * sum_e (c_e / (T k)) * (sum_rows partial[row][e] / T).
// One block of 1024 threads. With E a multiple of 4 (rows 16-byte aligned),
// thread (g, c) (c fastest over the E/4 float4 columns, RG = the largest power
// of two <= 1024 / (E/4) row groups) adds rows g, g + RG, ... of its four
// columns; the loads of a thread are independent of one another (unrolled, in
// flight together), the row groups are combined by a halving tree in shared
// memory. Otherwise thread (g, e) adds rows of one column in four independent
// accumulators. Then the experts are combined by a halving tree: a fixed order
// throughout.
__global__ void __launch_bounds__(1024) aux_loss_kernel(const float* __restrict__ partials, int nrows,
                                                        const int32_t* __restrict__ counts, int T, int E, int k,
                                                        float aux_coeff, float* __restrict__ out) {
  __shared__ float s_part[4096];
  __shared__ float s[256];
  const int tid = static_cast<int>(threadIdx.x);
  if ((E & 3) == 0 && (reinterpret_cast<uintptr_t>(partials) & 15) == 0) {
    const int C4 = E >> 2;
    int RG = 1;
    while (2 * RG * C4 <= 1024) RG *= 2;
    const int c = tid % C4, g = tid / C4;
    if (g < RG) {
      const float4* p4 = reinterpret_cast<const float4*>(partials);
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 16
      for (int i = g; i < nrows; i += RG) {
        const float4 v = __ldg(p4 + static_cast<size_t>(i) * C4 + c);
        acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
      }
      float* dst = s_part + g * E + 4 * c;
      dst[0] = acc.x; dst[1] = acc.y; dst[2] = acc.z; dst[3] = acc.w;
    }
    __syncthreads();
    for (int st = RG / 2; st >= 1; st >>= 1) {
      for (int i = tid; i < st * E; i += 1024) s_part[i] += s_part[i + st * E];
      __syncthreads();
    }
  } else {
    const int Eb = (E + 31) & ~31;
    const int G = 1024 / Eb;
    const int e = tid % Eb, g = tid / Eb;
    float P = 0.0f;
    if (g < G && e < E) {
      float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
      int i = g;
      for (; i + 3 * G < nrows; i += 4 * G) {
        a0 += partials[static_cast<size_t>(i) * E + e];
        a1 += partials[static_cast<size_t>(i + G) * E + e];
        a2 += partials[static_cast<size_t>(i + 2 * G) * E + e];
        a3 += partials[static_cast<size_t>(i + 3 * G) * E + e];
      }
      for (; i < nrows; i += G) a0 += partials[static_cast<size_t>(i) * E + e];
      P = (a0 + a1) + (a2 + a3);
    }
    s_part[tid] = P;
    __syncthreads();
    if (tid < E) {
      float Pe = 0.0f;
      for (int gg = 0; gg < G; ++gg) Pe += s_part[gg * Eb + tid];
      s_part[2048 + tid] = Pe;
    }
    __syncthreads();
    if (tid < E) s_part[tid] = s_part[2048 + tid];
    __syncthreads();
  }
  // s_part[e] = sum over the rows of column e
  if (tid < 256) {
    float v = 0.0f;
    if (tid < E)
      v = (static_cast<float>(counts[tid]) / (static_cast<float>(T) * k)) * (s_part[tid] / static_cast<float>(T));
    s[tid] = v;
  }
  __syncthreads();
  for (int d = 128; d > 0; d >>= 1) {
    if (tid < d) s[tid] += s[tid + d];
    __syncthreads();
  }
  if (tid == 0) *out = aux_coeff * static_cast<float>(E) * s[0];
}

// out[i] = sum_s partials[s][i], s in order.
__global__ void split_reduce_kernel(const float* __restrict__ partials, int splits, size_t n,
                                    float* __restrict__ out) {
  const size_t i4 = (static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 4;
  if (i4 >= n) return;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s = 0; s < splits; ++s) {
    const float4 v = *reinterpret_cast<const float4*>(partials + static_cast<size_t>(s) * n + i4);
    acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
  }
  *reinterpret_cast<float4*>(out + i4) = acc;
}

// ---------------------------------------------------------------------------
static int blocks_for(int T) { return (T + kWarpsPerBlock - 1) / kWarpsPerBlock; }

cudaError_t launch_combine(const moe_config& c, const void* y_perm, const int32_t* row_id_map, const float* gate,
                           const void* shared, void* y, cudaStream_t st, DevStatus* ds) {
  NvtxRange nvtx("moe.combine");
  const int b = blocks_for(c.T);
  const bool yp = c.inter_fp32 != 0, out = c.out_fp32 != 0;
  // the shared output has the storage type of y_perm
  if (yp && out) gather_sum_kernel<true, true, true><<<b, kWarpsPerBlock * 32, 0, st>>>(y_perm, row_id_map, gate, shared, y, c.T, c.H, c.k, nullptr, ds);
  else if (yp) gather_sum_kernel<true, true, false><<<b, kWarpsPerBlock * 32, 0, st>>>(y_perm, row_id_map, gate, shared, y, c.T, c.H, c.k, nullptr, ds);
  else if (out) gather_sum_kernel<false, false, true><<<b, kWarpsPerBlock * 32, 0, st>>>(y_perm, row_id_map, gate, shared, y, c.T, c.H, c.k, nullptr, ds);
  else gather_sum_kernel<false, false, false><<<b, kWarpsPerBlock * 32, 0, st>>>(y_perm, row_id_map, gate, shared, y, c.T, c.H, c.k, nullptr, ds);
  return cudaGetLastError();
}

cudaError_t launch_unpermute_sum(const moe_config& c, const void* dx_perm, const int32_t* row_id_map,
                                 const float* extra, void* dx, cudaStream_t st, const void* add, bool rows_fp32,
                                 DevStatus* ds) {
  NvtxRange nvtx("moe.permute_backward");
  const int b = blocks_for(c.T);
  const dim3 g(b), blk(kWarpsPerBlock * 32);
  if (rows_fp32 && c.out_fp32)
    gather_sum_kernel<true, true, true><<<g, blk, 0, st>>>(dx_perm, row_id_map, nullptr, extra, dx, c.T, c.H, c.k, add, ds);
  else if (rows_fp32)
    gather_sum_kernel<true, true, false><<<g, blk, 0, st>>>(dx_perm, row_id_map, nullptr, extra, dx, c.T, c.H, c.k, add, ds);
  else if (c.out_fp32)
    gather_sum_kernel<false, true, true><<<g, blk, 0, st>>>(dx_perm, row_id_map, nullptr, extra, dx, c.T, c.H, c.k, add, ds);
  else
    gather_sum_kernel<false, true, false><<<g, blk, 0, st>>>(dx_perm, row_id_map, nullptr, extra, dx, c.T, c.H, c.k,
                                                             add, ds);
  return cudaGetLastError();
}

cudaError_t launch_combine_bwd(const moe_config& c, const __nv_bfloat16* dO, const void* y_perm,
                               const int32_t* row_id_map, const float* gate, __nv_bfloat16* dy_perm, float* dgate,
                               cudaStream_t st, uint8_t* mq, uint8_t* msf, const int32_t* offsets,
                               const int32_t* topk_idx, DevStatus* ds, float* dy_amax) {
  NvtxRange nvtx("moe.combine_backward");
  const int b = blocks_for(c.T);
  const int th = kWarpsPerBlock * 32;
  unsigned* am = reinterpret_cast<unsigned*>(dy_amax);
  if (dy_amax != nullptr) {
    cudaError_t e = cudaMemsetAsync(dy_amax, 0, sizeof(float), st);
    if (e != cudaSuccess) return e;
  }
  if (mq != nullptr) {  // MXFP8 training step: dy_perm quantised as it is written
    cudaError_t e = cudaMemsetAsync(msf, 0, mx_sfa_bytes(static_cast<long long>(c.T) * c.k, c.E, c.H), st);
    if (e != cudaSuccess) return e;
    if (c.inter_fp32) {
      if (c.k <= 8) combine_bwd_kernel<true, 8, true, true><<<b, th, 0, st>>>(dO, y_perm, row_id_map, gate, dy_perm, dgate, c.T, c.H, c.k, mq, msf, offsets, topk_idx, c.E, ds);
      else combine_bwd_kernel<true, 16, true, true><<<b, th, 0, st>>>(dO, y_perm, row_id_map, gate, dy_perm, dgate, c.T, c.H, c.k, mq, msf, offsets, topk_idx, c.E, ds);
    } else {
      if (c.k <= 8) combine_bwd_kernel<false, 8, true, true><<<b, th, 0, st>>>(dO, y_perm, row_id_map, gate, dy_perm, dgate, c.T, c.H, c.k, mq, msf, offsets, topk_idx, c.E, ds);
      else combine_bwd_kernel<false, 16, true, true><<<b, th, 0, st>>>(dO, y_perm, row_id_map, gate, dy_perm, dgate, c.T, c.H, c.k, mq, msf, offsets, topk_idx, c.E, ds);
    }
    return cudaGetLastError();
  }
  if (y_perm == nullptr) {  // memory-saving backward: dy_perm only
    if (c.k <= 8) combine_bwd_kernel<false, 8, false><<<b, th, 0, st>>>(dO, nullptr, row_id_map, gate, dy_perm, nullptr, c.T, c.H, c.k, nullptr, nullptr, nullptr, nullptr, c.E, ds);
    else combine_bwd_kernel<false, 16, false><<<b, th, 0, st>>>(dO, nullptr, row_id_map, gate, dy_perm, nullptr, c.T, c.H, c.k, nullptr, nullptr, nullptr, nullptr, c.E, ds);
  } else if (c.inter_fp32) {
    if (c.k <= 8) combine_bwd_kernel<true, 8><<<b, th, 0, st>>>(dO, y_perm, row_id_map, gate, dy_perm, dgate, c.T, c.H, c.k, nullptr, nullptr, nullptr, nullptr, c.E, ds);
    else combine_bwd_kernel<true, 16><<<b, th, 0, st>>>(dO, y_perm, row_id_map, gate, dy_perm, dgate, c.T, c.H, c.k, nullptr, nullptr, nullptr, nullptr, c.E, ds);
  } else if (am != nullptr) {  // NVFP4 training step: with the maximum of dy_perm
    if (c.k <= 8) combine_bwd_kernel<false, 8, true, false, true><<<b, th, 0, st>>>(dO, y_perm, row_id_map, gate, dy_perm, dgate, c.T, c.H, c.k, nullptr, nullptr, nullptr, nullptr, c.E, ds, am);
    else combine_bwd_kernel<false, 16, true, false, true><<<b, th, 0, st>>>(dO, y_perm, row_id_map, gate, dy_perm, dgate, c.T, c.H, c.k, nullptr, nullptr, nullptr, nullptr, c.E, ds, am);
  } else {
    if (c.k <= 8) combine_bwd_kernel<false, 8><<<b, th, 0, st>>>(dO, y_perm, row_id_map, gate, dy_perm, dgate, c.T, c.H, c.k, nullptr, nullptr, nullptr, nullptr, c.E, ds);
    else combine_bwd_kernel<false, 16><<<b, th, 0, st>>>(dO, y_perm, row_id_map, gate, dy_perm, dgate, c.T, c.H, c.k, nullptr, nullptr, nullptr, nullptr, c.E, ds);
  }
  return cudaGetLastError();
}

cudaError_t launch_router_bwd(const moe_config& c, const float* logits, const int32_t* topk_idx, const float* gate,
                              const float* dgate, const float* dg_part, int n_part, const int32_t* row_id_map,
                              const int32_t* counts, int Ep, __nv_bfloat16* dL_hl, cudaStream_t st,
                              DevStatus* ds) {
  NvtxRange nvtx("moe.router_backward");
  const dim3 g(blocks_for(c.T)), b(kWarpsPerBlock * 32);
#define MOE_ROUTER_BWD(NJ)                                                                                  \
  router_bwd_kernel<NJ><<<g, b, 0, st>>>(logits, topk_idx, gate, dgate, dg_part, n_part, row_id_map, counts, \
                                         c.T, c.E, c.k, c.score, c.gate_scale, c.aux_coeff, Ep, dL_hl, ds)
  // Ep (a multiple of 64, <= 256) columns over 32 lanes
  if (Ep <= 64) MOE_ROUTER_BWD(2);
  else if (Ep <= 128) MOE_ROUTER_BWD(4);
  else MOE_ROUTER_BWD(8);
#undef MOE_ROUTER_BWD
  return cudaGetLastError();
}

cudaError_t launch_aux_loss(const moe_config& c, const float* aux_partials, const int32_t* counts, float* out,
                            cudaStream_t st) {
  NvtxRange nvtx("moe.aux_loss");
  aux_loss_kernel<<<1, 1024, 0, st>>>(aux_partials, 4 * ((c.T + 127) / 128), counts, c.T, c.E, c.k, c.aux_coeff, out);
  return cudaGetLastError();
}

cudaError_t launch_split_reduce(const float* partials, int splits, size_t n, float* out, cudaStream_t st) {
  NvtxRange nvtx("moe.router_weight_gradient_reduce");
  const size_t n4 = (n + 3) / 4;
  const int blocks = static_cast<int>((n4 + 255) / 256);
  split_reduce_kernel<<<blocks, 256, 0, st>>>(partials, splits, n, out);
  return cudaGetLastError();
}

}  // namespace moe

// ---------------------------------------------------------------------------
// Read ceiling (measurement helper): a grid-stride pass of 16-byte loads over
// a buffer, four loads in flight per thread, nothing stored unless the data
// hashes to a fixed word (so the loads cannot be dropped).
// ---------------------------------------------------------------------------
namespace moe {
__global__ void __launch_bounds__(512) read_ceiling_kernel(const uint4* __restrict__ p, size_t n16, unsigned* sink) {
  unsigned acc = 0;
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n16; i += 4 * stride) {
    const uint4 a = __ldg(p + i), b = __ldg(p + i + stride), c = __ldg(p + i + 2 * stride),
                d = __ldg(p + i + 3 * stride);
    acc += a.x ^ b.y ^ c.z ^ d.w;
  }
  for (; i < n16; i += stride) acc += __ldg(p + i).x;
  if (acc == 0x9e3779b9u) sink[blockIdx.x] = acc;
}
}  // namespace moe

namespace moe {
__global__ void __launch_bounds__(512) write_ceiling_kernel(uint4* __restrict__ p, size_t n16, uint32_t word) {
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  const uint4 v = make_uint4(word, word, word, word);
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16; i += stride) p[i] = v;
}
}  // namespace moe

extern "C" int moe_write_ceiling(void* buf, size_t bytes, unsigned word, void* stream) {
  using namespace moe;
  if (buf == nullptr || (reinterpret_cast<uintptr_t>(buf) & 15) != 0 || (bytes & 15) != 0) return MOE_ERR_INVALID_ARG;
  if (bytes == 0) return MOE_OK;
  NvtxRange nvtx("moe.write_ceiling");
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  write_ceiling_kernel<<<4 * num_sms(), 512, 0, st>>>(static_cast<uint4*>(buf), bytes / 16, word);
  const int rc = status_from_cuda(cudaGetLastError());
  record_stage(st, 31, 1);
  return rc;
}

extern "C" int moe_read_ceiling(const void* buf, size_t bytes, unsigned* sink, void* stream) {
  using namespace moe;
  if (buf == nullptr || sink == nullptr || (reinterpret_cast<uintptr_t>(buf) & 15) != 0 ||
      (reinterpret_cast<uintptr_t>(sink) & 15) != 0 || (bytes & 15) != 0)
    return MOE_ERR_INVALID_ARG;
  if (bytes == 0) return MOE_OK;
  NvtxRange nvtx("moe.read_ceiling");
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  read_ceiling_kernel<<<4 * num_sms(), 512, 0, st>>>(static_cast<const uint4*>(buf), bytes / 16, sink);
  const int rc = status_from_cuda(cudaGetLastError());
  record_stage(st, 30, 1);
  return rc;
}

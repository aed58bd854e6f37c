// Router selection: from the fp32 logits of the router GEMM to the top-k
// experts and gates of every token (figures & tables page of the report,
// Fig. 2: score function, top-k selection, load balancing).
//
// One warp per token, one CTA per 32-token slice (32 warps). Lane l holds the
// experts e = l + 32 j (j < 8, E <= 256) in registers. Per token:
//   L = logit + logit_bias; score = softmax(L) or sigmoid(L);
//   z = L (softmax without expert bias: same order as the probabilities) or
//       score + expert_bias;
//   group limit: group score = sum of its two largest z, keep the best
//       topk_groups groups (lower group index wins ties), z = -inf elsewhere;
//   k rounds of a warp arg-max over (z, -e): a lower expert index wins ties and
//       slot i holds the i-th largest z;
//   gates = gate_scale * score_i / sum of the selected scores (softmax: the
//       selected probabilities renormalised, computed from the selected logits).
// Optional outputs: the biased logits [T,E] and, for softmax, the column sums
// of the probabilities over the slice (aux_partials row = slice), reduced in a
// fixed order in shared memory.
#include "host_util.h"

namespace moe {

constexpr int kSel = 32;  // tokens (warps) per CTA = aux_partials slice

// warp arg-max of (v, e): larger v, then smaller e; every lane gets the result
__device__ __forceinline__ void warp_argmax(float& v, int& e) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oe = __shfl_xor_sync(0xffffffffu, e, o);
    if (ov > v || (ov == v && oe < e)) {
      v = ov;
      e = oe;
    }
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__global__ void __launch_bounds__(kSel * 32) router_select_kernel(
    const float* __restrict__ raw, int ld, int T, int E, int k, int score, int n_groups, int topk_groups,
    float gate_scale, const float* __restrict__ expert_bias, const float* __restrict__ logit_bias,
    int32_t* __restrict__ topk_idx, float* __restrict__ topk_gate, float* __restrict__ logits_out,
    float* __restrict__ aux_partials) {
  extern __shared__ float s_p[];  // [kSel][E] softmax values (aux only)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kSel + warp;
  const bool valid = t < T;
  const bool softmax = score == MOE_SCORE_SOFTMAX;
  const bool z_is_logit = softmax && expert_bias == nullptr;
  const bool want_aux = softmax && aux_partials != nullptr;
  const int nj = (E + 31) >> 5;

  float L[8], sc[8], z[8];
  float mx = -INFINITY;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int e = lane + 32 * j;
    L[j] = -INFINITY;
    if (j < nj && e < E && valid) {
      L[j] = raw[static_cast<size_t>(t) * ld + e] + (logit_bias != nullptr ? logit_bias[e] : 0.0f);
      mx = fmaxf(mx, L[j]);
    }
  }
  float inv_sum = 1.0f;
  if (softmax) {
    mx = warp_max(mx);
    float sum = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (j < nj && lane + 32 * j < E && valid) sum += __expf(L[j] - mx);
    inv_sum = 1.0f / warp_sum(sum);
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int e = lane + 32 * j;
    const bool in = j < nj && e < E && valid;
    sc[j] = !in ? 0.0f : (softmax ? __expf(L[j] - mx) * inv_sum : 1.0f / (1.0f + __expf(-L[j])));
    z[j] = !in ? -INFINITY : (z_is_logit ? L[j] : sc[j] + (expert_bias != nullptr ? expert_bias[e] : 0.0f));
  }
  if (valid && logits_out != nullptr) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = lane + 32 * j;
      if (j < nj && e < E) logits_out[static_cast<size_t>(t) * E + e] = L[j];
    }
  }
  if (want_aux) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = lane + 32 * j;
      if (j < nj && e < E) s_p[warp * E + e] = sc[j];  // 0 for tokens past T
    }
  }
  // group-limited selection
  if (n_groups > 1 && topk_groups < n_groups) {
    const int gsz = E / n_groups;
    uint32_t keep = 0u;
    float gscore[32];
#pragma unroll 1
    for (int g = 0; g < n_groups; ++g) {
      // this lane's two largest z of group g, then the warp's two largest
      float b1 = -INFINITY, b2 = -INFINITY;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int e = lane + 32 * j;
        if (j < nj && e < E && e / gsz == g) {
          if (z[j] > b1) { b2 = b1; b1 = z[j]; } else if (z[j] > b2) { b2 = z[j]; }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float o1 = __shfl_xor_sync(0xffffffffu, b1, o);
        const float o2 = __shfl_xor_sync(0xffffffffu, b2, o);
        // merge {b1, b2} and {o1, o2} into the two largest
        const float hi = fmaxf(b1, o1);
        const float lo = fmaxf(fminf(b1, o1), fmaxf(b2, o2));
        b1 = hi;
        b2 = lo;
      }
      gscore[g & 31] = (gsz >= 2) ? (b1 + b2) : b1;
    }
#pragma unroll 1
    for (int s = 0; s < topk_groups; ++s) {
      int bi = -1;
      float best = -INFINITY;
#pragma unroll 1
      for (int g = 0; g < n_groups; ++g)
        if (!((keep >> g) & 1u) && (bi < 0 || gscore[g] > best)) { best = gscore[g]; bi = g; }
      keep |= 1u << bi;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = lane + 32 * j;
      if (j < nj && e < E && !((keep >> (e / gsz)) & 1u)) z[j] = -INFINITY;
    }
  }
  // k rounds of arg-max; lane i keeps slot i
  int my_e = 0;
  float my_sc = 0.0f;
#pragma unroll 1
  for (int i = 0; i < k; ++i) {
    float v = -INFINITY;
    int e = 0x7fffffff;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int ej = lane + 32 * j;
      if (j < nj && ej < E && (z[j] > v || (z[j] == v && ej < e))) { v = z[j]; e = ej; }
    }
    warp_argmax(v, e);
    // the owner lane of e publishes its gate score and drops e from the race
    float own = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (lane + 32 * j == e) {
        own = z_is_logit ? L[j] : sc[j];
        z[j] = -INFINITY;
      }
    }
    const float sel_sc = __shfl_sync(0xffffffffu, own, e & 31);
    if (lane == i) {
      my_e = e;
      my_sc = sel_sc;
    }
  }
  // gates over the k slots (lanes 0..k-1)
  float w;
  if (z_is_logit) {
    const float top = __shfl_sync(0xffffffffu, my_sc, 0);
    w = lane < k ? __expf(my_sc - top) : 0.0f;
  } else {
    w = lane < k ? my_sc : 0.0f;
  }
  const float tot = warp_sum(w);
  if (valid && lane < k) {
    topk_idx[static_cast<size_t>(t) * k + lane] = my_e;
    topk_gate[static_cast<size_t>(t) * k + lane] = gate_scale * w / tot;
  }
  if (want_aux) {
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kSel * 32) {
      float acc = 0.0f;
      for (int r = 0; r < kSel; ++r) acc += s_p[r * E + e];
      aux_partials[static_cast<size_t>(blockIdx.x) * E + e] = acc;
    }
  }
}

cudaError_t launch_router_select(const moe_config& c, const float* raw, int ld, const float* expert_bias,
                                 const float* logit_bias, int32_t* topk_idx, float* topk_gate, float* logits_out,
                                 float* aux_partials, cudaStream_t st) {
  // one CTA per 32-token slice; aux_partials has 4*ceil(T/128) slice rows
  const int blocks = 4 * ((c.T + 127) / 128);
  const bool aux = c.score == MOE_SCORE_SOFTMAX && aux_partials != nullptr;
  const size_t smem = aux ? sizeof(float) * kSel * c.E : 0;
  router_select_kernel<<<blocks, kSel * 32, smem, st>>>(raw, ld, c.T, c.E, c.k, c.score, c.n_groups, c.topk_groups,
                                                        c.gate_scale, expert_bias, logit_bias, topk_idx,
                                                        topk_gate, logits_out, aux_partials);
  return cudaGetLastError();
}

}  // namespace moe

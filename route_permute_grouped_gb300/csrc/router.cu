// Router selection: from the fp32 logits of the router GEMM to the top-k
// experts and gates of every token (figures & tables page of the report,
// Fig. 2: score function, top-k selection, load balancing).
//
// One warp per token (a warp takes two tokens of its CTA's 32-token slice).
// Lane l holds the experts e = l + 32 j (j < 8, E <= 256) in registers. Per
// token:
//   L = logit + logit_bias; score = softmax(L) or sigmoid(L);
//   z = L (softmax without expert bias or group limit: the same order as the
//       probabilities) or score + expert_bias;
//   group limit: group score = sum of its two largest z, keep the best
//       topk_groups groups (lower group index wins ties), z = -inf elsewhere;
//   top-k of (z, -e) from per-lane sorted candidates and k rounds of warp
//       reductions (redux.sync): a lower expert index wins ties and slot i
//       holds the i-th largest z;
//   gates = gate_scale * score_i / sum of the selected scores (softmax: the
//       selected probabilities renormalised, computed from the selected logits).
// Optional outputs: the biased logits [T,E] and, for softmax, the column sums
// of the probabilities over the slice (aux_partials row = slice), reduced in a
// fixed order in shared memory.
#include "host_util.h"

namespace moe {

constexpr int kSel = 32;  // tokens (warps) per CTA = aux_partials slice

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
// warp maximum in one instruction (NaN inputs are ignored)
__device__ __forceinline__ float warp_max(float v) {
  float m;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(m) : "f"(v));
  return m;
}
__device__ __forceinline__ uint32_t warp_min_u32(uint32_t v) { return __reduce_min_sync(0xffffffffu, v); }

constexpr int kSelWarps = 16;                  // warps per CTA
constexpr int kTokPerWarp = kSel / kSelWarps;  // tokens per warp (2)

// Score modes of the selection kernel (compile-time):
//   SEL_SOFTMAX_LOGIT  softmax scores, no expert bias, no group limit: z = L
//                      (the logits order the probabilities), gates from the
//                      selected logits;
//   SEL_SOFTMAX_BIAS   softmax scores, with expert bias (z = p + b) or group
//                      limit (z = p);
//   SEL_SIGMOID        sigmoid scores (+ expert bias if given): z = s + b.
enum SelMode : int { SEL_SOFTMAX_LOGIT = 0, SEL_SOFTMAX_BIAS = 1, SEL_SIGMOID = 2 };

// Selection for one token. This lane holds the token's biased logits L[j] of
// experts lane + 32 j (j < NJ; -inf past E or past T). Writes the token's
// outputs and, when p_row != nullptr, its softmax values to p_row[e].
//
// Top-k: every lane sorts its NJ candidates by (z desc, e asc); a round takes
// the warp maximum of the lanes' heads (redux.sync), then the smallest expert
// among the lanes whose head equals it (a second redux.sync), and the winning
// lane drops its head. NaN values of z are taken as -inf.
template <int NJ, int MODE>
__device__ __forceinline__ void select_token(const float (&L)[NJ], int t, bool valid, int lane, int E, int k,
                                             bool force, int n_groups, int topk_groups, float gate_scale,
                                             const float* __restrict__ expert_bias, int32_t* __restrict__ topk_idx,
                                             float* __restrict__ topk_gate, float* __restrict__ logits_out,
                                             float* p_row) {
  constexpr bool kSoftmax = MODE != SEL_SIGMOID;
  constexpr bool kZL = MODE == SEL_SOFTMAX_LOGIT;
  float sc[NJ], z[NJ];
  // softmax probabilities: needed for the aux statistics or as the selection
  // scores; with z = L and no aux they are never formed
  if (kSoftmax && (!kZL || p_row != nullptr)) {
    float mx = -INFINITY;
#pragma unroll
    for (int j = 0; j < NJ; ++j)
      if (lane + 32 * j < E && valid) mx = fmaxf(mx, L[j]);
    mx = warp_max(mx);
    float ex[NJ], sum = 0.0f;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      ex[j] = (lane + 32 * j < E && valid) ? __expf(L[j] - mx) : 0.0f;
      sum += ex[j];
    }
    const float tot = warp_sum(sum);
    const float inv_sum = valid ? 1.0f / tot : 0.0f;  // tokens past T: all zero
#pragma unroll
    for (int j = 0; j < NJ; ++j) sc[j] = ex[j] * inv_sum;
  } else if (!kSoftmax) {
#pragma unroll
    for (int j = 0; j < NJ; ++j)
      sc[j] = (lane + 32 * j < E && valid) ? 1.0f / (1.0f + __expf(-L[j])) : 0.0f;
  } else {
#pragma unroll
    for (int j = 0; j < NJ; ++j) sc[j] = 0.0f;
  }
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const int e = lane + 32 * j;
    const bool in = e < E && valid;
    float zz = kZL ? L[j] : sc[j] + (expert_bias != nullptr && e < E ? expert_bias[e] : 0.0f);
    if (!in || zz != zz) zz = -INFINITY;
    z[j] = zz;
  }
  if (valid && logits_out != nullptr) {
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const int e = lane + 32 * j;
      if (e < E) logits_out[static_cast<size_t>(t) * E + e] = L[j];
    }
  }
  if (p_row != nullptr) {
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const int e = lane + 32 * j;
      if (e < E) p_row[e] = sc[j];  // 0 for tokens past T
    }
  }
  int my_e = 0;
  float my_sc = 0.0f;
  if (force) {
    // force-balanced routing: slot `lane` takes expert (t k + lane) mod E; its
    // score comes from the lane that holds that expert
    const int ei = static_cast<int>((static_cast<long long>(t) * k + lane) % E);
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const float v = __shfl_sync(0xffffffffu, kZL ? L[j] : sc[j], ei & 31);
      if ((ei >> 5) == j) my_sc = v;
    }
    my_e = ei;
  }
  // group-limited selection
  if (!force && n_groups > 1 && topk_groups < n_groups) {
    const int gsz = E / n_groups;
    uint32_t keep = 0u;
    float gscore[32];
#pragma unroll 1
    for (int g = 0; g < n_groups; ++g) {
      // this lane's two largest z of group g, then the warp's two largest
      float b1 = -INFINITY, b2 = -INFINITY;
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        const int e = lane + 32 * j;
        if (e < E && e / gsz == g) {
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
    for (int j = 0; j < NJ; ++j) {
      const int e = lane + 32 * j;
      if (e < E && !((keep >> (e / gsz)) & 1u)) z[j] = -INFINITY;
    }
  }
  // this lane's candidates (z, expert, published score), sorted by an
  // odd-even transposition network, descending by (z, -e); the padding past
  // E sorts last among equal values because its expert index is larger
  float cz[NJ], cv[NJ];
  int ce[NJ];
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    cz[j] = z[j];
    ce[j] = lane + 32 * j;
    cv[j] = sc[j];
  }
#pragma unroll
  for (int r = 0; r < NJ; ++r) {
#pragma unroll
    for (int j = r & 1; j + 1 < NJ; j += 2) {
      const bool sw = cz[j + 1] > cz[j] || (cz[j + 1] == cz[j] && ce[j + 1] < ce[j]);
      if (sw) {
        const float tz = cz[j]; cz[j] = cz[j + 1]; cz[j + 1] = tz;
        const int te = ce[j]; ce[j] = ce[j + 1]; ce[j + 1] = te;
        if (!kZL) { const float tv = cv[j]; cv[j] = cv[j + 1]; cv[j + 1] = tv; }
      }
    }
  }
  // k rounds; lane i keeps slot i
#pragma unroll 1
  for (int i = 0; i < (force ? 0 : k); ++i) {
    const float m = warp_max(cz[0]);
    const int e = static_cast<int>(warp_min_u32(cz[0] == m ? static_cast<uint32_t>(ce[0]) : 0xffffffffu));
    const float sel = kZL ? m : __shfl_sync(0xffffffffu, cv[0], e & 31);
    if (lane == i) {
      my_e = e;
      my_sc = sel;
    }
    if (ce[0] == e) {  // the winning lane drops its head
#pragma unroll
      for (int j = 0; j + 1 < NJ; ++j) {
        cz[j] = cz[j + 1];
        ce[j] = ce[j + 1];
        if (!kZL) cv[j] = cv[j + 1];
      }
      cz[NJ - 1] = -INFINITY;
      ce[NJ - 1] = lane + 32 * NJ;  // past every expert of this warp
    }
  }
  // gates over the k slots (lanes 0..k-1)
  float w;
  if (kZL) {
    const float top = warp_max(lane < k ? my_sc : -INFINITY);
    w = lane < k ? __expf(my_sc - top) : 0.0f;
  } else {
    w = lane < k ? my_sc : 0.0f;
  }
  const float tot = warp_sum(w);
  if (valid && lane < k) {
    topk_idx[static_cast<size_t>(t) * k + lane] = my_e;
    topk_gate[static_cast<size_t>(t) * k + lane] = gate_scale * w / tot;
  }
}

// One CTA of 16 warps per 32-token slice; warp w takes tokens 2w and 2w+1 of
// the slice, loading both tokens' logits before working on the first.
template <int NJ, int MODE>
__global__ void __launch_bounds__(kSelWarps * 32) router_select_kernel(
    const float* __restrict__ raw, int ld, int T, int E, int k, int force, int n_groups, int topk_groups,
    float gate_scale,
    const float* __restrict__ expert_bias, const float* __restrict__ logit_bias, int32_t* __restrict__ topk_idx,
    float* __restrict__ topk_gate, float* __restrict__ logits_out, float* __restrict__ aux_partials) {
  extern __shared__ float s_p[];  // [kSel][E] softmax values (aux only)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool want_aux = MODE != SEL_SIGMOID && aux_partials != nullptr;
  float bias[NJ];
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const int e = lane + 32 * j;
    bias[j] = (logit_bias != nullptr && e < E) ? logit_bias[e] : 0.0f;
  }
  float Ls[kTokPerWarp][NJ];
#pragma unroll
  for (int i = 0; i < kTokPerWarp; ++i) {
    const int t = blockIdx.x * kSel + warp * kTokPerWarp + i;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const int e = lane + 32 * j;
      Ls[i][j] = (t < T && e < E) ? raw[static_cast<size_t>(t) * ld + e] + bias[j] : -INFINITY;
    }
  }
#pragma unroll
  for (int i = 0; i < kTokPerWarp; ++i) {
    const int r = warp * kTokPerWarp + i;
    const int t = blockIdx.x * kSel + r;
    select_token<NJ, MODE>(Ls[i], t, t < T, lane, E, k, force != 0, n_groups, topk_groups, gate_scale, expert_bias,
                           topk_idx, topk_gate, logits_out, want_aux ? s_p + r * E : nullptr);
  }
  if (want_aux) {
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kSelWarps * 32) {
      float acc = 0.0f;
      for (int r = 0; r < kSel; ++r) acc += s_p[r * E + e];
      aux_partials[static_cast<size_t>(blockIdx.x) * E + e] = acc;
    }
  }
}

template <int MODE>
using SelKernel = void (*)(const float*, int, int, int, int, int, int, int, float, const float*, const float*,
                           int32_t*, float*, float*, float*);

template <int MODE>
static SelKernel<MODE> pick_select_kernel(int nj) {
  switch (nj) {
    case 1: return router_select_kernel<1, MODE>;
    case 2: return router_select_kernel<2, MODE>;
    case 3: return router_select_kernel<3, MODE>;
    case 4: return router_select_kernel<4, MODE>;
    case 5: return router_select_kernel<5, MODE>;
    case 6: return router_select_kernel<6, MODE>;
    case 7: return router_select_kernel<7, MODE>;
    default: return router_select_kernel<8, MODE>;
  }
}

cudaError_t launch_router_select(const moe_config& c, const float* raw, int ld, const float* expert_bias,
                                 const float* logit_bias, int32_t* topk_idx, float* topk_gate, float* logits_out,
                                 float* aux_partials, cudaStream_t st) {
  // one CTA per 32-token slice; aux_partials has 4*ceil(T/128) slice rows
  const int blocks = 4 * ((c.T + 127) / 128);
  const bool aux = c.score == MOE_SCORE_SOFTMAX && aux_partials != nullptr;
  const size_t smem = aux ? sizeof(float) * kSel * c.E : 0;
  const int nj = (c.E + 31) / 32;
  const bool softmax = c.score == MOE_SCORE_SOFTMAX;
  // a group limit ranks groups by sums of scores, which logits do not order
  const bool grouped = !c.force_balanced && c.n_groups > 1 && c.topk_groups < c.n_groups;
  if (softmax && expert_bias == nullptr && !grouped) {
    pick_select_kernel<SEL_SOFTMAX_LOGIT>(nj)<<<blocks, kSelWarps * 32, smem, st>>>(
        raw, ld, c.T, c.E, c.k, c.force_balanced, c.n_groups, c.topk_groups, c.gate_scale, expert_bias, logit_bias,
        topk_idx, topk_gate, logits_out, aux_partials);
  } else if (softmax) {
    pick_select_kernel<SEL_SOFTMAX_BIAS>(nj)<<<blocks, kSelWarps * 32, smem, st>>>(
        raw, ld, c.T, c.E, c.k, c.force_balanced, c.n_groups, c.topk_groups, c.gate_scale, expert_bias, logit_bias,
        topk_idx, topk_gate, logits_out, aux_partials);
  } else {
    pick_select_kernel<SEL_SIGMOID>(nj)<<<blocks, kSelWarps * 32, smem, st>>>(
        raw, ld, c.T, c.E, c.k, c.force_balanced, c.n_groups, c.topk_groups, c.gate_scale, expert_bias, logit_bias,
        topk_idx, topk_gate, logits_out, aux_partials);
  }
  return cudaGetLastError();
}

}  // namespace moe

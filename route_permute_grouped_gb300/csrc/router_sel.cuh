// Router selection in the epilogue of the router's logits GEMM (figures &
// tables page of the report: Fig. 2, linear projection -> score function ->
// top-k selection -> load balancing; Fig. 21, router fusion).
//
// One thread per token: the epilogue warp of TMEM lane quadrant q owns
// accumulator rows 32q .. 32q+31 of its CTA's 128-row tile and reads its row's
// logits 32 columns at a time (tcgen05.ld), so the fp32 logits never travel
// through HBM and no second kernel re-reads them. The row's selection values
// z are parked in the CTA's tensor memory past the accumulator (columns
// kRouterZCol + e) by the first pass that forms them; the later passes re-read
// them there instead of recomputing softmax or sigmoid.
//
// Per token (E experts, k <= 16 slots):
//   L = acc + logit_bias                                  (logits_out: L)
//   softmax statistics m = max L, S = sum exp(L - m)      (when probabilities
//       are needed: selection on probabilities, or the aux statistics)
//   z = L          softmax without expert bias or group limit (the logits
//                  order the probabilities)
//     = p + b      softmax otherwise (b = expert bias, selection only)
//     = s + b      sigmoid, s = 1 / (1 + exp(-L));       NaN -> -inf
//   group limit: group score = sum of the group's two largest z, the best
//       topk_groups groups kept (a lower group wins ties), z = -inf elsewhere
//   t = k-th largest z; selected = {z > t} and the lowest-index experts with
//       z == t up to k experts; slots ordered by (z desc, e asc), i.e. a lower
//       expert index wins every tie
//   force-balanced routing: slot i takes expert (t k + i) mod E instead
//   gates = gate_scale * w_i / sum_j w_j over the k slots, w = exp(L_i - max
//       selected L) (softmax: the selected probabilities renormalised) or
//       sigmoid(L_i) (sigmoid: the unbiased scores)
//   aux partials (softmax): column sums of p over the warp's 32 tokens (one
//       32-token slice row of aux_partials), reduced across the lanes by a
//       halving butterfly: after five exchange steps lane j holds column j of
//       the 32-column chunk.
#pragma once
#include "gemm_tc.cuh"

namespace moe {

// the router GEMM keeps one accumulator at TMEM column 0 (E <= 256 columns);
// the selection values of the tile's rows go to columns 256 ..
constexpr uint32_t kRouterZCol = 256;
constexpr int kRouterRows = 128;  // accumulator rows of a CTA = epilogue threads

// Shared memory of the router epilogue (in the epilogue staging region): the
// logit and expert biases (zero-padded to 256), and per thread the k selected
// (z, L, expert) stored slot-major ([slot][128], so the 32 lanes of a warp
// touch 32 consecutive words); the group scores ([group][128], up to 32
// groups) alias the z and L lists, which are filled only after the groups
// are chosen.
struct RouterSmem {
  float* lb;
  float* eb;
  float* sz;
  float* sL;
  int* se;
  __device__ __forceinline__ explicit RouterSmem(uint8_t* base)
      : lb(reinterpret_cast<float*>(base)),
        eb(lb + 256),
        sz(eb + 256),
        sL(sz + 16 * kRouterRows),
        se(reinterpret_cast<int*>(sL + 16 * kRouterRows)) {}
};
constexpr int kRouterSmemBytes = (512 + 3 * 16 * kRouterRows) * 4;

__device__ __forceinline__ void rs_ld(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  tmem_ld32(taddr, r);
  tmem_ld_wait();
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}
__device__ __forceinline__ void rs_st(uint32_t taddr, const float (&v)[32]) {
  uint32_t r[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(v[j]);
  tmem_st32(taddr, r);
  tmem_st_wait();
}

// Sum of v[j] over the warp's lanes, left in lane j (every lane passes its 32
// values; v is consumed).
__device__ __forceinline__ float lane_column_sums(float (&v)[32], int lane) {
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) {
    const bool upper = (lane & s) != 0;
#pragma unroll
    for (int j = 0; j < s; ++j) {
      const float send = upper ? v[j] : v[j + s];
      const float keep = upper ? v[j + s] : v[j];
      v[j] = keep + __shfl_xor_sync(0xffffffffu, send, s);
    }
  }
  return v[0];
}

// The whole selection of one accumulator row (token `row`, thread `tid` of the
// 128 epilogue threads). KM: capacity of the top-k list (8 or 16, >= k).
// Every tcgen05 access is executed by all 32 lanes (rows past T included).
template <int KM>
__device__ __forceinline__ void router_select_row(const GemmParams& p, uint32_t tacc, uint32_t tz, int row, int tid,
                                                  int lane, int slice, const RouterSmem& sm) {
  const int E = p.E, k = p.k, nch = (E + 31) >> 5;
  const bool valid = row < p.T;
  const int mode = p.r_mode;
  const bool force = p.r_force != 0;
  const bool grouped = !force && p.r_groups > 1 && p.r_topk_groups < p.r_groups;
  const bool want_aux = p.r_aux != nullptr;
  const bool need_p = mode == RSEL_SOFTMAX || want_aux;

  // pass 1: biased logits (out to logits_out), softmax statistics
  float m = -INFINITY, S = 0.0f;
  for (int c = 0; c < nch; ++c) {
    float v[32];
    rs_ld(tacc + 32 * c, v);
    float cm = -INFINITY;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      v[j] += sm.lb[32 * c + j];
      if (32 * c + j < E) cm = fmaxf(cm, v[j]);
    }
    if (p.r_logits != nullptr && valid) {
      float* dst = p.r_logits + static_cast<size_t>(row) * E + 32 * c;
      if (32 * c + 32 <= E && (E & 3) == 0) {
#pragma unroll
        for (int q = 0; q < 8; ++q)
          reinterpret_cast<float4*>(dst)[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (32 * c + j < E) dst[j] = v[j];
      }
    }
    if (need_p) {
      const float mn = fmaxf(m, cm);
      float cs = 0.0f;
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (32 * c + j < E) cs += __expf(v[j] - mn);
      S = S * __expf(m - mn) + cs;
      m = mn;
    }
  }
  const float inv = (valid && S > 0.0f) ? 1.0f / S : 0.0f;

  // pass 2: z parked in TMEM; group scores; aux column sums
  const int gsz = grouped ? E / p.r_groups : 1;
  int gcur = 0, gcnt = 0;
  float gb1 = -INFINITY, gb2 = -INFINITY;
  const int nslices = 4 * ((p.T + 127) >> 7);
  for (int c = 0; c < nch; ++c) {
    float v[32], z[32], pr[32];
    rs_ld(tacc + 32 * c, v);
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int e = 32 * c + j;
      const float L = v[j] + sm.lb[e];
      const float pe = need_p ? __expf(L - m) * inv : 0.0f;
      float zz = mode == RSEL_LOGIT ? L : (mode == RSEL_SOFTMAX ? pe + sm.eb[e] : 1.0f / (1.0f + __expf(-L)) + sm.eb[e]);
      if (zz != zz || e >= E) zz = -INFINITY;
      z[j] = zz;
      pr[j] = e < E ? pe : 0.0f;
      if (grouped && e < E) {
        if (zz > gb1) {
          gb2 = gb1;
          gb1 = zz;
        } else if (zz > gb2) {
          gb2 = zz;
        }
        if (++gcnt == gsz) {
          sm.sz[gcur * kRouterRows + tid] = gsz >= 2 ? gb1 + gb2 : gb1;
          ++gcur;
          gcnt = 0;
          gb1 = gb2 = -INFINITY;
        }
      }
    }
    if (!force) rs_st(tz + 32 * c, z);
    if (want_aux) {
      const float col = lane_column_sums(pr, lane);
      if (32 * c + lane < E && slice < nslices) p.r_aux[static_cast<size_t>(slice) * E + 32 * c + lane] = col;
    }
  }

  float sz_[KM], sl_[KM];
  int se_[KM];
  if (force) {
    // slot i: expert (row k + i) mod E, in slot order
    const int start = static_cast<int>((static_cast<long long>(row) * k) % E);
    for (int c = 0; c < nch; ++c) {
      float v[32];
      rs_ld(tacc + 32 * c, v);
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int e = 32 * c + j;
        int rel = e - start;
        if (rel < 0) rel += E;
        if (e < E && rel < k) {
          sm.sL[rel * kRouterRows + tid] = v[j] + sm.lb[e];
          sm.se[rel * kRouterRows + tid] = e;
        }
      }
    }
#pragma unroll
    for (int i = 0; i < KM; ++i) {
      sz_[i] = 0.0f;
      sl_[i] = i < k ? sm.sL[i * kRouterRows + tid] : 0.0f;
      se_[i] = i < k ? sm.se[i * kRouterRows + tid] : 0;
    }
  } else {
    if (grouped) {
      // keep the best topk_groups groups, then mask the others' z in TMEM
      uint32_t keep = 0u;
      for (int s = 0; s < p.r_topk_groups; ++s) {
        int bi = -1;
        float best = -INFINITY;
        for (int g = 0; g < p.r_groups; ++g) {
          if ((keep >> g) & 1u) continue;
          const float gs = sm.sz[g * kRouterRows + tid];
          if (bi < 0 || gs > best) {
            best = gs;
            bi = g;
          }
        }
        keep |= 1u << bi;
      }
      int g = 0, cnt = 0;
      for (int c = 0; c < nch; ++c) {
        float z[32];
        rs_ld(tz + 32 * c, z);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if (32 * c + j < E) {
            if (!((keep >> g) & 1u)) z[j] = -INFINITY;
            if (++cnt == gsz) {
              cnt = 0;
              ++g;
            }
          }
        }
        rs_st(tz + 32 * c, z);
      }
    }
    // pass 3: t = k-th largest z (a sorted list of the KM largest values)
    float b[KM];
#pragma unroll
    for (int i = 0; i < KM; ++i) b[i] = -INFINITY;
    for (int c = 0; c < nch; ++c) {
      float z[32];
      rs_ld(tz + 32 * c, z);
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        float cnd = 32 * c + j < E ? z[j] : -INFINITY;
#pragma unroll
        for (int i = 0; i < KM; ++i) {
          const float hi = fmaxf(b[i], cnd);
          cnd = fminf(b[i], cnd);
          b[i] = hi;
        }
      }
    }
    float t = b[0];
#pragma unroll
    for (int i = 1; i < KM; ++i)
      if (i == k - 1) t = b[i];
    // pass 4: how many lie strictly above t
    int ngt = 0;
    for (int c = 0; c < nch; ++c) {
      float z[32];
      rs_ld(tz + 32 * c, z);
#pragma unroll
      for (int j = 0; j < 32; ++j) ngt += (32 * c + j < E && z[j] > t) ? 1 : 0;
    }
    // pass 5: collect in ascending expert order: every z > t, and z == t
    // while slots remain (the lowest indices win the tie)
    int n = 0, eq_left = k - ngt;
    for (int c = 0; c < nch; ++c) {
      float z[32], v[32];
      rs_ld(tz + 32 * c, z);
      rs_ld(tacc + 32 * c, v);
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int e = 32 * c + j;
        if (e >= E) continue;
        bool take = z[j] > t;
        if (!take && z[j] == t && eq_left > 0) {
          take = true;
          --eq_left;
        }
        if (take && n < k) {
          sm.sz[n * kRouterRows + tid] = z[j];
          sm.sL[n * kRouterRows + tid] = v[j] + sm.lb[e];
          sm.se[n * kRouterRows + tid] = e;
          ++n;
        }
      }
    }
    // slots by (z desc, e asc): odd-even transposition over the list
#pragma unroll
    for (int i = 0; i < KM; ++i) {
      sz_[i] = i < n ? sm.sz[i * kRouterRows + tid] : -INFINITY;
      sl_[i] = i < n ? sm.sL[i * kRouterRows + tid] : 0.0f;
      se_[i] = i < n ? sm.se[i * kRouterRows + tid] : (1 << 20) + i;
    }
#pragma unroll
    for (int r = 0; r < KM; ++r) {
#pragma unroll
      for (int j = r & 1; j + 1 < KM; j += 2) {
        const bool sw = sz_[j + 1] > sz_[j] || (sz_[j + 1] == sz_[j] && se_[j + 1] < se_[j]);
        if (sw) {
          const float tz_ = sz_[j]; sz_[j] = sz_[j + 1]; sz_[j + 1] = tz_;
          const float tl = sl_[j]; sl_[j] = sl_[j + 1]; sl_[j + 1] = tl;
          const int te = se_[j]; se_[j] = se_[j + 1]; se_[j + 1] = te;
        }
      }
    }
  }

  // gates over the k slots
  float w[KM];
  float sum = 0.0f;
  if (mode != RSEL_SIGMOID) {
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < KM; ++i)
      if (i < k) mx = fmaxf(mx, sl_[i]);
#pragma unroll
    for (int i = 0; i < KM; ++i) w[i] = i < k ? __expf(sl_[i] - mx) : 0.0f;
  } else {
#pragma unroll
    for (int i = 0; i < KM; ++i) w[i] = i < k ? 1.0f / (1.0f + __expf(-sl_[i])) : 0.0f;
  }
#pragma unroll
  for (int i = 0; i < KM; ++i) sum += w[i];
  if (valid) {
    const float sc = p.r_gate_scale / sum;
#pragma unroll
    for (int i = 0; i < KM; ++i) {
      if (i < k) {
        p.r_idx[static_cast<size_t>(row) * k + i] = se_[i];
        p.r_gate[static_cast<size_t>(row) * k + i] = sc * w[i];
      }
    }
  }
}

}  // namespace moe

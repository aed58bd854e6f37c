// Router selection in the epilogue of the router's logits GEMM (figures &
// tables page of the report: Fig. 2, linear projection -> score function ->
// top-k selection -> load balancing; Fig. 21, router fusion).
//
// A token's row of the accumulator is worked on by the two epilogue warps of
// its TMEM lane quadrant ("parts"): part h reads the row's logits in the
// 32-column chunks [h * cpp, (h + 1) * cpp) of the E experts (cpp = half the
// chunks, rounded up), so lower parts hold lower expert indices. The parts
// exchange per-row partial results through shared memory at named barriers
// (one per quadrant, the quadrant's 64 threads). The fp32 logits never travel
// through HBM and no second kernel re-reads them. Selection values that are
// not the logits themselves are parked in the CTA's tensor memory past the
// accumulator (columns kRouterZCol + e) by the pass that forms them.
//
// Per token (E experts, k <= 16 slots):
//   L = acc + logit_bias                                  (logits_out: L)
//   softmax statistics m = max L, S = sum exp(L - m)      (when probabilities
//       are needed: selection on probabilities, or the aux statistics); each
//       part forms them over its chunks, then both combine the two
//   z = L          RSEL_LOGIT: softmax without expert bias or group limit (the
//                  logits order the probabilities)
//     = p + b      RSEL_SOFTMAX (b = expert bias, selection only)
//     = s + b      RSEL_SIGMOID, s = 1 / (1 + exp(-L));   NaN -> -inf
//   group limit: group score = sum of the group's two largest z, the best
//       topk_groups groups kept (a lower group wins ties), z = -inf elsewhere
//       (part 0 scores every group; each part masks its own chunks)
//   t = k-th largest z (each part keeps the KM largest values of its chunks,
//       then both merge the two lists); selected = {z > t} and the
//       lowest-index experts with z == t up to k experts; slots ordered by
//       (z desc, e asc), i.e. a lower expert index wins every tie
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
// the parked selection values of the tile's rows go to columns 256 ..
constexpr uint32_t kRouterZCol = 256;
constexpr int kRouterRows = 128;  // accumulator rows of a CTA
constexpr int kRouterParts = 2;   // epilogue warps per TMEM lane quadrant

// Shared memory of the router epilogue (in the epilogue staging region),
// every per-row array stored [entry][128 rows] so the 32 lanes of a warp touch
// 32 consecutive words:
//   lb, eb     logit and expert biases, zero-padded to 256 experts;
//   st_m, st_s each part's softmax maximum and sum;
//   gt, eq     each part's count of values above / equal to the threshold;
//   keep       the kept groups of each row (bit mask);
//   a union, used at different times: the parts' top-KM value lists
//   top[part][KM], the group scores gs[32], or the k selected slots
//   (sz, sL: selection value and logit; se: expert).
struct RouterSmem {
  float* lb;
  float* eb;
  float* st_m;
  float* st_s;
  int* gt;
  int* eq;
  uint32_t* keep;
  float* top;
  float* gs;
  float* sz;
  float* sL;
  int* se;
  __device__ __forceinline__ explicit RouterSmem(uint8_t* base) {
    float* f = reinterpret_cast<float*>(base);
    lb = f;
    eb = f + 256;
    st_m = f + 512;
    st_s = st_m + kRouterParts * kRouterRows;
    gt = reinterpret_cast<int*>(st_s + kRouterParts * kRouterRows);
    eq = gt + kRouterParts * kRouterRows;
    keep = reinterpret_cast<uint32_t*>(eq + kRouterParts * kRouterRows);
    float* u = reinterpret_cast<float*>(keep + kRouterRows);
    top = u;
    gs = u;
    sz = u;
    sL = u + 16 * kRouterRows;
    se = reinterpret_cast<int*>(u + 32 * kRouterRows);
  }
};
constexpr int kRouterSmemBytes = (512 + 4 * kRouterParts * kRouterRows + kRouterRows + 48 * kRouterRows) * 4;

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

// insert c into the descending list b[KM] (the smallest value drops out)
template <int KM>
__device__ __forceinline__ void topk_insert(float (&b)[KM], float c) {
#pragma unroll
  for (int i = 0; i < KM; ++i) {
    const float hi = fmaxf(b[i], c);
    c = fminf(b[i], c);
    b[i] = hi;
  }
}

// The selection values of chunk c of this thread's row (32 experts), from
// the accumulator (RSEL_LOGIT) or the parked values.
template <int MODE>
__device__ __forceinline__ void chunk_z(uint32_t tacc, uint32_t tz, int c, int E, const RouterSmem& sm,
                                        float (&z)[32]) {
  if constexpr (MODE == RSEL_LOGIT) {
    rs_ld(tacc + 32 * c, z);
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float L = z[j] + sm.lb[32 * c + j];
      z[j] = (32 * c + j < E && L == L) ? L : -INFINITY;
    }
  } else {
    rs_ld(tz + 32 * c, z);
  }
}

// One part's share of the selection of accumulator row `row` (thread `tid`
// of the quadrant's rows 32q .. 32q+31, lane `lane`). Both parts of a quadrant
// run it in lockstep: every named barrier below is reached by both.
template <int KM, int MODE>
__device__ __forceinline__ void router_select_part(const GemmParams& p, uint32_t tacc, uint32_t tz, int row, int tid,
                                                   int lane, int q, int part, int slice, const RouterSmem& sm) {
  const int E = p.E, k = p.k, nch = (E + 31) >> 5;
  const int cpp = (nch + 1) >> 1;
  const int c0 = part * cpp, c1 = min(nch, c0 + cpp);
  const bool valid = row < p.T;
  const bool force = p.r_force != 0;
  const bool grouped = MODE != RSEL_LOGIT && !force && p.r_groups > 1 && p.r_topk_groups < p.r_groups;
  const bool want_aux = p.r_aux != nullptr;
  const bool need_p = MODE == RSEL_SOFTMAX || want_aux;
  const int bar = 2 + q;  // named barrier of the quadrant's two warps
  const int me = part * kRouterRows + tid;
  const int other = (part ^ 1) * kRouterRows + tid;

  // pass 1: biased logits (out to logits_out), softmax statistics of the part
  // (skipped when there is neither)
  float m = -INFINITY, S = 0.0f;
  const bool pass1 = need_p || p.r_logits != nullptr;
  for (int c = c0; pass1 && c < c1; ++c) {
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
        for (int w = 0; w < 8; ++w)
          reinterpret_cast<float4*>(dst)[w] = make_float4(v[4 * w], v[4 * w + 1], v[4 * w + 2], v[4 * w + 3]);
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
      S = (m == -INFINITY ? 0.0f : S * __expf(m - mn)) + cs;
      m = mn;
    }
  }
  if (need_p) {
    sm.st_m[me] = m;
    sm.st_s[me] = S;
  }
  named_bar_sync(bar, 64);
  float inv = 0.0f;
  if (need_p) {
    const float mo = sm.st_m[other], so = sm.st_s[other];
    const float mm = fmaxf(m, mo);
    const float tot = (m == -INFINITY ? 0.0f : S * __expf(m - mm)) + (mo == -INFINITY ? 0.0f : so * __expf(mo - mm));
    m = mm;
    inv = (valid && tot > 0.0f) ? 1.0f / tot : 0.0f;
  }

  // pass 2: selection values (parked unless they are the logits); aux sums;
  // with a group limit whose groups lie inside this part's chunks, the part
  // also scores its own groups here (top-2 sum each) as the values pass by
  const int nslices = 4 * ((p.T + 127) >> 7);
  const int gsz = grouped ? E / p.r_groups : 1;
  const bool own_groups = grouped && (32 * cpp) % gsz == 0;
  if (MODE != RSEL_LOGIT || want_aux) {
    int og = (32 * c0) / gsz, ocnt = 0;
    float ob1 = -INFINITY, ob2 = -INFINITY;
    for (int c = c0; c < c1; ++c) {
      float v[32], z[32], pr[32];
      rs_ld(tacc + 32 * c, v);
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int e = 32 * c + j;
        const float L = v[j] + sm.lb[e];
        const float pe = need_p ? __expf(L - m) * inv : 0.0f;
        float zz;
        if constexpr (MODE == RSEL_SOFTMAX) zz = pe + sm.eb[e];
        else if constexpr (MODE == RSEL_SIGMOID) zz = __fdividef(1.0f, 1.0f + __expf(-L)) + sm.eb[e];
        else zz = L;
        if (zz != zz || e >= E) zz = -INFINITY;
        z[j] = zz;
        pr[j] = e < E ? pe : 0.0f;
      }
      if (MODE != RSEL_LOGIT && !force) rs_st(tz + 32 * c, z);
      if (own_groups) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if (32 * c + j < E) {
            if (z[j] > ob1) {
              ob2 = ob1;
              ob1 = z[j];
            } else if (z[j] > ob2) {
              ob2 = z[j];
            }
            if (++ocnt == gsz) {
              sm.gs[og * kRouterRows + tid] = gsz >= 2 ? ob1 + ob2 : ob1;
              ++og;
              ocnt = 0;
              ob1 = ob2 = -INFINITY;
            }
          }
        }
      }
      if (want_aux) {
        const float col = lane_column_sums(pr, lane);
        if (32 * c + lane < E && slice < nslices) p.r_aux[static_cast<size_t>(slice) * E + 32 * c + lane] = col;
      }
    }
  }

  if (force) {
    // slot i: expert (row k + i) mod E, in slot order; part 0 writes it
    if (part == 0) {
      const int start = static_cast<int>((static_cast<long long>(row) * k) % E);
      float wsum = 0.0f, mx = -INFINITY;
      float Ls[16];
      int es[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        es[i] = 0;
        Ls[i] = 0.0f;
      }
      for (int c = 0; c < nch; ++c) {
        float v[32];
        rs_ld(tacc + 32 * c, v);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int e = 32 * c + j;
          int rel = e - start;
          if (rel < 0) rel += E;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            if (i < k && e < E && rel == i) {
              Ls[i] = v[j] + sm.lb[e];
              es[i] = e;
            }
          }
        }
      }
      float w[16];
#pragma unroll
      for (int i = 0; i < 16; ++i)
        if (i < k) mx = fmaxf(mx, Ls[i]);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        w[i] = i >= k ? 0.0f : (MODE == RSEL_SIGMOID ? __fdividef(1.0f, 1.0f + __expf(-Ls[i])) : __expf(Ls[i] - mx));
        wsum += w[i];
      }
      if (valid) {
        const float sc = p.r_gate_scale / wsum;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          if (i < k) {
            p.r_idx[static_cast<size_t>(row) * k + i] = es[i];
            p.r_gate[static_cast<size_t>(row) * k + i] = sc * w[i];
          }
        }
      }
    }
    return;
  }

  uint32_t kp = 0xffffffffu;  // kept groups of this row
  if (grouped) {
    kp = 0u;
    named_bar_sync(bar, 64);  // both parts' values are parked (and own group scores written)
    if (!own_groups && part == 0) {
      // groups straddle the parts: part 0 scores every group from the parked values
      int g = 0, cnt = 0;
      float b1 = -INFINITY, b2 = -INFINITY;
      for (int c = 0; c < nch; ++c) {
        float z[32];
        rs_ld(tz + 32 * c, z);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if (32 * c + j < E) {
            if (z[j] > b1) {
              b2 = b1;
              b1 = z[j];
            } else if (z[j] > b2) {
              b2 = z[j];
            }
            if (++cnt == gsz) {
              sm.gs[g * kRouterRows + tid] = gsz >= 2 ? b1 + b2 : b1;
              ++g;
              cnt = 0;
              b1 = b2 = -INFINITY;
            }
          }
        }
      }
    }
    if (!own_groups) named_bar_sync(bar, 64);
    // the best topk_groups groups (a lower group wins ties), by both parts
    // from the shared scores
    for (int sg = 0; sg < p.r_topk_groups; ++sg) {
      int bi = -1;
      float best = -INFINITY;
      for (int gg = 0; gg < p.r_groups; ++gg) {
        if ((kp >> gg) & 1u) continue;
        const float v = sm.gs[gg * kRouterRows + tid];
        if (bi < 0 || v > best) {
          best = v;
          bi = gg;
        }
      }
      kp |= 1u << bi;
    }
    // each part masks its own parked chunks (groups of whole chunks are
    // masked per chunk where the passes below load them instead)
    for (int c = c0; c < c1 && gsz % 32 != 0; ++c) {
      float z[32];
      rs_ld(tz + 32 * c, z);
      int g = (32 * c) / gsz, cnt = (32 * c) % gsz;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (32 * c + j < E) {
          if (!((kp >> g) & 1u)) z[j] = -INFINITY;
          if (++cnt == gsz) {
            cnt = 0;
            ++g;
          }
        }
      }
      rs_st(tz + 32 * c, z);
    }
    named_bar_sync(bar, 64);  // both parts are done reading the group scores
  }

  // pass 3: the KM largest values of the part's chunks; both lists merged
  float b[KM];
#pragma unroll
  for (int i = 0; i < KM; ++i) b[i] = -INFINITY;
  for (int c = c0; c < c1; ++c) {
    float z[32];
    chunk_z<MODE>(tacc, tz, c, E, sm, z);
    if (grouped && gsz % 32 == 0 && !((kp >> ((32 * c) / gsz)) & 1u)) {
#pragma unroll
      for (int j = 0; j < 32; ++j) z[j] = -INFINITY;
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) topk_insert<KM>(b, z[j]);
  }
#pragma unroll
  for (int i = 0; i < KM; ++i) sm.top[(part * KM + i) * kRouterRows + tid] = b[i];
  named_bar_sync(bar, 64);
#pragma unroll
  for (int i = 0; i < KM; ++i) topk_insert<KM>(b, sm.top[((part ^ 1) * KM + i) * kRouterRows + tid]);
  float t = b[0];
#pragma unroll
  for (int i = 1; i < KM; ++i)
    if (i == k - 1) t = b[i];

  // pass 4: counts above / at the threshold per part
  int ngt = 0, neq = 0;
  for (int c = c0; c < c1; ++c) {
    float z[32];
    chunk_z<MODE>(tacc, tz, c, E, sm, z);
    if (grouped && gsz % 32 == 0 && !((kp >> ((32 * c) / gsz)) & 1u)) {
#pragma unroll
      for (int j = 0; j < 32; ++j) z[j] = -INFINITY;
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      ngt += z[j] > t ? 1 : 0;
      neq += (z[j] == t && 32 * c + j < E) ? 1 : 0;
    }
  }
  sm.gt[me] = ngt;
  sm.eq[me] = neq;
  named_bar_sync(bar, 64);  // also: every part is done reading the top lists
  const int gt0 = sm.gt[tid], gt1 = sm.gt[kRouterRows + tid];
  const int eq0 = sm.eq[tid];
  const int eq_left = k - gt0 - gt1;
  const int a0 = min(eq0, eq_left);
  int allow = part == 0 ? a0 : eq_left - a0;
  int n = part == 0 ? 0 : gt0 + a0;

  // pass 5: the part's selected experts in ascending index order
  for (int c = c0; c < c1; ++c) {
    float z[32], v[32];
    chunk_z<MODE>(tacc, tz, c, E, sm, z);
    if (grouped && gsz % 32 == 0 && !((kp >> ((32 * c) / gsz)) & 1u)) {
#pragma unroll
      for (int j = 0; j < 32; ++j) z[j] = -INFINITY;
    }
    if constexpr (MODE == RSEL_LOGIT) {
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = z[j];
    } else {
      rs_ld(tacc + 32 * c, v);
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] += sm.lb[32 * c + j];
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int e = 32 * c + j;
      bool take = z[j] > t;
      if (!take && z[j] == t && e < E && allow > 0) {
        take = true;
        --allow;
      }
      if (take && n < k) {
        sm.sz[n * kRouterRows + tid] = z[j];
        sm.sL[n * kRouterRows + tid] = v[j];
        sm.se[n * kRouterRows + tid] = e;
        ++n;
      }
    }
  }
  named_bar_sync(bar, 64);
  if (part != 0) return;

  // slots by (z desc, e asc): odd-even transposition over the list; gates
  float sz_[KM], sl_[KM];
  int se_[KM];
#pragma unroll
  for (int i = 0; i < KM; ++i) {
    sz_[i] = i < k ? sm.sz[i * kRouterRows + tid] : -INFINITY;
    sl_[i] = i < k ? sm.sL[i * kRouterRows + tid] : 0.0f;
    se_[i] = i < k ? sm.se[i * kRouterRows + tid] : (1 << 20) + i;
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
  float w[KM];
  float sum = 0.0f;
  if constexpr (MODE != RSEL_SIGMOID) {
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < KM; ++i)
      if (i < k) mx = fmaxf(mx, sl_[i]);
#pragma unroll
    for (int i = 0; i < KM; ++i) w[i] = i < k ? __expf(sl_[i] - mx) : 0.0f;
  } else {
#pragma unroll
    for (int i = 0; i < KM; ++i) w[i] = i < k ? __fdividef(1.0f, 1.0f + __expf(-sl_[i])) : 0.0f;
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

template <int MODE>
__device__ __forceinline__ void router_select_mode(const GemmParams& p, uint32_t tacc, uint32_t tz, int row, int tid,
                                                   int lane, int q, int part, int slice, const RouterSmem& sm) {
  if (p.k <= 8) router_select_part<8, MODE>(p, tacc, tz, row, tid, lane, q, part, slice, sm);
  else router_select_part<16, MODE>(p, tacc, tz, row, tid, lane, q, part, slice, sm);
}

}  // namespace moe

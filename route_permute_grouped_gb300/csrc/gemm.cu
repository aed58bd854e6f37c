// The persistent tcgen05 GEMM kernel and its epilogues (see gemm_tc.cuh for the
// structure). One template, instantiated once per kind.
#include <math.h>

#include "epilogue.cuh"
#include "gemm_tc.cuh"
#include "host_util.h"
#include "router_sel.cuh"

namespace moe {

// ---------------------------------------------------------------------------
// shared-memory layout
// ---------------------------------------------------------------------------
template <int KIND>
struct SmemLayout {
  static constexpr int kStages = KindTraits<KIND>::kStages;
  // output staging for the TMA-store epilogue: 2 (DGRAD2R: 3) x 4 KB per epilogue warp
  static constexpr int kOutOff = KindTraits<KIND>::kStages * KindTraits<KIND>::kStageBytesK;
  static constexpr int kOutBytes = KindTraits<KIND>::kEpiWarps * KindTraits<KIND>::kOutWarpBytes;
  static constexpr int kBarOff = kOutOff + kOutBytes;
  static constexpr int kNumBars = 2 * KindTraits<KIND>::kMaxStages + 5;  // full, empty, tfull[2],
                                                                        // tempty[2], drain
  static constexpr int kTmemSlot = kBarOff + kNumBars * 8;  // u32 TMEM base, int abort flag
  static constexpr int kCumOff = kTmemSlot + 16;
  static constexpr int kOffOff = kCumOff + (kMaxGroups + 1) * 4;
  // WGRAD: the experts in descending order of their rows (one byte each)
  static constexpr int kOrderOff = kOffOff + (kMaxGroups + 1) * 4;
  // WGRAD: 1 when the tiles are walked long / short alternately (skewed rows)
  static constexpr int kSkewOff = kOrderOff + kMaxGroups;
  static constexpr int kBytes = kSkewOff + 4;
  // the dynamic shared memory starts 1024-byte aligned (checked at kernel
  // entry): the 128-byte-swizzled tiles and staging boxes need that alignment
  static constexpr int kDynBytes = kBytes;
  static_assert(kDynBytes <= 232448, "shared memory per CTA");
  static_assert(KIND != KIND_ROUTER || kOutBytes >= kRouterSmemBytes, "router epilogue scratch");
};

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + __expf(-z)); }

// ---------------------------------------------------------------------------
// epilogues (thread = one accumulator row r of the 128-row tile)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void store_bf16x32(__nv_bfloat16* dst, const float* f) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 w;
    w.x = pack_bf16x2(f[8 * q + 0], f[8 * q + 1]);
    w.y = pack_bf16x2(f[8 * q + 2], f[8 * q + 3]);
    w.z = pack_bf16x2(f[8 * q + 4], f[8 * q + 5]);
    w.w = pack_bf16x2(f[8 * q + 6], f[8 * q + 7]);
    d[q] = w;
  }
}
__device__ __forceinline__ void store_f32x32(float* dst, const float* f) {
  float4* d = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int q = 0; q < 8; ++q) d[q] = make_float4(f[4 * q], f[4 * q + 1], f[4 * q + 2], f[4 * q + 3]);
}
__device__ __forceinline__ void load_bf16x32(const __nv_bfloat16* src, float* f) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 w = s[q];
    f[8 * q + 0] = bf16_lo(w.x); f[8 * q + 1] = bf16_hi(w.x);
    f[8 * q + 2] = bf16_lo(w.y); f[8 * q + 3] = bf16_hi(w.y);
    f[8 * q + 4] = bf16_lo(w.z); f[8 * q + 5] = bf16_hi(w.z);
    f[8 * q + 6] = bf16_lo(w.w); f[8 * q + 7] = bf16_hi(w.w);
  }
}
__device__ __forceinline__ void tmem_ld32f(uint32_t taddr, float* f) {
  uint32_t v[32];
  tmem_ld32(taddr, v);
  tmem_ld_wait();
#pragma unroll
  for (int j = 0; j < 32; ++j) f[j] = __uint_as_float(v[j]);
}

// FFN1: columns [0,128) of the accumulator hold h1 = x W1 for F columns
// n0..n0+127, columns [128,256) hold h3 = x W3 for the same F columns (a half
// tile: 64 columns each, h3 from column `up` = 64; nc = 2 chunks of 32).
__device__ __forceinline__ void epi_ffn1(const GemmParams& p, int n0, int row, int m_end, uint32_t tacc,
                                         int nc = 4, int up = 128) {
  const bool valid = row < m_end;
  __nv_bfloat16* a = reinterpret_cast<__nv_bfloat16*>(p.out0);
  __nv_bfloat16* h13 = reinterpret_cast<__nv_bfloat16*>(p.out1);
#pragma unroll 1
  for (int c = 0; c < nc; ++c) {
    float g[32], u[32];
    tmem_ld32f(tacc + c * 32, g);
    tmem_ld32f(tacc + up + c * 32, u);
    const int col = n0 + c * 32;
    if (valid && col < p.F) {
      float o[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) o[j] = silu_f(g[j]) * u[j];
      store_bf16x32(a + static_cast<size_t>(row) * p.F + col, o);
      if (h13 != nullptr) {
        store_bf16x32(h13 + static_cast<size_t>(row) * 2 * p.F + col, g);
        store_bf16x32(h13 + static_cast<size_t>(row) * 2 * p.F + p.F + col, u);
      }
    }
  }
}

// Plain store of a 128 x bn tile: bf16 or fp32, row-major with `ld` columns.
__device__ __forceinline__ void epi_store(const TileInfo& ti, uint32_t tacc, int r, int nchunks, int ncols,
                                          int ld, void* out, bool fp32, size_t row_base, float alpha = 1.0f) {
  const int row = ti.m0 + r;
  const bool valid = row < ti.m_end;
  const bool zero = ti.nkb == 0;  // no k blocks: the product is zero
#pragma unroll 1
  for (int c = 0; c < nchunks; ++c) {
    float f[32];
    if (!zero) {
      tmem_ld32f(tacc + c * 32, f);
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) f[j] = 0.0f;
    }
    const int col = ti.n0 + c * 32;
    if (alpha != 1.0f) {
#pragma unroll
      for (int j = 0; j < 32; ++j) f[j] *= alpha;
    }
    if (valid && col < ncols) {
      const size_t off = (row_base + static_cast<size_t>(row)) * ld + col;
      if (col + 32 <= ncols) {
        if (fp32) store_f32x32(reinterpret_cast<float*>(out) + off, f);
        else store_bf16x32(reinterpret_cast<__nv_bfloat16*>(out) + off, f);
      } else {
        // the matrix ends inside this chunk: columns past it belong to the
        // next row
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if (j >= ncols - col) break;
          if (fp32) reinterpret_cast<float*>(out)[off + j] = f[j];
          else reinterpret_cast<__nv_bfloat16*>(out)[off + j] = __float2bfloat16_rn(f[j]);
        }
      }
    }
  }
}

// Plain store of a half tile (an M = 128 pair MMA): warp q's 32 rows row0..
// (of the CTA's 64) hold output columns n0 + 128 (q / 2) .. at TMEM columns
// 0..127 (lanes 64.. carry the odd CTA's B half).
__device__ __forceinline__ void epi_store_half(const GemmParams& p, const TileInfo& ti, uint32_t tacc, int lane, int q,
                                            int r, int row0, bool full_rows, bool any_rows, Stager& st,
                                            const CUtensorMap* map) {
  TileInfo tw = ti;
  tw.n0 = ti.n0 + 128 * (q >> 1);
  if (full_rows) {
    if (p.out_fp32) epi_store_tma<true, false>(tw, tacc, lane, row0, p.H, st, map, 2);
    else epi_store_tma<false, false>(tw, tacc, lane, row0, p.H, st, map, 2);
  } else if (any_rows) {
    tw.m0 = row0 - 32 * q;  // epi_store takes row = m0 + r, r = 32 q + lane
    epi_store(tw, tacc, r, 4, p.H, p.H, p.out0, p.out_fp32 != 0, 0);
  }
}

// NVFP4 gate/up epilogue, thread = row r of this CTA's 128 rows of the pair
// tile, block b (0..2) of the tile's 96 F columns: h = bf16(g_x g_e acc) for
// the gate (columns 32 b..) and up (96 + 32 b..) halves, a = bf16(SiLU(h1) h3)
// stored to a[row, col..] (rows of this expert only), h stored to out1
// [rows, 2F] when set (training), and max |a| of the warp's rows into
// *nv_amax.
__device__ __forceinline__ void epi_ffn1_nv(const GemmParams& p, const TileInfo& ti, uint32_t tacc, int r, int b) {
  const int col = ti.n0 + 32 * b;
  if (col >= p.F) return;  // uniform: the last tile of a ragged F
  const int row = ti.m0 + r;
  const bool valid = row < ti.m_end;
  const float alpha = __ldg(p.nv_ga) * __ldg(p.nv_gb + ti.g);
  uint32_t v1[32], v3[32];
  tmem_ld32(tacc + 32 * b, v1);
  tmem_ld32(tacc + kMxTileF1 + 32 * b, v3);
  tmem_ld_wait();
  uint32_t o[16];
  float m = 0.0f;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    float a2[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const float h1 = __bfloat162float(__float2bfloat16_rn(alpha * __uint_as_float(v1[2 * j + u])));
      const float h3 = __bfloat162float(__float2bfloat16_rn(alpha * __uint_as_float(v3[2 * j + u])));
      a2[u] = h1 / (1.0f + expf(-h1)) * h3;
    }
    o[j] = pack_bf16x2(a2[0], a2[1]);
    m = fmaxf(m, fmaxf(fabsf(bf16_lo(o[j])), fabsf(bf16_hi(o[j]))));
  }
  if (valid) {
    uint4* d = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out0) + static_cast<size_t>(row) * p.F + col);
#pragma unroll
    for (int q = 0; q < 4; ++q) d[q] = make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
    if (p.out1 != nullptr) {  // training: the stored h1, h3 (bf16) for the backward
      __nv_bfloat16* h13 = reinterpret_cast<__nv_bfloat16*>(p.out1) + static_cast<size_t>(row) * 2 * p.F + col;
      float f[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) f[j] = alpha * __uint_as_float(v1[j]);
      store_bf16x32(h13, f);
#pragma unroll
      for (int j = 0; j < 32; ++j) f[j] = alpha * __uint_as_float(v3[j]);
      store_bf16x32(h13 + p.F, f);
    }
  } else {
    m = 0.0f;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  if ((threadIdx.x & 31) == 0) atomicMax(p.nv_amax, __float_as_uint(m));
}

// MXFP8 gate/up epilogue, thread = row r of this CTA's 128 rows of the pair
// tile, block b (0..2) of the tile's 96 F columns: a = SiLU(h1) h3 (h1 from
// accumulator columns 32 b.., h3 from 96 + 32 b..) is quantised as one MXFP8
// block of the down GEMM's K: codes to a_q[row, col..] (rows of this expert
// only) and the scale to the down GEMM's A scale block 2 * pair tile + rank
// (every row of the tile, so rows past the expert carry a valid scale).
__device__ __forceinline__ void epi_ffn1_mx(const GemmParams& p, const TileInfo& ti, uint32_t tacc, int r,
                                            int rank, int b) {
  const int col = ti.n0 + 32 * b;
  if (col >= p.F) return;  // uniform: the last tile of a ragged F
  const int row = ti.m0 + r;
  uint32_t v1[32], v3[32];
  tmem_ld32(tacc + 32 * b, v1);
  tmem_ld32(tacc + kMxTileF1 + 32 * b, v3);
  tmem_ld_wait();
  float a[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const float h1 = __uint_as_float(v1[j]);
    a[j] = __fdividef(h1, 1.0f + __expf(-h1)) * __uint_as_float(v3[j]);
  }
  uint32_t w[8];
  const uint32_t sb = mx_quant32(a, w);
  if (row < ti.m_end) {
    uint4* d = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(p.out0) + static_cast<size_t>(row) * p.F + col);
    d[0] = make_uint4(w[0], w[1], w[2], w[3]);
    d[1] = make_uint4(w[4], w[5], w[6], w[7]);
    if (p.out1 != nullptr) {  // training: the pre-activations h1, h3 in bf16
      __nv_bfloat16* h13 = reinterpret_cast<__nv_bfloat16*>(p.out1) + static_cast<size_t>(row) * 2 * p.F + col;
      float f[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) f[j] = __uint_as_float(v1[j]);
      store_bf16x32(h13, f);
#pragma unroll
      for (int j = 0; j < 32; ++j) f[j] = __uint_as_float(v3[j]);
      store_bf16x32(h13 + p.F, f);
    }
  }
  const int fb = col / 32;
  p.sfa_out[(static_cast<size_t>(2 * ti.mt + rank) * (p.F / kMxKB) + fb / 4) * kMxSfBytes + mx_sf_pos(r, fb & 3)] =
      static_cast<uint8_t>(sb);
}

// DGRAD2_MX, thread = row r of this CTA's 128 rows of the pair tile, 64-column
// part `part` (0..2) of the tile's 192 F columns (p.H = F here): da from the
// accumulator and the row's saved bf16 h1, h3 give
//   dh1 = da h3 SiLU'(h1), dh3 = da SiLU(h1) -> dh13 (bf16, out0 [rows, 2F])
//   a = SiLU(h1) h3                          -> out1 (bf16, [rows, F])
// and the MXFP8 codes of the bf16 dh1 and dh3 blocks -> q_out [rows, 2F], their
// scales in the gate/up data gradient's A layout (sfa_out, K = 2F: dh1 block
// f / 32, dh3 block F / 32 + f / 32). Rows past the expert's end load nothing
// and store no codes; their scale bytes stay in this expert's own blocks.
// one 32-column block of dh13 (columns c2.. of [0, 2F)) of DGRAD2_MX's row
__device__ __forceinline__ void dgrad2_mx_out(const GemmParams& p, const float (&d)[32], int c2, size_t sblk, int r,
                                              int step, size_t rb, bool valid, __nv_bfloat16* dh13) {
  uint32_t w[8];
  const uint32_t sb = mx_quant32(d, w);
  p.sfa_out[(sblk + c2 / kMxKB) * kMxSfBytes + mx_sf_pos(r, step)] = static_cast<uint8_t>(sb);
  if (valid) {
    uint4* q = reinterpret_cast<uint4*>(p.q_out + rb + c2);
    q[0] = make_uint4(w[0], w[1], w[2], w[3]);
    q[1] = make_uint4(w[4], w[5], w[6], w[7]);
    store_bf16x32(dh13 + rb + c2, d);
  }
}
__device__ __forceinline__ void epi_dgrad2_mx(const GemmParams& p, const TileInfo& ti, uint32_t tacc, int r,
                                              int rank, int part) {
  const int F = p.H;
  const int row = ti.m0 + r;
  const bool valid = row < ti.m_end;
  const int nkb = 2 * F / kMxKB;
  const size_t sblk = static_cast<size_t>(2 * ti.mt + rank) * nkb;
  const __nv_bfloat16* h13 = reinterpret_cast<const __nv_bfloat16*>(p.in_aux);
  __nv_bfloat16* dh13 = reinterpret_cast<__nv_bfloat16*>(p.out0);
  __nv_bfloat16* aout = reinterpret_cast<__nv_bfloat16*>(p.out1);
  const size_t rb = static_cast<size_t>(row) * 2 * F;
#pragma unroll 1
  for (int h = 0; h < 2; ++h) {
    const int c = 2 * part + h;  // 32-column block of the tile
    const int col = ti.n0 + 32 * c;
    if (col >= F) break;  // uniform: the last tile of a ragged F
    float g[32], u[32], v[32];
    // the saved h1, h3 first: their loads are in flight during the TMEM load
    if (valid) {
      load_bf16x32(h13 + rb + col, u);
      load_bf16x32(h13 + rb + F + col, v);
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) u[j] = v[j] = 0.0f;
    }
    tmem_ld32f(tacc + 32 * c, g);
    // in place: g <- dh1, u <- dh3, v <- a
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float s = 1.0f / (1.0f + __expf(-u[j]));
      const float si = u[j] * s;
      const float d1 = g[j] * v[j] * (s * (1.0f + u[j] * (1.0f - s)));
      const float d3 = g[j] * si;
      v[j] = si * v[j];
      g[j] = __bfloat162float(__float2bfloat16_rn(d1));
      u[j] = __bfloat162float(__float2bfloat16_rn(d3));
    }
    if (valid) store_bf16x32(aout + static_cast<size_t>(row) * F + col, v);
    // dh1 (columns col..) then dh3 (F + col..): codes from the bf16 values,
    // the scale, the bf16 values
    const int step = (col / kMxBlock) & 3;
    dgrad2_mx_out(p, g, col, sblk, r, step, rb, valid, dh13);
    dgrad2_mx_out(p, u, F + col, sblk, r, step, rb, valid, dh13);
  }
}

// DGRAD2: accumulator = da for F columns n0..n0+255; SwiGLU backward with the
// saved bf16 pre-activations h1 (columns [0,F) of h13) and h3 ([F,2F)):
//   dh1 = da * h3 * SiLU'(h1),  dh3 = da * SiLU(h1).
// `recompute` (DGRAD2R): also a = bf16(SiLU(h1) h3) into out1 [rows, F] and
// this row's partial <da, a> over the tile into dg_part[row, n0 / 256].
__device__ __forceinline__ void epi_dgrad2(const GemmParams& p, const TileInfo& ti, uint32_t tacc, int r,
                                           bool recompute, int c_begin, int c_end) {
  const int row = ti.m0 + r;
  const bool valid = row < ti.m_end;
  const __nv_bfloat16* h13 = reinterpret_cast<const __nv_bfloat16*>(p.in_aux);
  __nv_bfloat16* dh13 = reinterpret_cast<__nv_bfloat16*>(p.out0);
  __nv_bfloat16* aout = reinterpret_cast<__nv_bfloat16*>(p.out1);
  float dg = 0.0f;
#pragma unroll 1
  for (int c = c_begin; c < c_end; ++c) {
    float da[32];
    tmem_ld32f(tacc + c * 32, da);
    const int col = ti.n0 + c * 32;
    if (valid && col < p.F) {
      const size_t base = static_cast<size_t>(row) * 2 * p.F;
      float h1[32], h3[32], d1[32], d3[32], av[32];
      load_bf16x32(h13 + base + col, h1);
      load_bf16x32(h13 + base + p.F + col, h3);
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float s = 1.0f / (1.0f + __expf(-h1[j]));
        const float si = h1[j] * s;
        d1[j] = da[j] * h3[j] * (s * (1.0f + h1[j] * (1.0f - s)));
        d3[j] = da[j] * si;
        av[j] = __bfloat162float(__float2bfloat16_rn(si * h3[j]));
        dg = fmaf(da[j], av[j], dg);
      }
      store_bf16x32(dh13 + base + col, d1);
      store_bf16x32(dh13 + base + p.F + col, d3);
      if (recompute) store_bf16x32(aout + static_cast<size_t>(row) * p.F + col, av);
    }
  }
  if (recompute && valid) p.dg_part[static_cast<size_t>(row) * p.n_part + ti.n0 / 256] = dg;
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
// Order in which a CTA (pair) walks the tiles. Weight gradients: every expert
// has the same number of tiles, but a tile's k blocks are the expert's rows,
// so with skewed routing a hot expert's tiles are long (tensor-bound) and a
// cold expert's short (bound by its fp32 output). When the routing is skewed
// (`skew`: the largest expert above four times the mean rows), position
// v = k P + c of CTA c (P CTAs, k-th tile of each) takes the next tile from the
// front of the experts sorted by rows (descending) when k + c is even and from
// the back otherwise, so every CTA alternates long and short tiles and at any
// moment about half the CTAs compute while the others write. A bijection onto
// [0, ntiles): the front and back take disjoint ranges. Balanced routing keeps
// the expert-major order (one expert's operands hot in L2 at a time, measured
// faster there); other kinds: as is.
template <int KIND>
__device__ __forceinline__ int schedule_tile(int v, int P, int ntiles, const GemmParams& p, const uint8_t* s_order,
                                             int skew) {
  if constexpr (KIND == KIND_WGRAD) {
    if (!skew) return v;
    const int k = v / P, c = v - k * P;
    // front positions before v: rows 0..k-1 hold ceil(P/2) (k' even) or
    // floor(P/2) (k' odd) each; row k those c' < c with c' + k even
    const int front_rows = ((k + 1) / 2) * ((P + 1) / 2) + (k / 2) * (P / 2);
    const int front_before = front_rows + ((k & 1) == 0 ? (c + 1) / 2 : c / 2);
    const int j = ((k + c) & 1) == 0 ? front_before : ntiles - 1 - (v - front_before);
    const int tpg = p.m_tiles_fixed * p.n_tiles;
    const int e = j / tpg;
    return static_cast<int>(s_order[e]) * tpg + (j - e * tpg);
  } else {
    return v;
  }
}

template <int KIND>
__global__ void __launch_bounds__(KindTraits<KIND>::kThreadsK, 1)
    gemm_kernel(const __grid_constant__ GemmParams p, const __grid_constant__ CUtensorMap ma,
                const __grid_constant__ CUtensorMap mb0, const __grid_constant__ CUtensorMap mb1,
                const __grid_constant__ CUtensorMap mo0, const __grid_constant__ CUtensorMap mo1) {
  using TR = KindTraits<KIND>;
  using SL = SmemLayout<KIND>;
  constexpr int NSTMAX = TR::kMaxStages;
  constexpr bool PAIR = TR::kPair;
  const int NST = (KIND == KIND_ROUTER) ? router_stages(p.bn) : TR::kStages;
  const int SBYTES = (KIND == KIND_ROUTER) ? router_stage_bytes(p.bn) : TR::kStageBytesK;
  // CTA pairs: rank in the cluster (the even CTA issues the MMAs); tiles are
  // walked per cluster
  const int rank = PAIR ? static_cast<int>(cluster_ctarank()) : 0;
  const bool leader = rank == 0;
  const int tile_first = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int tile_step = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  // This kernel declares no static shared memory: the dynamic region must start
  // the CTA's shared window (1024-byte aligned) and its layout uses up to the
  // per-CTA maximum.
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {  // layout assumption broken: report, touch nothing
    if (threadIdx.x == 0) set_status(p.status, MOE_ERR_CUDA, 99);
    return;
  }
  uint8_t* smem = smem_raw;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + SL::kBarOff);
  uint64_t* empty = full + NSTMAX;
  uint64_t* tfull = empty + NSTMAX;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + SL::kTmemSlot);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + SL::kTmemSlot + 4);
  int* s_cum = reinterpret_cast<int*>(smem + SL::kCumOff);
  int* s_off = reinterpret_cast<int*>(smem + SL::kOffOff);
  uint8_t* s_order = smem + SL::kOrderOff;
  int* s_skew = reinterpret_cast<int*>(smem + SL::kSkewOff);

  const int warp = warp_id(), lane = lane_id();

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull + b, 1);
      mbar_init(tempty + b, (PAIR ? 2 : 1) * TR::kEpiWarps);  // pairs: the epilogue warps of both CTAs
    }
    mbar_init(drain, 1);
    *s_abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc2(s_tmem, kTmemCols);
      tmem_relinquish2();
    } else {
      tmem_alloc(s_tmem, kTmemCols);
      tmem_relinquish();
    }
  }
  if (warp == 0) {
    // tile schedule: s_off = row offsets of the groups, s_cum = prefix of tiles
    const int ng = p.ngroups;
    constexpr int PER = (kMaxGroups + 32) / 32;  // groups per lane (ceil(257/32))
    int cnt[PER];
    int local = 0;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int g = lane * PER + i;
      int c = 0;
      if (g <= ng) {
        int o;
        if (p.offsets != nullptr && KIND != KIND_ROUTER_DW) o = p.offsets[g];
        else o = (g == 0) ? 0 : p.M_total;
        s_off[g] = o;
      }
      if (g < ng) {
        if constexpr (KIND == KIND_WGRAD || KIND == KIND_WGRAD_MX || KIND == KIND_ROUTER_DW) {
          c = p.m_tiles_fixed * p.n_tiles;
        } else {
          int lo, hi;
          if (p.offsets != nullptr) { lo = p.offsets[g]; hi = p.offsets[g + 1]; }
          else { lo = 0; hi = p.M_total; }
          const int rows = max(hi - lo, 0);
          c = ((rows + TR::kTileM - 1) / TR::kTileM) * p.n_tiles;
        }
      }
      cnt[i] = c;
      local += c;
    }
    int incl = local;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += v;
    }
    int run = incl - local;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int g = lane * PER + i;
      if (g <= ng) s_cum[g] = run;
      run += cnt[i];
    }
    if constexpr (KIND == KIND_WGRAD) {
      // rank of each expert by its rows (descending, lower index first), and
      // whether the largest expert has more than four times the mean rows
      __syncwarp();
      int mx = 0;
      for (int g = lane; g < ng; g += 32) {
        const int rg = s_off[g + 1] - s_off[g];
        mx = max(mx, rg);
        int rank = 0;
        for (int h = 0; h < ng; ++h) {
          const int rh = s_off[h + 1] - s_off[h];
          rank += (rh > rg || (rh == rg && h < g)) ? 1 : 0;
        }
        s_order[rank] = static_cast<uint8_t>(g);
      }
#pragma unroll
      for (int d = 16; d >= 1; d >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, d));
      if (lane == 0) *s_skew = (static_cast<long long>(mx) * ng > 4ll * (s_off[ng] - s_off[0])) ? 1 : 0;
    }
  }
  tc_fence_before();
  __syncthreads();
  // pairs: the peer's barriers are initialised before any signal crosses over
  if constexpr (PAIR) cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;
  const int ntiles = s_cum[p.ngroups];
  const int skew = KIND == KIND_WGRAD ? *s_skew : 0;
  const uint64_t lim = p.wait_limit_ns;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&ma);
      tma_prefetch_desc(&mb0);
      if (KIND == KIND_FFN1 || KIND == KIND_DGRAD1) tma_prefetch_desc(&mb1);
      int stage = 0;
      uint32_t phase = 0;
      int issued_phase[NSTMAX];
#pragma unroll
      for (int s = 0; s < NSTMAX; ++s) issued_phase[s] = -1;
      bool ok = true;
      for (int tile = tile_first; tile < ntiles && ok; tile += tile_step) {
        const int t = schedule_tile<KIND>(tile, tile_step, ntiles, p, s_order, skew);
        const TileInfo ti = decode_tile<KIND>(p, s_cum, s_off, t, rank);
        for (int kb = 0; kb < ti.nkb; ++kb) {
          if (!mbar_wait_bounded(empty + stage, phase ^ 1u, s_abort, lim, p.status, 1)) { ok = false; break; }
          if constexpr (PAIR) {
            uint8_t* sA = smem + stage * SBYTES;
            // router: every pair reads the same router weight; start each pair at
            // a different k block (the sum runs over all k blocks either way)
            const int kbp = (KIND == KIND_ROUTER) ? (kb + tile_first * 5) % ti.nkb : kb;
            const CUtensorMap* amap = &ma;
            if constexpr (KIND == KIND_WGRAD) {
              if (ti.krow_end - (ti.krow0 + kb * kBK) < kBK) {
                // the expert's last, partial k block: A comes through the
                // expert's copy of its map (written before this launch by
                // tmap_rows_kernel), whose row extent ends at the expert's
                // last row, so the TMA reads zeros past it and those rows
                // contribute nothing whatever B holds there
                const uint8_t* slot = p.tmap_slots + static_cast<size_t>(ti.g) * 128;
                asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(slot) : "memory");
                amap = reinterpret_cast<const CUtensorMap*>(slot);
              }
            }
            // both CTAs' shares complete on the even CTA's barrier, which
            // expects them; a share may land before the expectation (the
            // transaction count goes below zero meanwhile)
            if (leader) mbar_arrive_expect_tx(full + stage, stage_tx_bytes<KIND>(p));
            issue_loads_pair<KIND>(p, ti, kbp, rank, sA, sA + kABytes, mapa_shared(smem_u32(full + stage), 0), amap,
                                   &mb0, &mb1, &mo1);
            issued_phase[stage] = static_cast<int>(phase);
            if (++stage == NST) { stage = 0; phase ^= 1u; }
            continue;
          }
          mbar_arrive_expect_tx(full + stage, stage_tx_bytes<KIND>(p));
          uint8_t* sA = smem + stage * SBYTES;
          // router: every CTA reads the same router weight; start each CTA at a
          // different k block so the CTAs do not all hit the same L2 lines
          // at once (the sum runs over all k blocks either way)
          const int kbl = (KIND == KIND_ROUTER) ? (kb + static_cast<int>(blockIdx.x) * 5) % ti.nkb : kb;
          issue_loads<KIND>(p, ti, kbl, sA, sA + TR::kBOff, full + stage, &ma, &mb0, &mb1);
          issued_phase[stage] = static_cast<int>(phase);
          if (++stage == NST) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok && PAIR) {
        // drain: pair shares complete on the even CTA's barriers, out of this
        // thread's sight; give copies in flight time to land
        const uint64_t t0 = globaltimer();
        while (globaltimer() - t0 < 200000ull) __nanosleep(1000);
      } else if (!ok) {
        // drain: wait (bounded, regardless of the abort flag) for copies in flight
        int zero = 0;
#pragma unroll
        for (int s = 0; s < NSTMAX; ++s)
          if (issued_phase[s] >= 0)
            mbar_wait_bounded(full + s, static_cast<uint32_t>(issued_phase[s]), reinterpret_cast<volatile int*>(&zero),
                              lim, nullptr, 0);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t idesc = TR::kNv ? idesc_nvf4_f32(TR::kTileM, kNvTileN)
                           : TR::kMx ? idesc_mxf8_f32(TR::kTileM, kMxBN)
                                     : idesc_bf16_f32(TR::kTileM, p.bn, TR::A_MN, TR::B_MN);
    // half tiles (kHalfTiles): M = 128 over the pair
    const uint32_t idesc_half = idesc_bf16_f32(TR::kTileM / 2, p.bn, TR::A_MN, TR::B_MN);
    // MXFP8: descriptors of the stage's scale blocks (32 rows of 16 bytes,
    // no swizzle, 8-row groups 128 bytes apart) for the copies into TMEM
    const uint32_t sf_lo0 = sdesc_lo(smem_u32(smem) + (TR::kNv ? kNvSfOff : kMxSfOff), 128);
    const uint64_t sf_hi = static_cast<uint64_t>((128u >> 4) | (1u << 14)) << 32;
    // operand descriptors: stage 0's low words, advanced per stage and per
    // 16-deep k step (K-major: 32 bytes; MN-major: 16 rows of 128 bytes)
    const uint32_t d_hi = sdesc_hi_sw128(1024);
    const uint32_t a_lo0 = sdesc_lo(smem_u32(smem), TR::A_MN ? 8192u : 16u);
    const uint32_t b_lo0 = sdesc_lo(smem_u32(smem) + TR::kBOff, TR::B_MN ? 8192u : 16u);
    constexpr uint32_t kAStep = TR::A_MN ? (2048u >> 4) : (32u >> 4);
    constexpr uint32_t kBStep = TR::B_MN ? (2048u >> 4) : (32u >> 4);
    const uint32_t stage_lo = static_cast<uint32_t>(SBYTES) >> 4;
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    // pairs: only the even CTA issues MMAs; its peer's MMA warp holds the
    // tensor memory allocation and waits at the end
    for (int tile = tile_first; tile < ntiles && ok && leader; tile += tile_step) {
      const int t = schedule_tile<KIND>(tile, tile_step, ntiles, p, s_order, skew);
      const TileInfo ti = decode_tile<KIND>(p, s_cum, s_off, t, rank);
      if constexpr (PAIR) {
        // the accumulator is free once the epilogue warps of both CTAs are done
        // with it (the odd CTA's arrive from across the cluster)
        const uint64_t t0 = globaltimer();
        bool got = mbar_try_wait_cluster(tempty + acc, acc_phase ^ 1u);
        while (!got && !*s_abort) {
          got = mbar_try_wait_cluster(tempty + acc, acc_phase ^ 1u);
          if (!got && globaltimer() - t0 > lim) {
            *s_abort = 1;
            set_status(p.status, MOE_ERR_DEVICE_TIMEOUT, 2);
          }
        }
        if (!got) { ok = false; break; }
      } else if (!mbar_wait_bounded(tempty + acc, acc_phase ^ 1u, s_abort, lim, p.status, 2)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kAccStride);
      if constexpr (TR::kNv) {
        // NVFP4: four K=64 steps per 256-element k block, each with its own
        // scale cells (A: 4 columns, B: 8); the twelve copies of block kb+1
        // go to the other scale region before the MMAs of block kb
        auto copy_scales = [&](int st_, uint32_t region) {
          const uint32_t sf_lo = sf_lo0 + static_cast<uint32_t>(st_) * stage_lo;
#pragma unroll
          for (int s4 = 0; s4 < 4; ++s4) {
            tmem_cp2_32x128b_x4(tmem_base + region + 4 * s4, sf_hi | (sf_lo + (512u * s4 >> 4)));
            tmem_cp2_32x128b_x4(tmem_base + region + 16 + 8 * s4, sf_hi | (sf_lo + ((kNvSfBytes + 512u * s4) >> 4)));
            tmem_cp2_32x128b_x4(tmem_base + region + 20 + 8 * s4,
                                sf_hi | (sf_lo + ((2 * kNvSfBytes + 512u * s4) >> 4)));
          }
        };
        if (ti.nkb > 0) {
          if (!mbar_wait_bounded(full + stage, phase, s_abort, lim, p.status, 3)) { ok = false; break; }
          tc_fence_after();
          if (lane == 0) copy_scales(stage, kNvSfRegion0);
          __syncwarp();
        }
        for (int kb = 0; kb < ti.nkb; ++kb) {
          const int cur = stage;
          const uint32_t region = (kb & 1) ? kNvSfRegion1 : kNvSfRegion0;
          if (++stage == NST) { stage = 0; phase ^= 1u; }
          if (kb + 1 < ti.nkb) {
            if (!mbar_wait_bounded(full + stage, phase, s_abort, lim, p.status, 3)) { ok = false; break; }
            tc_fence_after();
            if (lane == 0) copy_scales(stage, (kb & 1) ? kNvSfRegion0 : kNvSfRegion1);
          }
          if (lane == 0) {
            const uint32_t a_lo = a_lo0 + static_cast<uint32_t>(cur) * stage_lo;
            const uint32_t b_lo = b_lo0 + static_cast<uint32_t>(cur) * stage_lo;
#pragma unroll
            for (int s4 = 0; s4 < 4; ++s4)
              umma2_nv_w(d_tmem, a_lo + s4 * kAStep, b_lo + s4 * kBStep, d_hi, idesc, tmem_base + region + 4 * s4,
                         tmem_base + region + 16 + 8 * s4, (kb > 0 || s4 > 0) ? 1u : 0u);
            umma2_commit_mc(empty + cur, 3);  // frees the stage in both CTAs
          }
          __syncwarp();
        }
      }
      if constexpr (TR::kMx) {
        // MXFP8: the scale copy of k block kb+1 (into the other of two scale
        // regions) is issued before the MMAs of block kb, so no MMA waits for
        // the copy its scales come from (a copy takes about as long as a
        // quarter of a block's MMAs); region r holds the scales of the blocks
        // kb with kb % 2 == r
        auto copy_scales = [&](int st_, uint32_t region) {
          const uint32_t sf_lo = sf_lo0 + static_cast<uint32_t>(st_) * stage_lo;
          const uint32_t col = region * kMxSfRegion;
          tmem_cp2_32x128b_x4(tmem_base + kMxSfaCol + col, sf_hi | sf_lo);
          tmem_cp2_32x128b_x4(tmem_base + kMxSfbCol + col, sf_hi | (sf_lo + (kMxSfBytes >> 4)));
          tmem_cp2_32x128b_x4(tmem_base + kMxSfbCol + 4 + col, sf_hi | (sf_lo + (2 * kMxSfBytes >> 4)));
        };
        if (ti.nkb > 0) {
          if (!mbar_wait_bounded(full + stage, phase, s_abort, lim, p.status, 3)) { ok = false; break; }
          tc_fence_after();
          if (lane == 0) copy_scales(stage, 0u);
          __syncwarp();
        }
        for (int kb = 0; kb < ti.nkb; ++kb) {
          const int cur = stage;
          const uint32_t region = static_cast<uint32_t>(kb & 1);
          if (++stage == NST) { stage = 0; phase ^= 1u; }
          if (kb + 1 < ti.nkb) {
            if (!mbar_wait_bounded(full + stage, phase, s_abort, lim, p.status, 3)) { ok = false; break; }
            tc_fence_after();
            if (lane == 0) copy_scales(stage, region ^ 1u);
          }
          if (lane == 0) {
            const uint32_t a_lo = a_lo0 + static_cast<uint32_t>(cur) * stage_lo;
            const uint32_t b_lo = b_lo0 + static_cast<uint32_t>(cur) * stage_lo;
            const uint32_t col = region * kMxSfRegion;
#pragma unroll
            for (int kk = 0; kk < kMxKB / 32; ++kk)
              umma2_mx_w(d_tmem, a_lo + kk * kAStep, b_lo + kk * kBStep, d_hi,
                         idesc | (static_cast<uint32_t>(kk) << 29) | (static_cast<uint32_t>(kk) << 4),
                         tmem_base + kMxSfaCol + col, tmem_base + kMxSfbCol + col, (kb > 0 || kk > 0) ? 1u : 0u);
            umma2_commit_mc(empty + cur, 3);  // frees the stage in both CTAs
          }
          __syncwarp();
        }
      }
      for (int kb = 0; kb < ((TR::kMx || TR::kNv) ? 0 : ti.nkb); ++kb) {
        if (!mbar_wait_bounded(full + stage, phase, s_abort, lim, p.status, 3)) { ok = false; break; }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t a_lo = a_lo0 + static_cast<uint32_t>(stage) * stage_lo;
          const uint32_t b_lo = b_lo0 + static_cast<uint32_t>(stage) * stage_lo;
          const uint32_t id = (kHalfTiles<KIND> && ti.half) ? idesc_half : idesc;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            if constexpr (PAIR)
              umma2_bf16_w(d_tmem, a_lo + kk * kAStep, b_lo + kk * kBStep, d_hi, id, (kb > 0 || kk > 0) ? 1u : 0u);
            else
              umma_bf16_w(d_tmem, a_lo + kk * kAStep, b_lo + kk * kBStep, d_hi, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
          }
          if constexpr (KIND == KIND_ROUTER_DW) {
            // the lo part of dL against the same box of x
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
              umma_bf16_w(d_tmem, a_lo + (kABytes >> 4) + kk * kAStep, b_lo + kk * kBStep, d_hi, idesc, 1u);
          }
          if constexpr (PAIR) umma2_commit_mc(empty + stage, 3);  // frees the stage in both CTAs
          else umma_commit(empty + stage);
        }
        __syncwarp();
        if (++stage == NST) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      if (lane == 0) {
        if constexpr (PAIR) umma2_commit_mc(tfull + acc, 3);  // with no MMA (nkb = 0) it arrives at once
        else if (ti.nkb > 0) umma_commit(tfull + acc);
        else mbar_arrive(tfull + acc);
      }
      __syncwarp();
      if constexpr (KIND == KIND_ROUTER) {
        acc_phase ^= 1u;  // one accumulator: the columns past it hold the epilogue's selection values
      } else {
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
    }
    // drain every MMA issued by this CTA before the TMEM is released
    if (leader) {
      if (lane == 0) {
        if constexpr (PAIR) umma2_commit_mc(drain, 1);
        else umma_commit(drain);
      }
      __syncwarp();
      int zero = 0;
      mbar_wait_bounded(drain, 0, reinterpret_cast<volatile int*>(&zero), lim, nullptr, 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quadrant of this warp
    const int part = (warp - 2) >> 2;  // DGRAD2, ROUTER: which half of the tile's columns
    const int r = q * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    Stager st{smem + SL::kOutOff + (warp - 2) * TR::kOutWarpBytes, 0u};
    // pairs: the odd CTA's epilogue frees the even CTA's accumulator slot
    const uint32_t tempty_even = PAIR ? mapa_shared(smem_u32(tempty), 0) : 0u;
    if constexpr (KIND == KIND_ROUTER) {
      // the logit and expert biases, zero-padded to 256 experts, for every tile
      RouterSmem rsm(smem + SL::kOutOff);
      for (int i = static_cast<int>(threadIdx.x) - 64; i < 256; i += 32 * TR::kEpiWarps) {
        rsm.lb[i] = (p.r_lbias != nullptr && i < p.E) ? p.r_lbias[i] : 0.0f;
        rsm.eb[i] = (p.r_ebias != nullptr && i < p.E) ? p.r_ebias[i] : 0.0f;
      }
      named_bar_sync(1, 32 * TR::kEpiWarps);
    }
    for (int tile = tile_first; tile < ntiles; tile += tile_step) {
      const int t = schedule_tile<KIND>(tile, tile_step, ntiles, p, s_order, skew);
      const TileInfo ti = decode_tile<KIND>(p, s_cum, s_off, t, rank);
      // this warp's 32 rows: a full block leaves through TMA boxes; a block
      // that crosses the end of the expert's rows uses masked per-thread stores
      // a half tile: this warp's 32 of the CTA's 64 rows, and the columns of
      // the B half its TMEM lanes hold (lanes 64.. : the odd CTA's half)
      const bool half = kHalfTiles<KIND> && ti.half;
      const int row0 = ti.m0 + 32 * (half ? (q & 1) : q);
      const bool full_rows = row0 + 32 <= ti.m_end;
      const bool any_rows = row0 < ti.m_end;
      if (!mbar_wait_bounded(tfull + acc, acc_phase, s_abort, lim, p.status, 4)) break;
      tc_fence_after();
      const uint32_t tacc = tmem_base + static_cast<uint32_t>(acc * kAccStride) + (static_cast<uint32_t>(q * 32) << 16);
      if constexpr (KIND == KIND_FFN1) {
        if (half) {
          // 64 F columns n0 + 64 (q / 2) ..: h1 at TMEM columns 0..63, h3 at 64..127
          const int n0h = ti.n0 + 64 * (q >> 1);
          if (full_rows) epi_ffn1_tma(p, n0h, tacc, lane, row0, st, &mo0, &mo1, 1, 64);
          else if (any_rows) epi_ffn1(p, n0h, row0 + lane, ti.m_end, tacc, 2, 64);
        } else {
          if (full_rows) epi_ffn1_tma(p, ti.n0, tacc, lane, row0, st, &mo0, &mo1);
          else if (any_rows) epi_ffn1(p, ti.n0, ti.m0 + r, ti.m_end, tacc);
        }
      } else if constexpr (KIND == KIND_FFN2) {
        if (half) {
          epi_store_half(p, ti, tacc, lane, q, r, row0, full_rows, any_rows, st, &mo0);
        } else if (full_rows) {
          if (p.out_fp32) epi_store_tma<true, false>(ti, tacc, lane, row0, p.H, st, &mo0);
          else epi_store_tma<false, false>(ti, tacc, lane, row0, p.H, st, &mo0);
        } else if (any_rows) {
          epi_store(ti, tacc, r, 8, p.H, p.H, p.out0, p.out_fp32 != 0, 0);
        }
      } else if constexpr (KIND == KIND_FFN1_MX) {
        epi_ffn1_mx(p, ti, tacc, r, rank, part);
      } else if constexpr (KIND == KIND_FFN2_MX) {
        if (full_rows) {
          if (p.out_fp32) epi_store_tma<true, false>(ti, tacc, lane, row0, p.H, st, &mo0, kMxBN / 64);
          else epi_store_tma<false, false>(ti, tacc, lane, row0, p.H, st, &mo0, kMxBN / 64);
        } else if (any_rows) {
          epi_store(ti, tacc, r, kMxBN / 32, p.H, p.H, p.out0, p.out_fp32 != 0, 0);
        }
      } else if constexpr (KIND == KIND_WGRAD_MX) {
        // 3-D output maps clip rows past M per expert; six 32-column boxes
        epi_wgrad_tma(p, ti, tacc, lane, row0, st, &mo0, &mo1, 0, kMxBN / 32);
      } else if constexpr (KIND == KIND_DGRAD2_MX) {
        epi_dgrad2_mx(p, ti, tacc, r, rank, part);
      } else if constexpr (KIND == KIND_FFN1_NV) {
        epi_ffn1_nv(p, ti, tacc, r, part);
      } else if constexpr (KIND == KIND_GEMM_NV) {
        // y = g_x g_e (sum of the block-scaled products)
        // (fp32 out: the data gradient da of the NVFP4 training step)
        const float alpha = __ldg(p.nv_ga) * __ldg(p.nv_gb + ti.g);
        if (full_rows) {
          if (p.out_fp32) epi_store_tma<true, false>(ti, tacc, lane, row0, p.H, st, &mo0, kNvTileN / 64, alpha);
          else epi_store_tma<false, false>(ti, tacc, lane, row0, p.H, st, &mo0, kNvTileN / 64, alpha);
        } else if (any_rows) {
          epi_store(ti, tacc, r, kNvTileN / 32, p.H, p.H, p.out0, p.out_fp32 != 0, 0, alpha);
        }
      } else if constexpr (KIND == KIND_ROUTER) {
        // score, selection, gates (and aux statistics, logits) per token
        const RouterSmem rsm(smem + SL::kOutOff);
        const int tid = q * 32 + lane;
        const uint32_t tz = tmem_base + kRouterZCol + (static_cast<uint32_t>(q * 32) << 16);
        const int row = ti.m0 + tid, slice = ti.m0 / 32 + q;
        if (p.r_mode == RSEL_LOGIT) router_select_mode<RSEL_LOGIT>(p, tacc, tz, row, tid, lane, q, part, slice, rsm);
        else if (p.r_mode == RSEL_SOFTMAX)
          router_select_mode<RSEL_SOFTMAX>(p, tacc, tz, row, tid, lane, q, part, slice, rsm);
        else router_select_mode<RSEL_SIGMOID>(p, tacc, tz, row, tid, lane, q, part, slice, rsm);
      } else if constexpr (KIND == KIND_DGRAD2R) {
        if (full_rows) epi_dgrad2r_tma(p, ti, tacc, lane, row0, st, &mo0, &mo1);
        else if (any_rows) epi_dgrad2(p, ti, tacc, r, true, 0, 8);
      } else if constexpr (KIND == KIND_DGRAD2) {
        if (full_rows) epi_dgrad2_tma(p, ti, tacc, lane, row0, st, &mo0, 2 * part, 2 * part + 2);
        else if (any_rows) epi_dgrad2(p, ti, tacc, r, false, 4 * part, 4 * part + 4);
      } else if constexpr (KIND == KIND_DGRAD1) {
        if (half) {
          epi_store_half(p, ti, tacc, lane, q, r, row0, full_rows, any_rows, st, &mo0);
        } else if (full_rows) {
          if (p.out_fp32) epi_store_tma<true, false>(ti, tacc, lane, row0, p.H, st, &mo0);
          else epi_store_tma<false, false>(ti, tacc, lane, row0, p.H, st, &mo0);
        } else if (any_rows) {
          epi_store(ti, tacc, r, 8, p.H, p.H, p.out0, p.out_fp32 != 0, 0);
        }
      } else if constexpr (KIND == KIND_WGRAD) {
        // 3-D output maps clip rows past M per expert
        epi_wgrad_direct(p, ti, tacc, q, lane);
      } else if constexpr (KIND == KIND_ROUTER_DX) {
        // the map's row extent is T: rows past it are clipped
        epi_store_tma<true, false>(ti, tacc, lane, row0, p.H, st, &mo0);
      } else {  // ROUTER_DW partial of split g: 3-D map {H, E, splits} clips rows >= E
        epi_store_tma<true, true>(ti, tacc, lane, row0, p.H, st, &mo0);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (KIND == KIND_WGRAD) {
          // the tile's TMEM loads are complete (tcgen05.wait::ld in every
          // lane before the warp sync): release the accumulator without
          // waiting for this warp's fp32 stores to drain
          if (PAIR && !leader) mbar_arrive_cluster_relaxed(tempty_even + 8u * acc);
          else mbar_arrive_relaxed(tempty + acc);
        } else {
          if (PAIR && !leader) mbar_arrive_cluster(tempty_even + 8u * acc);
          else mbar_arrive(tempty + acc);
        }
      }
      if constexpr (KIND == KIND_ROUTER) {
        acc_phase ^= 1u;
      } else {
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
    }
    st.drain(lane);  // this warp's stores are complete
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) {
    // neither CTA leaves (or frees the pair's tensor memory) while its peer may
    // still read its shared memory or signal its barriers
    if (*s_abort) {
      const uint64_t t0 = globaltimer();
      while (globaltimer() - t0 < 200000ull) __nanosleep(1000);
    }
    cluster_sync_all();
  }
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR) tmem_dealloc2(tmem_base, kTmemCols);
    else tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// host launch
// ---------------------------------------------------------------------------
template <int KIND>
static cudaError_t launch_kind(const GemmParams& p, const CUtensorMap& ma, const CUtensorMap& mb0,
                               const CUtensorMap& mb1, const CUtensorMap& mo0, const CUtensorMap& mo1, int grid,
                               cudaStream_t st) {
  auto kern = gemm_kernel<KIND>;
  const int smem = SmemLayout<KIND>::kDynBytes;
  static int configured_dev = -1;
  static int max_pairs = 0;  // clusters of two CTAs resident at once (pair kinds)
  int dev = 0;
  cudaGetDevice(&dev);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.blockDim = dim3(KindTraits<KIND>::kThreadsK);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  if (KindTraits<KIND>::kPair) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  if (configured_dev != dev) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (KindTraits<KIND>::kPair) {
      cfg.gridDim = dim3(2 * (num_sms() / 2));
      e = cudaOccupancyMaxActiveClusters(&max_pairs, kern, &cfg);
      if (e != cudaSuccess) return e;
      if (max_pairs < 1) return cudaErrorInvalidConfiguration;
    }
    configured_dev = dev;
  }
  if (KindTraits<KIND>::kPair) {
    // a persistent grid of resident pairs (tiles are walked per cluster)
    const int pairs = (grid + 1) / 2;
    grid = 2 * (pairs < max_pairs ? pairs : max_pairs);
  }
  cfg.gridDim = dim3(grid);
  return cudaLaunchKernelEx(&cfg, kern, p, ma, mb0, mb1, mo0, mo1);
}

// Per-expert copies of the weight gradients' A tensor map: maps[e] (128 bytes)
// = tmpl with its row extent set to expert e's end row offsets[e + 1] (one
// group of `rows` rows when offsets == nullptr), released to the TMA unit (the
// GEMM launched next acquires each copy before its first use).
__global__ void tmap_rows_kernel(const __grid_constant__ CUtensorMap tmpl, const int32_t* __restrict__ offsets, int E,
                                 int rows, uint8_t* __restrict__ maps) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= E) return;
  tmap_set_rows(&tmpl, maps + static_cast<size_t>(e) * 128, offsets != nullptr ? offsets[e + 1] : rows);
}

cudaError_t launch_tmap_rows(const CUtensorMap& tmpl, const int32_t* offsets, int E, uint8_t* maps, cudaStream_t st,
                             int rows) {
  NvtxRange nvtx("moe.weight_gradient_maps");
  tmap_rows_kernel<<<(E + 127) / 128, 128, 0, st>>>(tmpl, offsets, E, rows, maps);
  return cudaGetLastError();
}

static const char* gemm_range_name(int kind) {
  switch (kind) {
    case KIND_FFN1: return "moe.gemm.gate_up_swiglu";
    case KIND_FFN2: return "moe.gemm.down";
    case KIND_ROUTER: return "moe.router";
    case KIND_DGRAD2: return "moe.gemm.dgrad_down_swiglu_bwd";
    case KIND_DGRAD2R: return "moe.gemm.dgrad_down_swiglu_bwd_recompute";
    case KIND_DGRAD1: return "moe.gemm.dgrad_gate_up";
    case KIND_WGRAD: return "moe.gemm.weight_gradient";
    case KIND_ROUTER_DX: return "moe.router_dgrad";
    case KIND_ROUTER_DW: return "moe.router_wgrad";
    case KIND_FFN1_MX: return "moe.gemm.mxfp8_gate_up_swiglu";
    case KIND_FFN2_MX: return "moe.gemm.mxfp8_down";
    case KIND_DGRAD2_MX: return "moe.gemm.mxfp8_dgrad_down_swiglu_bwd";
    case KIND_WGRAD_MX: return "moe.gemm.mxfp8_weight_gradient";
    case KIND_GEMM_NV: return "moe.gemm.nvfp4";
    case KIND_FFN1_NV: return "moe.gemm.nvfp4_gate_up_swiglu";
    default: return "moe.gemm";
  }
}

cudaError_t launch_gemm(int kind, const GemmParams& p, const CUtensorMap& ma, const CUtensorMap& mb0,
                        const CUtensorMap& mb1, int grid, cudaStream_t st, const CUtensorMap* out0,
                        const CUtensorMap* out1) {
  NvtxRange nvtx(gemm_range_name(kind));
  static const CUtensorMap kNone = {};
  const CUtensorMap& mo0 = out0 ? *out0 : kNone;
  const CUtensorMap& mo1 = out1 ? *out1 : kNone;
  switch (kind) {
    case KIND_FFN1: return launch_kind<KIND_FFN1>(p, ma, mb0, mb1, mo0, mo1, grid, st);
    case KIND_FFN2: return launch_kind<KIND_FFN2>(p, ma, mb0, mb1, mo0, mo1, grid, st);
    case KIND_ROUTER: return launch_kind<KIND_ROUTER>(p, ma, mb0, mb1, mo0, mo1, grid, st);
    case KIND_DGRAD2: return launch_kind<KIND_DGRAD2>(p, ma, mb0, mb1, mo0, mo1, grid, st);
    case KIND_DGRAD2R: return launch_kind<KIND_DGRAD2R>(p, ma, mb0, mb1, mo0, mo1, grid, st);
    case KIND_DGRAD1: return launch_kind<KIND_DGRAD1>(p, ma, mb0, mb1, mo0, mo1, grid, st);
    case KIND_WGRAD: return launch_kind<KIND_WGRAD>(p, ma, mb0, mb1, mo0, mo1, grid, st);
    case KIND_ROUTER_DX: return launch_kind<KIND_ROUTER_DX>(p, ma, mb0, mb1, mo0, mo1, grid, st);
    case KIND_ROUTER_DW: return launch_kind<KIND_ROUTER_DW>(p, ma, mb0, mb1, mo0, mo1, grid, st);
    case KIND_FFN1_MX: return launch_kind<KIND_FFN1_MX>(p, ma, mb0, mb1, mo0, mo1, grid, st);
    case KIND_FFN2_MX: return launch_kind<KIND_FFN2_MX>(p, ma, mb0, mb1, mo0, mo1, grid, st);
    case KIND_DGRAD2_MX: return launch_kind<KIND_DGRAD2_MX>(p, ma, mb0, mb1, mo0, mo1, grid, st);
    case KIND_WGRAD_MX: return launch_kind<KIND_WGRAD_MX>(p, ma, mb0, mb1, mo0, mo1, grid, st);
    case KIND_GEMM_NV: return launch_kind<KIND_GEMM_NV>(p, ma, mb0, mb1, mo0, mo1, grid, st);
    case KIND_FFN1_NV: return launch_kind<KIND_FFN1_NV>(p, ma, mb0, mb1, mo0, mo1, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace moe

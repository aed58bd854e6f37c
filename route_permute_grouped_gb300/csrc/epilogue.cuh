// GEMM epilogues that leave through the TMA: each epilogue warp owns the 32
// accumulator rows of its TMEM lane quarter and two 4 KB shared-memory staging
// buffers. A 32-row x 128-byte box (32 fp32 or 64 bf16 columns) is written to a
// buffer in the 128-byte swizzled layout (16-byte chunk j of row r lands at
// chunk j ^ (r & 7), so the 32 lanes' writes spread over all banks), then one
// lane stores the box with a bulk tensor copy. Two buffers let the copy of one
// box overlap the staging of the next. Blocks that cross the end of an expert's
// rows use the per-thread masked stores instead (a box would overwrite the next
// expert's rows).
#pragma once
#include "gemm_tc.cuh"

namespace moe {

__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int c0, int c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(src)), "r"(c0), "r"(c1)
               : "memory");
}
// wait until at most one committed bulk store of this thread still reads
// shared memory
__device__ __forceinline__ void bulk_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }

struct Stager {
  uint8_t* base;  // 8 KB, 1024-byte aligned: two boxes
  uint32_t n;     // boxes committed so far by this warp

  // a free buffer: the one whose previous box (two boxes ago) has been read
  __device__ __forceinline__ uint8_t* next(int lane) {
    if (n >= 2 && lane == 0) bulk_wait_read1();
    __syncwarp();
    return base + ((n & 1u) << 12);
  }
  // both buffers free (every committed box has been read)
  __device__ __forceinline__ void both(int lane, uint8_t*& b0, uint8_t*& b1) {
    if (lane == 0) bulk_wait_read0();
    __syncwarp();
    b0 = base;
    b1 = base + 4096;
  }
  __device__ __forceinline__ void commit2d(int lane, const CUtensorMap* m, const uint8_t* buf, int c0, int c1) {
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(m, buf, c0, c1);
      bulk_commit();
    }
    ++n;
  }
  __device__ __forceinline__ void commit3d(int lane, const CUtensorMap* m, const uint8_t* buf, int c0, int c1,
                                           int c2) {
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_3d(m, buf, c0, c1, c2);
      bulk_commit();
    }
    ++n;
  }
  __device__ __forceinline__ void drain(int lane) {
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }
};

// row `lane` of a box: 32 fp32 (the whole 128-byte row)
__device__ __forceinline__ void stage_f32x32(uint8_t* buf, int lane, const float* f) {
  uint8_t* row = buf + lane * 128;
#pragma unroll
  for (int j = 0; j < 8; ++j)
    *reinterpret_cast<float4*>(row + ((j ^ (lane & 7)) << 4)) =
        make_float4(f[4 * j], f[4 * j + 1], f[4 * j + 2], f[4 * j + 3]);
}
// row `lane` of a box: 32 bf16 into half `half` (bytes 64*half..) of the row
__device__ __forceinline__ void stage_bf16x32(uint8_t* buf, int lane, int half, const float* f) {
  uint8_t* row = buf + lane * 128;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint4 w;
    w.x = pack_bf16x2(f[8 * j + 0], f[8 * j + 1]);
    w.y = pack_bf16x2(f[8 * j + 2], f[8 * j + 3]);
    w.z = pack_bf16x2(f[8 * j + 4], f[8 * j + 5]);
    w.w = pack_bf16x2(f[8 * j + 6], f[8 * j + 7]);
    *reinterpret_cast<uint4*>(row + (((4 * half + j) ^ (lane & 7)) << 4)) = w;
  }
}

__device__ __forceinline__ void tmem_ld32_f(uint32_t taddr, float* f) {
  uint32_t v[32];
  tmem_ld32(taddr, v);
  tmem_ld_wait();
#pragma unroll
  for (int j = 0; j < 32; ++j) f[j] = __uint_as_float(v[j]);
}

__device__ __forceinline__ float silu_fast(float z) { return z / (1.0f + __expf(-z)); }

// FFN1, rows row0..row0+31 all inside the expert: a = SiLU(h1) h3 (and h1, h3
// when saving) for the 64 * nch F-columns n0.. (h1 at TMEM columns 0.., h3 at
// `up` ..), in 64-column boxes.
__device__ __forceinline__ void epi_ffn1_tma(const GemmParams& p, int n0, uint32_t tacc, int lane, int row0,
                                             Stager& st, const CUtensorMap* map_a, const CUtensorMap* map_h13,
                                             int nch = 2, int up = 128) {
  const bool save = p.out1 != nullptr;
#pragma unroll 1
  for (int cc = 0; cc < nch; ++cc) {
    const int col = n0 + cc * 64;
    if (col >= p.F) break;  // uniform over the warp
    uint8_t* buf = st.next(lane);
#pragma unroll 1
    for (int h = 0; h < 2; ++h) {
      float g[32], u[32];
      tmem_ld32_f(tacc + (cc * 2 + h) * 32, g);
      tmem_ld32_f(tacc + up + (cc * 2 + h) * 32, u);
#pragma unroll
      for (int j = 0; j < 32; ++j) g[j] = silu_fast(g[j]) * u[j];
      stage_bf16x32(buf, lane, h, g);
    }
    st.commit2d(lane, map_a, buf, col, row0);
    if (save) {
#pragma unroll 1
      for (int part = 0; part < 2; ++part) {  // h1 then h3
        uint8_t* b = st.next(lane);
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
          float v[32];
          tmem_ld32_f(tacc + part * up + (cc * 2 + h) * 32, v);
          stage_bf16x32(b, lane, h, v);
        }
        st.commit2d(lane, map_h13, b, part * p.F + col, row0);
      }
    }
  }
}

// Plain store of the 32 x 256 block of this warp: bf16 in 64-column boxes or
// fp32 in 32-column boxes. 3-D maps (weight gradients, router partials) take
// the group as the third coordinate and clip rows per group.
template <bool F32, bool THREE_D>
__device__ __forceinline__ void epi_store_tma(const TileInfo& ti, uint32_t tacc, int lane, int row0, int ncols,
                                              Stager& st, const CUtensorMap* map, int nch64 = 4, float alpha = 1.0f) {
  const bool zero = ti.nkb == 0;
  if constexpr (F32) {
#pragma unroll 1
    for (int c = 0; c < 2 * nch64; ++c) {
      const int col = ti.n0 + c * 32;
      if (col >= ncols) break;
      float f[32];
      if (!zero) {
        tmem_ld32_f(tacc + c * 32, f);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) f[j] = 0.0f;
      }
      if (alpha != 1.0f) {
#pragma unroll
        for (int j = 0; j < 32; ++j) f[j] *= alpha;
      }
      uint8_t* buf = st.next(lane);
      stage_f32x32(buf, lane, f);
      if (THREE_D) st.commit3d(lane, map, buf, col, row0, ti.g);
      else st.commit2d(lane, map, buf, col, row0);
    }
  } else {
#pragma unroll 1
    for (int cc = 0; cc < nch64; ++cc) {
      const int col = ti.n0 + cc * 64;
      if (col >= ncols) break;
      uint8_t* buf = st.next(lane);
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        float f[32];
        if (!zero) {
          tmem_ld32_f(tacc + (cc * 2 + h) * 32, f);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) f[j] = 0.0f;
        }
        if (alpha != 1.0f) {
#pragma unroll
          for (int j = 0; j < 32; ++j) f[j] *= alpha;
        }
        stage_bf16x32(buf, lane, h, f);
      }
      if (THREE_D) st.commit3d(lane, map, buf, col, row0, ti.g);
      else st.commit2d(lane, map, buf, col, row0);
    }
  }
}

// Weight gradient: 32 fp32 columns per box (boxes c_begin .. c_end - 1 of the
// tile), into dW1 (n < F) or dW3 (n >= F) in mode 1, into dW2 in mode 0; 3-D
// maps {N, M, experts}.
__device__ __forceinline__ void epi_wgrad_tma(const GemmParams& p, const TileInfo& ti, uint32_t tacc, int lane,
                                              int row0, Stager& st, const CUtensorMap* mo0,
                                              const CUtensorMap* mo1, int c_begin = 0, int c_end = 8) {
  const bool zero = ti.nkb == 0;
#pragma unroll 1
  for (int c = c_begin; c < c_end; ++c) {
    const int n = ti.n0 + c * 32;
    if (n >= p.wg_N) break;
    float f[32];
    if (!zero) {
      tmem_ld32_f(tacc + c * 32, f);
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) f[j] = 0.0f;
    }
    uint8_t* buf = st.next(lane);
    stage_f32x32(buf, lane, f);
    const CUtensorMap* m = mo0;
    int col = n;
    if (p.wg_mode == 1 && n >= p.wg_N / 2) {
      m = mo1;
      col = n - p.wg_N / 2;
    }
    st.commit3d(lane, m, buf, col, row0, ti.g);
  }
}

// WGRAD (bf16 operands), fp32 output stored straight from tensor memory: the
// warp of lane quadrant q reads its 32 rows in two 16-lane halves and 64-column
// blocks with the 16x256b shape, so each store instruction of the warp writes
// 32 contiguous bytes (one full sector) in each of 8 rows; no shared-memory
// staging. Rows past wg_M are skipped (the tile's rows of the next m tile do
// not exist); a tile with no k blocks (an expert with no rows) stores zeros.
// Mode 0: out0 = dW [E][wg_M][wg_N]; mode 1: columns [0, wg_N/2) go to out0 and
// [wg_N/2, wg_N) to out1, each [E][wg_M][wg_N/2].
__device__ __forceinline__ void st_f32x2(float* dst, uint32_t a, uint32_t b) {
  asm volatile("st.global.v2.b32 [%0], {%1, %2};" ::"l"(dst), "r"(a), "r"(b) : "memory");
}
__device__ __forceinline__ void epi_wgrad_direct(const GemmParams& p, const TileInfo& ti, uint32_t tacc_q, int q,
                                                 int lane) {
  const bool zero = ti.nkb == 0;
  const int half_n = p.wg_N / 2;
  const int ld = p.wg_mode == 1 ? half_n : p.wg_N;
#pragma unroll 1
  for (int h = 0; h < 2; ++h) {
    const int ra = ti.m0 + 32 * q + 16 * h + (lane >> 2);  // rows ra and ra + 8
#pragma unroll 1
    for (int cb = 0; cb < 4; ++cb) {
      const int n = ti.n0 + 64 * cb;
      if (n >= p.wg_N) break;  // uniform
      uint32_t r[32];
      if (!zero) {
        tmem_ld16x256b_x8(tacc_q + (static_cast<uint32_t>(16 * h) << 16) + 64 * cb, r);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) r[j] = 0u;
      }
      float* out = reinterpret_cast<float*>(p.out0);
      int col = n;
      if (p.wg_mode == 1 && n >= half_n) {
        out = reinterpret_cast<float*>(p.out1);
        col = n - half_n;
      }
      const size_t base_a = (static_cast<size_t>(ti.g) * p.wg_M + ra) * ld + col + 2 * (lane & 3);
      const size_t base_b = base_a + static_cast<size_t>(8) * ld;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (ra < p.wg_M) st_f32x2(out + base_a + 8 * j, r[4 * j], r[4 * j + 1]);
        if (ra + 8 < p.wg_M) st_f32x2(out + base_b + 8 * j, r[4 * j + 2], r[4 * j + 3]);
      }
    }
  }
}

// DGRAD2, rows all inside the expert: dh1 = da h3 SiLU'(h1), dh3 = da SiLU(h1).
// Per 64-column chunk each thread reads its row's 64 values of the saved h1
// and h3 with vector loads (not through the TMA unit, whose queue holds the
// operand loads of the main loop), reads da from TMEM, and the warp's one
// staging box carries dh1 to a TMA store, then dh3 (held in registers
// meanwhile).
__device__ __forceinline__ uint4 ldg_nc_v4(const void* ptr) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(ptr));
  return v;
}
// chunks cc_begin .. cc_end - 1 of the tile's four 64-column chunks
__device__ __forceinline__ void epi_dgrad2_tma(const GemmParams& p, const TileInfo& ti, uint32_t tacc, int lane,
                                               int row0, Stager& st, const CUtensorMap* map_out, int cc_begin,
                                               int cc_end) {
  const __nv_bfloat16* hrow =
      reinterpret_cast<const __nv_bfloat16*>(p.in_aux) + static_cast<size_t>(row0 + lane) * (2 * p.F);
#pragma unroll 1
  for (int cc = cc_begin; cc < cc_end; ++cc) {
    const int col = ti.n0 + cc * 64;
    if (col >= p.F) break;
    uint4 v1[8], v3[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      v1[j] = ldg_nc_v4(hrow + col + 8 * j);
      v3[j] = ldg_nc_v4(hrow + p.F + col + 8 * j);
    }
    float da0[32], da1[32];
    tmem_ld32_f(tacc + (cc * 2) * 32, da0);
    tmem_ld32_f(tacc + (cc * 2 + 1) * 32, da1);
    // one 4 KB staging box per warp: dh1 leaves first, dh3 waits in registers
    uint8_t* b1 = st.base;
    if (lane == 0) bulk_wait_read0();
    __syncwarp();
    uint32_t keep[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float* da = j < 4 ? da0 : da1;
      const uint32_t a1[4] = {v1[j].x, v1[j].y, v1[j].z, v1[j].w};
      const uint32_t a3[4] = {v3[j].x, v3[j].y, v3[j].z, v3[j].w};
      uint32_t o1[4], o3[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float d1v[2], d3v[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float x1 = e ? bf16_hi(a1[q]) : bf16_lo(a1[q]);
          const float x3 = e ? bf16_hi(a3[q]) : bf16_lo(a3[q]);
          const float d = da[8 * (j & 3) + 2 * q + e];
          const float s = 1.0f / (1.0f + __expf(-x1));
          d1v[e] = d * x3 * (s * (1.0f + x1 * (1.0f - s)));
          d3v[e] = d * x1 * s;
        }
        o1[q] = pack_bf16x2(d1v[0], d1v[1]);
        o3[q] = pack_bf16x2(d3v[0], d3v[1]);
      }
      const int off = lane * 128 + ((j ^ (lane & 7)) << 4);
      *reinterpret_cast<uint4*>(b1 + off) = make_uint4(o1[0], o1[1], o1[2], o1[3]);
#pragma unroll
      for (int q = 0; q < 4; ++q) keep[j][q] = o3[q];
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(map_out, b1, col, row0);
      bulk_commit();
      bulk_wait_read0();
    }
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int off = lane * 128 + ((j ^ (lane & 7)) << 4);
      *reinterpret_cast<uint4*>(b1 + off) = make_uint4(keep[j][0], keep[j][1], keep[j][2], keep[j][3]);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(map_out, b1, p.F + col, row0);
      bulk_commit();
    }
    st.n += 2;
  }
}

// DGRAD2R (memory-saving backward), rows all inside the expert: as
// epi_dgrad2_tma, and also a = bf16(SiLU(h1) h3) recomputed from the saved
// pre-activations into a third staging box (TMA store through map_a), and this
// row's partial of the gate gradient, sum over the tile's columns of da * a
// (with a as stored), into dg_part[row, n0 / 256].
__device__ __forceinline__ void epi_dgrad2r_tma(const GemmParams& p, const TileInfo& ti, uint32_t tacc, int lane,
                                                int row0, Stager& st, const CUtensorMap* map_out,
                                                const CUtensorMap* map_a) {
  const __nv_bfloat16* hrow =
      reinterpret_cast<const __nv_bfloat16*>(p.in_aux) + static_cast<size_t>(row0 + lane) * (2 * p.F);
  float dg = 0.0f;
#pragma unroll 1
  for (int cc = 0; cc < 4; ++cc) {
    const int col = ti.n0 + cc * 64;
    if (col >= p.F) break;
    uint4 v1[8], v3[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      v1[j] = ldg_nc_v4(hrow + col + 8 * j);
      v3[j] = ldg_nc_v4(hrow + p.F + col + 8 * j);
    }
    float da0[32], da1[32];
    tmem_ld32_f(tacc + (cc * 2) * 32, da0);
    tmem_ld32_f(tacc + (cc * 2 + 1) * 32, da1);
    uint8_t *b1, *b3;
    st.both(lane, b1, b3);  // every previous box has left the three buffers
    uint8_t* ba = b1 + 8192;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float* da = j < 4 ? da0 : da1;
      const uint32_t a1[4] = {v1[j].x, v1[j].y, v1[j].z, v1[j].w};
      const uint32_t a3[4] = {v3[j].x, v3[j].y, v3[j].z, v3[j].w};
      uint32_t o1[4], o3[4], oa[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float d1v[2], d3v[2], av[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float x1 = e ? bf16_hi(a1[q]) : bf16_lo(a1[q]);
          const float x3 = e ? bf16_hi(a3[q]) : bf16_lo(a3[q]);
          const float d = da[8 * (j & 3) + 2 * q + e];
          const float s = 1.0f / (1.0f + __expf(-x1));
          const float si = x1 * s;
          d1v[e] = d * x3 * (s * (1.0f + x1 * (1.0f - s)));
          d3v[e] = d * si;
          av[e] = __bfloat162float(__float2bfloat16_rn(si * x3));
          dg = fmaf(d, av[e], dg);
        }
        o1[q] = pack_bf16x2(d1v[0], d1v[1]);
        o3[q] = pack_bf16x2(d3v[0], d3v[1]);
        oa[q] = pack_bf16x2(av[0], av[1]);
      }
      const int off = lane * 128 + ((j ^ (lane & 7)) << 4);
      *reinterpret_cast<uint4*>(b1 + off) = make_uint4(o1[0], o1[1], o1[2], o1[3]);
      *reinterpret_cast<uint4*>(b3 + off) = make_uint4(o3[0], o3[1], o3[2], o3[3]);
      *reinterpret_cast<uint4*>(ba + off) = make_uint4(oa[0], oa[1], oa[2], oa[3]);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(map_out, b1, col, row0);
      tma_store_2d(map_out, b3, p.F + col, row0);
      tma_store_2d(map_a, ba, col, row0);
      bulk_commit();
    }
    st.n += 3;
  }
  p.dg_part[static_cast<size_t>(row0 + lane) * p.n_part + ti.n0 / 256] = dg;
}

}  // namespace moe

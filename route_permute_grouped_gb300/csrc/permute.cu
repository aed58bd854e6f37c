// Local dispatch: per-expert histogram, single-pass decoupled-lookback scan
// over token chunks, and the 16-byte vectorised row scatter into
// expert-contiguous rows (dropless; rows of one expert in token order).
#include <stdio.h>

#include <initializer_list>
#include <mutex>

#include "host_util.h"
#include "mx.cuh"
#include "nv.cuh"

namespace moe {

constexpr int kChunk = 64;          // tokens per scan chunk (two rank warps)
constexpr int kScanThreads = 256;
constexpr uint32_t kFlagP = 0x80000000u;  // inclusive prefix published
constexpr uint32_t kFlagA = 0x40000000u;  // chunk aggregate published
constexpr uint32_t kValMask = 0x3fffffffu;

// counts[e] += number of (t,i) with topk_idx[t,i] == e. Warp-aggregated: lanes
// holding the same expert combine through __match_any_sync, then one shared
// atomic per group and one global atomic per (block, expert).
__global__ void __launch_bounds__(256) permute_hist_kernel(const int32_t* __restrict__ topk_idx, int n, int E,
                                                           int32_t* __restrict__ counts, DevStatus* st) {
  __shared__ int s_h[256];
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_h[e] = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int stride = gridDim.x * blockDim.x;
  const int iters = (n + stride - 1) / stride;
  for (int it = 0; it < iters; ++it) {
    const int i = it * stride + blockIdx.x * blockDim.x + threadIdx.x;
    int e = -1;
    if (i < n) {
      e = __ldg(topk_idx + i);
      if (e < 0 || e >= E) {
        set_status(st, MOE_ERR_DEVICE_INDEX, 10);
        e = -1;
      }
    }
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && lane == __ffs(peers) - 1) atomicAdd(&s_h[e], __popc(peers));
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    if (s_h[e] != 0) atomicAdd(&counts[e], s_h[e]);
}

__device__ __forceinline__ uint32_t ld_volatile_u32(const int32_t* p) {
  return static_cast<uint32_t>(*reinterpret_cast<const volatile int32_t*>(p));
}
__device__ __forceinline__ void st_volatile_u32(int32_t* p, uint32_t v) {
  *reinterpret_cast<volatile int32_t*>(p) = static_cast<int32_t>(v);
}

// training scatter with quantised rows: the bf16 copies of token t's row too
// (for the weight gradient), 16-byte vectors, lane l taking vectors l, l + 32,
// ... (the row is in cache); rows[i] < 0: slot dropped
__device__ __forceinline__ void scatter_row_bf16(const __nv_bfloat16* __restrict__ x,
                                                 __nv_bfloat16* __restrict__ x_perm, int t, int H, const int* rows,
                                                 int k, int lane) {
  const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * H);
  for (int vv = lane; vv < H / 8; vv += 32) {
    const uint4 w = __ldg(src + vv);
    for (int i = 0; i < k; ++i) {
      const int r = rows[i];
      if (r >= 0) reinterpret_cast<uint4*>(x_perm + static_cast<size_t>(r) * H)[vv] = w;
    }
  }
}

// One CTA per chunk of 64 tokens, chunks taken in ticket order (so every
// earlier chunk has started when a CTA looks back). For expert e the row of
// (t,i) is offsets[e] + (rows of e in earlier chunks) + (rank of t among this
// chunk's tokens routed to e). The earlier-chunk term comes from a decoupled
// lookback over per-(chunk, expert) words [flag | value].
//
// MX: the scattered rows are MXFP8 instead of bf16: each token's row is
// quantised once (32-element blocks along H) and its codes written to every
// destination row of x_q; the scale of row r (rel = r - offset of its expert),
// block j goes to scale block 2 P + h, P = the expert's first 256-row pair tile
// + rel / 256, h = (rel / 128) % 2, k block j / 4 in sfa (row rel % 128, K
// step j % 4): the blocks the CTA pairs of the expert GEMM read. With x_perm
// non-null (training) the bf16 rows are scattered as well.
//
// NV (the MX instance with nv_g != nullptr): the rows are NVFP4 with the
// tensor scale *nv_g: 16-element blocks quantised once per token, codes (two
// per byte) to every destination row, scales to the same pair-tile blocks (2 KB
// per 128 rows and k block of 256); the bf16 rows too with x_perm non-null.
template <bool MX>
__global__ void __launch_bounds__(kScanThreads) permute_scan_scatter_kernel(
    const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ topk_idx, int T, int H, int E, int k,
    const int32_t* __restrict__ counts, int32_t* __restrict__ offsets_out, int32_t* __restrict__ lookback,
    __nv_bfloat16* __restrict__ x_perm, int32_t* __restrict__ row_id_map, DevStatus* st,
    unsigned long long limit_ns, int fault, uint8_t* __restrict__ x_q, uint8_t* __restrict__ sfa,
    const float* __restrict__ nv_g) {
  __shared__ int s_ticket;
  __shared__ uint32_t s_mask[2][256];
  __shared__ int s_base[256];
  __shared__ int s_scan[256];
  __shared__ int s_tscan[MX ? 256 : 1];
  __shared__ int s_rows[kChunk * 16];
  __shared__ int s_exp[MX ? kChunk * 16 : 1];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int32_t* ticket_ctr = lookback;  // lookback[0] is the chunk ticket counter
  int32_t* flags = lookback + 64;  // [nchunks][E]
  if (tid == 0) s_ticket = atomicAdd(ticket_ctr, 1);
  for (int e = tid; e < 256; e += kScanThreads) {
    s_mask[0][e] = 0u;
    s_mask[1][e] = 0u;
  }
  // exclusive scan of the global counts (E <= 256): offsets of the experts
  const int cnt = (tid < E) ? counts[tid] : 0;
  s_scan[tid] = cnt;
  if (MX) s_tscan[tid] = (cnt + 2 * kBM - 1) / (2 * kBM);  // 256-row pair tiles per expert
  __syncthreads();
  for (int d = 1; d < 256; d <<= 1) {
    const int v = (tid >= d) ? s_scan[tid - d] : 0;
    const int vt = (MX && tid >= d) ? s_tscan[tid - d] : 0;
    __syncthreads();
    s_scan[tid] += v;
    if (MX) s_tscan[tid] += vt;
    __syncthreads();
  }
  const int b = s_ticket;
  const int t0 = b * kChunk;
  if (b == 0) {
    if (tid < E) offsets_out[tid] = (tid == 0) ? 0 : s_scan[tid - 1];
    if (tid == 0) offsets_out[E] = s_scan[E - 1];
  }
  // per-warp bitmasks: bit `lane` of s_mask[w][e] = token t0 + 32w + lane routes to e
  int my_e[16];
  if (warp < 2) {
    const int t = t0 + warp * 32 + lane;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      my_e[i] = -1;
      if (i < k && t < T) {
        int e = topk_idx[static_cast<size_t>(t) * k + i];
        if (e < 0 || e >= E) {
          set_status(st, MOE_ERR_DEVICE_INDEX, 11);
          e = -1;
        }
        my_e[i] = e;
        if (e >= 0) atomicOr(&s_mask[warp][e], 1u << lane);
      }
    }
  }
  __syncthreads();
  // publish this chunk's aggregate, look back for the earlier chunks' total
  for (int e = tid; e < E; e += kScanThreads) {
    const uint32_t c = __popc(s_mask[0][e]) + __popc(s_mask[1][e]);
    int32_t* mine = flags + static_cast<size_t>(b) * E + e;
    uint32_t excl = 0;
    if (b == 0) {
      if (!fault) st_volatile_u32(mine, kFlagP | c);
    } else {
      st_volatile_u32(mine, kFlagA | c);
      int bb = b - 1;
      uint64_t t_start = 0;
      uint32_t spins = 0;
      while (bb >= 0) {
        const uint32_t v = ld_volatile_u32(flags + static_cast<size_t>(bb) * E + e);
        if (v & kFlagP) {
          excl += v & kValMask;
          break;
        } else if (v & kFlagA) {
          excl += v & kValMask;
          --bb;
        } else {
          if (spins == 0) t_start = globaltimer();
          if ((++spins & 31u) == 0 && globaltimer() - t_start > limit_ns) {
            set_status(st, MOE_ERR_DEVICE_TIMEOUT, 12);
            break;  // give up: publish what we have so later chunks finish
          }
        }
      }
      st_volatile_u32(mine, kFlagP | ((excl + c) & kValMask));
    }
    s_base[e] = ((e == 0) ? 0 : s_scan[e - 1]) + static_cast<int>(excl);
  }
  __syncthreads();
  // rows of this chunk's (t,i)
  if (warp < 2) {
    const int t = t0 + warp * 32 + lane;
    const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (i < k && t < T) {
        const int e = my_e[i];
        int r = -1;
        if (e >= 0) {
          r = s_base[e] + (warp == 1 ? __popc(s_mask[0][e]) : 0) + __popc(s_mask[warp][e] & lt);
        }
        row_id_map[static_cast<size_t>(t) * k + i] = r;
        s_rows[(warp * 32 + lane) * k + i] = r;
        if (MX) s_exp[(warp * 32 + lane) * k + i] = e;
      }
    }
  }
  __syncthreads();
  if (MX && nv_g != nullptr) {
    // NVFP4: lane l takes the 16-element blocks l, l+32, ... of the row
    const float g = *nv_g;
    const int nblk = H / kNvBlock, nkb = H / kNvKB;
    for (int j = warp; j < kChunk; j += kScanThreads / 32) {
      const int t = t0 + j;
      if (t >= T) break;
      for (int b = lane; b < nblk; b += 32) {
        const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * H + b * kNvBlock);
        float v[16];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const uint4 w = __ldg(src + u);
          const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            v[8 * u + 2 * q] = bf16_lo(ww[q]);
            v[8 * u + 2 * q + 1] = bf16_hi(ww[q]);
          }
        }
        uint32_t c[2];
        const uint8_t sb = static_cast<uint8_t>(nv_quant16(v, g, c));
        for (int i = 0; i < k; ++i) {
          const int r = s_rows[j * k + i];
          if (r < 0) continue;
          *reinterpret_cast<uint2*>(x_q + static_cast<size_t>(r) * (H / 2) + b * 8) = make_uint2(c[0], c[1]);
          const int e = s_exp[j * k + i];
          const int rel = r - (e == 0 ? 0 : s_scan[e - 1]);
          const int blk = 2 * ((e == 0 ? 0 : s_tscan[e - 1]) + rel / (2 * kBM)) + ((rel / kBM) & 1);
          sfa[(static_cast<size_t>(blk) * nkb + b / 16) * kNvSfBytes + nv_sf_pos(rel % kBM, b & 15)] = sb;
        }
      }
      if (x_perm != nullptr) scatter_row_bf16(x, x_perm, t, H, s_rows + j * k, k, lane);
    }
    return;
  }
  if constexpr (MX) {
    // quantise and scatter: warp w takes tokens w, w+8, ...; lane l the
    // 32-element blocks l, l+32, ... of the row (64 contiguous bytes each)
    const int nblk = H / kMxBlock, nkb = H / kMxKB;
    for (int j = warp; j < kChunk; j += kScanThreads / 32) {
      const int t = t0 + j;
      if (t >= T) break;
      for (int b = lane; b < nblk; b += 32) {
        const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * H + b * kMxBlock);
        float v[32];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint4 w = __ldg(src + u);
          const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            v[8 * u + 2 * q] = bf16_lo(ww[q]);
            v[8 * u + 2 * q + 1] = bf16_hi(ww[q]);
          }
        }
        uint32_t c[8];
        const uint8_t sb = static_cast<uint8_t>(mx_quant32(v, c));
        for (int i = 0; i < k; ++i) {
          const int r = s_rows[j * k + i];
          if (r < 0) continue;
          uint4* dst = reinterpret_cast<uint4*>(x_q + static_cast<size_t>(r) * H + b * kMxBlock);
          dst[0] = make_uint4(c[0], c[1], c[2], c[3]);
          dst[1] = make_uint4(c[4], c[5], c[6], c[7]);
          const int e = s_exp[j * k + i];
          const int rel = r - (e == 0 ? 0 : s_scan[e - 1]);
          const int blk = 2 * ((e == 0 ? 0 : s_tscan[e - 1]) + rel / (2 * kBM)) + ((rel / kBM) & 1);
          sfa[(static_cast<size_t>(blk) * nkb + b / 4) * kMxSfBytes + mx_sf_pos(rel % kBM, b & 3)] = sb;
        }
      }
      if (x_perm != nullptr) scatter_row_bf16(x, x_perm, t, H, s_rows + j * k, k, lane);
    }
    return;
  }
  // scatter: warp w copies tokens w, w+8, ... of the chunk; 16-byte vectors
  const int nvec = H / 8;
  for (int j = warp; j < kChunk; j += kScanThreads / 32) {
    const int t = t0 + j;
    if (t >= T) break;
    const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * H);
    for (int v0 = 0; v0 < nvec; v0 += 32 * 8) {
      uint4 buf[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int v = v0 + u * 32 + lane;
        if (v < nvec) buf[u] = __ldg(src + v);
      }
      for (int i = 0; i < k; ++i) {
        const int r = s_rows[j * k + i];
        if (r < 0) continue;
        uint4* dst = reinterpret_cast<uint4*>(x_perm + static_cast<size_t>(r) * H);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int v = v0 + u * 32 + lane;
          if (v < nvec) dst[v] = buf[u];
        }
      }
    }
  }
}

cudaError_t launch_permute(const moe_config& c, const __nv_bfloat16* x, const int32_t* topk_idx,
                           __nv_bfloat16* x_perm, int32_t* row_id_map, int32_t* counts, int32_t* offsets,
                           int32_t* lookback, DevStatus* st, cudaStream_t stream, uint8_t* x_q, uint8_t* sfa,
                           const float* nv_g) {
  NvtxRange nvtx(x_q == nullptr ? "moe.permute" : "moe.permute_quantize");
  const int T = c.T, E = c.E, k = c.k;
  const int nchunks = (T + kChunk - 1) / kChunk;
  cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, stream);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(lookback, 0, sizeof(int32_t) * (64 + static_cast<size_t>(nchunks) * E), stream);
  if (e != cudaSuccess) return e;
  const int n = T * k;
  int hb = (n + 1023) / 1024;
  hb = hb < 4 * num_sms() ? hb : 4 * num_sms();
  if (hb < 1) hb = 1;
  permute_hist_kernel<<<hb, 256, 0, stream>>>(topk_idx, n, E, counts, st);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (x_q != nullptr) {
    // scale blocks of rows past an expert's count (the tail of its last m
    // tile) are not written by the scatter: zero scales
    e = cudaMemsetAsync(sfa, 0, nv_g != nullptr ? nv_act_sf_bytes(T * k, E, c.H) : mx_sfa_bytes(T * k, E, c.H),
                        stream);
    if (e != cudaSuccess) return e;
    permute_scan_scatter_kernel<true><<<nchunks, kScanThreads, 0, stream>>>(
        x, topk_idx, T, c.H, E, k, counts, offsets, lookback, x_perm, row_id_map, st, wait_limit_ns(),
        debug_fault(), x_q, sfa, nv_g);
  } else {
    permute_scan_scatter_kernel<false><<<nchunks, kScanThreads, 0, stream>>>(
        x, topk_idx, T, c.H, E, k, counts, offsets, lookback, x_perm, row_id_map, st, wait_limit_ns(),
        debug_fault(), nullptr, nullptr, nullptr);
  }
  return cudaGetLastError();
}

size_t permute_lookback_ints(int T, int E) {
  return 64 + static_cast<size_t>((T + kChunk - 1) / kChunk) * E;
}

// ---------------------------------------------------------------------------
// Allocation-free permute: the same kernels, with their scratch (status word,
// chunk ticket and the per-(chunk, expert) lookback words) in a fixed
// file-scope device array instead of a caller-provided workspace.
// ---------------------------------------------------------------------------
constexpr size_t kNoAllocStatusInts = sizeof(DevStatus) / sizeof(int32_t);  // 64
constexpr size_t kNoAllocMaxFlags = size_t(1) << 18;  // chunks x experts words (1 MiB)
constexpr size_t kNoAllocScratchInts = kNoAllocStatusInts + 64 + kNoAllocMaxFlags;

// Every GPU that loads the library holds this array (about 1 MiB) until exit.
static __device__ __align__(256) int32_t g_noalloc_scratch[kNoAllocScratchInts];

// Device address of g_noalloc_scratch per device (host code cannot use the
// symbol itself: on the host it names a stand-in, not device memory).
static int32_t* noalloc_scratch_ptr(int dev) {
  static std::mutex mu;
  static int32_t* ptrs[64] = {nullptr};
  if (dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (ptrs[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<int32_t*>(p);
  }
  return ptrs[dev];
}

int validate_config(const moe_config* c);

}  // namespace moe

extern "C" int moe_noalloc_get_device_status(void* stream, int* status_out) {
  using namespace moe;
  if (status_out == nullptr) return MOE_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  int32_t* scratch = noalloc_scratch_ptr(dev);
  if (scratch == nullptr) return MOE_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int e = status_from_cuda(cudaStreamSynchronize(s));
  if (e != MOE_OK) return e;
  DevStatus h;
  e = status_from_cuda(cudaMemcpy(&h, scratch, sizeof(h), cudaMemcpyDeviceToHost));
  if (e != MOE_OK) return e;
  *status_out = h.status;
  return status_from_cuda(cudaMemset(scratch, 0, sizeof(DevStatus)));
}

extern "C" int moe_permute_noalloc(const moe_config* cfg, const moe_bf16* x, const int32_t* topk_idx,
                                   moe_bf16* x_perm, int32_t* row_id_map, int32_t* counts, int32_t* offsets,
                                   void* stream) {
  using namespace moe;
  const int v = validate_config(cfg);
  if (v != MOE_OK) return v;
  const moe_config& c = *cfg;
  if (!x || !topk_idx || !x_perm || !row_id_map || !counts || !offsets) return MOE_ERR_INVALID_ARG;
  for (const void* ptr : {static_cast<const void*>(x), static_cast<const void*>(topk_idx),
                          static_cast<const void*>(x_perm), static_cast<const void*>(row_id_map),
                          static_cast<const void*>(counts), static_cast<const void*>(offsets)})
    if (reinterpret_cast<uintptr_t>(ptr) & 15u) return MOE_ERR_INVALID_ARG;
  const size_t flags = static_cast<size_t>((c.T + kChunk - 1) / kChunk) * c.E;
  if (flags > kNoAllocMaxFlags) {
    fprintf(stderr,
            "moe_permute_noalloc: ceil(T/64)*E = %zu exceeds the static scratch limit %zu "
            "(use moe_permute with a workspace)\n",
            flags, kNoAllocMaxFlags);
    return MOE_ERR_UNSUPPORTED_SHAPE;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  int32_t* scratch = noalloc_scratch_ptr(dev);
  if (scratch == nullptr) return MOE_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  DevStatus* st = reinterpret_cast<DevStatus*>(scratch);
  // the status word keeps the previous call's contents: start from zero
  if (status_from_cuda(cudaMemsetAsync(st, 0, sizeof(DevStatus), s)) != MOE_OK) return MOE_ERR_CUDA;
  // launch_permute zeroes the ticket and lookback words itself
  const int e = status_from_cuda(launch_permute(c, reinterpret_cast<const __nv_bfloat16*>(x), topk_idx,
                                                reinterpret_cast<__nv_bfloat16*>(x_perm), row_id_map, counts,
                                                offsets, scratch + kNoAllocStatusInts, st, s));
  if (e != MOE_OK) return e;
  record_stage(s, 2 /* the permute's profiling tag */, 2);
  return MOE_OK;
}

// Host-side helpers shared by the translation units: tensor-map encoding (via
// the driver entry point, so the library does not link libcuda), device
// properties, and the launchers each .cu file exports.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stddef.h>
#include <stdint.h>

#include "gemm_tc.cuh"

namespace moe {

// NVTX range for the lifetime of the object (header-only NVTX3: a no-op unless
// a profiler attaches). Every entry point opens one named after itself and
// every kernel launch one named after its stage, so timelines of Nsight tools
// show the layer's stages and ncu can filter launches by range.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// 2-D bf16 tensor map over a row-major [outer, inner] array with row pitch
// `row_bytes`, box {box_inner, box_outer}, 128-byte swizzle, zero fill outside
// the array. Returns false if the driver rejects it.
bool make_map_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                   uint32_t box_inner, uint32_t box_outer);

int num_sms();
// Bookkeeping every entry point does after enqueueing a stage: launch counter,
// profiling event (tag as in moe_profile_start), debug synchronisation.
void record_stage(cudaStream_t s, int tag, int launches);
// MOE_OK for cudaSuccess, else MOE_ERR_CUDA with the CUDA message on stderr.
int status_from_cuda(cudaError_t e);
unsigned long long wait_limit_ns();
int debug_fault();

// 3-D fp32 tensor map over [outer2, outer1, inner] (row-major), box
// {32, 32, 1}, 128-byte swizzle: the output map of the weight-gradient GEMM.
bool make_map_f32_3d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t mid, uint64_t outer);

// out0/out1: output tensor maps of kinds that store through TMA (weight
// gradients); nullptr for the others.
cudaError_t launch_gemm(int kind, const GemmParams& p, const CUtensorMap& ma, const CUtensorMap& mb0,
                        const CUtensorMap& mb1, int grid, cudaStream_t st, const CUtensorMap* out0 = nullptr,
                        const CUtensorMap* out1 = nullptr);

// permute.cu
// With x_q != nullptr the permute writes MXFP8 rows (x_q [R, H] codes and the
// tile-ready scales sfa, mx_sfa_bytes(R, E, H) bytes) instead of bf16 x_perm;
// with nv_g != nullptr too, NVFP4 rows with the tensor scale *nv_g (x_q
// [R, H/2], nv_act_sf_bytes(R, E, H) bytes of scales).
cudaError_t launch_permute(const moe_config& c, const __nv_bfloat16* x, const int32_t* topk_idx,
                           __nv_bfloat16* x_perm, int32_t* row_id_map, int32_t* counts, int32_t* offsets,
                           int32_t* lookback, DevStatus* st, cudaStream_t stream, uint8_t* x_q = nullptr,
                           uint8_t* sfa = nullptr, const float* nv_g = nullptr);

size_t permute_lookback_ints(int T, int E);

// elementwise.cu
// ds: the status word that a dropped-slot or (bounds-check build) out-of-range
// index read from row_id_map / topk_idx is recorded in; nullable
cudaError_t launch_combine(const moe_config& c, const void* y_perm, const int32_t* row_id_map,
                           const float* gate, const void* shared, void* y, cudaStream_t st, DevStatus* ds = nullptr);
// mq != nullptr (MXFP8 training step): also the MXFP8 rows of dy_perm (codes
// mq [R, H], tile-ready scales msf; offsets and topk_idx locate each row)
// dy_amax (bf16 dy_perm only): the largest |dy_perm| stored, as fp32 bits
cudaError_t launch_combine_bwd(const moe_config& c, const __nv_bfloat16* dO, const void* y_perm,
                               const int32_t* row_id_map, const float* gate, __nv_bfloat16* dy_perm, float* dgate,
                               cudaStream_t st, uint8_t* mq = nullptr, uint8_t* msf = nullptr,
                               const int32_t* offsets = nullptr, const int32_t* topk_idx = nullptr,
                               DevStatus* ds = nullptr, float* dy_amax = nullptr);
// dx = sum_i dx_perm[row(t,i)] + extra (fp32, nullable) + add ([T,H], nullable);
// dx_perm and add are fp32 with rows_fp32, else bf16
cudaError_t launch_unpermute_sum(const moe_config& c, const void* dx_perm, const int32_t* row_id_map,
                                 const float* extra, void* dx, cudaStream_t st, const void* add = nullptr,
                                 bool rows_fp32 = false, DevStatus* ds = nullptr);
cudaError_t launch_router_bwd(const moe_config& c, const float* logits, const int32_t* topk_idx,
                              const float* gate, const float* dgate, const float* dg_part, int n_part,
                              const int32_t* row_id_map, const int32_t* counts, int Ep, __nv_bfloat16* dL_hl,
                              cudaStream_t st, DevStatus* ds = nullptr);
cudaError_t launch_aux_loss(const moe_config& c, const float* aux_partials, const int32_t* counts, float* out,
                            cudaStream_t st);
cudaError_t launch_split_reduce(const float* partials, int splits, size_t n, float* out, cudaStream_t st);

// mx.cu: MXFP8 quantisers and the sizes of the tile-ready scale buffers
inline int mx_ntiles1(const moe_config& c) { return (c.F + kMxTileF1 - 1) / kMxTileF1; }
inline int mx_ntiles2(const moe_config& c) { return (c.H + kMxTileN2 - 1) / kMxTileN2; }
inline size_t mx_sf13_bytes(const moe_config& c) {
  return static_cast<size_t>(c.E) * mx_ntiles1(c) * (c.H / kMxKB) * 2 * kMxSfBytes;
}
inline size_t mx_sf2_bytes(const moe_config& c) {
  return static_cast<size_t>(c.E) * mx_ntiles2(c) * (c.F / kMxKB) * 2 * kMxSfBytes;
}
// scale blocks of the activations of a grouped GEMM with K = `K`: two per
// (256-row pair tile, k block); an expert's rows start a new pair tile, so
// there are at most ceil(R / 256) + E pair tiles
inline size_t mx_sfa_bytes(long long R, int E, int K) {
  return 2 * static_cast<size_t>((R + 2 * kBM - 1) / (2 * kBM) + E) * (K / kMxKB) * kMxSfBytes;
}
// weights of the MXFP8 data-gradient GEMMs: W2 along H (B rows F in tiles of
// 192) and W1 | W3 along F (one K = 2F operand, B rows H in tiles of 192)
inline int mx_ntiles_f(const moe_config& c) { return (c.F + kMxTileN2 - 1) / kMxTileN2; }
inline size_t mx_sf2h_bytes(const moe_config& c) {
  return static_cast<size_t>(c.E) * mx_ntiles_f(c) * (c.H / kMxKB) * 2 * kMxSfBytes;
}
inline size_t mx_sf13f_bytes(const moe_config& c) {
  return static_cast<size_t>(c.E) * mx_ntiles2(c) * (2 * c.F / kMxKB) * 2 * kMxSfBytes;
}
// operands of the MXFP8 weight gradients: the tokens of each expert padded to
// whole k blocks of 128, kbt = k blocks of the padded axis (at most
// ceil((R + 127 E) / 128)); scale bytes of a transposed operand of C rows in
// tiles of tile_rows
inline int mx_wg_kbt(long long R, int E) { return static_cast<int>((R + 127ll * E + kMxKB - 1) / kMxKB); }
inline size_t mx_tok_sf_bytes(int C, int tile_rows, int kbt) {
  return static_cast<size_t>((C + tile_rows - 1) / tile_rows) * kbt * ((tile_rows + 127) / 128) * kMxSfBytes;
}
// nv.cu: NVFP4 quantisers and the sizes of the tile-ready scale buffers
inline size_t nv_weight_sf_bytes(int E, int K, int N) {
  return static_cast<size_t>(E) * ((N + kNvTileN - 1) / kNvTileN) * (K / kNvKB) * 2 * kNvSfBytes;
}
// gate/up weights [W1 | W3] (K = H, 2F columns) in the gate/up GEMM's tiles
// of 96 W1 + 96 W3 columns
inline size_t nv_weight_sf_bytes_gu(int E, int K, int F) {
  return static_cast<size_t>(E) * ((F + kMxTileF1 - 1) / kMxTileF1) * (K / kNvKB) * 2 * kNvSfBytes;
}
inline size_t nv_act_sf_bytes(long long R, int E, int K) {
  return 2 * static_cast<size_t>((R + 2 * kBM - 1) / (2 * kBM) + E) * (K / kNvKB) * kNvSfBytes;
}
// tensor scales of `groups` tensors of n_per elements (x2: a second tensor of
// the same shape whose elements count too)
cudaError_t launch_nv_amax(const __nv_bfloat16* x, long long n_per, int groups, float* out_g, cudaStream_t st,
                           const __nv_bfloat16* x2 = nullptr);
cudaError_t launch_nv_scale_from_amax(float* g, int n, cudaStream_t st);
cudaError_t launch_nv_quantize_rows(const __nv_bfloat16* x, long long M, int K, const float* g, uint8_t* q,
                                    uint8_t* s, cudaStream_t st);
cudaError_t launch_nv_quantize_weights(const __nv_bfloat16* w, int E, int K, int N, const float* g, uint8_t* wq,
                                       uint8_t* sf, cudaStream_t st, const __nv_bfloat16* w_hi = nullptr,
                                       int split = 0);
cudaError_t launch_nv_quantize_grouped(const __nv_bfloat16* x, int R, int K, int E, const int32_t* offsets,
                                       const float* g, uint8_t* xq, uint8_t* sf, cudaStream_t st);
// row-major weights W[E][N][K] (columns [split, K) from w_hi [E][N][K - split])
// -> K-major codes and tile-ready scales as launch_nv_quantize_weights' plain layout
cudaError_t launch_nv_quantize_weight_rows(const __nv_bfloat16* w, int E, int K, int N, const float* g, uint8_t* wq,
                                           uint8_t* sf, cudaStream_t st, const __nv_bfloat16* w_hi = nullptr,
                                           int split = 0);
// dh13 = SwiGLU backward of da (fp32 [R, F]) on the saved h13 (first *n_rows
// rows), its tensor scale into *g
cudaError_t launch_nv_swiglu_bwd(const float* da, const __nv_bfloat16* h13, int R, int F, const int32_t* n_rows,
                                 __nv_bfloat16* dh13, float* g, cudaStream_t st);
cudaError_t launch_mx_quantize_rows(const __nv_bfloat16* x, long long M, int K, uint8_t* q, uint8_t* s,
                                    cudaStream_t st);
cudaError_t launch_mx_quantize_weights(const moe_config& c, const __nv_bfloat16* W1, const __nv_bfloat16* W3,
                                       const __nv_bfloat16* W2, uint8_t* w13q, uint8_t* sf13, uint8_t* w2q,
                                       uint8_t* sf2, cudaStream_t st);
// gemm.cu: per-expert copies of a 2-D tensor map with the row extent set to
// each expert's end row (for the weight gradients' partial k blocks); one copy
// ending at `rows` when offsets == nullptr
cudaError_t launch_tmap_rows(const CUtensorMap& tmpl, const int32_t* offsets, int E, uint8_t* maps, cudaStream_t st,
                             int rows = 0);
cudaError_t launch_mx_quantize_tokens(const __nv_bfloat16* X, int R, int C, int ldx, int E, const int32_t* offsets,
                                      uint8_t* XT, uint8_t* sf, int tile_rows, int32_t* pad_off, cudaStream_t st);
cudaError_t launch_mx_quantize_bwd_weights(const moe_config& c, const __nv_bfloat16* W1, const __nv_bfloat16* W3,
                                           const __nv_bfloat16* W2, uint8_t* w2h, uint8_t* sf2h, uint8_t* w13f,
                                           uint8_t* sf13f, cudaStream_t st);
}  // namespace moe

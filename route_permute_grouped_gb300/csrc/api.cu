// The C ABI: argument checks, workspace layout, tensor maps and the
// composition of the kernels into the layer forward and backward.
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <initializer_list>
#include <mutex>
#include <vector>

#include "host_util.h"

namespace moe {

// ---------------------------------------------------------------------------
// process-wide settings
// ---------------------------------------------------------------------------
static unsigned long long g_wait_limit_ns = 2000000000ull;
static int g_fault = 0;

// Stage timing log (benchmark support): when enabled, every stage of the
// layer calls records a CUDA event on the caller's stream, tagged with the
// stage; the elapsed time between consecutive events is the stage's time.
struct ProfLog {
  bool on = false;
  int n = 0;
  std::vector<cudaEvent_t> ev;
  std::vector<int> tag;
};
static ProfLog g_prof;
static unsigned long long g_launches = 0;

static void prof_mark(cudaStream_t s, int tag) {
  if (!g_prof.on || g_prof.n >= static_cast<int>(g_prof.ev.size())) return;
  cudaEventRecord(g_prof.ev[g_prof.n], s);
  g_prof.tag[g_prof.n] = tag;
  ++g_prof.n;
}
static void count_launches(int n) { g_launches += static_cast<unsigned long long>(n); }

enum StageTag : int {
  STAGE_BEGIN = 0, STAGE_ROUTER = 1, STAGE_PERMUTE = 2, STAGE_FFN1 = 3, STAGE_FFN2 = 4, STAGE_SHARED1 = 5,
  STAGE_SHARED2 = 6, STAGE_COMBINE = 7,
  STAGE_COMBINE_BWD = 10, STAGE_ROUTER_BWD = 11, STAGE_DGRAD2 = 12, STAGE_WGRAD2 = 13, STAGE_DGRAD1 = 14,
  STAGE_WGRAD13 = 15, STAGE_ROUTER_DX = 16, STAGE_UNPERMUTE = 17, STAGE_ROUTER_DW = 18, STAGE_AUX = 19,
  STAGE_NV_QUANT = 20, STAGE_NV_GEMM = 21,
  STAGE_MX_QUANT_TOK = 22, STAGE_MX_DGRAD2 = 24, STAGE_MX_DGRAD1 = 25,
  STAGE_SHARED_DGRAD2 = 26, STAGE_SHARED_WGRAD2 = 27, STAGE_SHARED_DGRAD1 = 28, STAGE_SHARED_WGRAD13 = 29,
  STAGE_NV_DGRAD2 = 32, STAGE_NV_SWIGLU_BWD = 33, STAGE_NV_DGRAD1 = 34,
};
// MOE_DEBUG_SYNC=1 in the environment: synchronise after every stage and
// report the first stage whose kernels failed (debugging aid, off by default).
static bool debug_sync() {
  static int v = -1;
  if (v < 0) {
    const char* e = getenv("MOE_DEBUG_SYNC");
    v = (e != nullptr && e[0] == '1') ? 1 : 0;
  }
  return v == 1;
}
static void stage_done(cudaStream_t s, int tag, int launches) {
  count_launches(launches);
  prof_mark(s, tag);
  if (debug_sync()) {
    cudaError_t e = cudaStreamSynchronize(s);
    fprintf(stderr, "moe: stage %d done: %s\n", tag, cudaGetErrorString(e));
  }
}
void record_stage(cudaStream_t s, int tag, int launches) { stage_done(s, tag, launches); }
unsigned long long wait_limit_ns() { return g_wait_limit_ns; }
int debug_fault() { return g_fault; }

int num_sms() {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (cached[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 1;
  }
  return cached[dev];
}

// ---------------------------------------------------------------------------
// tensor maps through the driver entry point (no link-time libcuda)
// ---------------------------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool make_map_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                   uint32_t box_inner, uint32_t box_outer) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D map over a row-major [outer, inner] array of bytes (E4M3 codes), box
// {box_inner, box_outer}, 128-byte swizzle (or none: scale blocks as rows of
// 256 bytes), zero fill outside the array.
static bool make_map_u8(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
                        uint32_t box_outer, bool swizzle = true) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_map_f32_3d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t mid, uint64_t outer) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {inner, mid, outer};
  cuuint64_t strides[2] = {inner * 4, inner * mid * 4};
  cuuint32_t box[3] = {32, 32, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Store map of a row-major [rows, cols] output for the TMA-store epilogue:
// 32-row boxes of 128 bytes (64 bf16 or 32 fp32 columns), 128-byte swizzle.
static bool make_map_store(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, bool fp32) {
  if (!fp32) return make_map_bf16(m, base, cols, rows, 2 * cols, 64, 32);
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 4};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// ---------------------------------------------------------------------------
// workspace layout
// ---------------------------------------------------------------------------
static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct WsLayout {
  size_t status, lookback;
  // forward intermediates (inference, or standalone grouped FFN without a_save)
  size_t topk_idx, topk_gate, row_id_map, counts, offsets, x_perm, a, y_perm, as, s_out;
  // backward
  size_t dy_perm, dgate, dh13, dx_perm, dL_hl, dx_r, dwr_part, dg_part, tmap_slots;
  // backward of the shared expert: dh13 [T, 2Fs] and its input gradient [T, H] (bf16)
  size_t dh13_s, dx_s;
  // MXFP8 forward: E4M3 rows of x_perm and a, and their tile-ready scales
  size_t x_q, sfa1, a_q, sfa2;
  // MXFP8 backward: E4M3 rows of dy_perm and dh13 with their scales; the
  // transposed token-axis operands of the weight gradients (A, B) with their
  // scales and the padded token offsets
  size_t dy_q, sfa_dy, dh_q, sfa_dh, tok_a, sf_a, tok_b, sf_b, pad_off;
  // NVFP4: codes and scales of the current GEMM's activations (x_perm, then
  // a; training: then dy_perm, then dh13), their tensor scales (x, a, dy,
  // dh13); training: da (fp32)
  size_t nv_q, nv_sf, nv_g, nv_da;
  size_t total;
};

static int padded_experts(int E) { return ((E + 63) / 64) * 64; }
// K splits of the router weight gradient (at most 16, at most one per token
// block); the workspace holds this many partials, a launch may use fewer
static int router_dw_splits(int T) {
  const int kbh = (T + kBK - 1) / kBK;
  int s = 16;
  if (kbh < s) s = kbh;
  return s < 1 ? 1 : s;
}

// the weight-gradient kernels' per-expert tensor-map copies (128 bytes each)
constexpr size_t kTmapSlotBytes = 128;

static WsLayout ws_layout(const moe_config& c, bool training, bool mx = false, bool nv = false) {
  WsLayout L{};
  const size_t T = c.T, H = c.H, E = c.E, k = c.k, F = c.F, R = T * k;
  const size_t inter = c.inter_fp32 ? 4 : 2;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o += align256(bytes);
    return at;
  };
  L.status = take(sizeof(DevStatus));
  L.lookback = take(sizeof(int32_t) * permute_lookback_ints(c.T, c.E));
  L.topk_idx = take(4 * T * k);
  L.topk_gate = take(4 * T * k);
  L.row_id_map = take(4 * T * k);
  L.counts = take(4 * E);
  L.offsets = take(4 * (E + 1));
  if (mx) {
    L.x_q = take(R * H);
    L.sfa1 = take(mx_sfa_bytes(c.T * c.k, c.E, c.H));
    L.a_q = take(R * F);
    L.sfa2 = take(mx_sfa_bytes(c.T * c.k, c.E, c.F));
    if (training) {
      L.a = take(2 * R * F);  // a recomputed from h13 for the down weight gradient
      L.dy_q = take(R * H);
      L.sfa_dy = take(mx_sfa_bytes(c.T * c.k, c.E, c.H));
      L.dh_q = take(2 * R * F);
      L.sfa_dh = take(mx_sfa_bytes(c.T * c.k, c.E, 2 * c.F));
      const int kbt = mx_wg_kbt(static_cast<long long>(R), c.E);
      const size_t ldk = static_cast<size_t>(kbt) * kMxKB;
      const int CA = c.H > c.F ? c.H : c.F;  // A: a (F rows) or x_perm (H rows)
      const int CB = c.H > c.F ? c.H : c.F;  // B: dy_perm (H rows), dh1 or dh3 (F rows)
      L.tok_a = take(static_cast<size_t>(CA) * ldk);
      L.sf_a = take(mx_tok_sf_bytes(CA, 128, kbt));
      L.tok_b = take(static_cast<size_t>(CB) * ldk);
      L.sf_b = take(mx_tok_sf_bytes(CB, kMxBN, kbt));
      L.pad_off = take(sizeof(int32_t) * (E + 1));
    }
  } else {
    if (!nv) L.x_perm = take(2 * R * H);  // the NVFP4 permute writes codes only
    if (!(nv && training)) L.a = take(2 * R * F);  // NVFP4 training: a lives in the saved buffers
  }
  if (nv) {
    // the widest activation operand: x_perm or a (H or F columns); training
    // also dh13 (2F)
    const size_t kq = training ? (H > 2 * F ? H : 2 * F) : (H > F ? H : F);
    L.nv_q = take(R * kq / 2);
    L.nv_sf = take(nv_act_sf_bytes(static_cast<long long>(R), c.E, static_cast<int>(kq)));
    L.nv_g = take(4 * sizeof(float));
    if (training) L.nv_da = take(4 * R * F);
  }
  L.y_perm = take(inter * R * H);
  L.as = c.F_shared ? take(2 * T * c.F_shared) : 0;
  L.s_out = c.F_shared ? take(inter * T * H) : 0;
  if (training) {
    const size_t Ep = padded_experts(c.E);
    L.dy_perm = take(2 * R * H);
    L.dgate = take(4 * T * k);
    L.dg_part = take(4 * R * ((F + 255) / 256));  // memory-saving backward: gate-gradient partials
    L.dh13 = take(2 * R * 2 * F);
    L.dx_perm = take(inter * R * H);  // fp32 with inter_fp32 (the bf16 backward)
    L.dL_hl = take(2 * T * 2 * Ep);
    L.dx_r = take(4 * T * H);
    L.dwr_part = take(4 * static_cast<size_t>(router_dw_splits(c.T)) * E * H);
    L.tmap_slots = take(kTmapSlotBytes * (E + 1));  // weight gradients: per-expert A-map copies (+ shared)
    if (c.F_shared) {
      L.dh13_s = take(2 * T * 2 * static_cast<size_t>(c.F_shared));
      L.dx_s = take(inter * T * H);
    }
  }
  L.total = o;
  return L;
}

template <class P>
static P* at(void* ws, size_t off) {
  return reinterpret_cast<P*>(reinterpret_cast<uint8_t*>(ws) + off);
}

// ---------------------------------------------------------------------------
// checks
// ---------------------------------------------------------------------------
static int check_cfg(const moe_config* c) {
  if (c == nullptr) return MOE_ERR_INVALID_ARG;
  if (c->T < 1 || c->H < 1 || c->E < 1 || c->k < 1 || c->F < 1 || c->F_shared < 0) return MOE_ERR_INVALID_ARG;
  if (c->k > c->E) return MOE_ERR_INVALID_ARG;
  if (c->score != MOE_SCORE_SOFTMAX && c->score != MOE_SCORE_SIGMOID) return MOE_ERR_INVALID_ARG;
  if (!(c->gate_scale > 0.0f)) return MOE_ERR_INVALID_ARG;
  if (c->n_groups < 1 || c->topk_groups < 1 || c->topk_groups > c->n_groups) return MOE_ERR_INVALID_ARG;
  if (c->force_balanced != 0 && c->force_balanced != 1) return MOE_ERR_INVALID_ARG;
  if (c->E % c->n_groups != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (c->n_groups > 32) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (c->n_groups > 1 && c->topk_groups < c->n_groups && c->k > c->topk_groups * (c->E / c->n_groups))
    return MOE_ERR_INVALID_ARG;
  if (c->k > 16 || c->E > 256) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (c->H % 64 != 0 || c->F % 64 != 0 || c->F_shared % 64 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (static_cast<long long>(c->T) * c->k >= (1ll << 30)) return MOE_ERR_UNSUPPORTED_SHAPE;
  return MOE_OK;
}

int validate_config(const moe_config* c) { return check_cfg(c); }

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
// Every device pointer an entry point takes must be 16-byte aligned: the
// kernels reach them with 16-byte vector accesses and TMA copies, which fault
// on a misaligned address. Null passes here (the null checks are separate).
static bool all_aligned16(std::initializer_list<const void*> ps) {
  for (const void* p : ps)
    if (!aligned16(p)) return false;
  return true;
}
static bool saved_aligned16(const moe_fwd_saved* sv) {
  return sv == nullptr || all_aligned16({sv->topk_idx, sv->topk_gate, sv->logits, sv->row_id_map, sv->counts,
                                         sv->offsets, sv->x_perm, sv->h13, sv->a, sv->y_perm, sv->aux_partials,
                                         sv->h13_shared, sv->a_shared});
}

static int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return MOE_OK;
  fprintf(stderr, "moe: CUDA error %s\n", cudaGetErrorString(e));
  return MOE_ERR_CUDA;
}
int status_from_cuda(cudaError_t e) { return cuda_status(e); }

static GemmParams base_params(const moe_config& c, DevStatus* st) {
  GemmParams p;
  memset(&p, 0, sizeof(p));
  p.T = c.T; p.H = c.H; p.E = c.E; p.k = c.k; p.F = c.F;
  p.bn = 256;
  p.splits = 1;
  p.status = st;
  p.wait_limit_ns = g_wait_limit_ns;
  return p;
}

#define MOE_TRY(x)                 \
  do {                             \
    int _s = (x);                  \
    if (_s != MOE_OK) return _s;   \
  } while (0)
#define MOE_CUDA(x) MOE_TRY(cuda_status(x))
#define MOE_MAP(...)                                   \
  do {                                                 \
    if (!make_map_bf16(__VA_ARGS__)) return MOE_ERR_CUDA; \
  } while (0)

// ---------------------------------------------------------------------------
// stages
// ---------------------------------------------------------------------------
static int run_router(const moe_config& c, const __nv_bfloat16* x, const __nv_bfloat16* w_r, const float* eb,
                      const float* lb, int32_t* idx, float* gate, float* logits, float* aux, DevStatus* st,
                      cudaStream_t s) {
  // logits GEMM with the score, selection and gates in its epilogue: one CTA
  // per 128-row tile of x against the whole router weight (E <= 256 columns)
  GemmParams p = base_params(c, st);
  p.bn = ((c.E + 31) / 32) * 32;
  p.n_tiles = 1;
  p.ngroups = 1;
  p.M_total = c.T;
  p.kb_total = c.H / kBK;
  p.offsets = nullptr;
  const bool softmax = c.score == MOE_SCORE_SOFTMAX;
  // a group limit ranks groups by sums of scores, which logits do not order
  const bool grouped = !c.force_balanced && c.n_groups > 1 && c.topk_groups < c.n_groups;
  p.r_mode = !softmax ? RSEL_SIGMOID : ((eb == nullptr && !grouped) ? RSEL_LOGIT : RSEL_SOFTMAX);
  p.r_lbias = lb;
  p.r_ebias = eb;
  p.r_idx = idx;
  p.r_gate = gate;
  p.r_logits = logits;
  p.r_aux = softmax ? aux : nullptr;
  p.r_groups = c.n_groups;
  p.r_topk_groups = c.topk_groups;
  p.r_force = c.force_balanced;
  p.r_gate_scale = c.gate_scale;
  CUtensorMap ma, mb;
  MOE_MAP(&ma, x, c.H, c.T, 2ull * c.H, 64, 128);
  MOE_MAP(&mb, w_r, c.H, c.E, 2ull * c.H, 64, p.bn);  // rows past E read as zero
  const int tiles = (c.T + kBM - 1) / kBM;
  const int grid = tiles < num_sms() ? tiles : num_sms();
  return cuda_status(launch_gemm(KIND_ROUTER, p, ma, mb, mb, grid, s));
}

// grouped (offsets != nullptr, rows of x_rows grouped by expert) or single-group
// (offsets == nullptr, M rows) SwiGLU FFN: a = SiLU(x W1) * (x W3), y = a W2.
static int run_ffn(const moe_config& c, int F, int ngroups, const int32_t* offsets, int M,
                   const __nv_bfloat16* x_rows, const __nv_bfloat16* W1, const __nv_bfloat16* W3,
                   const __nv_bfloat16* W2, __nv_bfloat16* h13, __nv_bfloat16* a, void* y, bool y_fp32,
                   DevStatus* st, cudaStream_t s, int tag1 = STAGE_FFN1, int tag2 = STAGE_FFN2) {
  GemmParams p = base_params(c, st);
  p.F = F;
  p.ngroups = ngroups;
  p.offsets = offsets;
  p.M_total = M;
  // h = x [W1 | W3], 128 gate + 128 up columns per tile
  p.n_tiles = (F + 127) / 128;
  p.kb_total = c.H / kBK;
  p.out0 = a;
  p.out1 = h13;
  CUtensorMap ma, m1, m3, m2;
  MOE_MAP(&ma, x_rows, c.H, M, 2ull * c.H, 64, 128);
  MOE_MAP(&m1, W1, F, static_cast<uint64_t>(ngroups) * c.H, 2ull * F, 64, 64);
  MOE_MAP(&m3, W3, F, static_cast<uint64_t>(ngroups) * c.H, 2ull * F, 64, 64);
  CUtensorMap oa, oh;
  if (!make_map_store(&oa, a, F, M, false)) return MOE_ERR_CUDA;
  if (h13 != nullptr && !make_map_store(&oh, h13, 2ull * F, M, false)) return MOE_ERR_CUDA;
  MOE_CUDA(launch_gemm(KIND_FFN1, p, ma, m1, m3, num_sms(), s, &oa, h13 != nullptr ? &oh : nullptr));
  stage_done(s, tag1, 1);
  // y = a W2
  GemmParams q = base_params(c, st);
  q.F = F;
  q.ngroups = ngroups;
  q.offsets = offsets;
  q.M_total = M;
  q.n_tiles = (c.H + 255) / 256;
  q.kb_total = F / kBK;
  q.out0 = y;
  q.out_fp32 = y_fp32;
  CUtensorMap mA;
  MOE_MAP(&mA, a, F, M, 2ull * F, 64, 128);
  MOE_MAP(&m2, W2, c.H, static_cast<uint64_t>(ngroups) * F, 2ull * c.H, 64, 64);
  CUtensorMap oy;
  if (!make_map_store(&oy, y, c.H, M, y_fp32)) return MOE_ERR_CUDA;
  MOE_CUDA(launch_gemm(KIND_FFN2, q, mA, m2, m2, num_sms(), s, &oy));
  stage_done(s, tag2, 1);
  return MOE_OK;
}

static int check_mx_shape(const moe_config& c) {
  // k blocks of 128 codes along H (gate/up GEMM) and F (down GEMM)
  if (c.H % kMxKB != 0 || c.F % kMxKB != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  return MOE_OK;
}

// MXFP8 grouped SwiGLU FFN over the permuted rows: a = SiLU(Q(x) Q(W1)) * (Q(x)
// Q(W3)) quantised in the epilogue, y_perm = Q(a) Q(W2). Scale blocks are read
// as rows of 256 bytes (A: 2 per block, B: 4 per tile's pair of blocks).
static int run_ffn_mx(const moe_config& c, const int32_t* offsets, int R, const uint8_t* x_q, const uint8_t* sfa1,
                      const moe_mx_weights& w, uint8_t* a_q, uint8_t* sfa2, void* y, bool y_fp32, DevStatus* st,
                      cudaStream_t s, __nv_bfloat16* h13 = nullptr) {
  GemmParams p = base_params(c, st);
  p.F = c.F;
  p.ngroups = c.E;
  p.offsets = offsets;
  p.M_total = R;
  p.bn = kMxBN;
  p.n_tiles = mx_ntiles1(c);
  p.nt_w = mx_ntiles1(c);
  p.kb_total = c.H / kMxKB;
  p.out0 = a_q;
  p.out1 = h13;  // training: bf16 h1 | h3 saved for the backward
  p.sfa_out = sfa2;
  CUtensorMap ma, mb, msa, msb;
  if (!make_map_u8(&ma, x_q, c.H, R, kMxKB, kBM)) return MOE_ERR_CUDA;
  if (!make_map_u8(&mb, w.w13, c.H, 2ull * c.E * c.F, kMxKB, kMxTileF1)) return MOE_ERR_CUDA;
  if (!make_map_u8(&msa, sfa1, 256, mx_sfa_bytes(R, c.E, c.H) / 256, 256, 2, false)) return MOE_ERR_CUDA;
  if (!make_map_u8(&msb, w.sf13, 256, mx_sf13_bytes(c) / 256, 256, 4, false)) return MOE_ERR_CUDA;
  MOE_CUDA(launch_gemm(KIND_FFN1_MX, p, ma, mb, msa, num_sms(), s, nullptr, &msb));
  stage_done(s, STAGE_FFN1, 1);
  GemmParams q = base_params(c, st);
  q.F = c.F;
  q.ngroups = c.E;
  q.offsets = offsets;
  q.M_total = R;
  q.bn = kMxBN;
  q.n_tiles = mx_ntiles2(c);
  q.nt_w = mx_ntiles2(c);
  q.kb_total = c.F / kMxKB;
  q.out0 = y;
  q.out_fp32 = y_fp32;
  CUtensorMap ma2, mb2, msa2, msb2, oy;
  if (!make_map_u8(&ma2, a_q, c.F, R, kMxKB, kBM)) return MOE_ERR_CUDA;
  if (!make_map_u8(&mb2, w.w2, c.F, static_cast<uint64_t>(c.E) * c.H, kMxKB, kMxBN / 2)) return MOE_ERR_CUDA;
  if (!make_map_u8(&msa2, sfa2, 256, mx_sfa_bytes(R, c.E, c.F) / 256, 256, 2, false)) return MOE_ERR_CUDA;
  if (!make_map_u8(&msb2, w.sf2, 256, mx_sf2_bytes(c) / 256, 256, 4, false)) return MOE_ERR_CUDA;
  if (!make_map_store(&oy, y, c.H, R, y_fp32)) return MOE_ERR_CUDA;
  MOE_CUDA(launch_gemm(KIND_FFN2_MX, q, ma2, mb2, msa2, num_sms(), s, &oy, &msb2));
  stage_done(s, STAGE_FFN2, 1);
  return MOE_OK;
}

// Grouped MXFP8 GEMM y [R, N] bf16 = Q(A) Q(W_e)^T (the down projection's
// kernel kind with N and K as given): A codes [R, K] with the activations'
// tile-ready scales (mx_sfa_bytes(R, E, K)), W codes [E][N][K] with the
// weights' tile-ready scales (tiles of 192 B rows, sfw_bytes in all).
static int run_gemm_mx(const moe_config& c, const int32_t* offsets, int R, int K, int N, const uint8_t* aq,
                       const uint8_t* sfa, const uint8_t* wq, const uint8_t* sfw, size_t sfw_bytes,
                       __nv_bfloat16* y, DevStatus* st, cudaStream_t s) {
  GemmParams q = base_params(c, st);
  q.H = N;
  q.ngroups = c.E;
  q.offsets = offsets;
  q.M_total = R;
  q.bn = kMxBN;
  q.n_tiles = (N + kMxTileN2 - 1) / kMxTileN2;
  q.nt_w = q.n_tiles;
  q.kb_total = K / kMxKB;
  q.out0 = y;
  CUtensorMap ma, mb, msa, msb, oy;
  if (!make_map_u8(&ma, aq, K, R, kMxKB, kBM)) return MOE_ERR_CUDA;
  if (!make_map_u8(&mb, wq, K, static_cast<uint64_t>(c.E) * N, kMxKB, kMxBN / 2)) return MOE_ERR_CUDA;
  if (!make_map_u8(&msa, sfa, 256, mx_sfa_bytes(R, c.E, K) / 256, 256, 2, false)) return MOE_ERR_CUDA;
  if (!make_map_u8(&msb, sfw, 256, sfw_bytes / 256, 256, 4, false)) return MOE_ERR_CUDA;
  if (!make_map_store(&oy, y, N, R, false)) return MOE_ERR_CUDA;
  return cuda_status(launch_gemm(KIND_FFN2_MX, q, ma, mb, msa, num_sms(), s, &oy, &msb));
}

// MXFP8 data gradient of the down projection with the SwiGLU backward in its
// epilogue: da = Q(dy_perm) Q(W2_e)^T (K = H, N = F) -> dh13, a (bf16) and the
// MXFP8 rows of dh13 with their tile-ready scales (K = 2F)
static int run_dgrad2_mx(const moe_config& c, const int32_t* offsets, int R, const uint8_t* dy_q,
                         const uint8_t* sfa_dy, const moe_mx_bwd_weights& w, const __nv_bfloat16* h13,
                         __nv_bfloat16* dh13, __nv_bfloat16* a, uint8_t* dh_q, uint8_t* sfa_dh, DevStatus* st,
                         cudaStream_t s) {
  GemmParams q = base_params(c, st);
  q.H = c.F;  // N of this GEMM
  q.ngroups = c.E;
  q.offsets = offsets;
  q.M_total = R;
  q.bn = kMxBN;
  q.n_tiles = mx_ntiles_f(c);
  q.nt_w = q.n_tiles;
  q.kb_total = c.H / kMxKB;
  q.in_aux = h13;
  q.out0 = dh13;
  q.out1 = a;
  q.q_out = dh_q;
  q.sfa_out = sfa_dh;
  CUtensorMap ma, mb, msa, msb;
  if (!make_map_u8(&ma, dy_q, c.H, R, kMxKB, kBM)) return MOE_ERR_CUDA;
  if (!make_map_u8(&mb, w.w2h, c.H, static_cast<uint64_t>(c.E) * c.F, kMxKB, kMxBN / 2)) return MOE_ERR_CUDA;
  if (!make_map_u8(&msa, sfa_dy, 256, mx_sfa_bytes(R, c.E, c.H) / 256, 256, 2, false)) return MOE_ERR_CUDA;
  if (!make_map_u8(&msb, w.sf2h, 256, mx_sf2h_bytes(c) / 256, 256, 4, false)) return MOE_ERR_CUDA;
  return cuda_status(launch_gemm(KIND_DGRAD2_MX, q, ma, mb, msa, num_sms(), s, nullptr, &msb));
}

// MXFP8 weight gradient out [E][M][N] fp32 = Q(A_e)^T Q(B_e) over each expert's
// tokens: X_A [R, M] (row stride lda) and X_B [R, N] (row stride ldb), bf16
// rows grouped by expert, are quantised along the tokens into the transposed
// operands (A: 128-row scale tiles, B: 192-row tiles; the padded token offsets
// become the GEMM's group offsets), then one ragged-K block-scaled GEMM
static int run_wgrad_mx(const moe_config& c, const int32_t* offsets, int R, const __nv_bfloat16* XA, int M, int lda,
                        const __nv_bfloat16* XB, int N, int ldb, float* out, void* ws, const WsLayout& L,
                        DevStatus* st, cudaStream_t s, bool quantise_a = true) {
  const int kbt = mx_wg_kbt(static_cast<long long>(R), c.E);
  const uint64_t ldk = static_cast<uint64_t>(kbt) * kMxKB;
  uint8_t* ta = at<uint8_t>(ws, L.tok_a);
  uint8_t* sa = at<uint8_t>(ws, L.sf_a);
  uint8_t* tb = at<uint8_t>(ws, L.tok_b);
  uint8_t* sb = at<uint8_t>(ws, L.sf_b);
  int32_t* pad = at<int32_t>(ws, L.pad_off);
  if (quantise_a) MOE_CUDA(launch_mx_quantize_tokens(XA, R, M, lda, c.E, offsets, ta, sa, 128, pad, s));
  MOE_CUDA(launch_mx_quantize_tokens(XB, R, N, ldb, c.E, offsets, tb, sb, kMxBN, pad, s));
  stage_done(s, STAGE_MX_QUANT_TOK, quantise_a ? 2 : 1);
  GemmParams p = base_params(c, st);
  p.ngroups = c.E;
  p.offsets = pad;
  p.wg_M = M; p.wg_N = N; p.wg_mode = 0;
  p.m_tiles_fixed = (M + 255) / 256;
  p.n_tiles = (N + kMxBN - 1) / kMxBN;
  p.bn = kMxBN;
  p.kb_total = kbt;
  p.out0 = out;
  CUtensorMap ma, mb, msa, msb, mo;
  if (!make_map_u8(&ma, ta, ldk, static_cast<uint64_t>(M), kMxKB, kBM)) return MOE_ERR_CUDA;
  if (!make_map_u8(&mb, tb, ldk, static_cast<uint64_t>(N), kMxKB, kMxBN / 2)) return MOE_ERR_CUDA;
  if (!make_map_u8(&msa, sa, 256, mx_tok_sf_bytes(M, 128, kbt) / 256, 256, 2, false)) return MOE_ERR_CUDA;
  if (!make_map_u8(&msb, sb, 256, mx_tok_sf_bytes(N, kMxBN, kbt) / 256, 256, 4, false)) return MOE_ERR_CUDA;
  if (!make_map_f32_3d(&mo, out, N, M, c.E)) return MOE_ERR_CUDA;
  const long long tiles = static_cast<long long>(c.E) * p.m_tiles_fixed * p.n_tiles;
  return cuda_status(launch_gemm(KIND_WGRAD_MX, p, ma, mb, msa,
                                 static_cast<int>(tiles < num_sms() ? tiles : num_sms()), s, &mo, &msb));
}

// NVFP4 grouped GEMM on quantised activations: y [R, N] = g_x g_e (Q(x) Q(W_e)),
// bf16 (fp32 with out_fp32)
static int run_gemm_nv(int E, long long R, int K, int N, const int32_t* offsets, const uint8_t* xq,
                       const uint8_t* sfx, const float* gx, const uint8_t* wq, const uint8_t* sf, const float* g,
                       void* y, DevStatus* st, cudaStream_t s, bool out_fp32 = false) {
  moe_config c{};
  c.T = 1; c.H = N; c.E = E; c.k = 1; c.F = K;
  GemmParams p = base_params(c, st);
  p.H = N;
  p.ngroups = E;
  p.offsets = offsets;
  p.M_total = static_cast<int>(R);
  p.bn = kNvTileN;
  p.n_tiles = (N + kNvTileN - 1) / kNvTileN;
  p.nt_w = p.n_tiles;
  p.kb_total = K / kNvKB;
  p.out0 = y;
  p.out_fp32 = out_fp32 ? 1 : 0;
  p.nv_ga = gx;
  p.nv_gb = g;
  CUtensorMap ma, mb, msa, msb, oy;
  if (!make_map_u8(&ma, xq, K / 2, R, 128, kBM)) return MOE_ERR_CUDA;
  if (!make_map_u8(&mb, wq, K / 2, static_cast<uint64_t>(E) * N, 128, kNvTileN / 2)) return MOE_ERR_CUDA;
  if (!make_map_u8(&msa, sfx, 256, nv_act_sf_bytes(R, E, K) / 256, 256, 8, false)) return MOE_ERR_CUDA;
  if (!make_map_u8(&msb, sf, 256, nv_weight_sf_bytes(E, K, N) / 256, 256, 16, false)) return MOE_ERR_CUDA;
  if (!make_map_store(&oy, y, N, R, out_fp32)) return MOE_ERR_CUDA;
  return cuda_status(launch_gemm(KIND_GEMM_NV, p, ma, mb, msa, num_sms(), s, &oy, &msb));
}

// NVFP4 layer: k blocks of 256 along H and F; bf16 intermediates (y_perm
// too); no shared expert
static int check_nv_layer_shape(const moe_config& c) {
  if (c.H % kNvKB != 0 || c.F % kNvKB != 0 || c.F_shared != 0 || c.inter_fp32 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  return MOE_OK;
}

}  // namespace moe

using namespace moe;

// ---------------------------------------------------------------------------
// exported C ABI
// ---------------------------------------------------------------------------
extern "C" {

size_t moe_workspace_bytes(const moe_config* cfg, int training) {
  if (check_cfg(cfg) != MOE_OK) return 0;
  return ws_layout(*cfg, training != 0).total;
}

size_t moe_abi_struct_bytes(int which) {
  return which == 0 ? sizeof(moe_config) : (which == 1 ? sizeof(moe_fwd_saved) : 0);
}

const char* moe_status_string(int s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE_TIMEOUT: return "device: bounded wait ran out";
    case MOE_ERR_DEVICE_INDEX: return "device: index out of range";
    default: return "unknown status";
  }
}

void moe_debug_set_wait_limit_ns(long long ns) { g_wait_limit_ns = ns > 0 ? static_cast<unsigned long long>(ns) : 2000000000ull; }
void moe_debug_set_fault(int fault) { g_fault = fault; }

void moe_profile_start(int capacity) {
  for (cudaEvent_t e : g_prof.ev) cudaEventDestroy(e);
  g_prof.ev.assign(capacity > 0 ? capacity : 0, nullptr);
  g_prof.tag.assign(g_prof.ev.size(), -1);
  for (auto& e : g_prof.ev) cudaEventCreate(&e);
  g_prof.n = 0;
  g_prof.on = true;
}

void moe_profile_stop(void) { g_prof.on = false; }

int moe_bounds_checked(void) { return kBoundsCheck ? 1 : 0; }

int moe_profile_read(int* tags, float* ms, int max) {
  const int n = g_prof.n < max ? g_prof.n : max;
  for (int i = 0; i < n; ++i) {
    if (cudaEventSynchronize(g_prof.ev[i]) != cudaSuccess) return -1;
    tags[i] = g_prof.tag[i];
    ms[i] = 0.0f;
    if (i > 0 && g_prof.tag[i] != STAGE_BEGIN) cudaEventElapsedTime(&ms[i], g_prof.ev[i - 1], g_prof.ev[i]);
  }
  return n;
}

unsigned long long moe_debug_launch_count(void) { return g_launches; }

size_t moe_debug_workspace_offset(const moe_config* cfg, int training, int which) {
  if (check_cfg(cfg) != MOE_OK) return static_cast<size_t>(-1);
  const WsLayout L = ws_layout(*cfg, training != 0);
  if (training == 0 && which != 2) return static_cast<size_t>(-1);
  switch (which) {
    case 0: return L.dy_perm;
    case 1: return L.dh13;
    case 2: return L.a;
    case 3: return L.dx_perm;
    default: return static_cast<size_t>(-1);
  }
}

int moe_get_device_status(void* ws, void* stream, int* status_out) {
  if (ws == nullptr || status_out == nullptr) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  MOE_CUDA(cudaStreamSynchronize(s));
  DevStatus h;
  MOE_CUDA(cudaMemcpy(&h, ws, sizeof(h), cudaMemcpyDeviceToHost));
  *status_out = h.status;
  MOE_CUDA(cudaMemset(ws, 0, sizeof(DevStatus)));
  return MOE_OK;
}

int moe_router_topk(const moe_config* cfg, const moe_bf16* x, const moe_bf16* router_w, const float* expert_bias,
                    const float* logit_bias, int32_t* topk_idx, float* topk_gate, float* logits_out,
                    float* aux_partials, void* ws, size_t ws_bytes, void* stream) {
  NvtxRange nvtx("moe_router_topk");
  MOE_TRY(check_cfg(cfg));
  const moe_config& c = *cfg;
  if (!x || !router_w || !topk_idx || !topk_gate || !ws) return MOE_ERR_INVALID_ARG;
  if (!all_aligned16({x, router_w, expert_bias, logit_bias, topk_idx, topk_gate, logits_out, aux_partials, ws}))
    return MOE_ERR_INVALID_ARG;
  if (ws_bytes < ws_layout(c, false).total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  MOE_TRY(run_router(c, reinterpret_cast<const __nv_bfloat16*>(x), reinterpret_cast<const __nv_bfloat16*>(router_w),
                     expert_bias, logit_bias, topk_idx, topk_gate, logits_out, aux_partials,
                     at<DevStatus>(ws, 0),
                     static_cast<cudaStream_t>(stream)));
  stage_done(static_cast<cudaStream_t>(stream), STAGE_ROUTER, 1);
  return MOE_OK;
}

int moe_permute(const moe_config* cfg, const moe_bf16* x, const int32_t* topk_idx, moe_bf16* x_perm,
                int32_t* row_id_map, int32_t* counts, int32_t* offsets, void* ws, size_t ws_bytes, void* stream) {
  NvtxRange nvtx("moe_permute");
  MOE_TRY(check_cfg(cfg));
  const moe_config& c = *cfg;
  if (!x || !topk_idx || !x_perm || !row_id_map || !counts || !offsets || !ws) return MOE_ERR_INVALID_ARG;
  if (!all_aligned16({x, topk_idx, x_perm, row_id_map, counts, offsets, ws})) return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(c, false);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  MOE_CUDA(launch_permute(c, reinterpret_cast<const __nv_bfloat16*>(x), topk_idx,
                          reinterpret_cast<__nv_bfloat16*>(x_perm), row_id_map, counts, offsets,
                          at<int32_t>(ws, L.lookback), at<DevStatus>(ws, 0), static_cast<cudaStream_t>(stream)));
  stage_done(static_cast<cudaStream_t>(stream), STAGE_PERMUTE, 2);
  return MOE_OK;
}

int moe_grouped_swiglu_ffn(const moe_config* cfg, const moe_bf16* x_perm, const int32_t* offsets,
                           const moe_bf16* W1, const moe_bf16* W3, const moe_bf16* W2, moe_bf16* h13_save,
                           moe_bf16* a_save, void* y_perm, void* ws, size_t ws_bytes, void* stream) {
  NvtxRange nvtx("moe_grouped_swiglu_ffn");
  MOE_TRY(check_cfg(cfg));
  const moe_config& c = *cfg;
  if (!x_perm || !offsets || !W1 || !W3 || !W2 || !y_perm || !ws) return MOE_ERR_INVALID_ARG;
  if (!all_aligned16({x_perm, offsets, W1, W3, W2, h13_save, a_save, y_perm, ws}))
    return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(c, false);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  __nv_bfloat16* a = a_save ? reinterpret_cast<__nv_bfloat16*>(a_save) : at<__nv_bfloat16>(ws, L.a);
  return run_ffn(c, c.F, c.E, offsets, c.T * c.k, reinterpret_cast<const __nv_bfloat16*>(x_perm),
                 reinterpret_cast<const __nv_bfloat16*>(W1), reinterpret_cast<const __nv_bfloat16*>(W3),
                 reinterpret_cast<const __nv_bfloat16*>(W2), reinterpret_cast<__nv_bfloat16*>(h13_save), a, y_perm,
                 c.inter_fp32 != 0, at<DevStatus>(ws, 0), static_cast<cudaStream_t>(stream));
}

int moe_unpermute_combine(const moe_config* cfg, const void* y_perm, const int32_t* row_id_map,
                          const float* topk_gate, const void* shared_out, void* y, void* stream) {
  NvtxRange nvtx("moe_unpermute_combine");
  MOE_TRY(check_cfg(cfg));
  const moe_config& c = *cfg;
  if (!y_perm || !row_id_map || !topk_gate || !y) return MOE_ERR_INVALID_ARG;
  if (!all_aligned16({y_perm, row_id_map, topk_gate, shared_out, y})) return MOE_ERR_INVALID_ARG;
  MOE_CUDA(launch_combine(c, y_perm, row_id_map, topk_gate, shared_out, y, static_cast<cudaStream_t>(stream)));
  stage_done(static_cast<cudaStream_t>(stream), STAGE_COMBINE, 1);
  return MOE_OK;
}

int moe_layer_fwd(const moe_config* cfg, const moe_bf16* x, const moe_bf16* router_w, const float* expert_bias,
                  const float* logit_bias, const moe_bf16* W1, const moe_bf16* W3, const moe_bf16* W2,
                  const moe_bf16* Ws1, const moe_bf16* Ws3, const moe_bf16* Ws2, void* y, const moe_fwd_saved* saved,
                  void* ws, size_t ws_bytes, void* stream) {
  NvtxRange nvtx("moe_layer_fwd");
  MOE_TRY(check_cfg(cfg));
  const moe_config& c = *cfg;
  if (!x || !router_w || !W1 || !W3 || !W2 || !y || !ws) return MOE_ERR_INVALID_ARG;
  if (c.F_shared && (!Ws1 || !Ws3 || !Ws2)) return MOE_ERR_INVALID_ARG;
  if (!all_aligned16({x, router_w, expert_bias, logit_bias, W1, W3, W2, Ws1, Ws3, Ws2, y, ws}) ||
      !saved_aligned16(saved))
    return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(c, false);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  DevStatus* st = at<DevStatus>(ws, 0);
  int32_t *idx, *rows, *counts, *offs;
  float *gate, *logits = nullptr, *aux = nullptr;
  __nv_bfloat16 *xp, *a, *h13 = nullptr;
  void* yp;
  if (saved != nullptr) {
    if (!saved->topk_idx || !saved->topk_gate || !saved->logits || !saved->row_id_map || !saved->counts ||
        !saved->offsets || !saved->x_perm || !saved->h13 || (!saved->a) != (!saved->y_perm))
      return MOE_ERR_INVALID_ARG;
    if (c.aux_coeff != 0.0f && !saved->aux_partials) return MOE_ERR_INVALID_ARG;
    if (c.F_shared && (!saved->h13_shared || !saved->a_shared)) return MOE_ERR_INVALID_ARG;
    idx = saved->topk_idx; gate = saved->topk_gate; logits = saved->logits; rows = saved->row_id_map;
    counts = saved->counts; offs = saved->offsets;
    xp = reinterpret_cast<__nv_bfloat16*>(saved->x_perm);
    h13 = reinterpret_cast<__nv_bfloat16*>(saved->h13);
    // memory-saving mode (a and y_perm NULL): both stay in the workspace
    a = saved->a ? reinterpret_cast<__nv_bfloat16*>(saved->a) : at<__nv_bfloat16>(ws, L.a);
    yp = saved->y_perm ? saved->y_perm : at<void>(ws, L.y_perm);
    aux = c.aux_coeff != 0.0f ? saved->aux_partials : nullptr;
  } else {
    idx = at<int32_t>(ws, L.topk_idx); gate = at<float>(ws, L.topk_gate); rows = at<int32_t>(ws, L.row_id_map);
    counts = at<int32_t>(ws, L.counts); offs = at<int32_t>(ws, L.offsets);
    xp = at<__nv_bfloat16>(ws, L.x_perm); a = at<__nv_bfloat16>(ws, L.a); yp = at<void>(ws, L.y_perm);
  }
  const __nv_bfloat16* xb = reinterpret_cast<const __nv_bfloat16*>(x);
  prof_mark(s, STAGE_BEGIN);
  MOE_TRY(run_router(c, xb, reinterpret_cast<const __nv_bfloat16*>(router_w), expert_bias, logit_bias, idx, gate,
                     logits, aux, st, s));
  stage_done(s, STAGE_ROUTER, 1);
  MOE_CUDA(launch_permute(c, xb, idx, xp, rows, counts, offs, at<int32_t>(ws, L.lookback), st, s));
  stage_done(s, STAGE_PERMUTE, 2);
  MOE_TRY(run_ffn(c, c.F, c.E, offs, c.T * c.k, xp, reinterpret_cast<const __nv_bfloat16*>(W1),
                  reinterpret_cast<const __nv_bfloat16*>(W3), reinterpret_cast<const __nv_bfloat16*>(W2), h13, a, yp,
                  c.inter_fp32 != 0, st, s, STAGE_FFN1, STAGE_FFN2));
  void* shared = nullptr;
  if (c.F_shared) {
    // training: the shared expert's pre-activations and activation are saved
    // for the backward
    shared = at<void>(ws, L.s_out);
    __nv_bfloat16* h13s = saved ? reinterpret_cast<__nv_bfloat16*>(saved->h13_shared) : nullptr;
    __nv_bfloat16* as = saved ? reinterpret_cast<__nv_bfloat16*>(saved->a_shared) : at<__nv_bfloat16>(ws, L.as);
    MOE_TRY(run_ffn(c, c.F_shared, 1, nullptr, c.T, xb, reinterpret_cast<const __nv_bfloat16*>(Ws1),
                    reinterpret_cast<const __nv_bfloat16*>(Ws3), reinterpret_cast<const __nv_bfloat16*>(Ws2), h13s, as,
                    shared, c.inter_fp32 != 0, st, s, STAGE_SHARED1, STAGE_SHARED2));
  }
  MOE_CUDA(launch_combine(c, yp, rows, gate, shared, y, s, st));
  stage_done(s, STAGE_COMBINE, 1);
  return MOE_OK;
}

// The layer backward after the checks. mx != nullptr: the backward of the
// MXFP8 training step (the data-gradient GEMMs on MXFP8 operands with the
// weights in mx; W1, W3, W2 unused); with mx_wgrad the weight gradients too
// (operands quantised along each expert's tokens).
// Backward of the shared expert S(x) = (SiLU(x Ws1) * (x Ws3)) Ws2, added
// ungated to every token (figures & tables page, Fig. 40): its output gradient
// is dO itself. Four GEMMs over the T tokens as one group:
//   da_s = dO Ws2^T -> SwiGLU backward with the saved h13_s -> dh13_s  (bf16)
//   dWs2 = a_s^T dO                                                    (fp32)
//   dx_s = dh13_s [Ws1 | Ws3]^T                          (bf16, fp32 with inter_fp32)
//   dWs1 | dWs3 = x^T dh13_s                                           (fp32)
// dx_s is added to dx by the permute backward.
static int shared_bwd(const moe_config& c, const __nv_bfloat16* dO, const __nv_bfloat16* x,
                      const __nv_bfloat16* Ws1, const __nv_bfloat16* Ws3, const __nv_bfloat16* Ws2,
                      const moe_fwd_saved* saved, float* dWs1, float* dWs3, float* dWs2, void* ws, const WsLayout& L,
                      cudaStream_t s) {
  DevStatus* st = at<DevStatus>(ws, 0);
  const int Fs = c.F_shared;
  __nv_bfloat16* dh13s = at<__nv_bfloat16>(ws, L.dh13_s);
  void* dxs = at<void>(ws, L.dx_s);
  uint8_t* slot = at<uint8_t>(ws, L.tmap_slots) + kTmapSlotBytes * c.E;  // after the routed experts' copies
  {
    GemmParams p = base_params(c, st);
    p.F = Fs; p.ngroups = 1; p.offsets = nullptr; p.M_total = c.T;
    p.n_tiles = (Fs + 255) / 256; p.kb_total = c.H / kBK;
    p.out0 = dh13s; p.in_aux = saved->h13_shared;
    CUtensorMap ma, mb, od;
    MOE_MAP(&ma, dO, c.H, c.T, 2ull * c.H, 64, 128);
    MOE_MAP(&mb, Ws2, c.H, Fs, 2ull * c.H, 64, 128);  // CTA pairs: 128 rows each
    if (!make_map_store(&od, dh13s, 2ull * Fs, c.T, false)) return MOE_ERR_CUDA;
    MOE_CUDA(launch_gemm(KIND_DGRAD2, p, ma, mb, mb, num_sms(), s, &od));
    stage_done(s, STAGE_SHARED_DGRAD2, 1);
  }
  {
    GemmParams p = base_params(c, st);
    p.ngroups = 1; p.offsets = nullptr; p.M_total = c.T;
    p.wg_M = Fs; p.wg_N = c.H; p.wg_mode = 0;
    p.tmap_slots = slot;
    p.m_tiles_fixed = (Fs + 255) / 256; p.n_tiles = (c.H + 255) / 256;
    p.out0 = dWs2;
    CUtensorMap ma, mb, mo;
    MOE_MAP(&ma, saved->a_shared, Fs, c.T, 2ull * Fs, 64, 64);
    MOE_MAP(&mb, dO, c.H, c.T, 2ull * c.H, 64, 64);
    if (!make_map_f32_3d(&mo, dWs2, c.H, Fs, 1)) return MOE_ERR_CUDA;
    const int tiles = p.m_tiles_fixed * p.n_tiles;
    MOE_CUDA(launch_tmap_rows(ma, nullptr, 1, slot, s, c.T));
    MOE_CUDA(launch_gemm(KIND_WGRAD, p, ma, mb, mb, tiles < num_sms() ? tiles : num_sms(), s, &mo, &mo));
    stage_done(s, STAGE_SHARED_WGRAD2, 2);
  }
  {
    GemmParams p = base_params(c, st);
    p.F = Fs; p.ngroups = 1; p.offsets = nullptr; p.M_total = c.T;
    p.n_tiles = (c.H + 255) / 256; p.kb_total = 2 * Fs / kBK;
    p.out0 = dxs;
    p.out_fp32 = c.inter_fp32;
    CUtensorMap ma, m1, m3, od;
    MOE_MAP(&ma, dh13s, 2ull * Fs, c.T, 4ull * Fs, 64, 128);
    MOE_MAP(&m1, Ws1, Fs, c.H, 2ull * Fs, 64, 128);  // CTA pairs: 128 rows each
    MOE_MAP(&m3, Ws3, Fs, c.H, 2ull * Fs, 64, 128);
    if (!make_map_store(&od, dxs, c.H, c.T, c.inter_fp32 != 0)) return MOE_ERR_CUDA;
    MOE_CUDA(launch_gemm(KIND_DGRAD1, p, ma, m1, m3, num_sms(), s, &od));
    stage_done(s, STAGE_SHARED_DGRAD1, 1);
  }
  {
    GemmParams p = base_params(c, st);
    p.ngroups = 1; p.offsets = nullptr; p.M_total = c.T;
    p.wg_M = c.H; p.wg_N = 2 * Fs; p.wg_mode = 1;
    p.tmap_slots = slot;
    p.m_tiles_fixed = (c.H + 255) / 256; p.n_tiles = (2 * Fs + 255) / 256;
    p.out0 = dWs1; p.out1 = dWs3;
    CUtensorMap ma, mb, mo1, mo3;
    MOE_MAP(&ma, x, c.H, c.T, 2ull * c.H, 64, 64);
    MOE_MAP(&mb, dh13s, 2ull * Fs, c.T, 4ull * Fs, 64, 64);
    if (!make_map_f32_3d(&mo1, dWs1, Fs, c.H, 1) || !make_map_f32_3d(&mo3, dWs3, Fs, c.H, 1)) return MOE_ERR_CUDA;
    const int tiles = p.m_tiles_fixed * p.n_tiles;
    MOE_CUDA(launch_tmap_rows(ma, nullptr, 1, slot, s, c.T));
    MOE_CUDA(launch_gemm(KIND_WGRAD, p, ma, mb, mb, tiles < num_sms() ? tiles : num_sms(), s, &mo1, &mo3));
    stage_done(s, STAGE_SHARED_WGRAD13, 2);
  }
  return MOE_OK;
}

static int layer_bwd_core(const moe_config& c, const moe_bf16* dO, const moe_bf16* x, const moe_bf16* router_w,
                          const moe_bf16* W1, const moe_bf16* W3, const moe_bf16* W2, const moe_fwd_saved* saved,
                          void* dx, float* dW_router, float* dW1, float* dW3, float* dW2, float* aux_loss_out,
                          void* ws, const WsLayout& L, const moe_mx_bwd_weights* mx, cudaStream_t s,
                          bool mx_wgrad = false, const moe_bf16* Ws1 = nullptr, const moe_bf16* Ws3 = nullptr,
                          const moe_bf16* Ws2 = nullptr, float* dWs1 = nullptr, float* dWs3 = nullptr,
                          float* dWs2 = nullptr, const moe_nv_bwd_weights* nv = nullptr) {
  // memory-saving backward: a recomputed from h13, gate gradient from the dgrad
  const bool recompute = mx == nullptr && saved->a == nullptr;
  DevStatus* st = at<DevStatus>(ws, 0);
  const int R = c.T * c.k;
  const int Ep = padded_experts(c.E);
  __nv_bfloat16* dy_perm = at<__nv_bfloat16>(ws, L.dy_perm);
  float* dgate = at<float>(ws, L.dgate);
  __nv_bfloat16* dh13 = at<__nv_bfloat16>(ws, L.dh13);
  __nv_bfloat16* dx_perm = at<__nv_bfloat16>(ws, L.dx_perm);
  // the bf16 backward keeps the per-row input gradients in fp32 with
  // inter_fp32 (layers whose activations reach magnitudes where one bf16
  // rounding exceeds the accuracy bar); the MXFP8 backward stores them in bf16
  const bool dxp32 = mx == nullptr && c.inter_fp32 != 0;
  __nv_bfloat16* dL_hl = at<__nv_bfloat16>(ws, L.dL_hl);
  float* dx_r = at<float>(ws, L.dx_r);
  float* dwr_part = at<float>(ws, L.dwr_part);

  prof_mark(s, STAGE_BEGIN);
  // 1. combine backward (memory-saving: dy_perm only; MXFP8: dy_perm also
  //    quantised, blocks of 32 along H)
  //    NVFP4: with the largest |dy_perm| for its tensor scale
  float* nv_dy_g = nv != nullptr ? at<float>(ws, L.nv_g) + 2 : nullptr;
  MOE_CUDA(launch_combine_bwd(c, reinterpret_cast<const __nv_bfloat16*>(dO), saved->y_perm, saved->row_id_map,
                              saved->topk_gate, dy_perm, dgate, s, mx ? at<uint8_t>(ws, L.dy_q) : nullptr,
                              mx ? at<uint8_t>(ws, L.sfa_dy) : nullptr, saved->offsets, saved->topk_idx, st, nv_dy_g));
  if (nv != nullptr) MOE_CUDA(launch_nv_scale_from_amax(nv_dy_g, 1, s));
  stage_done(s, STAGE_COMBINE_BWD, nv != nullptr ? 2 : 1);
  const int n_part = (c.F + 255) / 256;
  float* dg_part = at<float>(ws, L.dg_part);
  __nv_bfloat16* a_used =
      (recompute || mx != nullptr) ? at<__nv_bfloat16>(ws, L.a) : reinterpret_cast<__nv_bfloat16*>(saved->a);
  if (recompute) {
    // 3'. da = dy_perm W2_e^T: SwiGLU backward -> dh13, recomputed a -> workspace,
    //     gate-gradient partials <da, a> per row and 256-column tile
    GemmParams p = base_params(c, st);
    p.ngroups = c.E; p.offsets = saved->offsets; p.M_total = R;
    p.n_tiles = n_part; p.kb_total = c.H / kBK;
    p.out0 = dh13; p.in_aux = saved->h13; p.out1 = a_used; p.dg_part = dg_part; p.n_part = n_part;
    CUtensorMap ma, mb;
    MOE_MAP(&ma, dy_perm, c.H, R, 2ull * c.H, 64, 128);
    MOE_MAP(&mb, W2, c.H, static_cast<uint64_t>(c.E) * c.F, 2ull * c.H, 64, 128);  // CTA pairs: 128 rows each
    CUtensorMap od, oa;
    if (!make_map_store(&od, dh13, 2ull * c.F, R, false) || !make_map_store(&oa, a_used, c.F, R, false))
      return MOE_ERR_CUDA;
    MOE_CUDA(launch_gemm(KIND_DGRAD2R, p, ma, mb, mb, num_sms(), s, &od, &oa));
    stage_done(s, STAGE_DGRAD2, 1);
  }
  // 2. router backward (element-wise): dL as bf16 hi/lo
  MOE_CUDA(launch_router_bwd(c, saved->logits, saved->topk_idx, saved->topk_gate, dgate, recompute ? dg_part : nullptr,
                             n_part, saved->row_id_map, saved->counts, Ep, dL_hl, s, st));
  stage_done(s, STAGE_ROUTER_BWD, 1);
  // 3. da = dy_perm W2_e^T with the SwiGLU backward epilogue -> dh13
  if (nv != nullptr) {
    // NVFP4: dy_perm quantised as one tensor (blocks along H, the tensor
    // scale from the combine backward's maximum); da = Q(dy_perm)
    // Q(W2_e)^T in fp32; the SwiGLU backward -> dh13 (bf16) and its maximum;
    // dh13 quantised as one tensor (blocks along 2F) for step 5
    uint8_t* q = at<uint8_t>(ws, L.nv_q);
    uint8_t* sfq = at<uint8_t>(ws, L.nv_sf);
    float* gq = at<float>(ws, L.nv_g);
    float* da = at<float>(ws, L.nv_da);
    const int32_t* n_rows = saved->offsets + c.E;
    MOE_CUDA(launch_nv_quantize_grouped(dy_perm, R, c.H, c.E, saved->offsets, gq + 2, q, sfq, s));
    stage_done(s, STAGE_NV_QUANT, 1);
    MOE_TRY(run_gemm_nv(c.E, R, c.H, c.F, saved->offsets, q, sfq, gq + 2, nv->w2h, nv->sf2h, nv->g2h, da, st, s,
                        true));
    stage_done(s, STAGE_NV_DGRAD2, 1);
    MOE_CUDA(launch_nv_swiglu_bwd(da, reinterpret_cast<const __nv_bfloat16*>(saved->h13), R, c.F, n_rows, dh13,
                                  gq + 3, s));
    stage_done(s, STAGE_NV_SWIGLU_BWD, 2);
    MOE_CUDA(launch_nv_quantize_grouped(dh13, R, 2 * c.F, c.E, saved->offsets, gq + 3, q, sfq, s));
    stage_done(s, STAGE_NV_QUANT, 1);
  } else if (mx != nullptr) {
    // MXFP8: da = Q(dy_perm) Q(W2_e)^T with the SwiGLU backward in the GEMM's
    // epilogue -> dh13 bf16, a (for dW2) and the E4M3 rows of dh13 (blocks
    // along 2F)
    MOE_TRY(run_dgrad2_mx(c, saved->offsets, R, at<uint8_t>(ws, L.dy_q), at<uint8_t>(ws, L.sfa_dy), *mx,
                          reinterpret_cast<const __nv_bfloat16*>(saved->h13), dh13, a_used, at<uint8_t>(ws, L.dh_q),
                          at<uint8_t>(ws, L.sfa_dh), st, s));
    stage_done(s, STAGE_MX_DGRAD2, 1);
  } else if (!recompute) {
    GemmParams p = base_params(c, st);
    p.ngroups = c.E; p.offsets = saved->offsets; p.M_total = R;
    p.n_tiles = (c.F + 255) / 256; p.kb_total = c.H / kBK;
    p.out0 = dh13; p.in_aux = saved->h13;
    CUtensorMap ma, mb;
    MOE_MAP(&ma, dy_perm, c.H, R, 2ull * c.H, 64, 128);
    MOE_MAP(&mb, W2, c.H, static_cast<uint64_t>(c.E) * c.F, 2ull * c.H, 64, 128);  // CTA pairs: 128 rows each
    CUtensorMap od;
    if (!make_map_store(&od, dh13, 2ull * c.F, R, false)) return MOE_ERR_CUDA;
    MOE_CUDA(launch_gemm(KIND_DGRAD2, p, ma, mb, mb, num_sms(), s, &od));
    stage_done(s, STAGE_DGRAD2, 1);
  }
  // 4. dW2_e = a_e^T dy_perm_e
  if (mx != nullptr && mx_wgrad) {
    // MXFP8: both operands quantised along the expert's tokens
    MOE_TRY(run_wgrad_mx(c, saved->offsets, R, a_used, c.F, c.F, dy_perm, c.H, c.H, dW2, ws, L, st, s));
    stage_done(s, STAGE_WGRAD2, 1);
  } else {
    GemmParams p = base_params(c, st);
    p.ngroups = c.E; p.offsets = saved->offsets;
    p.wg_M = c.F; p.wg_N = c.H; p.wg_mode = 0;
    p.tmap_slots = at<uint8_t>(ws, L.tmap_slots);
    p.m_tiles_fixed = (c.F + 255) / 256; p.n_tiles = (c.H + 255) / 256;  // CTA-pair tiles of 256 rows
    p.out0 = dW2;
    CUtensorMap ma, mb;
    MOE_MAP(&ma, a_used, c.F, R, 2ull * c.F, 64, 64);
    MOE_MAP(&mb, dy_perm, c.H, R, 2ull * c.H, 64, 64);
    CUtensorMap mo;
    if (!make_map_f32_3d(&mo, dW2, c.H, c.F, c.E)) return MOE_ERR_CUDA;
    const long long tiles = static_cast<long long>(c.E) * p.m_tiles_fixed * p.n_tiles;
    MOE_CUDA(launch_tmap_rows(ma, saved->offsets, c.E, p.tmap_slots, s));
    MOE_CUDA(launch_gemm(KIND_WGRAD, p, ma, mb, mb, static_cast<int>(tiles < num_sms() ? tiles : num_sms()), s,
                         &mo, &mo));
    stage_done(s, STAGE_WGRAD2, 2);
  }
  // 5. dx_perm = dh13 [W1_e | W3_e]^T
  if (nv != nullptr) {
    MOE_TRY(run_gemm_nv(c.E, R, 2 * c.F, c.H, saved->offsets, at<uint8_t>(ws, L.nv_q), at<uint8_t>(ws, L.nv_sf),
                        at<float>(ws, L.nv_g) + 3, nv->w13f, nv->sf13f, nv->g13f, dx_perm, st, s));
    stage_done(s, STAGE_NV_DGRAD1, 1);
  } else if (mx != nullptr) {
    MOE_TRY(run_gemm_mx(c, saved->offsets, R, 2 * c.F, c.H, at<uint8_t>(ws, L.dh_q), at<uint8_t>(ws, L.sfa_dh),
                        mx->w13f, mx->sf13f, mx_sf13f_bytes(c), dx_perm, st, s));
    stage_done(s, STAGE_MX_DGRAD1, 1);
  } else {
    GemmParams p = base_params(c, st);
    p.ngroups = c.E; p.offsets = saved->offsets; p.M_total = R;
    p.n_tiles = (c.H + 255) / 256; p.kb_total = 2 * c.F / kBK;
    p.out0 = dx_perm;
    p.out_fp32 = dxp32;
    CUtensorMap ma, m1, m3;
    MOE_MAP(&ma, dh13, 2ull * c.F, R, 4ull * c.F, 64, 128);
    MOE_MAP(&m1, W1, c.F, static_cast<uint64_t>(c.E) * c.H, 2ull * c.F, 64, 128);  // CTA pairs: 128 rows each
    MOE_MAP(&m3, W3, c.F, static_cast<uint64_t>(c.E) * c.H, 2ull * c.F, 64, 128);
    CUtensorMap od;
    if (!make_map_store(&od, dx_perm, c.H, R, dxp32)) return MOE_ERR_CUDA;
    MOE_CUDA(launch_gemm(KIND_DGRAD1, p, ma, m1, m3, num_sms(), s, &od));
    stage_done(s, STAGE_DGRAD1, 1);
  }
  // 6. dW1_e | dW3_e = x_perm_e^T dh13_e
  if (mx != nullptr && mx_wgrad) {
    // MXFP8: dW1 from dh1 (columns [0, F) of dh13), then dW3 from dh3 with
    // the quantised x_perm kept
    const __nv_bfloat16* xp = reinterpret_cast<const __nv_bfloat16*>(saved->x_perm);
    MOE_TRY(run_wgrad_mx(c, saved->offsets, R, xp, c.H, c.H, dh13, c.F, 2 * c.F, dW1, ws, L, st, s));
    stage_done(s, STAGE_WGRAD13, 1);
    MOE_TRY(run_wgrad_mx(c, saved->offsets, R, xp, c.H, c.H, dh13 + c.F, c.F, 2 * c.F, dW3, ws, L, st, s, false));
    stage_done(s, STAGE_WGRAD13, 1);
  } else {
    GemmParams p = base_params(c, st);
    p.ngroups = c.E; p.offsets = saved->offsets;
    p.wg_M = c.H; p.wg_N = 2 * c.F; p.wg_mode = 1;
    p.tmap_slots = at<uint8_t>(ws, L.tmap_slots);
    p.m_tiles_fixed = (c.H + 255) / 256; p.n_tiles = (2 * c.F + 255) / 256;  // CTA-pair tiles of 256 rows
    p.out0 = dW1; p.out1 = dW3;
    CUtensorMap ma, mb;
    MOE_MAP(&ma, saved->x_perm, c.H, R, 2ull * c.H, 64, 64);
    MOE_MAP(&mb, dh13, 2ull * c.F, R, 4ull * c.F, 64, 64);
    CUtensorMap mo1, mo3;
    if (!make_map_f32_3d(&mo1, dW1, c.F, c.H, c.E) || !make_map_f32_3d(&mo3, dW3, c.F, c.H, c.E))
      return MOE_ERR_CUDA;
    const long long tiles = static_cast<long long>(c.E) * p.m_tiles_fixed * p.n_tiles;
    MOE_CUDA(launch_tmap_rows(ma, saved->offsets, c.E, p.tmap_slots, s));
    MOE_CUDA(launch_gemm(KIND_WGRAD, p, ma, mb, mb, static_cast<int>(tiles < num_sms() ? tiles : num_sms()), s,
                         &mo1, &mo3));
    stage_done(s, STAGE_WGRAD13, 2);
  }
  // 7. router part of dx: dx_r = dL W_r (fp32)
  {
    GemmParams p = base_params(c, st);
    p.ngroups = 1; p.offsets = nullptr; p.M_total = c.T;
    p.n_tiles = (c.H + 255) / 256; p.kb_total = 2 * Ep / kBK; p.Ep = Ep;
    p.out0 = dx_r;
    CUtensorMap ma, mb;
    MOE_MAP(&ma, dL_hl, 2ull * Ep, c.T, 4ull * Ep, 64, 128);
    MOE_MAP(&mb, router_w, c.H, c.E, 2ull * c.H, 64, 64);
    const int tiles = ((c.T + kBM - 1) / kBM) * p.n_tiles;
    CUtensorMap od;
    if (!make_map_store(&od, dx_r, c.H, c.T, true)) return MOE_ERR_CUDA;
    MOE_CUDA(launch_gemm(KIND_ROUTER_DX, p, ma, mb, mb, tiles < num_sms() ? tiles : num_sms(), s, &od));
    stage_done(s, STAGE_ROUTER_DX, 1);
  }
  // 7'. the shared expert's backward (its input gradient dx_s in the workspace)
  const bool shared = c.F_shared != 0 && mx == nullptr;
  if (shared) {
    MOE_TRY(shared_bwd(c, reinterpret_cast<const __nv_bfloat16*>(dO), reinterpret_cast<const __nv_bfloat16*>(x),
                       reinterpret_cast<const __nv_bfloat16*>(Ws1), reinterpret_cast<const __nv_bfloat16*>(Ws3),
                       reinterpret_cast<const __nv_bfloat16*>(Ws2), saved, dWs1, dWs3, dWs2, ws, L, s));
  }
  // 8. dx = sum_i dx_perm[row(t,i)] + dx_r (+ dx_s)
  MOE_CUDA(launch_unpermute_sum(c, dx_perm, saved->row_id_map, dx_r, dx, s,
                                shared ? at<void>(ws, L.dx_s) : nullptr, dxp32, st));
  stage_done(s, STAGE_UNPERMUTE, 1);
  // 9. dW_r = dL^T x (each token block: dL's hi and lo parts against one box
  // of x), split over the token blocks, then reduced in split order; as many
  // splits as keep one wave of tiles on the SMs
  {
    const int m_tiles = (c.E + 127) / 128, n_tiles = (c.H + 255) / 256;
    int splits = num_sms() / (m_tiles * n_tiles);
    if (splits > router_dw_splits(c.T)) splits = router_dw_splits(c.T);
    if (splits < 1) splits = 1;
    const int total_kb = (c.T + kBK - 1) / kBK;
    GemmParams p = base_params(c, st);
    p.ngroups = splits; p.offsets = nullptr; p.splits = splits;
    p.kb_total = (total_kb + splits - 1) / splits;
    p.m_tiles_fixed = m_tiles; p.n_tiles = n_tiles; p.Ep = Ep;
    p.out0 = dwr_part;
    CUtensorMap ma, mb;
    MOE_MAP(&ma, dL_hl, 2ull * Ep, c.T, 4ull * Ep, 64, 64);
    MOE_MAP(&mb, x, c.H, c.T, 2ull * c.H, 64, 64);
    const int tiles = splits * p.m_tiles_fixed * p.n_tiles;
    CUtensorMap od;
    if (!make_map_f32_3d(&od, dwr_part, c.H, c.E, splits)) return MOE_ERR_CUDA;
    MOE_CUDA(launch_gemm(KIND_ROUTER_DW, p, ma, mb, mb, tiles < num_sms() ? tiles : num_sms(), s, &od));
    MOE_CUDA(launch_split_reduce(dwr_part, splits, static_cast<size_t>(c.E) * c.H, dW_router, s));
    stage_done(s, STAGE_ROUTER_DW, 2);
  }
  // 10. aux loss value
  if (c.aux_coeff != 0.0f && aux_loss_out != nullptr) {
    MOE_CUDA(launch_aux_loss(c, saved->aux_partials, saved->counts, aux_loss_out, s));
    stage_done(s, STAGE_AUX, 1);
  }
  return MOE_OK;
}

int moe_layer_bwd(const moe_config* cfg, const moe_bf16* dO, const moe_bf16* x, const moe_bf16* router_w,
                  const moe_bf16* W1, const moe_bf16* W3, const moe_bf16* W2, const moe_bf16* Ws1,
                  const moe_bf16* Ws3, const moe_bf16* Ws2, const moe_fwd_saved* saved, void* dx, float* dW_router,
                  float* dW1, float* dW3, float* dW2, float* dWs1, float* dWs3, float* dWs2, float* aux_loss_out,
                  void* ws, size_t ws_bytes, void* stream) {
  NvtxRange nvtx("moe_layer_bwd");
  MOE_TRY(check_cfg(cfg));
  const moe_config& c = *cfg;
  if (!dO || !x || !router_w || !W1 || !W3 || !W2 || !saved || !dx || !dW_router || !dW1 || !dW3 || !dW2 || !ws)
    return MOE_ERR_INVALID_ARG;
  if (!all_aligned16({dO, x, router_w, W1, W3, W2, Ws1, Ws3, Ws2, dx, dW_router, dW1, dW3, dW2, dWs1, dWs3, dWs2,
                      aux_loss_out, ws}) ||
      !saved_aligned16(saved))
    return MOE_ERR_INVALID_ARG;
  if (!saved->topk_idx || !saved->topk_gate || !saved->logits || !saved->row_id_map || !saved->counts ||
      !saved->offsets || !saved->x_perm || !saved->h13 || (!saved->a) != (!saved->y_perm))
    return MOE_ERR_INVALID_ARG;
  if (c.aux_coeff != 0.0f && !saved->aux_partials) return MOE_ERR_INVALID_ARG;
  if (c.F_shared != 0) {
    if (!Ws1 || !Ws3 || !Ws2 || !dWs1 || !dWs3 || !dWs2 || !saved->h13_shared || !saved->a_shared)
      return MOE_ERR_INVALID_ARG;
  }
  const WsLayout L = ws_layout(c, true);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  return layer_bwd_core(c, dO, x, router_w, W1, W3, W2, saved, dx, dW_router, dW1, dW3, dW2, aux_loss_out, ws, L,
                        nullptr, static_cast<cudaStream_t>(stream), false, Ws1, Ws3, Ws2, dWs1, dWs3, dWs2);
}

// ---------------------------------------------------------------------------
// MXFP8 forward
// ---------------------------------------------------------------------------
size_t moe_mx_weight_bytes(const moe_config* cfg, int which) {
  if (check_cfg(cfg) != MOE_OK || check_mx_shape(*cfg) != MOE_OK) return 0;
  const moe_config& c = *cfg;
  switch (which) {
    case 0: return 2ull * c.E * c.F * c.H;
    case 1: return mx_sf13_bytes(c);
    case 2: return static_cast<size_t>(c.E) * c.H * c.F;
    case 3: return mx_sf2_bytes(c);
    default: return 0;
  }
}

int moe_mx_quantize_weights(const moe_config* cfg, const moe_bf16* W1, const moe_bf16* W3, const moe_bf16* W2,
                            const moe_mx_weights* w, void* stream) {
  NvtxRange nvtx("moe_mx_quantize_weights");
  MOE_TRY(check_cfg(cfg));
  MOE_TRY(check_mx_shape(*cfg));
  if (!W1 || !W3 || !W2 || !w || !w->w13 || !w->sf13 || !w->w2 || !w->sf2) return MOE_ERR_INVALID_ARG;
  if (!all_aligned16({W1, W3, W2, w->w13, w->sf13, w->w2, w->sf2}))
    return MOE_ERR_INVALID_ARG;
  MOE_CUDA(launch_mx_quantize_weights(*cfg, reinterpret_cast<const __nv_bfloat16*>(W1),
                                      reinterpret_cast<const __nv_bfloat16*>(W3),
                                      reinterpret_cast<const __nv_bfloat16*>(W2), w->w13, w->sf13, w->w2, w->sf2,
                                      static_cast<cudaStream_t>(stream)));
  count_launches(3);
  return MOE_OK;
}

int moe_mx_quantize(const moe_bf16* x, long long M, int K, uint8_t* q, uint8_t* scales, void* stream) {
  NvtxRange nvtx("moe_mx_quantize");
  if (!x || !q || !scales || M < 0 || K < kMxBlock || K % kMxBlock != 0) return MOE_ERR_INVALID_ARG;
  if (!all_aligned16({x, q, scales})) return MOE_ERR_INVALID_ARG;
  MOE_CUDA(launch_mx_quantize_rows(reinterpret_cast<const __nv_bfloat16*>(x), M, K, q, scales,
                                   static_cast<cudaStream_t>(stream)));
  count_launches(M > 0 ? 1 : 0);
  return MOE_OK;
}

size_t moe_mx_workspace_bytes(const moe_config* cfg) {
  if (check_cfg(cfg) != MOE_OK || check_mx_shape(*cfg) != MOE_OK) return 0;
  return ws_layout(*cfg, false, true).total;
}

int moe_layer_fwd_mxfp8(const moe_config* cfg, const moe_bf16* x, const moe_bf16* router_w,
                        const float* expert_bias, const float* logit_bias, const moe_mx_weights* w,
                        const moe_bf16* Ws1, const moe_bf16* Ws3, const moe_bf16* Ws2, void* y, void* ws,
                        size_t ws_bytes, void* stream) {
  NvtxRange nvtx("moe_layer_fwd_mxfp8");
  MOE_TRY(check_cfg(cfg));
  const moe_config& c = *cfg;
  MOE_TRY(check_mx_shape(c));
  if (!x || !router_w || !w || !w->w13 || !w->sf13 || !w->w2 || !w->sf2 || !y || !ws) return MOE_ERR_INVALID_ARG;
  if (c.F_shared && (!Ws1 || !Ws3 || !Ws2)) return MOE_ERR_INVALID_ARG;
  if (!all_aligned16({x, router_w, expert_bias, logit_bias, w->w13, w->sf13, w->w2, w->sf2, Ws1, Ws3, Ws2, y,
                      ws}))
    return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(c, false, true);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  DevStatus* st = at<DevStatus>(ws, 0);
  int32_t* idx = at<int32_t>(ws, L.topk_idx);
  float* gate = at<float>(ws, L.topk_gate);
  int32_t* rows = at<int32_t>(ws, L.row_id_map);
  int32_t* counts = at<int32_t>(ws, L.counts);
  int32_t* offs = at<int32_t>(ws, L.offsets);
  uint8_t* x_q = at<uint8_t>(ws, L.x_q);
  uint8_t* sfa1 = at<uint8_t>(ws, L.sfa1);
  uint8_t* a_q = at<uint8_t>(ws, L.a_q);
  uint8_t* sfa2 = at<uint8_t>(ws, L.sfa2);
  void* yp = at<void>(ws, L.y_perm);
  const __nv_bfloat16* xb = reinterpret_cast<const __nv_bfloat16*>(x);
  prof_mark(s, STAGE_BEGIN);
  MOE_TRY(run_router(c, xb, reinterpret_cast<const __nv_bfloat16*>(router_w), expert_bias, logit_bias, idx, gate,
                     nullptr, nullptr, st, s));
  stage_done(s, STAGE_ROUTER, 1);
  MOE_CUDA(launch_permute(c, xb, idx, nullptr, rows, counts, offs, at<int32_t>(ws, L.lookback), st, s, x_q, sfa1));
  stage_done(s, STAGE_PERMUTE, 2);
  MOE_TRY(run_ffn_mx(c, offs, c.T * c.k, x_q, sfa1, *w, a_q, sfa2, yp, c.inter_fp32 != 0, st, s));
  void* shared = nullptr;
  if (c.F_shared) {
    shared = at<void>(ws, L.s_out);
    MOE_TRY(run_ffn(c, c.F_shared, 1, nullptr, c.T, xb, reinterpret_cast<const __nv_bfloat16*>(Ws1),
                    reinterpret_cast<const __nv_bfloat16*>(Ws3), reinterpret_cast<const __nv_bfloat16*>(Ws2), nullptr,
                    at<__nv_bfloat16>(ws, L.as), shared, c.inter_fp32 != 0, st, s, STAGE_SHARED1, STAGE_SHARED2));
  }
  MOE_CUDA(launch_combine(c, yp, rows, gate, shared, y, s, st));
  stage_done(s, STAGE_COMBINE, 1);
  return MOE_OK;
}

// ---------------------------------------------------------------------------
// MXFP8 training step
// ---------------------------------------------------------------------------
size_t moe_mx_bwd_weight_bytes(const moe_config* cfg, int which) {
  if (check_cfg(cfg) != MOE_OK || check_mx_shape(*cfg) != MOE_OK) return 0;
  const moe_config& c = *cfg;
  switch (which) {
    case 0: return static_cast<size_t>(c.E) * c.F * c.H;
    case 1: return mx_sf2h_bytes(c);
    case 2: return 2ull * c.E * c.H * c.F;
    case 3: return mx_sf13f_bytes(c);
    default: return 0;
  }
}

int moe_mx_quantize_bwd_weights(const moe_config* cfg, const moe_bf16* W1, const moe_bf16* W3, const moe_bf16* W2,
                                const moe_mx_bwd_weights* w, void* stream) {
  NvtxRange nvtx("moe_mx_quantize_bwd_weights");
  MOE_TRY(check_cfg(cfg));
  MOE_TRY(check_mx_shape(*cfg));
  if (!W1 || !W3 || !W2 || !w || !w->w2h || !w->sf2h || !w->w13f || !w->sf13f) return MOE_ERR_INVALID_ARG;
  if (!all_aligned16({W1, W3, W2, w->w2h, w->sf2h, w->w13f, w->sf13f}))
    return MOE_ERR_INVALID_ARG;
  MOE_CUDA(launch_mx_quantize_bwd_weights(*cfg, reinterpret_cast<const __nv_bfloat16*>(W1),
                                          reinterpret_cast<const __nv_bfloat16*>(W3),
                                          reinterpret_cast<const __nv_bfloat16*>(W2), w->w2h, w->sf2h, w->w13f,
                                          w->sf13f, static_cast<cudaStream_t>(stream)));
  count_launches(3);
  return MOE_OK;
}

size_t moe_mx_train_workspace_bytes(const moe_config* cfg) {
  if (check_cfg(cfg) != MOE_OK || check_mx_shape(*cfg) != MOE_OK || cfg->F_shared != 0) return 0;
  return ws_layout(*cfg, true, true).total;
}

static bool mx_saved_ok(const moe_config& c, const moe_fwd_saved* sv) {
  return sv && sv->topk_idx && sv->topk_gate && sv->logits && sv->row_id_map && sv->counts && sv->offsets &&
         sv->x_perm && sv->h13 && sv->y_perm && (c.aux_coeff == 0.0f || sv->aux_partials) &&
         saved_aligned16(sv);
}

int moe_layer_fwd_mxfp8_train(const moe_config* cfg, const moe_bf16* x, const moe_bf16* router_w,
                              const float* expert_bias, const float* logit_bias, const moe_mx_weights* w, void* y,
                              const moe_fwd_saved* saved, void* ws, size_t ws_bytes, void* stream) {
  NvtxRange nvtx("moe_layer_fwd_mxfp8_train");
  MOE_TRY(check_cfg(cfg));
  const moe_config& c = *cfg;
  MOE_TRY(check_mx_shape(c));
  if (c.F_shared != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!x || !router_w || !w || !w->w13 || !w->sf13 || !w->w2 || !w->sf2 || !y || !ws || !mx_saved_ok(c, saved))
    return MOE_ERR_INVALID_ARG;
  if (!all_aligned16({x, router_w, expert_bias, logit_bias, w->w13, w->sf13, w->w2, w->sf2, y, ws}))
    return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(c, true, true);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  DevStatus* st = at<DevStatus>(ws, 0);
  const moe_fwd_saved& sv = *saved;
  uint8_t* x_q = at<uint8_t>(ws, L.x_q);
  uint8_t* sfa1 = at<uint8_t>(ws, L.sfa1);
  const __nv_bfloat16* xb = reinterpret_cast<const __nv_bfloat16*>(x);
  prof_mark(s, STAGE_BEGIN);
  MOE_TRY(run_router(c, xb, reinterpret_cast<const __nv_bfloat16*>(router_w), expert_bias, logit_bias, sv.topk_idx,
                     sv.topk_gate, sv.logits, c.aux_coeff != 0.0f ? sv.aux_partials : nullptr,
                     st, s));
  stage_done(s, STAGE_ROUTER, 1);
  MOE_CUDA(launch_permute(c, xb, sv.topk_idx, reinterpret_cast<__nv_bfloat16*>(sv.x_perm), sv.row_id_map, sv.counts,
                          sv.offsets, at<int32_t>(ws, L.lookback), st, s, x_q, sfa1));
  stage_done(s, STAGE_PERMUTE, 2);
  MOE_TRY(run_ffn_mx(c, sv.offsets, c.T * c.k, x_q, sfa1, *w, at<uint8_t>(ws, L.a_q), at<uint8_t>(ws, L.sfa2),
                     sv.y_perm, c.inter_fp32 != 0, st, s, reinterpret_cast<__nv_bfloat16*>(sv.h13)));
  MOE_CUDA(launch_combine(c, sv.y_perm, sv.row_id_map, sv.topk_gate, nullptr, y, s, st));
  stage_done(s, STAGE_COMBINE, 1);
  return MOE_OK;
}

int moe_layer_bwd_mxfp8(const moe_config* cfg, const moe_bf16* dO, const moe_bf16* x, const moe_bf16* router_w,
                        const moe_mx_bwd_weights* w, const moe_fwd_saved* saved, void* dx, float* dW_router,
                        float* dW1, float* dW3, float* dW2, float* aux_loss_out, int mx_wgrad, void* ws,
                        size_t ws_bytes, void* stream) {
  NvtxRange nvtx("moe_layer_bwd_mxfp8");
  MOE_TRY(check_cfg(cfg));
  const moe_config& c = *cfg;
  MOE_TRY(check_mx_shape(c));
  if (c.F_shared != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!dO || !x || !router_w || !w || !w->w2h || !w->sf2h || !w->w13f || !w->sf13f || !mx_saved_ok(c, saved) ||
      !dx || !dW_router || !dW1 || !dW3 || !dW2 || !ws)
    return MOE_ERR_INVALID_ARG;
  if (!all_aligned16({dO, x, router_w, w->w2h, w->sf2h, w->w13f, w->sf13f, dx, dW_router, dW1, dW3, dW2,
                      aux_loss_out, ws}))
    return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(c, true, true);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  return layer_bwd_core(c, dO, x, router_w, nullptr, nullptr, nullptr, saved, dx, dW_router, dW1, dW3, dW2,
                        aux_loss_out, ws, L, w, static_cast<cudaStream_t>(stream), mx_wgrad != 0);
}

// ---------------------------------------------------------------------------
// NVFP4 grouped expert GEMM
// ---------------------------------------------------------------------------
static int check_nv_shape(int E, long long R, int K, int N) {
  if (E < 1 || R < 0 || K < 1 || N < 1) return MOE_ERR_INVALID_ARG;
  if (E > kMaxGroups || K % kNvKB != 0 || N % 8 != 0 || R >= (1ll << 30)) return MOE_ERR_UNSUPPORTED_SHAPE;
  return MOE_OK;
}

size_t moe_nv_weight_bytes(int E, int K, int N, int which) {
  if (check_nv_shape(E, 0, K, N) != MOE_OK) return 0;
  switch (which) {
    case 0: return static_cast<size_t>(E) * N * (K / 2);
    case 1: return nv_weight_sf_bytes(E, K, N);
    case 2: return sizeof(float) * E;
    default: return 0;
  }
}

int moe_nv_quantize_weights(int E, int K, int N, const moe_bf16* W, uint8_t* wq, uint8_t* sf, float* g,
                            void* stream) {
  NvtxRange nvtx("moe_nv_quantize_weights");
  MOE_TRY(check_nv_shape(E, 0, K, N));
  if (!W || !wq || !sf || !g || !all_aligned16({W, wq, sf, g})) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const __nv_bfloat16* w = reinterpret_cast<const __nv_bfloat16*>(W);
  MOE_CUDA(launch_nv_amax(w, static_cast<long long>(K) * N, E, g, s));
  MOE_CUDA(launch_nv_quantize_weights(w, E, K, N, g, wq, sf, s));
  count_launches(3);
  return MOE_OK;
}

int moe_nv_quantize(const moe_bf16* x, long long M, int K, uint8_t* q, uint8_t* scales, float* g, void* stream) {
  NvtxRange nvtx("moe_nv_quantize");
  if (!x || !q || !scales || !g || M < 1 || K < kNvBlock || K % kNvBlock != 0) return MOE_ERR_INVALID_ARG;
  if (!all_aligned16({x, q, scales, g}) || (M * K) % 8 != 0) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const __nv_bfloat16* xb = reinterpret_cast<const __nv_bfloat16*>(x);
  MOE_CUDA(launch_nv_amax(xb, M * K, 1, g, s));
  MOE_CUDA(launch_nv_quantize_rows(xb, M, K, g, q, scales, s));
  count_launches(3);
  return MOE_OK;
}

struct NvWs {
  size_t status, g, xq, sf, total;
};
static NvWs nv_ws_layout(int E, long long R, int K) {
  NvWs L{};
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o += align256(bytes);
    return at;
  };
  L.status = take(sizeof(DevStatus));
  L.g = take(sizeof(float));
  L.xq = take(static_cast<size_t>(R) * (K / 2));
  L.sf = take(nv_act_sf_bytes(R, E, K));
  L.total = o;
  return L;
}

size_t moe_nv_workspace_bytes(int E, long long R, int K) {
  if (check_nv_shape(E, R, K, 8) != MOE_OK) return 0;
  return nv_ws_layout(E, R, K).total;
}

int moe_nv_grouped_gemm(int E, long long R, int K, int N, const moe_bf16* x, const int32_t* offsets,
                        const uint8_t* wq, const uint8_t* sf, const float* g, moe_bf16* y, void* ws,
                        size_t ws_bytes, void* stream) {
  NvtxRange nvtx("moe_nv_grouped_gemm");
  MOE_TRY(check_nv_shape(E, R, K, N));
  if (!x || !offsets || !wq || !sf || !g || !y || !ws) return MOE_ERR_INVALID_ARG;
  if (!all_aligned16({x, offsets, wq, sf, g, y, ws}))
    return MOE_ERR_INVALID_ARG;
  const NvWs L = nv_ws_layout(E, R, K);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (R == 0) return MOE_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  DevStatus* st = at<DevStatus>(ws, L.status);
  float* gx = at<float>(ws, L.g);
  uint8_t* xq = at<uint8_t>(ws, L.xq);
  uint8_t* sfx = at<uint8_t>(ws, L.sf);
  const __nv_bfloat16* xb = reinterpret_cast<const __nv_bfloat16*>(x);
  prof_mark(s, STAGE_BEGIN);
  MOE_CUDA(launch_nv_amax(xb, R * K, 1, gx, s));
  MOE_CUDA(launch_nv_quantize_grouped(xb, static_cast<int>(R), K, E, offsets, gx, xq, sfx, s));
  stage_done(s, STAGE_NV_QUANT, 3);
  MOE_TRY(run_gemm_nv(E, R, K, N, offsets, xq, sfx, gx, wq, sf, g, reinterpret_cast<__nv_bfloat16*>(y), st, s));
  stage_done(s, STAGE_NV_GEMM, 1);
  return MOE_OK;
}

// ---------------------------------------------------------------------------
// NVFP4 layer forward
// ---------------------------------------------------------------------------
size_t moe_nv_layer_weight_bytes(const moe_config* cfg, int which) {
  if (check_cfg(cfg) != MOE_OK || check_nv_layer_shape(*cfg) != MOE_OK) return 0;
  const moe_config& c = *cfg;
  switch (which) {
    case 0: return moe_nv_weight_bytes(c.E, c.H, 2 * c.F, 0);
    case 1: return nv_weight_sf_bytes_gu(c.E, c.H, c.F);
    case 2: return moe_nv_weight_bytes(c.E, c.H, 2 * c.F, 2);
    case 3: return moe_nv_weight_bytes(c.E, c.F, c.H, 0);
    case 4: return moe_nv_weight_bytes(c.E, c.F, c.H, 1);
    case 5: return moe_nv_weight_bytes(c.E, c.F, c.H, 2);
    default: return 0;
  }
}

int moe_nv_quantize_layer_weights(const moe_config* cfg, const moe_bf16* W1, const moe_bf16* W3, const moe_bf16* W2,
                                  const moe_nv_weights* w, void* stream) {
  NvtxRange nvtx("moe_nv_quantize_layer_weights");
  MOE_TRY(check_cfg(cfg));
  const moe_config& c = *cfg;
  MOE_TRY(check_nv_layer_shape(c));
  if (!W1 || !W3 || !W2 || !w || !w->w13 || !w->sf13 || !w->g13 || !w->w2 || !w->sf2 || !w->g2)
    return MOE_ERR_INVALID_ARG;
  if (!all_aligned16({W1, W3, W2, w->w13, w->sf13, w->g13, w->w2, w->sf2, w->g2}))
    return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const __nv_bfloat16* w1 = reinterpret_cast<const __nv_bfloat16*>(W1);
  const __nv_bfloat16* w3 = reinterpret_cast<const __nv_bfloat16*>(W3);
  const __nv_bfloat16* w2 = reinterpret_cast<const __nv_bfloat16*>(W2);
  // gate/up: [W1_e | W3_e] (H x 2F) is one tensor per expert
  MOE_CUDA(launch_nv_amax(w1, static_cast<long long>(c.H) * c.F, c.E, w->g13, s, w3));
  MOE_CUDA(launch_nv_quantize_weights(w1, c.E, c.H, 2 * c.F, w->g13, w->w13, w->sf13, s, w3, c.F));
  MOE_CUDA(launch_nv_amax(w2, static_cast<long long>(c.F) * c.H, c.E, w->g2, s));
  MOE_CUDA(launch_nv_quantize_weights(w2, c.E, c.F, c.H, w->g2, w->w2, w->sf2, s));
  count_launches(7);
  return MOE_OK;
}

static WsLayout nv_layer_ws(const moe_config& c) { return ws_layout(c, false, false, true); }

size_t moe_nv_workspace_bytes_layer(const moe_config* cfg) {
  if (check_cfg(cfg) != MOE_OK || check_nv_layer_shape(*cfg) != MOE_OK) return 0;
  return nv_layer_ws(*cfg).total;
}

int moe_layer_fwd_nvfp4(const moe_config* cfg, const moe_bf16* x, const moe_bf16* router_w,
                        const float* expert_bias, const float* logit_bias, const moe_nv_weights* w, void* y, void* ws,
                        size_t ws_bytes, void* stream) {
  NvtxRange nvtx("moe_layer_fwd_nvfp4");
  MOE_TRY(check_cfg(cfg));
  const moe_config& c = *cfg;
  MOE_TRY(check_nv_layer_shape(c));
  if (!x || !router_w || !w || !w->w13 || !w->sf13 || !w->g13 || !w->w2 || !w->sf2 || !w->g2 || !y || !ws)
    return MOE_ERR_INVALID_ARG;
  if (!all_aligned16({x, router_w, expert_bias, logit_bias, w->w13, w->sf13, w->g13, w->w2, w->sf2, w->g2, y,
                      ws}))
    return MOE_ERR_INVALID_ARG;
  const WsLayout L = nv_layer_ws(c);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  DevStatus* st = at<DevStatus>(ws, 0);
  const long long R = static_cast<long long>(c.T) * c.k;
  int32_t* idx = at<int32_t>(ws, L.topk_idx);
  float* gate = at<float>(ws, L.topk_gate);
  int32_t* rows = at<int32_t>(ws, L.row_id_map);
  int32_t* counts = at<int32_t>(ws, L.counts);
  int32_t* offs = at<int32_t>(ws, L.offsets);
  __nv_bfloat16* a = at<__nv_bfloat16>(ws, L.a);
  uint8_t* q = at<uint8_t>(ws, L.nv_q);
  uint8_t* sfq = at<uint8_t>(ws, L.nv_sf);
  float* gq = at<float>(ws, L.nv_g);
  void* yp = at<void>(ws, L.y_perm);
  const __nv_bfloat16* xb = reinterpret_cast<const __nv_bfloat16*>(x);
  prof_mark(s, STAGE_BEGIN);
  MOE_TRY(run_router(c, xb, reinterpret_cast<const __nv_bfloat16*>(router_w), expert_bias, logit_bias, idx, gate,
                     nullptr, nullptr, st, s));
  stage_done(s, STAGE_ROUTER, 1);
  // the routed rows are copies of x's rows: the tensor maximum of x, then the
  // permute quantises as it scatters
  MOE_CUDA(launch_nv_amax(xb, static_cast<long long>(c.T) * c.H, 1, gq, s));
  MOE_CUDA(launch_permute(c, xb, idx, nullptr, rows, counts, offs, at<int32_t>(ws, L.lookback), st, s, q, sfq, gq));
  stage_done(s, STAGE_PERMUTE, 4);
  // gate/up GEMM with SiLU * up and the maximum of a in its epilogue
  MOE_CUDA(cudaMemsetAsync(gq + 1, 0, sizeof(float), s));
  {
    GemmParams p = base_params(c, st);
    p.F = c.F;
    p.ngroups = c.E;
    p.offsets = offs;
    p.M_total = static_cast<int>(R);
    p.bn = kNvTileN;
    p.n_tiles = (c.F + kMxTileF1 - 1) / kMxTileF1;
    p.nt_w = p.n_tiles;
    p.kb_total = c.H / kNvKB;
    p.out0 = a;
    p.nv_ga = gq;
    p.nv_gb = w->g13;
    p.nv_amax = reinterpret_cast<unsigned*>(gq + 1);
    CUtensorMap ma, mb, msa, msb;
    if (!make_map_u8(&ma, q, c.H / 2, R, 128, kBM)) return MOE_ERR_CUDA;
    if (!make_map_u8(&mb, w->w13, c.H / 2, 2ull * c.E * c.F, 128, kMxTileF1)) return MOE_ERR_CUDA;
    if (!make_map_u8(&msa, sfq, 256, nv_act_sf_bytes(R, c.E, c.H) / 256, 256, 8, false)) return MOE_ERR_CUDA;
    if (!make_map_u8(&msb, w->sf13, 256, nv_weight_sf_bytes_gu(c.E, c.H, c.F) / 256, 256, 16, false))
      return MOE_ERR_CUDA;
    MOE_CUDA(launch_gemm(KIND_FFN1_NV, p, ma, mb, msa, num_sms(), s, nullptr, &msb));
  }
  MOE_CUDA(launch_nv_scale_from_amax(gq + 1, 1, s));
  stage_done(s, STAGE_FFN1, 2);
  MOE_CUDA(launch_nv_quantize_grouped(a, static_cast<int>(R), c.F, c.E, offs, gq + 1, q, sfq, s));
  stage_done(s, STAGE_NV_QUANT, 1);
  MOE_TRY(run_gemm_nv(c.E, R, c.F, c.H, offs, q, sfq, gq + 1, w->w2, w->sf2, w->g2,
                      reinterpret_cast<__nv_bfloat16*>(yp), st, s));
  stage_done(s, STAGE_FFN2, 1);
  MOE_CUDA(launch_combine(c, yp, rows, gate, nullptr, y, s, st));
  stage_done(s, STAGE_COMBINE, 1);
  return MOE_OK;
}

// ---------------------------------------------------------------------------
// NVFP4 training step
// ---------------------------------------------------------------------------
size_t moe_nv_bwd_weight_bytes(const moe_config* cfg, int which) {
  if (check_cfg(cfg) != MOE_OK || check_nv_layer_shape(*cfg) != MOE_OK) return 0;
  const moe_config& c = *cfg;
  switch (which) {
    case 0: return moe_nv_weight_bytes(c.E, c.H, c.F, 0);      // W2_e rows along H: K = H, N = F
    case 1: return moe_nv_weight_bytes(c.E, c.H, c.F, 1);
    case 2: return moe_nv_weight_bytes(c.E, c.H, c.F, 2);
    case 3: return moe_nv_weight_bytes(c.E, 2 * c.F, c.H, 0);  // [W1_e | W3_e] rows along 2F: K = 2F, N = H
    case 4: return moe_nv_weight_bytes(c.E, 2 * c.F, c.H, 1);
    case 5: return moe_nv_weight_bytes(c.E, 2 * c.F, c.H, 2);
    default: return 0;
  }
}

int moe_nv_quantize_bwd_weights(const moe_config* cfg, const moe_bf16* W1, const moe_bf16* W3, const moe_bf16* W2,
                                const moe_nv_bwd_weights* w, void* stream) {
  NvtxRange nvtx("moe_nv_quantize_bwd_weights");
  MOE_TRY(check_cfg(cfg));
  const moe_config& c = *cfg;
  MOE_TRY(check_nv_layer_shape(c));
  if (!W1 || !W3 || !W2 || !w || !w->w2h || !w->sf2h || !w->g2h || !w->w13f || !w->sf13f || !w->g13f)
    return MOE_ERR_INVALID_ARG;
  if (!all_aligned16({W1, W3, W2, w->w2h, w->sf2h, w->g2h, w->w13f, w->sf13f, w->g13f}))
    return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const __nv_bfloat16* w1 = reinterpret_cast<const __nv_bfloat16*>(W1);
  const __nv_bfloat16* w3 = reinterpret_cast<const __nv_bfloat16*>(W3);
  const __nv_bfloat16* w2 = reinterpret_cast<const __nv_bfloat16*>(W2);
  // W2_e [F, H] row-wise along H, one tensor per expert
  MOE_CUDA(launch_nv_amax(w2, static_cast<long long>(c.F) * c.H, c.E, w->g2h, s));
  MOE_CUDA(launch_nv_quantize_weight_rows(w2, c.E, c.H, c.F, w->g2h, w->w2h, w->sf2h, s));
  // [W1_e | W3_e] [H, 2F] row-wise along 2F, one tensor per expert
  MOE_CUDA(launch_nv_amax(w1, static_cast<long long>(c.H) * c.F, c.E, w->g13f, s, w3));
  MOE_CUDA(launch_nv_quantize_weight_rows(w1, c.E, 2 * c.F, c.H, w->g13f, w->w13f, w->sf13f, s, w3, c.F));
  count_launches(7);
  return MOE_OK;
}

int moe_nv_quantize_train_weights(const moe_config* cfg, const moe_bf16* W1, const moe_bf16* W3,
                                  const moe_bf16* W2, const moe_nv_weights* fw, const moe_nv_bwd_weights* bw,
                                  void* stream) {
  NvtxRange nvtx("moe_nv_quantize_train_weights");
  MOE_TRY(check_cfg(cfg));
  const moe_config& c = *cfg;
  MOE_TRY(check_nv_layer_shape(c));
  if (!W1 || !W3 || !W2 || !fw || !fw->w13 || !fw->sf13 || !fw->g13 || !fw->w2 || !fw->sf2 || !fw->g2 || !bw ||
      !bw->w2h || !bw->sf2h || !bw->g2h || !bw->w13f || !bw->sf13f || !bw->g13f)
    return MOE_ERR_INVALID_ARG;
  if (!all_aligned16({W1, W3, W2, fw->w13, fw->sf13, fw->g13, fw->w2, fw->sf2, fw->g2, bw->w2h, bw->sf2h, bw->g2h,
                      bw->w13f, bw->sf13f, bw->g13f}))
    return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const __nv_bfloat16* w1 = reinterpret_cast<const __nv_bfloat16*>(W1);
  const __nv_bfloat16* w3 = reinterpret_cast<const __nv_bfloat16*>(W3);
  const __nv_bfloat16* w2 = reinterpret_cast<const __nv_bfloat16*>(W2);
  // both copies quantise the same per-expert tensors ([W1_e | W3_e] and
  // W2_e), so they share one tensor scale each: the maxima are taken once
  MOE_CUDA(launch_nv_amax(w1, static_cast<long long>(c.H) * c.F, c.E, fw->g13, s, w3));
  MOE_CUDA(launch_nv_amax(w2, static_cast<long long>(c.F) * c.H, c.E, fw->g2, s));
  MOE_CUDA(cudaMemcpyAsync(bw->g13f, fw->g13, sizeof(float) * c.E, cudaMemcpyDeviceToDevice, s));
  MOE_CUDA(cudaMemcpyAsync(bw->g2h, fw->g2, sizeof(float) * c.E, cudaMemcpyDeviceToDevice, s));
  // forward operands: codes along H (gate/up) and F (down)
  MOE_CUDA(launch_nv_quantize_weights(w1, c.E, c.H, 2 * c.F, fw->g13, fw->w13, fw->sf13, s, w3, c.F));
  MOE_CUDA(launch_nv_quantize_weights(w2, c.E, c.F, c.H, fw->g2, fw->w2, fw->sf2, s));
  // data-gradient operands: W2_e row-wise along H, [W1_e | W3_e] row-wise along 2F
  MOE_CUDA(launch_nv_quantize_weight_rows(w2, c.E, c.H, c.F, bw->g2h, bw->w2h, bw->sf2h, s));
  MOE_CUDA(launch_nv_quantize_weight_rows(w1, c.E, 2 * c.F, c.H, bw->g13f, bw->w13f, bw->sf13f, s, w3, c.F));
  count_launches(9);
  return MOE_OK;
}

size_t moe_nv_train_workspace_bytes(const moe_config* cfg) {
  if (check_cfg(cfg) != MOE_OK || check_nv_layer_shape(*cfg) != MOE_OK) return 0;
  return ws_layout(*cfg, true, false, true).total;
}

static bool nv_saved_ok(const moe_config& c, const moe_fwd_saved* sv) {
  return sv && sv->topk_idx && sv->topk_gate && sv->logits && sv->row_id_map && sv->counts && sv->offsets &&
         sv->x_perm && sv->h13 && sv->a && sv->y_perm && (c.aux_coeff == 0.0f || sv->aux_partials) &&
         saved_aligned16(sv);
}

int moe_layer_fwd_nvfp4_train(const moe_config* cfg, const moe_bf16* x, const moe_bf16* router_w,
                              const float* expert_bias, const float* logit_bias, const moe_nv_weights* w, void* y,
                              const moe_fwd_saved* saved, void* ws, size_t ws_bytes, void* stream) {
  NvtxRange nvtx("moe_layer_fwd_nvfp4_train");
  MOE_TRY(check_cfg(cfg));
  const moe_config& c = *cfg;
  MOE_TRY(check_nv_layer_shape(c));
  if (!x || !router_w || !w || !w->w13 || !w->sf13 || !w->g13 || !w->w2 || !w->sf2 || !w->g2 || !y || !ws ||
      !nv_saved_ok(c, saved))
    return MOE_ERR_INVALID_ARG;
  if (!all_aligned16({x, router_w, expert_bias, logit_bias, w->w13, w->sf13, w->g13, w->w2, w->sf2, w->g2, y,
                      ws}))
    return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(c, true, false, true);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  DevStatus* st = at<DevStatus>(ws, 0);
  const moe_fwd_saved& sv = *saved;
  const long long R = static_cast<long long>(c.T) * c.k;
  uint8_t* q = at<uint8_t>(ws, L.nv_q);
  uint8_t* sfq = at<uint8_t>(ws, L.nv_sf);
  float* gq = at<float>(ws, L.nv_g);
  const __nv_bfloat16* xb = reinterpret_cast<const __nv_bfloat16*>(x);
  prof_mark(s, STAGE_BEGIN);
  MOE_TRY(run_router(c, xb, reinterpret_cast<const __nv_bfloat16*>(router_w), expert_bias, logit_bias, sv.topk_idx,
                     sv.topk_gate, sv.logits, c.aux_coeff != 0.0f ? sv.aux_partials : nullptr, st, s));
  stage_done(s, STAGE_ROUTER, 1);
  // the permute quantises the routed rows (x's tensor scale) and scatters
  // their bf16 copies for the weight gradient
  MOE_CUDA(launch_nv_amax(xb, static_cast<long long>(c.T) * c.H, 1, gq, s));
  MOE_CUDA(launch_permute(c, xb, sv.topk_idx, reinterpret_cast<__nv_bfloat16*>(sv.x_perm), sv.row_id_map, sv.counts,
                          sv.offsets, at<int32_t>(ws, L.lookback), st, s, q, sfq, gq));
  stage_done(s, STAGE_PERMUTE, 4);
  MOE_CUDA(cudaMemsetAsync(gq + 1, 0, sizeof(float), s));
  {
    GemmParams p = base_params(c, st);
    p.F = c.F;
    p.ngroups = c.E;
    p.offsets = sv.offsets;
    p.M_total = static_cast<int>(R);
    p.bn = kNvTileN;
    p.n_tiles = (c.F + kMxTileF1 - 1) / kMxTileF1;
    p.nt_w = p.n_tiles;
    p.kb_total = c.H / kNvKB;
    p.out0 = sv.a;
    p.out1 = sv.h13;
    p.nv_ga = gq;
    p.nv_gb = w->g13;
    p.nv_amax = reinterpret_cast<unsigned*>(gq + 1);
    CUtensorMap ma, mb, msa, msb;
    if (!make_map_u8(&ma, q, c.H / 2, R, 128, kBM)) return MOE_ERR_CUDA;
    if (!make_map_u8(&mb, w->w13, c.H / 2, 2ull * c.E * c.F, 128, kMxTileF1)) return MOE_ERR_CUDA;
    if (!make_map_u8(&msa, sfq, 256, nv_act_sf_bytes(R, c.E, c.H) / 256, 256, 8, false)) return MOE_ERR_CUDA;
    if (!make_map_u8(&msb, w->sf13, 256, nv_weight_sf_bytes_gu(c.E, c.H, c.F) / 256, 256, 16, false))
      return MOE_ERR_CUDA;
    MOE_CUDA(launch_gemm(KIND_FFN1_NV, p, ma, mb, msa, num_sms(), s, nullptr, &msb));
  }
  MOE_CUDA(launch_nv_scale_from_amax(gq + 1, 1, s));
  stage_done(s, STAGE_FFN1, 2);
  MOE_CUDA(launch_nv_quantize_grouped(reinterpret_cast<const __nv_bfloat16*>(sv.a), static_cast<int>(R), c.F, c.E,
                                      sv.offsets, gq + 1, q, sfq, s));
  stage_done(s, STAGE_NV_QUANT, 1);
  MOE_TRY(run_gemm_nv(c.E, R, c.F, c.H, sv.offsets, q, sfq, gq + 1, w->w2, w->sf2, w->g2, sv.y_perm, st, s));
  stage_done(s, STAGE_FFN2, 1);
  MOE_CUDA(launch_combine(c, sv.y_perm, sv.row_id_map, sv.topk_gate, nullptr, y, s, st));
  stage_done(s, STAGE_COMBINE, 1);
  return MOE_OK;
}

int moe_layer_bwd_nvfp4(const moe_config* cfg, const moe_bf16* dO, const moe_bf16* x, const moe_bf16* router_w,
                        const moe_nv_bwd_weights* w, const moe_fwd_saved* saved, void* dx, float* dW_router,
                        float* dW1, float* dW3, float* dW2, float* aux_loss_out, void* ws, size_t ws_bytes,
                        void* stream) {
  NvtxRange nvtx("moe_layer_bwd_nvfp4");
  MOE_TRY(check_cfg(cfg));
  const moe_config& c = *cfg;
  MOE_TRY(check_nv_layer_shape(c));
  if (!dO || !x || !router_w || !w || !w->w2h || !w->sf2h || !w->g2h || !w->w13f || !w->sf13f || !w->g13f ||
      !nv_saved_ok(c, saved) || !dx || !dW_router || !dW1 || !dW3 || !dW2 || !ws)
    return MOE_ERR_INVALID_ARG;
  if (!all_aligned16({dO, x, router_w, w->w2h, w->sf2h, w->g2h, w->w13f, w->sf13f, w->g13f, dx, dW_router, dW1,
                      dW3, dW2, aux_loss_out, ws}))
    return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(c, true, false, true);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  return layer_bwd_core(c, dO, x, router_w, nullptr, nullptr, nullptr, saved, dx, dW_router, dW1, dW3, dW2,
                        aux_loss_out, ws, L, nullptr, static_cast<cudaStream_t>(stream), false, nullptr, nullptr,
                        nullptr, nullptr, nullptr, nullptr, w);
}

}  // extern "C"

// Persistent, warp-specialised tcgen05 GEMM for the MoE layer.
//
// One CTA per SM (192 threads):
//   warp 0      TMA producer: 128-byte-swizzled tiles of A and B into a ring of
//               shared-memory stages (mbarrier full/empty pairs);
//   warp 1      TMEM owner and MMA issuer: 128 (pairs: 256) x BN x 16 bf16 MMAs
//               into one of two fp32 accumulators in tensor memory (2 x 256
//               columns), so the epilogue of tile i overlaps the main loop of
//               tile i+1;
//   warps 2-5   epilogue: each thread owns one accumulator row (TMEM lane),
//               reads 32 columns at a time and applies the kind's epilogue.
//
// CTA pairs (every kind but the router gradients): clusters of two CTAs run
// M=256 tiles with tcgen05.mma.cta_group::2. Each CTA stages its own 128 rows
// of A and one half of B; both CTAs' loads complete on the even CTA's full
// barrier; the even CTA issues the MMAs and signals stage release, accumulator
// ready and drain to both CTAs with multicast commits; the odd CTA's epilogue
// frees the accumulator with cluster-scope arrivals on the even CTA's barrier.
// An SM then receives 32 KB per 64-deep k block instead of 48 KB, which keeps
// the operand stream within the L2-to-SM bandwidth.
//
// Tiles come from a device-side schedule: every CTA reads the per-expert row
// offsets produced by the permute (no host synchronisation), builds the
// prefix of tile counts in shared memory, and walks tiles blockIdx.x (pairs:
// its cluster's index), + gridDim.x (pairs: the number of clusters), ... .
// Each kind below fixes which global tensors feed A and B, how a tile maps to
// coordinates, and what the epilogue writes.
//
// Operand staging (both operands as 128-byte swizzled boxes of 64 bf16):
//   K-major operand with R rows: one box {64 (k), R} -> R rows of 128 B;
//   MN-major operand with R (m or n) extent: R/64 boxes {64 (mn), 64 (k)}, each
//   64 K-rows of 128 B (8 KB), placed 8 KB apart.
#pragma once
#include "common.cuh"
#include "mx.cuh"
#include "nv.cuh"

namespace moe {

enum GemmKind : int {
  KIND_FFN1 = 0,       // h = x_perm [W1_e | W3_e]  -> a = SiLU(h1) h3 (+ h13 save)
  KIND_FFN2 = 1,       // y_perm = a W2_e
  KIND_ROUTER = 2,     // router: logits L = x W_r^T, score, selection and gates in the epilogue (router_sel.cuh)
  KIND_DGRAD2 = 3,     // da = dy_perm W2_e^T -> SwiGLU backward -> dh13
  KIND_DGRAD1 = 4,     // dx_perm = dh13 [W1_e | W3_e]^T
  KIND_WGRAD = 5,      // dW_e = X_e^T Y_e over the expert's rows (ragged K)
  KIND_ROUTER_DX = 6,  // dx_r = dL W_r     (dL as bf16 hi + lo parts)
  KIND_ROUTER_DW = 7,  // dW_r partial = dL^T x over one K split
  KIND_DGRAD2R = 8,    // DGRAD2 of the memory-saving backward: also stores a = SiLU(h1) h3 recomputed from
                       // h13 and the per-row partials of the gate gradient <da, a> over each 256-column tile
  KIND_FFN1_MX = 9,    // MXFP8 gate/up: h = Q(x_perm) [Q(W1_e) | Q(W3_e)] -> a = SiLU(h1) h3, stored as MXFP8
                       // (codes + the down GEMM's tile-ready scales); 256 x (96 gate + 96 up) pair tiles
  KIND_FFN2_MX = 10,   // MXFP8 down: y_perm = Q(a) Q(W2_e), bf16 out; 256 x 192 pair tiles
  KIND_GEMM_NV = 11,   // NVFP4 grouped expert GEMM: y = g_x g_e Q(x_e) Q(W_e), bf16 or fp32 out; 256 x 192 pair tiles
  KIND_FFN1_NV = 12,   // NVFP4 gate/up: h = g_x g_e Q(x_perm) Q([W1_e | W3_e]) -> a = bf16(SiLU(h1) h3) and max |a|;
                       // 256 x (96 gate + 96 up) pair tiles
  KIND_DGRAD2_MX = 13, // MXFP8 down-projection data gradient: da = Q(dy_perm) Q(W2_e)^T -> SwiGLU backward ->
                       // dh13 and a (bf16) and dh13 as MXFP8 (codes + the gate/up data gradient's scales);
                       // 256 x 192 pair tiles
  KIND_WGRAD_MX = 14,  // MXFP8 weight gradient dW_e = Q(X_e)^T Q(Y_e) over the expert's tokens (K-major
                       // transposed operands, k blocks of 128 padded tokens per expert), fp32 out;
                       // 256 x 192 pair tiles
};

// Score modes of the router's selection (router_sel.cuh): selection on the
// logits (softmax, no expert bias, no group limit), on softmax probabilities
// (+ expert bias), or on sigmoid scores (+ expert bias).
enum RouterSelMode : int { RSEL_LOGIT = 0, RSEL_SOFTMAX = 1, RSEL_SIGMOID = 2 };

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kThreads = 192;
constexpr int kABytes = kBM * 128;        // 16 KB
constexpr int kBBytesMax = 256 * 128;     // 32 KB
constexpr int kStageBytes = kABytes + kBBytesMax;
constexpr int kRingBytes = 4 * kStageBytes;  // shared memory of the operand stage ring
constexpr int kMaxGroups = 256;
constexpr int kTmemCols = 512;
// MXFP8 pair stage (per CTA): A 16 KB at 0, B (96 rows x 128 B) at 16 KB, scale
// blocks of A (512 B) and B (1 KB) at 28 KB; 31 KB keeps every stage
// 1024-byte aligned
constexpr int kMxSfOff = 28672;
constexpr int kMxStageBytes = 31744;
constexpr uint32_t kMxStageTx = 16384 + (kMxBN / 2) * 128 + 3 * kMxSfBytes;  // one CTA's share
// TMEM columns of the scale cells (past both 192-column accumulators): two
// regions of 12 columns (A: 4, B: 8), alternating per k block
constexpr uint32_t kMxSfaCol = 448;
constexpr uint32_t kMxSfbCol = 452;
constexpr uint32_t kMxSfRegion = 12;
// NVFP4 pair stage (per CTA): A 16 KB, B 12 KB at 16 KB, A scales (2 KB) and
// B scales (4 KB) at 28 KB. TMEM scale regions of 48 columns (A: 4 steps x 4,
// B: 4 steps x 8) in the gaps after the two 192-column accumulators.
constexpr int kNvSfOff = 28672;
constexpr int kNvStageBytes = 34816;
constexpr uint32_t kNvStageTx = kNvStageBytes;  // one CTA's share
constexpr uint32_t kNvSfRegion0 = 192;
constexpr uint32_t kNvSfRegion1 = 448;
constexpr int kAccStride = 256;           // TMEM column distance of the two accumulators

template <int KIND>
struct KindTraits {
  static constexpr bool A_MN = (KIND == KIND_WGRAD || KIND == KIND_ROUTER_DW);
  static constexpr bool B_MN = (KIND == KIND_FFN1 || KIND == KIND_FFN2 || KIND == KIND_WGRAD ||
                                KIND == KIND_ROUTER_DX || KIND == KIND_ROUTER_DW);
  // CTA pairs: the expert GEMMs with a fixed K run as M=256 tiles on two SMs
  // (cta_group::2); each CTA stages its own 128 rows of A and half of B
  // MXFP8 kinds: CTA pairs on 256 x 192 tiles; a CTA's stage holds 128 k
  // elements (one byte each) of its 128 A rows (16 KB) and 96 B rows (12 KB),
  // its A scale block (0.5 KB) and the tile's B scale blocks (1 KB)
  static constexpr bool kMx =
      (KIND == KIND_FFN1_MX || KIND == KIND_FFN2_MX || KIND == KIND_DGRAD2_MX || KIND == KIND_WGRAD_MX);
  // NVFP4: like MXFP8 with 256-element k blocks (128 bytes of codes per row)
  // and four scale blocks per operand block (2 KB of A, 4 KB of B scales)
  static constexpr bool kNv = (KIND == KIND_GEMM_NV || KIND == KIND_FFN1_NV);
  static constexpr bool kPair = (KIND == KIND_FFN1 || KIND == KIND_FFN2 || KIND == KIND_DGRAD2 ||
                                 KIND == KIND_DGRAD1 || KIND == KIND_WGRAD || KIND == KIND_DGRAD2R || kMx || kNv);
  static constexpr int kTileM = kPair ? 2 * kBM : kBM;  // rows of one (pair) tile
  // stage ring of kRingBytes: single-CTA stages of kStageBytes; pair stages of
  // 16 KB of A + 16 KB of B
  // ROUTER_DW: both bf16 parts of dL (hi, lo) with one box of x, so x is
  // read once for the two products
  static constexpr int kStageBytesK = kNv ? kNvStageBytes
                                      : kMx ? kMxStageBytes
                                      : kPair ? (kABytes + kBBytesMax / 2)
                                      : (KIND == KIND_ROUTER_DW) ? (2 * kABytes + kBBytesMax) : kStageBytes;
  // offset of B in a stage
  static constexpr int kBOff = (KIND == KIND_ROUTER_DW) ? 2 * kABytes : kABytes;
  // DGRAD2 runs eight epilogue warps (two per TMEM lane quadrant, each taking
  // half of the tile's columns) to hide the latency of its loads of the saved
  // pre-activations, with one 4 KB staging box each (dh1 leaves before dh3
  // is staged), which keeps six stages; DGRAD2R (third staging box) gives up
  // one stage
  // FFN1_MX runs twelve (three per TMEM lane quadrant, one 32-column block of
  // the 96 SwiGLU columns each): its tiles are short (K / 128 blocks of
  // 128) and its epilogue (SiLU, quantisation) long
  // DGRAD2_MX runs twelve (three per quadrant, 64 of the tile's 192 columns
  // each) for the same reasons
  // ROUTER runs eight (two per quadrant, each on half of a token's experts):
  // its selection follows the tile's main loop with nothing to overlap it
  static constexpr int kEpiWarps =
      (KIND == KIND_DGRAD2 || KIND == KIND_ROUTER) ? 8
      : (KIND == KIND_FFN1_MX || KIND == KIND_FFN1_NV || KIND == KIND_DGRAD2_MX) ? 12 : 4;
  static constexpr int kThreadsK = 64 + 32 * kEpiWarps;
  // WGRAD stores its fp32 output straight from tensor memory (no staging
  // boxes), which leaves room for a seventh stage
  static constexpr int kStages = (KIND == KIND_DGRAD2R || kNv) ? 5
                                 : (KIND == KIND_WGRAD)                            ? 7
                                 : kPair                                           ? 6
                                 : (KIND == KIND_ROUTER_DW)                        ? 3
                                                                                   : 4;
  static constexpr int kOutWarpBytes =
      (KIND == KIND_DGRAD2R) ? 3 * 4096
      : (KIND == KIND_ROUTER) ? 4096  // selection scratch, 32 KB in all
      : (KIND == KIND_FFN1_MX || KIND == KIND_FFN1_NV || KIND == KIND_DGRAD2_MX || KIND == KIND_WGRAD) ? 0
      : (KIND == KIND_DGRAD2)                                                                           ? 4096
                                                                                                       : 2 * 4096;  // staging
  // the router's B is bn x 64 (bn <= 256): its stages are packed at
  // router_stage_bytes(bn) so narrow routers keep more k blocks in flight
  static constexpr int kMaxStages = (KIND == KIND_ROUTER) ? 8 : kStages;
  static constexpr bool kGroupedRows = (KIND == KIND_FFN1 || KIND == KIND_FFN2 || KIND == KIND_DGRAD2 ||
                                        KIND == KIND_DGRAD1 || KIND == KIND_DGRAD2R || (kMx && KIND != KIND_WGRAD_MX) || kNv);
};

struct GemmParams {
  // problem sizes
  int T, H, E, k, F;
  int M_total;           // rows of the single group when offsets == nullptr
  int ngroups;           // groups (experts) in the schedule
  int bn;                // UMMA N (multiple of 32, <= 256)
  int n_tiles;           // N tiles per m tile (uniform over groups)
  int m_tiles_fixed;     // WGRAD / ROUTER_DW: m tiles per group
  int wg_M, wg_N;        // WGRAD: output rows / columns of one expert's gradient
  int wg_mode;           // WGRAD: 0 = dW2 [E,F,H]; 1 = dW1|dW3 from N = 2F
  int kb_total;          // k blocks (non-ragged kinds); ROUTER_DW: per split
  int splits;            // ROUTER_DW: number of K splits
  int Ep;                // ROUTER_DX / ROUTER_DW: padded expert count (multiple of 64)
  const int32_t* offsets;  // [ngroups+1] device row offsets (grouped kinds, WGRAD)
  // outputs / epilogue inputs
  void* out0;            // FFN1: a; FFN2: y_perm; DGRAD2: dh13; DGRAD1: dx_perm;
                         // WGRAD: dW2 or dW1; ROUTER_DX: dx_r (fp32); ROUTER_DW: partials
  void* out1;            // FFN1: h13 save (nullable); WGRAD mode 1: dW3
  const void* in_aux;    // DGRAD2, DGRAD2R: h13 (saved pre-activations)
  float* dg_part;        // DGRAD2R: gate-gradient partials [rows, n_part] (DGRAD2R also stores a in out1)
  uint8_t* q_out;        // DGRAD2_MX: MXFP8 codes of dh13 [rows, 2F] (scales in sfa_out)
  uint8_t* tmap_slots;   // WGRAD: per-expert copies of the A map (128 bytes each) for the partial k blocks
  int n_part;            // DGRAD2R: 256-column tiles of F
  int out_fp32;          // FFN2: y_perm fp32; DGRAD1: dx_perm fp32
  // MXFP8 kinds: the activations' scale blocks are read through a tensor map;
  // FFN1_MX writes the down GEMM's A scale blocks to sfa_out; nt_w = n tiles
  // per expert of the weight scales (the weight scales: map msfb)
  uint8_t* sfa_out;
  int nt_w;
  const float* nv_ga;    // GEMM_NV: tensor scale of the activations (one value)
  const float* nv_gb;    // GEMM_NV: tensor scales of the experts' weights [ngroups]
  unsigned* nv_amax;     // FFN1_NV: running max |a| (fp32 bits)
  // ROUTER: the selection in the epilogue (router_sel.cuh)
  const float* r_lbias;  // logit bias [E] (added to the logits), nullable
  const float* r_ebias;  // expert bias [E] (selection only), nullable
  int32_t* r_idx;        // topk_idx [T, k]
  float* r_gate;         // topk_gate [T, k]
  float* r_logits;       // biased logits [T, E], nullable
  float* r_aux;          // softmax column sums per 32-token slice [4 ceil(T/128), E], nullable
  int r_mode;            // RouterSelMode
  int r_groups, r_topk_groups, r_force;
  float r_gate_scale;
  // status
  DevStatus* status;
  unsigned long long wait_limit_ns;
};

struct TileInfo {
  int g;       // group (expert) or split
  int m0;      // first row of the tile (global row for grouped kinds; m offset otherwise)
  int m_end;   // one past the last valid row
  int n0;      // first output column of the tile
  int kb0;     // first k block
  int nkb;     // k blocks of this tile
  int krow0;   // WGRAD: first row of the expert (K origin); ROUTER_DW: unused
  int krow_end;
  int mt;      // grouped kinds: global m tile (tiles of all earlier groups + this group's)
  int nb;      // n tile within the group
  int half;    // an expert's last m tile with at most 128 rows: an M = 128 pair MMA (64 rows per CTA)
};

// Kinds whose last m tile of an expert runs as an M = 128 pair MMA when it
// holds at most 128 rows (the tail of a ragged expert then costs half the
// tensor work). With cta_group::2 and M = 128 each CTA supplies 64 rows of A
// and holds its 64 rows' accumulator twice over in tensor memory: lanes 0..63
// with the N columns of the even CTA's B half, lanes 64..127 with the odd
// CTA's, both at columns 0 .. N/2 - 1 (measured on the GB300 with an in-bounds
// probe before use).
template <int KIND>
constexpr bool kHalfTiles = (KIND == KIND_FFN1 || KIND == KIND_FFN2 || KIND == KIND_DGRAD1);

template <int KIND>
__device__ __forceinline__ TileInfo decode_tile(const GemmParams& p, const int* s_cum, const int* s_off,
                                                int tile, int rank = 0) {
  TileInfo ti;
  int lo = 0, hi = p.ngroups;  // find g with s_cum[g] <= tile < s_cum[g+1]
  while (hi - lo > 1) {
    int mid = (lo + hi) >> 1;
    if (s_cum[mid] <= tile) lo = mid; else hi = mid;
  }
  ti.g = lo;
  const int local = tile - s_cum[lo];
  int mb, nb;
  if constexpr (KindTraits<KIND>::kGroupedRows && !KindTraits<KIND>::kMx && !KindTraits<KIND>::kNv) {
    // bf16 kinds: n-major inside an expert: its m tiles of one n tile are
    // consecutive, so CTA pairs that start together share that n tile's weight
    // block in L2 (m-major, an expert whose tiles straddle two rounds of the
    // persistent CTAs read the weight blocks of the later round from DRAM
    // again). The MXFP8 and NVFP4 kinds, whose weight blocks are half or a
    // quarter the bytes, measured 1% faster m-major and keep it.
    const int me = (s_cum[lo + 1] - s_cum[lo]) / p.n_tiles;
    nb = local / me;
    mb = local - nb * me;
  } else {
    mb = local / p.n_tiles;
    nb = local - mb * p.n_tiles;
  }
  ti.mt = s_cum[lo] / p.n_tiles + mb;
  ti.nb = nb;
  ti.half = 0;
  if constexpr (kHalfTiles<KIND>) {
    const int me = (s_cum[lo + 1] - s_cum[lo]) / p.n_tiles;
    ti.half = (mb == me - 1 && s_off[lo + 1] - s_off[lo] - mb * KindTraits<KIND>::kTileM <= kBM) ? 1 : 0;
  }
  if constexpr (KindTraits<KIND>::kGroupedRows || KIND == KIND_ROUTER || KIND == KIND_ROUTER_DX) {
    // a pair tile spans 256 rows: this CTA's 128 start at rank * 128 (a half
    // tile's 64 at rank * 64)
    ti.m0 = s_off[lo] + mb * KindTraits<KIND>::kTileM + rank * (ti.half ? kBM / 2 : kBM);
    ti.m_end = s_off[lo + 1];
    ti.kb0 = 0;
    ti.nkb = p.kb_total;
    ti.krow0 = 0;
    ti.krow_end = 0;
  } else if constexpr (KIND == KIND_WGRAD) {
    ti.m0 = mb * KindTraits<KIND>::kTileM + rank * kBM;
    ti.m_end = p.wg_M;
    ti.krow0 = s_off[lo];
    ti.krow_end = s_off[lo + 1];
    ti.kb0 = 0;
    ti.nkb = (ti.krow_end - ti.krow0 + kBK - 1) / kBK;
  } else if constexpr (KIND == KIND_WGRAD_MX) {
    // fixed M per expert; K = the expert's padded tokens (group offsets are
    // padded token offsets, multiples of 128), whole k blocks from kb0
    ti.mt = mb;
    ti.m0 = mb * KindTraits<KIND>::kTileM + rank * kBM;
    ti.m_end = p.wg_M;
    ti.kb0 = s_off[lo] / kMxKB;
    ti.nkb = (s_off[lo + 1] - s_off[lo]) / kMxKB;
    ti.krow0 = 0;
    ti.krow_end = 0;
  } else {  // ROUTER_DW: group = split of the token blocks
    ti.m0 = mb * kBM;
    ti.m_end = p.E;
    int total = (p.T + kBK - 1) / kBK;
    int per = p.kb_total;
    ti.kb0 = lo * per;
    ti.nkb = min(per, total - ti.kb0);
    if (ti.nkb < 0) ti.nkb = 0;
    ti.krow0 = 0;
    ti.krow_end = 0;
  }
  if constexpr (KIND == KIND_FFN1) {
    ti.n0 = nb * 128;  // F columns (gate and up halves of the 256-wide tile)
  } else if constexpr (KIND == KIND_FFN1_MX || KIND == KIND_FFN1_NV) {
    ti.n0 = nb * kMxTileF1;  // F columns (gate and up halves of the 192-wide tile)
  } else {
    ti.n0 = nb * p.bn;
  }
  return ti;
}

// CTA pairs: this CTA's share of k block `kb`: its 128 rows of A and half of B
// (FFN1: the W1 (even CTA) or W3 (odd CTA) columns of the tile; FFN2: columns
// n0 + 128 rank ..; DGRAD2 / DGRAD1: B rows n0 + 128 rank .., boxes of 128
// rows; WGRAD: A columns m0 .. m0 + 127 and B columns n0 + 128 rank .. of the
// expert's rows kb*64 .., A through the map `ma` given), completing on the even
// CTA's barrier `bar_cluster`.
template <int KIND>
__device__ __forceinline__ void issue_loads_pair(const GemmParams& p, const TileInfo& ti, int kb, int rank,
                                                 uint8_t* sA, uint8_t* sB, uint32_t bar_cluster, const CUtensorMap* ma,
                                                 const CUtensorMap* mb0, const CUtensorMap* mb1,
                                                 const CUtensorMap* msfb = nullptr) {
  if constexpr (KindTraits<KIND>::kNv) {
    // 256 k elements (128 bytes) of this CTA's 128 A rows and its 96 B rows
    // (rows n0 + 96 rank .. of expert g's [N] weight rows), its A scale block
    // (2 KB = 8 rows of the activations' scale map) and the tile's two B scale
    // blocks (4 KB = 16 rows of msfb)
    const int kc = kb * (kNvKB / 2);
    tma_load_2d_pair(sA, ma, bar_cluster, kc, ti.m0);
    if constexpr (KIND == KIND_FFN1_NV) {
      // W1 rows n0.. (even CTA) or W3 rows n0.. (odd CTA) of expert g ([E][2F] rows)
      tma_load_2d_pair(sB, mb0, bar_cluster, kc, ti.g * 2 * p.F + rank * p.F + ti.n0);
    } else {
      tma_load_2d_pair(sB, mb0, bar_cluster, kc, ti.g * p.H + ti.n0 + rank * (kNvTileN / 2));
    }
    uint8_t* sSF = sA + kNvSfOff;
    tma_load_2d_pair(sSF, mb1, bar_cluster, 0, 8 * ((2 * ti.mt + rank) * p.kb_total + kb));
    tma_load_2d_pair(sSF + kNvSfBytes, msfb, bar_cluster, 0, 16 * ((ti.g * p.nt_w + ti.nb) * p.kb_total + kb));
    return;
  }
  if constexpr (KindTraits<KIND>::kMx) {
    // 128 k elements (bytes) of this CTA's 128 A rows and its 96 B rows, its A
    // scale block (block 2 * pair tile + rank of the activations' scales: map
    // mb1, 256-byte rows) and the tile's two B scale blocks (map msfb)
    // WGRAD_MX: k block kb0 + kb of the padded token axis shared by all
    // experts (its operands and scales carry no expert index)
    const int kbg = (KIND == KIND_WGRAD_MX) ? ti.kb0 + kb : kb;
    const int kc = kbg * kMxKB;
    tma_load_2d_pair(sA, ma, bar_cluster, kc, ti.m0);
    if constexpr (KIND == KIND_FFN1_MX) {
      // W1 rows n0.. (even CTA) or W3 rows n0.. (odd CTA) of expert g
      tma_load_2d_pair(sB, mb0, bar_cluster, kc, ti.g * 2 * p.F + rank * p.F + ti.n0);
    } else if constexpr (KIND == KIND_WGRAD_MX) {
      // rows n0 + 96 rank .. of the transposed B operand
      tma_load_2d_pair(sB, mb0, bar_cluster, kc, ti.n0 + rank * (kMxBN / 2));
    } else {
      // W2 rows (H index) n0 + 96 rank .. of expert g
      tma_load_2d_pair(sB, mb0, bar_cluster, kc, ti.g * p.H + ti.n0 + rank * (kMxBN / 2));
    }
    uint8_t* sSF = sA + kMxSfOff;
    const int ablk = (2 * ti.mt + rank) * p.kb_total + kbg;
    tma_load_2d_pair(sSF, mb1, bar_cluster, 0, 2 * ablk);
    const int bblk = ((KIND == KIND_WGRAD_MX) ? ti.nb : ti.g * p.nt_w + ti.nb) * p.kb_total + kbg;
    tma_load_2d_pair(sSF + kMxSfBytes, msfb, bar_cluster, 0, 4 * bblk);
    return;
  }
  const int kk = kb * kBK;
  if constexpr (KIND == KIND_WGRAD) {
    const int r = ti.krow0 + kk;
    const int n = ti.n0 + 128 * rank;
    // the operands are re-read by the expert's other tiles while the fp32
    // output streams through L2: they stay, the output goes first
    const uint64_t keep = l2_policy_evict_last();
    tma_load_2d_pair_hint(sA, ma, bar_cluster, ti.m0, r, keep);
    tma_load_2d_pair_hint(sA + 8192, ma, bar_cluster, ti.m0 + 64, r, keep);
    tma_load_2d_pair_hint(sB, mb0, bar_cluster, n, r, keep);
    tma_load_2d_pair_hint(sB + 8192, mb0, bar_cluster, n + 64, r, keep);
    return;
  }
  tma_load_2d_pair(sA, ma, bar_cluster, kk, ti.m0);
  if constexpr (KIND == KIND_FFN1) {
    const int brow = ti.g * p.H + kk;
    if (ti.half) {
      // half tile: this CTA's B half holds W1 and W3 columns n0 + 64 rank ..
      // (64 each), so a row's gate and up values share a TMEM lane
      tma_load_2d_pair(sB, mb0, bar_cluster, ti.n0 + 64 * rank, brow);
      tma_load_2d_pair(sB + 8192, mb1, bar_cluster, ti.n0 + 64 * rank, brow);
      return;
    }
    const CUtensorMap* m = rank == 0 ? mb0 : mb1;
    tma_load_2d_pair(sB, m, bar_cluster, ti.n0, brow);
    tma_load_2d_pair(sB + 8192, m, bar_cluster, ti.n0 + 64, brow);
  } else if constexpr (KIND == KIND_FFN2) {
    const int brow = ti.g * p.F + kk;
    const int n = ti.n0 + 128 * rank;
    tma_load_2d_pair(sB, mb0, bar_cluster, n, brow);
    tma_load_2d_pair(sB + 8192, mb0, bar_cluster, n + 64, brow);
  } else if constexpr (KIND == KIND_DGRAD2 || KIND == KIND_DGRAD2R) {
    tma_load_2d_pair(sB, mb0, bar_cluster, kk, ti.g * p.F + ti.n0 + 128 * rank);
  } else {  // DGRAD1
    const int brow = ti.g * p.H + ti.n0 + 128 * rank;
    if (kk < p.F) tma_load_2d_pair(sB, mb0, bar_cluster, kk, brow);
    else tma_load_2d_pair(sB, mb1, bar_cluster, kk - p.F, brow);
  }
}

// Issue the TMA loads of k block `kb` of tile `ti` into stage buffers sA, sB.
template <int KIND>
__device__ __forceinline__ void issue_loads(const GemmParams& p, const TileInfo& ti, int kb, uint8_t* sA,
                                            uint8_t* sB, uint64_t* bar, const CUtensorMap* ma,
                                            const CUtensorMap* mb0, const CUtensorMap* mb1) {
  const int kk = kb * kBK;
  if constexpr (KIND == KIND_FFN1) {
    tma_load_2d(sA, ma, bar, kk, ti.m0);
    const int brow = ti.g * p.H + kk;
    tma_load_2d(sB + 0 * 8192, mb0, bar, ti.n0, brow);
    tma_load_2d(sB + 1 * 8192, mb0, bar, ti.n0 + 64, brow);
    tma_load_2d(sB + 2 * 8192, mb1, bar, ti.n0, brow);
    tma_load_2d(sB + 3 * 8192, mb1, bar, ti.n0 + 64, brow);
  } else if constexpr (KIND == KIND_FFN2) {
    tma_load_2d(sA, ma, bar, kk, ti.m0);
    const int brow = ti.g * p.F + kk;
#pragma unroll
    for (int j = 0; j < 4; ++j) tma_load_2d(sB + j * 8192, mb0, bar, ti.n0 + 64 * j, brow);
  } else if constexpr (KIND == KIND_ROUTER) {
    // x is read once here: its lines go first when L2 needs room, so that
    // streaming it does not push other kernels' data (or their dirty lines)
    // out; the router weight, read by every CTA, stays
    tma_load_2d_hint(sA, ma, bar, kk, ti.m0, l2_policy_evict_first());
    tma_load_2d_hint(sB, mb0, bar, kk, 0, l2_policy_evict_last());
  } else if constexpr (KIND == KIND_DGRAD2) {
    tma_load_2d(sA, ma, bar, kk, ti.m0);
    tma_load_2d(sB, mb0, bar, kk, ti.g * p.F + ti.n0);
  } else if constexpr (KIND == KIND_DGRAD1) {
    tma_load_2d(sA, ma, bar, kk, ti.m0);
    if (kk < p.F) tma_load_2d(sB, mb0, bar, kk, ti.g * p.H + ti.n0);
    else tma_load_2d(sB, mb1, bar, kk - p.F, ti.g * p.H + ti.n0);
  } else if constexpr (KIND == KIND_WGRAD) {
    const int r = ti.krow0 + kk;
    tma_load_2d(sA, ma, bar, ti.m0, r);
    tma_load_2d(sA + 8192, ma, bar, ti.m0 + 64, r);
#pragma unroll
    for (int j = 0; j < 4; ++j) tma_load_2d(sB + j * 8192, mb0, bar, ti.n0 + 64 * j, r);
  } else if constexpr (KIND == KIND_ROUTER_DX) {
    tma_load_2d(sA, ma, bar, kk, ti.m0);
    const int erow = kk % p.Ep;
#pragma unroll
    for (int j = 0; j < 4; ++j) tma_load_2d(sB + j * 8192, mb0, bar, ti.n0 + 64 * j, erow);
  } else {  // ROUTER_DW: token block kb0 + kb; dL hi at sA, lo at sA + kABytes
    const int trow = (ti.kb0 + kb) * kBK;
    const int col = ti.m0;
    if (p.Ep <= kBM) {
      // one tile of experts: each box of x is read by one CTA; x goes first
      // when L2 needs room, dL (re-read by every tile of H) stays
      const uint64_t keep = l2_policy_evict_last(), stream = l2_policy_evict_first();
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        tma_load_2d_hint(sA + part * kABytes, ma, bar, col + part * p.Ep, trow, keep);
        tma_load_2d_hint(sA + part * kABytes + 8192, ma, bar, col + part * p.Ep + 64, trow, keep);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) tma_load_2d_hint(sB + j * 8192, mb0, bar, ti.n0 + 64 * j, trow, stream);
    } else {
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        tma_load_2d(sA + part * kABytes, ma, bar, col + part * p.Ep, trow);
        tma_load_2d(sA + part * kABytes + 8192, ma, bar, col + part * p.Ep + 64, trow);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) tma_load_2d(sB + j * 8192, mb0, bar, ti.n0 + 64 * j, trow);
    }
  }
}

// Bulk tensor store shared -> global (3-D box), tracked by bulk groups.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// wait until no committed bulk store of this thread still reads shared memory
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// wait until every committed bulk store of this thread has completed
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// router stage stride (128 x 64 of x and bn x 64 of the router weight; a
// multiple of 1024 bytes: bn is a multiple of 32) and the number of such
// stages in the ring
__host__ __device__ __forceinline__ int router_stage_bytes(int bn) { return kABytes + bn * 128; }
__host__ __device__ __forceinline__ int router_stages(int bn) {
  const int n = kRingBytes / router_stage_bytes(bn);
  return n < 8 ? n : 8;
}

template <int KIND>
__device__ __forceinline__ uint32_t stage_tx_bytes(const GemmParams& p) {
  if constexpr (KindTraits<KIND>::kNv) return 2 * kNvStageTx;                    // both CTAs' shares
  else if constexpr (KindTraits<KIND>::kMx) return 2 * kMxStageTx;               // both CTAs' shares
  else if constexpr (KIND == KIND_ROUTER) return router_stage_bytes(p.bn);
  else if constexpr (KindTraits<KIND>::kPair) return 2 * KindTraits<KIND>::kStageBytesK;  // both CTAs' shares
  else return KindTraits<KIND>::kStageBytesK;
}

}  // namespace moe

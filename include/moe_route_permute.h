/*
 * moe_route_permute.h -- C ABI of the GB300 (sm_103a) MoE layer hot path.
 *
 * The path is the single-GPU Route -> Dispatch -> Compute -> Combine of an MoE
 * layer, with a local permute in place of the all-to-all (report "Scalable
 * Training of Mixture-of-Experts Models with Megatron Core": summary page,
 * "Problem Definition", "Pipeline Flow" and "System Modules"; figures & tables
 * page, Fig. 1 and Fig. 2), and its training backward.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensors are dense, row-major, in DEVICE memory of the current CUDA
 *    device, and allocated by the caller. The library allocates nothing on the
 *    GPU and keeps no per-call state. Pointers must be 16-byte aligned
 *    (every device pointer an entry point takes, the fields of the structs
 *    it takes included, is checked: a misaligned one is MOE_ERR_INVALID_ARG).
 *  - bf16 tensors are passed as moe_bf16* (IEEE bfloat16 bit patterns).
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Every call only enqueues work on `stream` and returns; nothing synchronises
 *    the host, and counts/offsets stay on the device.
 *  - Return value: MOE_OK or a host-detected error (invalid argument,
 *    unsupported shape, workspace too small, CUDA launch error). On an error
 *    nothing has been enqueued. Errors detected on the device (a bounded wait
 *    that ran out, an index out of range) are recorded in a status word in the
 *    workspace and read back with moe_get_device_status().
 *  - Sizes: T tokens, H hidden, E experts, k experts per token, F expert FFN
 *    width, R = T*k routed rows, Fs shared-expert width.
 *  - Supported shapes: H and F multiples of 64; 1 <= k <= min(E, 16);
 *    E <= 256; E divisible by n_groups; Fs multiple of 64 (or 0);
 *    T >= 1 and T*k < 2^30.
 */
#ifndef MOE_ROUTE_PERMUTE_H
#define MOE_ROUTE_PERMUTE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t moe_bf16;

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,        /* null pointer, k > E, bad enum, ...        */
  MOE_ERR_UNSUPPORTED_SHAPE = 2,  /* outside the supported shapes above        */
  MOE_ERR_WORKSPACE_TOO_SMALL = 3,
  MOE_ERR_CUDA = 4,               /* a CUDA runtime/driver call failed          */
  MOE_ERR_DEVICE_TIMEOUT = 5,     /* device: a bounded wait ran out             */
  MOE_ERR_DEVICE_INDEX = 6        /* device: an expert or row index out of range */
} moe_status;

typedef enum { MOE_SCORE_SOFTMAX = 0, MOE_SCORE_SIGMOID = 1 } moe_score_fn;

/* Layer description. Router options (figures & tables page, Fig. 2: linear
 * projection, score function, top-k selection, load balancing):
 *   score        softmax over the E experts, or element-wise sigmoid;
 *   n_groups,
 *   topk_groups  group-limited selection: experts split into n_groups
 *                contiguous groups, a group scored by the sum of its two best
 *                selection values, only the best topk_groups groups eligible
 *                (1,1 = plain top-k);
 *   gate_scale   gates = gate_scale * score_i / sum over the k selected scores;
 *   aux_coeff    coefficient alpha of the load-balancing loss
 *                alpha * E * sum_e (c_e / (T k)) * mean_t p[t,e] (training);
 *   out_fp32     y (forward) and dx (backward) written as fp32 instead of bf16;
 *   inter_fp32   expert outputs y_perm and the shared-expert output kept in
 *                fp32 instead of bf16, and in the backward the input
 *                gradients of the routed rows (dx_perm) and of the shared
 *                expert likewise;
 *   force_balanced  force-balanced routing (throughput page, Table 11, where
 *                every benchmark configuration uses it): slot i of token t goes
 *                to expert (t k + i) mod E instead of the top-k, so each expert
 *                receives floor(T k / E) or one more rows; the scores, gates
 *                (renormalised over the assigned experts), aux statistics and
 *                the backward are computed as usual; the group limit and the
 *                expert bias do not apply. 0 or 1. */
typedef struct {
  int T, H, E, k, F;
  int F_shared;      /* 0 = no shared expert */
  int score;         /* moe_score_fn */
  int n_groups, topk_groups;
  float gate_scale;
  float aux_coeff;
  int out_fp32;
  int inter_fp32;
  int force_balanced;
} moe_config;

/* Tensors the training forward keeps for the backward (all caller-owned).
 * Shapes: topk_idx, row_id_map [T,k] int32; topk_gate [T,k] fp32;
 * logits [T,E] fp32 (router logits incl. logit_bias); counts [E] int32;
 * offsets [E+1] int32; x_perm [R,H] bf16; h13 [R,2F] bf16 (gate
 * pre-activation x W1 in columns [0,F), up projection x W3 in [F,2F));
 * a [R,F] bf16 (SiLU(h1)*h3); y_perm [R,H] bf16 (fp32 if inter_fp32);
 * aux_partials [4*ceil(T/128), E] fp32 (column sums of the full softmax over
 * consecutive 32-token slices; only when aux_coeff != 0, else may be NULL).
 * Memory-saving mode (captions page, Fig. 7 memory-efficient permutation and
 * Table 4 SwiGLU recompute): a and y_perm both NULL (one NULL alone is
 * MOE_ERR_INVALID_ARG). The forward then keeps them in the workspace only; the
 * backward, given the same NULLs, recomputes a = bf16(SiLU(h1) h3) from h13 in
 * the epilogue of the down-projection dgrad and takes the gate gradient there
 * as <da, a> / g (da = dy_perm W2^T, dy_perm = g dO; 0 where g = 0), which
 * equals <dO, y_perm> in exact arithmetic. Saves 2 R (F + H) bytes (bf16).
 * With a shared expert (F_shared > 0; figures & tables page, Fig. 40):
 * h13_shared [T,2Fs] bf16 (x Ws1 in columns [0,Fs), x Ws3 in [Fs,2Fs)) and
 * a_shared [T,Fs] bf16 (SiLU(h1) * h3) are required; otherwise unused. */
typedef struct {
  int32_t* topk_idx;
  float* topk_gate;
  float* logits;
  int32_t* row_id_map;
  int32_t* counts;
  int32_t* offsets;
  moe_bf16* x_perm;
  moe_bf16* h13;
  moe_bf16* a;
  void* y_perm;
  float* aux_partials;
  moe_bf16* h13_shared;
  moe_bf16* a_shared;
} moe_fwd_saved;

/* Bytes of device workspace the calls below need (training != 0: the
 * backward's needs included). The workspace is caller-owned scratch; its first
 * bytes hold the device status word. It must stay allocated until the enqueued
 * work has finished; two calls in flight at once must use two workspaces. */
size_t moe_workspace_bytes(const moe_config* cfg, int training);

/* Router (figures & tables page, Fig. 2; summary page, "System Modules",
 * Router: a learned linear layer + softmax choosing the top-k experts):
 *   L = x router_w^T (+ logit_bias),  x [T,H] bf16, router_w [E,H] bf16;
 *   scores = softmax(L) or sigmoid(L);
 *   selection on scores (+ expert_bias [E] fp32, selection only), optionally
 *   group-limited; ties go to the lower expert index; slots ordered by
 *   descending selection value;
 *   topk_gate[t,i] = gate_scale * score[e_i] / sum_j score[e_j].
 * Outputs topk_idx [T,k] int32, topk_gate [T,k] fp32; optional logits_out
 * [T,E] fp32 and aux_partials [4*ceil(T/128),E] fp32 (softmax column sums per
 * 32-token slice; rows past the last token are zero). expert_bias, logit_bias, logits_out, aux_partials may be
 * NULL. The bf16 products are exact and accumulate in fp32 on the tensor
 * cores. */
int moe_router_topk(const moe_config* cfg, const moe_bf16* x, const moe_bf16* router_w,
                    const float* expert_bias, const float* logit_bias,
                    int32_t* topk_idx, float* topk_gate, float* logits_out,
                    float* aux_partials, void* ws, size_t ws_bytes, void* stream);

/* Local dispatch (summary page, "Key Terms", Grouped GEMM; figures & tables
 * page, Fig. 7 and Fig. 20): counts[e] = number of (t,i) routed to e;
 * offsets [E+1] = exclusive prefix sum (offsets[E] = T*k); row_id_map[t,i] =
 * offsets[e] + number of tokens t' < t routed to e (rows grouped by expert, in
 * token order within an expert; dropless); x_perm[row_id_map[t,i]] = x[t].
 * Deterministic. Device errors: an index outside [0,E) sets
 * MOE_ERR_DEVICE_INDEX (that entry is skipped); a bounded wait of the scan sets
 * MOE_ERR_DEVICE_TIMEOUT. */
int moe_permute(const moe_config* cfg, const moe_bf16* x, const int32_t* topk_idx,
                moe_bf16* x_perm, int32_t* row_id_map, int32_t* counts, int32_t* offsets,
                void* ws, size_t ws_bytes, void* stream);

/* moe_permute without a workspace. The report has no counterpart of this
 * entry point; it exists for callers that cannot allocate device memory: a
 * serving engine that fixes its device memory at start-up and forbids
 * allocation afterwards, a plug-in whose host runtime owns every device
 * buffer, or code for which a cudaMalloc could fail or synchronise at the
 * wrong moment. Same arguments and results as moe_permute minus `ws`.
 * Its scratch (status word, chunk ticket, lookback words) is a fixed array of
 * about 1 MiB inside the library, held by every GPU that loads the library
 * until the process exits; it serves problems with ceil(T/64)*E <= 262144
 * (for example T <= 65536 with E = 256). Larger problems are rejected with
 * MOE_ERR_UNSUPPORTED_SHAPE (and a message on stderr) before any GPU work.
 * The first call on a device looks up the array's device address (set-up with
 * that device current); make that first call before any stream capture. The
 * call allocates nothing: it clears the part of the array it uses with
 * cudaMemsetAsync on `stream` and launches the permute kernels. All calls
 * share the one array, so calls that overlap on the GPU (other streams or
 * threads) race and give wrong results; serialise them. Device-side errors
 * (an index outside [0,E) skipped, a bounded wait that ran out) go to the
 * status word of that array, which each call clears first:
 * moe_noalloc_get_device_status reads the most recent call's. */
int moe_permute_noalloc(const moe_config* cfg, const moe_bf16* x, const int32_t* topk_idx,
                        moe_bf16* x_perm, int32_t* row_id_map, int32_t* counts, int32_t* offsets,
                        void* stream);

/* Synchronises `stream`, returns in *status_out the device-side status of the
 * most recent moe_permute_noalloc call on the current device (MOE_OK if none;
 * MOE_ERR_DEVICE_INDEX, MOE_ERR_DEVICE_TIMEOUT as for moe_permute) and
 * clears it. Allocates nothing; for tests and debugging. */
int moe_noalloc_get_device_status(void* stream, int* status_out);

/* Grouped SwiGLU experts (summary page, "Key Terms", Grouped GEMM and
 * "System Modules", Experts; figures & tables page, Table 4): for each expert
 * e, rows offsets[e]..offsets[e+1] of x_perm [R,H]:
 *   h1 = x W1[e], h3 = x W3[e]   (W1, W3 [E,H,F] bf16; W1 is the gate),
 *   a  = bf16(SiLU(h1) * h3),
 *   y_perm = a W2[e]             (W2 [E,F,H] bf16), bf16 (fp32 if inter_fp32).
 * `offsets` is read on the device (no host synchronisation). h13_save [R,2F]
 * and a_save [R,F] are optional outputs for the backward; without a_save the
 * activation lives in the workspace. */
int moe_grouped_swiglu_ffn(const moe_config* cfg, const moe_bf16* x_perm, const int32_t* offsets,
                           const moe_bf16* W1, const moe_bf16* W3, const moe_bf16* W2,
                           moe_bf16* h13_save, moe_bf16* a_save, void* y_perm,
                           void* ws, size_t ws_bytes, void* stream);

/* Combine (summary page, "Problem Definition" and "System Modules", Combiner;
 * figures & tables page, Fig. 40 for the shared expert):
 *   y[t] = sum_{i=0..k-1} topk_gate[t,i] * y_perm[row_id_map[t,i]] (+ shared_out[t]),
 * reduced in fp32 in slot order. y_perm and shared_out are bf16 (fp32 if
 * inter_fp32); y [T,H] is bf16 (fp32 if out_fp32). shared_out may be NULL. A
 * row index of -1 in row_id_map (a slot moe_permute dropped for an expert
 * index outside [0,E)) is weighted 0 (row 0 of y_perm is read in its place). */
int moe_unpermute_combine(const moe_config* cfg, const void* y_perm, const int32_t* row_id_map,
                          const float* topk_gate, const void* shared_out, void* y, void* stream);

/* Whole layer forward = router -> permute -> grouped SwiGLU -> (shared
 * expert) -> combine. Ws1, Ws3 [H,Fs], Ws2 [Fs,H] bf16 when F_shared > 0
 * (the shared expert processes every token and is added ungated).
 * saved != NULL (training): every field of *saved must be set (except a and
 * y_perm together, the memory-saving mode, and aux_partials when aux_coeff is
 * 0) and receives the tensors for moe_layer_bwd; saved == NULL (inference):
 * intermediates live in the workspace. */
int moe_layer_fwd(const moe_config* cfg, const moe_bf16* x, const moe_bf16* router_w,
                  const float* expert_bias, const float* logit_bias,
                  const moe_bf16* W1, const moe_bf16* W3, const moe_bf16* W2,
                  const moe_bf16* Ws1, const moe_bf16* Ws3, const moe_bf16* Ws2,
                  void* y, const moe_fwd_saved* saved, void* ws, size_t ws_bytes, void* stream);

/* Whole layer backward for the loss <dO, y> + L_aux (the chain rule of the
 * forward; top-k selection and counts carry no gradient). dO [T,H] bf16.
 * Outputs: dx [T,H] (bf16, fp32 if out_fp32); dW_router [E,H], dW1, dW3
 * [E,H,F], dW2 [E,F,H] fp32 (overwritten, zero for experts with no tokens);
 * aux_loss_out (1 fp32, may be NULL; written when aux_coeff != 0).
 * Shared expert (F_shared > 0; figures & tables page, Fig. 40: it processes
 * every token and is added ungated, so its output gradient is dO): Ws1, Ws3
 * [H,Fs], Ws2 [Fs,H] bf16 as in the forward, saved->h13_shared and
 * saved->a_shared from the training forward, and the outputs dWs1, dWs3
 * [H,Fs], dWs2 [Fs,H] fp32; its input gradient is added to dx. All six are
 * ignored (may be NULL) when F_shared == 0. With saved->a and saved->y_perm
 * NULL it runs the memory-saving backward of the routed experts (see
 * moe_fwd_saved); the workspace must be the training size either way. */
int moe_layer_bwd(const moe_config* cfg, const moe_bf16* dO, const moe_bf16* x,
                  const moe_bf16* router_w, const moe_bf16* W1, const moe_bf16* W3,
                  const moe_bf16* W2, const moe_bf16* Ws1, const moe_bf16* Ws3,
                  const moe_bf16* Ws2, const moe_fwd_saved* saved,
                  void* dx, float* dW_router, float* dW1, float* dW3, float* dW2,
                  float* dWs1, float* dWs3, float* dWs2,
                  float* aux_loss_out, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * MXFP8 expert GEMMs (forward). The report benchmarks its Blackwell runs with
 * MXFP8, microscaling FP8 (figures & tables page, Table 11 "Dtype" and
 * Fig. 30) without defining it; the format here is the OCP Microscaling (MX)
 * v1.0 MXFP8: blocks of 32 consecutive elements along a GEMM operand's K share
 * one E8M0 scale 2^s (byte s + 127), s = floor(log2 max|v|) - 8 clamped to
 * [-127, 127] (-127 for an all-zero block); elements are E4M3 (bias 7, no
 * infinities) v / 2^s rounded to nearest, ties to even, saturating at +-448.
 * Requires H and F multiples of 128.
 * ------------------------------------------------------------------------- */

/* Quantised expert weights, device buffers owned by the caller (sizes from
 * moe_mx_weight_bytes), written by moe_mx_quantize_weights:
 *   w13  [E][2][F][H] E4M3: per expert W1[e]^T then W3[e]^T (K = H contiguous);
 *   w2   [E][H][F]    E4M3: W2[e]^T (K = F contiguous);
 *   sf13, sf2: their E8M0 scales in the tile-ready layout of the FP8 GEMMs
 *   (opaque: blocks of 2 x 512 bytes per expert, 96-column (w13: 96 W1 +
 *   96 W3 rows) or 192-column (w2) tile and 128-element k block; byte
 *   512 b + 16 r + 4 c + s holds the scale of tile row 128 b + 32 c + r,
 *   32-element K block 4 kb + s; unused bytes zero). */
typedef struct {
  uint8_t* w13;
  uint8_t* sf13;
  uint8_t* w2;
  uint8_t* sf2;
} moe_mx_weights;

/* Bytes of the moe_mx_weights buffers: which = 0 w13, 1 sf13, 2 w2, 3 sf2
 * (0 for an invalid config or shape). */
size_t moe_mx_weight_bytes(const moe_config* cfg, int which);

/* Quantise the bf16 expert weights W1, W3 [E,H,F] (blocks along H) and W2
 * [E,F,H] (blocks along F) into *w. Enqueues on `stream`. */
int moe_mx_quantize_weights(const moe_config* cfg, const moe_bf16* W1, const moe_bf16* W3,
                            const moe_bf16* W2, const moe_mx_weights* w, void* stream);

/* Row-major MXFP8 quantisation of x [M,K] bf16 (K a multiple of 32, blocks
 * along K): q [M,K] E4M3 codes, scales [M,K/32] E8M0 bytes. */
int moe_mx_quantize(const moe_bf16* x, long long M, int K, uint8_t* q, uint8_t* scales, void* stream);

/* Workspace bytes of moe_layer_fwd_mxfp8. */
size_t moe_mx_workspace_bytes(const moe_config* cfg);

/* Whole layer forward with MXFP8 expert GEMMs: router and combine as in
 * moe_layer_fwd; the permute quantises x's rows (blocks along H) as it
 * scatters them; gate/up GEMM h = Q(x_perm) [Q(W1_e) | Q(W3_e)] (fp32
 * accumulation) with a = SiLU(h1) h3 quantised in its epilogue (blocks along
 * F); down GEMM y_perm = Q(a) Q(W2_e), stored bf16 (fp32 if inter_fp32); the
 * shared expert (F_shared > 0) runs in bf16. y [T,H] bf16 (fp32 if out_fp32).
 * Inference: intermediates live in the workspace. */
int moe_layer_fwd_mxfp8(const moe_config* cfg, const moe_bf16* x, const moe_bf16* router_w,
                        const float* expert_bias, const float* logit_bias, const moe_mx_weights* w,
                        const moe_bf16* Ws1, const moe_bf16* Ws3, const moe_bf16* Ws2, void* y,
                        void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * MXFP8 training step: the forward above saving what the backward needs, and
 * a backward whose two data-gradient GEMMs run on MXFP8 operands, each
 * quantised along that GEMM's contraction axis (the report's Blackwell
 * training runs use MXFP8, figures & tables page, Table 11 and Fig. 30; the
 * split of the recipe is this library's reading):
 *   da      = Q(dy_perm) Q(W2_e)^T                  (blocks along H; fp32, not stored)
 *   dh1     = da h3 SiLU'(h1), dh3 = da SiLU(h1)    (saved bf16 h13; bf16)
 *   dx_perm = bf16(Q([dh1 | dh3]) Q([W1_e | W3_e])^T)  (blocks along 2F)
 * and the weight gradients (fp32 out) dW2_e = a_e^T dy_perm_e, with
 * a = bf16(SiLU(h1) h3) recomputed from the saved h13, and
 * dW1_e | dW3_e = x_perm_e^T [dh1 | dh3]: in bf16 on the tensor cores, or with
 * mx_wgrad set as MXFP8 GEMMs whose operands are quantised along each
 * expert's tokens (blocks of 32 from the expert's first row, a last partial
 * block zero-padded). Routing, combine, their backward and the router
 * backward are those of the bf16 layer. Requires H and F multiples of 128
 * and F_shared == 0.
 * Every call below enqueues on `stream` and returns without a host sync; it
 * returns MOE_ERR_INVALID_ARG for a null or misaligned pointer,
 * MOE_ERR_UNSUPPORTED_SHAPE for a shape outside the above,
 * MOE_ERR_WORKSPACE_TOO_SMALL for ws_bytes below moe_mx_train_workspace_bytes
 * (which includes the buffers of the MXFP8 weight gradients), before any CUDA
 * work; device-detected errors go to the workspace's status word.
 * ------------------------------------------------------------------------- */

/* The weights of the two data-gradient GEMMs, device buffers owned by the
 * caller (sizes from moe_mx_bwd_weight_bytes), written by
 * moe_mx_quantize_bwd_weights:
 *   w2h  [E][F][H]  E4M3: W2[e] quantised along H (K = H contiguous);
 *   w13f [E][H][2F] E4M3: row h = W1[e][h][:] then W3[e][h][:], quantised
 *                   along F (K = 2F contiguous);
 *   sf2h, sf13f: their E8M0 scales in the tile-ready layout of moe_mx_weights
 *   (192-row tiles: F rows for w2h, H rows for w13f; w13f's k blocks
 *   0 .. F/128 - 1 hold W1, the rest W3). */
typedef struct {
  uint8_t* w2h;
  uint8_t* sf2h;
  uint8_t* w13f;
  uint8_t* sf13f;
} moe_mx_bwd_weights;

/* Bytes of the moe_mx_bwd_weights buffers: which = 0 w2h, 1 sf2h, 2 w13f,
 * 3 sf13f (0 for an invalid config or shape). */
size_t moe_mx_bwd_weight_bytes(const moe_config* cfg, int which);

/* Quantise W1, W3 [E,H,F] (blocks along F) and W2 [E,F,H] (blocks along H)
 * into *w. Enqueues on `stream`. */
int moe_mx_quantize_bwd_weights(const moe_config* cfg, const moe_bf16* W1, const moe_bf16* W3,
                                const moe_bf16* W2, const moe_mx_bwd_weights* w, void* stream);

/* Workspace bytes of moe_layer_fwd_mxfp8_train and moe_layer_bwd_mxfp8 (one
 * workspace serves both; 0 for an unsupported config). */
size_t moe_mx_train_workspace_bytes(const moe_config* cfg);

/* Training forward of the MXFP8 layer: the computation of
 * moe_layer_fwd_mxfp8 (no shared expert) that also fills *saved: topk_idx,
 * topk_gate, logits, row_id_map, counts, offsets, x_perm (bf16 rows, for the
 * weight gradient), h13 (bf16 h1 | h3 from the gate/up GEMM's fp32
 * accumulators), y_perm, aux_partials (when aux_coeff != 0). saved->a is
 * not used. Every saved buffer is required (MOE_ERR_INVALID_ARG otherwise). */
int moe_layer_fwd_mxfp8_train(const moe_config* cfg, const moe_bf16* x, const moe_bf16* router_w,
                              const float* expert_bias, const float* logit_bias, const moe_mx_weights* w,
                              void* y, const moe_fwd_saved* saved, void* ws, size_t ws_bytes, void* stream);

/* Backward of the MXFP8 training step for the loss <dO, y> + L_aux, given the
 * forward's saved tensors (the workspace need not hold the forward's): outputs as moe_layer_bwd
 * (dx, dW_router, dW1, dW3, dW2 fp32, aux_loss_out). mx_wgrad != 0: MXFP8
 * weight gradients (see above), else bf16. */
int moe_layer_bwd_mxfp8(const moe_config* cfg, const moe_bf16* dO, const moe_bf16* x,
                        const moe_bf16* router_w, const moe_mx_bwd_weights* w,
                        const moe_fwd_saved* saved, void* dx, float* dW_router, float* dW1,
                        float* dW3, float* dW2, float* aux_loss_out, int mx_wgrad, void* ws,
                        size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * NVFP4 grouped expert GEMM. The report lists NVFP4 among its precisions
 * (summary page, "Modeling" and "Key Terms") without defining it; the format
 * here is NVIDIA's NVFP4: E2M1 elements (magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6,
 * round to nearest even, saturating), a positive E4M3 scale per 16 consecutive
 * elements along K and an fp32 tensor scale g = amax / (6 * 448) (1 for a zero
 * tensor); in fp32: s_b = E4M3(fp32(amax_b / 6) / g), q = E2M1(v / fp32(s_b g)).
 * Codes are packed two per byte, element 2j in the low nibble.
 * Requires K a multiple of 256, N a multiple of 8, E <= 256.
 * ------------------------------------------------------------------------- */

/* Bytes of the quantised weights of E experts W[E][K][N]: which = 0 codes
 * [E][N][K/2] (K-major), 1 tile-ready scales (opaque: per expert, 192-row n
 * tile and 256-element k block, two blocks of 4 x 512 bytes; byte
 * 2048 b + 512 s + 16 r + 4 c + j = scale of tile row 128 b + 32 c + r,
 * 16-element block 4 s + j; unused bytes zero), 2 tensor scales [E] fp32. */
size_t moe_nv_weight_bytes(int E, int K, int N, int which);

/* Quantise W [E][K][N] bf16 (each expert a tensor of its own, blocks along K)
 * into wq, sf and g. */
int moe_nv_quantize_weights(int E, int K, int N, const moe_bf16* W, uint8_t* wq, uint8_t* sf, float* g,
                            void* stream);

/* Row-major NVFP4 quantisation of x [M,K] bf16 as one tensor (blocks along K):
 * q [M][K/2] codes, scales [M][K/16] E4M3 bytes, *g the tensor scale. */
int moe_nv_quantize(const moe_bf16* x, long long M, int K, uint8_t* q, uint8_t* scales, float* g, void* stream);

/* Workspace bytes of moe_nv_grouped_gemm. */
size_t moe_nv_workspace_bytes(int E, long long R, int K);

/* Grouped expert GEMM on NVFP4 operands: rows offsets[e]..offsets[e+1] of
 * x [R,K] bf16 (quantised here as one tensor, blocks along K) times expert
 * e's quantised weights (moe_nv_quantize_weights): y [R,N] bf16 =
 * g_x g_e sum_k Q(x)[r,k] Q(W_e)[k,n], fp32 accumulation. offsets [E+1] is
 * read on the device. */
int moe_nv_grouped_gemm(int E, long long R, int K, int N, const moe_bf16* x, const int32_t* offsets,
                        const uint8_t* wq, const uint8_t* sf, const float* g, moe_bf16* y, void* ws,
                        size_t ws_bytes, void* stream);

/* NVFP4 layer forward. Quantised weights (device buffers owned by the caller,
 * sizes from moe_nv_layer_weight_bytes, which = 0..5 in field order): w13 /
 * g13 are [W1_e | W3_e] (H x 2F, one tensor per expert: codes [E][2F][H/2],
 * W1's columns then W3's) and sf13 their scales in the gate/up GEMM's tiles
 * (opaque: tile t = 96 W1 columns 96 t .. then the same W3 columns, blocks as
 * in moe_nv_quantize_weights); w2 / sf2 / g2 are W2 (K = F, N = H) in the
 * layout of moe_nv_quantize_weights. */
typedef struct {
  uint8_t* w13;
  uint8_t* sf13;
  float* g13;
  uint8_t* w2;
  uint8_t* sf2;
  float* g2;
} moe_nv_weights;

size_t moe_nv_layer_weight_bytes(const moe_config* cfg, int which);

/* Quantise W1, W3 [E,H,F] and W2 [E,F,H] bf16 into *w. */
int moe_nv_quantize_layer_weights(const moe_config* cfg, const moe_bf16* W1, const moe_bf16* W3, const moe_bf16* W2,
                                  const moe_nv_weights* w, void* stream);

/* Workspace bytes of moe_layer_fwd_nvfp4. */
size_t moe_nv_workspace_bytes_layer(const moe_config* cfg);

/* Whole layer forward with NVFP4 expert GEMMs: router, permute and combine as
 * in moe_layer_fwd; the routed rows x_perm (one tensor: x's maximum) are
 * quantised, the gate/up GEMM forms h = bf16(g_x g_e Q(x_perm) Q([W1|W3]))
 * and writes a = bf16(SiLU(h1) h3) [R, F] with its maximum, a is quantised as
 * one tensor, and the down GEMM writes y_perm = bf16(g_a g_e Q(a) Q(W2)). y [T,H]
 * bf16 (fp32 if out_fp32). Requires H and F multiples of 256, F_shared = 0 and
 * inter_fp32 = 0. Inference: intermediates live in the workspace. */
int moe_layer_fwd_nvfp4(const moe_config* cfg, const moe_bf16* x, const moe_bf16* router_w,
                        const float* expert_bias, const float* logit_bias, const moe_nv_weights* w, void* y, void* ws,
                        size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * NVFP4 training step. The report trains in NVFP4 (summary page, "Modeling";
 * "Key Terms") without giving a recipe; the reading here follows the NVFP4
 * forward: each data-gradient GEMM quantises both operands along its own
 * contraction axis, the operand made of routed rows as ONE tensor (one tensor
 * scale over every routed row), each expert's weight as a tensor of its own;
 * the weight gradients stay bf16 x bf16 with fp32 output.
 * ------------------------------------------------------------------------- */

/* The data gradients' quantised weights (device buffers owned by the caller,
 * sizes from moe_nv_bwd_weight_bytes, which = 0..5 in field order): w2h /
 * sf2h / g2h are W2_e [F, H] row-wise along H (codes [E][F][H/2]; scales in
 * the layout of moe_nv_quantize_weights with K = H, N = F); w13f / sf13f /
 * g13f are [W1_e | W3_e] [H, 2F] row-wise along 2F, one tensor per expert
 * (codes [E][H][F]: W1's F columns then W3's; K = 2F, N = H). */
typedef struct {
  uint8_t* w2h;
  uint8_t* sf2h;
  float* g2h;
  uint8_t* w13f;
  uint8_t* sf13f;
  float* g13f;
} moe_nv_bwd_weights;

size_t moe_nv_bwd_weight_bytes(const moe_config* cfg, int which);

/* Quantise W1, W3 [E,H,F] and W2 [E,F,H] bf16 into *w (the data gradients'
 * weights). */
int moe_nv_quantize_bwd_weights(const moe_config* cfg, const moe_bf16* W1, const moe_bf16* W3, const moe_bf16* W2,
                                const moe_nv_bwd_weights* w, void* stream);

/* Both weight copies of the NVFP4 training step in one call, as a training
 * loop refreshes them once per optimizer step: the same codes, scales and
 * tensor scales as moe_nv_quantize_layer_weights into *fw and
 * moe_nv_quantize_bwd_weights into *bw, with each per-expert maximum taken once
 * (the two copies quantise the same per-expert tensors, so g13f = g13 and
 * g2h = g2). Buffers as those two calls take them. Returns MOE_ERR_INVALID_ARG
 * for a null or misaligned pointer, MOE_ERR_UNSUPPORTED_SHAPE where the NVFP4
 * layer does not apply. */
int moe_nv_quantize_train_weights(const moe_config* cfg, const moe_bf16* W1, const moe_bf16* W3,
                                  const moe_bf16* W2, const moe_nv_weights* fw, const moe_nv_bwd_weights* bw,
                                  void* stream);

/* Workspace bytes of moe_layer_fwd_nvfp4_train / moe_layer_bwd_nvfp4 (one
 * workspace serves both). 0 for an unsupported shape. */
size_t moe_nv_train_workspace_bytes(const moe_config* cfg);

/* NVFP4 layer forward that keeps what the backward needs: as
 * moe_layer_fwd_nvfp4, with the router's logits (and aux partials when
 * aux_coeff != 0), routing, x_perm (bf16 rows), h13 (the stored bf16 gate/up
 * output), a and y_perm (bf16) written to *saved (all of them required). */
int moe_layer_fwd_nvfp4_train(const moe_config* cfg, const moe_bf16* x, const moe_bf16* router_w,
                              const float* expert_bias, const float* logit_bias, const moe_nv_weights* w, void* y,
                              const moe_fwd_saved* saved, void* ws, size_t ws_bytes, void* stream);

/* Backward of the NVFP4 layer for the loss <dO, y> + L_aux (outputs as in
 * moe_layer_bwd, no shared expert): dy_perm = g dO (bf16); da = Q(dy_perm)
 * Q(W2_e)^T (fp32, blocks along H); dh1 = da h3 SiLU'(h1), dh3 = da SiLU(h1)
 * (bf16); dx_perm = Q([dh1 | dh3]) Q([W1_e | W3_e])^T (bf16, blocks along
 * 2F); dW2 = a^T dy_perm, dW1 | dW3 = x_perm^T [dh1 | dh3] (bf16 operands,
 * fp32); the router backward and dx as in moe_layer_bwd. `saved` is the one
 * moe_layer_fwd_nvfp4_train filled, `ws` the same workspace. */
int moe_layer_bwd_nvfp4(const moe_config* cfg, const moe_bf16* dO, const moe_bf16* x, const moe_bf16* router_w,
                        const moe_nv_bwd_weights* w, const moe_fwd_saved* saved, void* dx, float* dW_router,
                        float* dW1, float* dW3, float* dW2, float* aux_loss_out, void* ws, size_t ws_bytes,
                        void* stream);

/* Synchronises `stream`, returns in *status_out the first device-side error
 * recorded in `ws` since the last read (MOE_OK if none) and clears it. For
 * tests and debugging; the hot path never calls it. */
int moe_get_device_status(void* ws, void* stream, int* status_out);

/* Static text for a moe_status value. */
const char* moe_status_string(int status);

/* Size in bytes of the ABI structs as this library was compiled:
 * which = 0 -> sizeof(moe_config), 1 -> sizeof(moe_fwd_saved), else 0.
 * For bindings that mirror the structs to check their layout. */
size_t moe_abi_struct_bytes(int which);

/* Test hooks (not for production use). moe_debug_set_wait_limit_ns sets the
 * limit of every bounded device wait (default 2e9 ns = 2 s; 0 restores the
 * default). moe_debug_set_fault(1) makes the permute scan's first token chunk
 * skip publishing its counts, so that the other chunks' waits run out and the
 * device status reports MOE_ERR_DEVICE_TIMEOUT; moe_debug_set_fault(0) turns
 * it off. Both are process-wide. */
void moe_debug_set_wait_limit_ns(long long ns);
void moe_debug_set_fault(int fault);

/* Benchmark support. moe_profile_start(capacity) makes the entry points above
 * record a CUDA event on the caller's stream at the start of each layer call
 * and after each of its stages (up to `capacity` events; stage tags: 0 call
 * start, 1 router, 2 permute, 3/4 expert GEMM 1/2, 5/6 shared expert GEMM 1/2,
 * 7 combine, 10 combine backward, 11 router backward (element-wise), 12 down
 * projection data gradient + SwiGLU backward, 13 down projection weight
 * gradient, 14 gate/up data gradient, 15 gate/up weight gradient, 16 router
 * data gradient, 17 permute backward, 18 router weight gradient, 19 aux loss,
 * 20 NVFP4 quantisation of a GEMM's activations, 21 NVFP4 grouped GEMM, 22
 * MXFP8 token-axis quantisation, 24 MXFP8 down data gradient + SwiGLU
 * backward, 25 MXFP8 gate/up data gradient, 26-29 the shared expert's down
 * data gradient + SwiGLU backward, down weight gradient, gate/up data
 * gradient, gate/up weight gradient; 30 moe_read_ceiling, 31
 * moe_write_ceiling; 32 NVFP4 down data gradient (da), 33 NVFP4 SwiGLU
 * backward, 34 NVFP4 gate/up data gradient).
 * moe_profile_stop() stops recording. moe_profile_read() waits for the events
 * and returns their number; ms[i] is the time from event i-1 to event i
 * (0 for call starts). moe_debug_launch_count() returns the number of kernels
 * the library has launched in this process. */
void moe_profile_start(int capacity);
void moe_profile_stop(void);
int moe_profile_read(int* tags, float* ms, int max);
unsigned long long moe_debug_launch_count(void);

/* 1 when this library is the bounds-check build (compiled with
 * -DMOE_BOUNDS_CHECK): its element-wise kernels (combine, combine backward,
 * permute backward, router backward) range-check every row index they read
 * from row_id_map against [-1, T*k) and every expert index from topk_idx
 * against [0, E); an index outside records MOE_ERR_DEVICE_INDEX in the
 * workspace status word (read by moe_get_device_status; the standalone
 * moe_unpermute_combine has none and only skips it) and is skipped instead of
 * read. 0 for the default build, which skips the row index -1 (a slot
 * moe_permute dropped) and trusts the rest. */
int moe_bounds_checked(void);

/* Measurement helper, not a step of the layer: reads the `bytes` bytes at
 * `buf` (device memory, 16-byte aligned, bytes a multiple of 16) once, with
 * coalesced 16-byte loads from a grid of four 512-thread CTAs per SM, and
 * stores nothing unless the data hashes to one fixed word (then one word per
 * CTA into `sink`, device memory of at least 16 * SMs bytes). One launch timed
 * alone (cold L2) gives the rate at which a single kernel reading that many
 * bytes can stream them: the practical ceiling of a read-bound kernel of that
 * size, below the long-copy peak by the launch's ramp-up and tail. Returns
 * MOE_ERR_INVALID_ARG for a null or misaligned pointer or size. */
int moe_read_ceiling(const void* buf, size_t bytes, unsigned* sink, void* stream);

/* Measurement helper, not a step of the layer: fills the `bytes` bytes at
 * `buf` (device memory, 16-byte aligned, bytes a multiple of 16) with the
 * 32-bit `word`, 16-byte stores from a grid of four 512-thread CTAs per SM. One
 * launch over a buffer much larger than L2, timed alone, gives the rate at
 * which HBM absorbs writes: the bound of a kernel whose time goes to storing
 * its output (the fp32 weight gradients). Returns MOE_ERR_INVALID_ARG for a
 * null or misaligned pointer or size. */
int moe_write_ceiling(void* buf, size_t bytes, unsigned word, void* stream);

/* Test hook: byte offset, inside a workspace of moe_workspace_bytes(cfg,
 * training), of an intermediate the layer keeps there, so that tests can read
 * the bf16 operands the backward's GEMMs consumed: which = 0 dy_perm [R,H]
 * (g * dO per routed row), 1 dh13 [R,2F] (dh1 in columns [0,F), dh3 in
 * [F,2F)), 2 a [R,F] (the activation of the memory-saving mode), 3 dx_perm
 * [R,H], all bf16 (dx_perm fp32 with inter_fp32), rows grouped by expert as
 * x_perm. Valid until the next call
 * that uses the workspace. Returns (size_t)-1 for an invalid config, an
 * unknown `which`, or a buffer the workspace does not hold (training == 0 and
 * which != 2). */
size_t moe_debug_workspace_offset(const moe_config* cfg, int training, int which);

#ifdef __cplusplus
}
#endif
#endif /* MOE_ROUTE_PERMUTE_H */

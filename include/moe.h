/*
 * moe.h - C ABI of the GB300 (sm_103a) dropless mixture-of-experts expert
 * layer: router, permutation builder, grouped expert GEMMs (forward and
 * backward) and the MXFP8 quantiser.
 *
 * Sources of the operations (web pages on the method, cited by title and
 * section):
 *   [MM] "Prime Intellect releases Prime Mega MoE: a trainable fused MoE
 *        kernel" (MarkTechPost): "In brief" (128 experts, top-8 routing;
 *        BF16 and MXFP8 on Blackwell), "How does the fused kernel work?"
 *        (dispatch, two expert linears, SwiGLU, combine in one fused path;
 *        GPU-only scratch buffers; the trainable backward; fp8_bwd = BF16
 *        forward with FP8 backward).
 *   [OB] "Prime Intellect Mega MoE" digest (neurobober), "Overlapping
 *        Backward Pass": activation gradients need the weights but not the
 *        weight gradients, so the two halves of the backward can overlap.
 *   [TE] "Accelerating dropless MoE in JAX with NVIDIA Transformer Engine"
 *        (aikraft): 02 dropless routing over ragged per-expert groups; 03
 *        group-aware MXFP8 quantisation; "Optimisation 1: grouped GEMM" (all
 *        experts in one launch over their real token counts, counts never
 *        copied to the host); "Optimisation 2" (local reordering on dispatch,
 *        summation of expert outputs on combine).
 *
 * Conventions shared by every call
 *   - All pointers except `dims`, `route` and the pointer-holding structs
 *     themselves are DEVICE pointers, 16-byte aligned, row-major, owned by
 *     the caller.  The library never allocates, never frees and never
 *     synchronises the stream; every call is asynchronous on `stream` (a
 *     cudaStream_t, passed as void*; NULL is the legacy default stream).
 *   - The return value reports only checks done on the host before any
 *     launch (MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED) and launch failures
 *     (MOE_ERR_CUDA).  Errors found on the device (MOE_ERR_TIMEOUT,
 *     MOE_ERR_BAD_INDEX, ...) are written to `*dev_status`, a device int32
 *     that the caller zeroes before the call and reads when it chooses; the
 *     first error written wins.  Device-detected errors never trap: the
 *     failing kernel skips the bad access, records the code and returns.
 *   - Token counts stay on the device: no call copies data to the host, so
 *     every call can be captured in a CUDA graph.
 *   - Storage dtype follows dims->mode: MOE_F32 uses float for X, W13, W2, Y,
 *     dY, dX, dW13, dW2 (tensor cores run TF32); the other modes use bf16 for
 *     those tensors (MOE_MXFP8 and MOE_FP8_BWD quantise internally).
 *   - Gradients overwrite their outputs; they do not accumulate.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,  /* bad size, null or misaligned pointer, short buffer */
  MOE_ERR_UNSUPPORTED = 2,  /* valid request this build does not implement      */
  MOE_ERR_CUDA = 3,         /* a CUDA launch or driver call failed              */
  MOE_ERR_TIMEOUT = 4,      /* device: a bounded wait ran out (kernel returned) */
  MOE_ERR_BAD_INDEX = 5,    /* device: an expert index outside [0, E) was seen  */
  MOE_ERR_BAD_INPUT = 6     /* device: an input the operation is not defined for
                               (a NaN logit; a token whose logits are all -inf) */
} moe_status;

typedef enum {
  MOE_F32 = 0,      /* fp32 storage, TF32 tensor-core GEMMs                       */
  MOE_BF16 = 1,     /* bf16 storage, bf16 GEMMs with fp32 accumulation            */
  MOE_MXFP8 = 2,    /* bf16 storage, MXFP8 GEMMs in forward and backward          */
  MOE_FP8_BWD = 3   /* bf16 storage, bf16 forward GEMMs, MXFP8 backward GEMMs     */
} moe_mode;
/* The MXFP8 GEMMs (MOE_MXFP8 forward and backward, MOE_FP8_BWD backward)
 * need I a multiple of 384 and H of 128; other shapes return
 * MOE_ERR_UNSUPPORTED from the call that would run them. */

/* Problem shape.  T tokens of width H, E experts of intermediate size I, each
 * token routed to top_k experts ([MM] "In brief": top-8 of 128).  Limits:
 * 1 <= top_k <= min(E, 32); 1 <= E <= 1024; H and I multiples of 64;
 * T*top_k + 128*E < 2^31. */
typedef struct {
  int T, H, E, I, top_k;
  moe_mode mode;
  int save_for_backward;   /* forward also stores H13 (needed by moe_backward) */
} moe_dims;

/* Routing result (moe_route output, moe_forward / moe_backward input).
 * Assignment a = t*top_k + j is slot j of token t; slot order is descending
 * logit with ties to the lower expert index.  Rows of expert e occupy the
 * storage range [padded_offsets[e], padded_offsets[e+1]) whose length is
 * counts[e] rounded up to 128; within an expert, rows follow ascending a.
 *   topk_idx       int32 [T, top_k]
 *   gate           float [T, top_k]  softmax over E, renormalised over the k
 *   counts         int32 [E]
 *   offsets        int32 [E+1]       exclusive scan of counts
 *   padded_offsets int32 [E+1]       exclusive scan of roundup(counts, 128)
 *   row_of_assign  int32 [T*top_k]
 *   assign_of_row  int32 [moe_max_rows(dims)]  a of each row, -1 on pad rows
 *                                    and on rows >= padded_offsets[E] */
typedef struct {
  int32_t* topk_idx;
  float* gate;
  int32_t* counts;
  int32_t* offsets;
  int32_t* padded_offsets;
  int32_t* row_of_assign;
  int32_t* assign_of_row;
} moe_route_out;

/* Byte offsets of the tensors inside the `saved` buffer written by
 * moe_forward and read by moe_backward (rows = moe_max_rows(dims), elem =
 * 4 bytes for MOE_F32, else 2):
 *   x_perm [rows, H]   gathered tokens, expert-major, zero pad rows
 *                      (zero-sized in MOE_MXFP8 mode: the dispatch gather
 *                      goes straight into its MXFP8 encodings, x_col below)
 *   h13    [rows, 2I]  X_perm_e W13_e before the activation (if save_for_backward)
 *   act    [rows, I]   A = silu(h13[:, :I]) * h13[:, I:]; in MOE_BF16 mode
 *                      gate * A (the gate of the row's assignment, 0 on pad
 *                      rows), the form both the down GEMM and dW2 consume;
 *                      zero-sized in MOE_MXFP8 mode (the gate/up epilogue
 *                      writes A's MXFP8 encodings directly: act_col below,
 *                      and a row-wise copy in the forward workspace)
 * MOE_MXFP8 only (zero-sized in the other modes): the backward's MXFP8
 * operands, which the forward quantises in the same passes as its own
 * (E4M3 codes *_q, tensor-core scale atoms *_sf; written only with
 * save_for_backward):
 *   x_col   X_perm, 32-row blocks per expert group       (dW13 operand)
 *   act_col A, 32-row blocks per expert group             (dW2 operand)
 *   w13_row W13 [E*H, 2I], 32-column blocks along 2I      (dX operand)
 *   w2_row  W2 [E*I, H], 32-column blocks along H          (D operand)
 * The block-scaled GEMMs run tiles 192 columns wide, so the scales of the
 * two weight operands (the GEMMs' B) sit in tile slots: row r of a weight
 * with S rows per expert (S = H for w13_row, I for w2_row) has the scale
 * MN index (r / S) * ceil(S / 192) * 256 + ((r % S) / 192) * 256 +
 * (r % S) % 192 in the atom layout of moe_quantize_mxfp8_dual (each tile
 * owns two whole atoms); the row-wise activations' scales use MN = row.   */
typedef struct {
  size_t x_perm, h13, act;
  size_t x_col_q, x_col_sf, act_col_q, act_col_sf;
  size_t w13_row_q, w13_row_sf, w2_row_q, w2_row_sf;
  size_t total;
} moe_saved_layout;

enum { MOE_WS_ROUTE = 0, MOE_WS_FORWARD = 1, MOE_WS_BACKWARD = 2 };

/* Upper bound of padded_offsets[E]: T*top_k + 128*E rows. */
int64_t moe_max_rows(const moe_dims* dims);

/* Size in bytes of the caller-provided workspace of one call kind
 * (MOE_WS_ROUTE / MOE_WS_FORWARD / MOE_WS_BACKWARD); 0 on invalid dims. */
size_t moe_workspace_size(const moe_dims* dims, int which);

/* Layout of the saved-activation buffer; returns MOE_ERR_INVALID_ARG on bad
 * dims. */
moe_status moe_saved_layout_of(const moe_dims* dims, moe_saved_layout* out);

/* Router and permutation builder ([MM] "In brief"; [TE] 02 and
 * "Optimisation 2": local reordering of token copies by expert).
 *   logits  float [T, E] (device).  -inf experts are never chosen while
 *           top_k finite logits remain (a token with fewer finite logits
 *           gets its -inf slots in ascending expert order, with gate 0).
 *           A token whose logits are all -inf has no softmax: it is routed
 *           to experts 0..top_k-1 with every gate 0 (it contributes nothing
 *           to the layer's output) and *dev_status gets MOE_ERR_BAD_INPUT.
 *           A NaN logit is read as -inf and also reported as
 *           MOE_ERR_BAD_INPUT.
 *   out     all seven arrays of moe_route_out (device, caller-owned).
 *   ws      MOE_WS_ROUTE workspace.
 * Indices, counts and offsets are deterministic and independent of the GPU. */
moe_status moe_route(const moe_dims* dims, const float* logits,
                     const moe_route_out* out, void* ws, size_t ws_bytes,
                     int32_t* dev_status, void* stream);

/* moe_route without a workspace argument, for callers that cannot allocate
 * device memory.  The pages have no counterpart: it exists for integrations
 * such as plugins inside a host framework that owns every device allocation
 * and exposes no workspace hook, or latency-critical loops that must not call
 * cudaMalloc (which can synchronise the device) after start-up.  Results are
 * identical to moe_route.
 *   Scratch: a library-owned device array of 512 KiB (131072 int32) that
 *   every GPU which loads the library holds until process exit.  Requires
 *   2 * E * ceil(T / 128) <= 131072, else MOE_ERR_INVALID_ARG (no launch).
 *   The first call in each CUDA context (each device's primary context,
 *   and again after a device reset, which creates a new context holding a
 *   new copy of the array) looks up the array's device address with that
 *   device current (no allocation) and caches it; make that first call
 *   before any stream capture (a call during capture that would need the
 *   lookup returns MOE_ERR_CUDA and launches nothing).  The library calls
 *   no cudaMalloc / cudaFree here; the cache is safe across host threads.
 *   All calls share the one array: calls whose work can overlap on the GPU
 *   (different streams, or different host threads) race and must be ordered
 *   by the caller.  Each call writes every scratch entry it reads. */
moe_status moe_route_noalloc(const moe_dims* dims, const float* logits,
                             const moe_route_out* out, int32_t* dev_status,
                             void* stream);

/* Router backward: d(logits) from d(gate) through the renormalised top-k
 * softmax, the selection held fixed.  For a selected expert i of token t,
 * gate_i = exp(l_i) / sum_{j in top-k} exp(l_j), so
 *   dlogits[t, i] = gate_i * (dgate_i - sum_j gate_j * dgate_j),
 * and every unselected expert gets 0 (the step upstream of moe_backward's
 * d(gate); [MM] "How does the fused kernel work?": the trainable backward).
 *   route    moe_route output (topk_idx and gate are read).
 *   dgate    float [T, top_k] (device), e.g. from moe_backward.
 *   dlogits  float [T, E] (device), fully overwritten. */
moe_status moe_route_backward(const moe_dims* dims, const moe_route_out* route,
                              const float* dgate, float* dlogits,
                              int32_t* dev_status, void* stream);

/* Forward of the expert layer ([MM] "How does the fused kernel work?";
 * [TE] "Optimisation 1" and "Optimisation 2"):
 *   X_perm = rows of X in expert-major order (pad rows 0)
 *   h13    = X_perm_e W13_e per expert (grouped GEMM),
 *   A      = silu(h13[:, :I]) * h13[:, I:]           (fused epilogue)
 *   Z      = gate * (A_e W2_e)                        (grouped GEMM + gate)
 *   Y[t]   = sum_j Z[row_of_assign[t*k + j]]          (deterministic combine)
 * In MOE_BF16 mode the gate is applied to A in the gate/up epilogue instead
 * (Z = (gate * A_e) W2_e, the same product).
 *   X    [T, H]; W13 [E, H, 2I]; W2 [E, I, H]; Y [T, H]  (device)
 *   route  moe_route output for the same dims.
 *   saved  moe_saved_layout_of(dims).total bytes (device).
 *   ws     MOE_WS_FORWARD workspace. */
moe_status moe_forward(const moe_dims* dims, const void* X, const void* W13,
                       const void* W2, const moe_route_out* route, void* Y,
                       void* saved, size_t saved_bytes, void* ws,
                       size_t ws_bytes, int32_t* dev_status, void* stream);

/* Backward of the expert layer with the routing held fixed ([MM] "How does
 * the fused kernel work?": the trainable backward; [OB] "Overlapping Backward
 * Pass"): with dY the gradient of Y,
 *   D      = dY_perm_e W2_e^T,  dgate = <A, D> per assignment,
 *   dA     = gate * D,  dh13 = [dA * v * silu'(u) | dA * silu(u)],
 *   dX[t]  = sum_j (dh13 W13_e^T)[row_of_assign[t*k + j]],
 *   dW13_e = X_perm_e^T dh13_e,  dW2_e = A_e^T (gate * dY)_perm_e,
 * experts with no token get zero weight gradients.  The activation-gradient
 * GEMMs and the weight-gradient GEMMs run as co-scheduled tiles of
 * persistent launches ({D + dSwiGLU, dW2}, then {dX, dW13}).  In MOE_BF16
 * mode dW2_e = (gate * A)_e^T dY_perm_e (the same product, from the gated
 * `act` the forward saved: no gated copy of dY is made).
 *   dY [T, H]; dX [T, H]; dW13 [E, H, 2I]; dW2 [E, I, H]; dgate float [T, k]
 *   saved  the buffer written by moe_forward with save_for_backward = 1.
 *   ws     MOE_WS_BACKWARD workspace. */
moe_status moe_backward(const moe_dims* dims, const void* dY, const void* W13,
                        const void* W2, const moe_route_out* route,
                        const void* saved, size_t saved_bytes, void* dX,
                        void* dW13, void* dW2, float* dgate, void* ws,
                        size_t ws_bytes, int32_t* dev_status, void* stream);

/* MXFP8 quantiser ([TE] 03: group-aware MXFP8 quantisation; OCP MX v1.0
 * E4M3 elements, 32-element blocks, E8M0 scales):
 *   for each 32-element block, s = floor(log2(amax)) - 8 clamped to
 *   [-127, 127] (-127 for an all-zero block); code = E4M3(x / 2^s) rounded to
 *   nearest even, saturating to +-448; scale byte = s + 127.
 *   src     bf16 [R, ld] (device), the first C columns are quantised.
 *   axis    1: blocks of 32 along each row, scales [R, C/32];
 *           0: blocks of 32 rows down each column, scales [R/32, C].
 *   group_offsets  optional (NULL allowed), device int32 [G+1], axis 0 only:
 *           rows are concatenated groups, blocks restart at each group start,
 *           and rows >= group_offsets[G] are not touched.  Every offset must
 *           be a multiple of 32 (else MOE_ERR_INVALID_ARG in *dev_status).
 *   q       uint8 [R, C] E4M3 codes (device).   scales  uint8 (device).
 * R must be a multiple of 32 for axis 0; C a multiple of 32 for axis 1. */
moe_status moe_quantize_mxfp8(const void* src, int R, int C, int ld, int axis,
                              const int32_t* group_offsets, int G, uint8_t* q,
                              uint8_t* scales, int32_t* dev_status,
                              void* stream);

/* Both MXFP8 encodings of one bf16 tensor from a single read (the rule of
 * moe_quantize_mxfp8), with the scales in the tensor-core atom layout that
 * the layer's block-scaled GEMMs read: 512-byte atoms of 128 MN indices x 128
 * K elements, the scale of MN index mn and 32-element K block kb at byte
 *   ((mn / 128) * kgroups + kb / 4) * 512 + (mn % 32) * 16 + ((mn / 32) % 4) * 4 + kb % 4.
 *   q_row, s_row  blocks of 32 along each row: MN = row, kgroups = C / 128;
 *                 s_row holds ceil(R / 128) * 128 * C / 32 bytes.
 *   q_col, s_col  blocks of 32 rows down each column: MN = column,
 *                 kgroups = ceil(R / 128); s_col holds C * ceil(R / 128) * 4 bytes.
 *   q_row, q_col  uint8 [R, C] E4M3 codes (device).
 *   src           bf16 [R, ld] (device).
 *   rows_limit    optional device int32 (NULL: R): rows at or past it are
 *                 neither read nor written (it must be a multiple of 32).
 * R must be a multiple of 32, C of 128, ld >= C a multiple of 8; other sizes
 * return MOE_ERR_INVALID_ARG. */
moe_status moe_quantize_mxfp8_dual(const void* src, int R, int C, int ld,
                                   const int32_t* rows_limit, uint8_t* q_row,
                                   uint8_t* s_row, uint8_t* q_col, uint8_t* s_col,
                                   int32_t* dev_status, void* stream);

/* Human-readable name of a status code (static string). */
const char* moe_status_string(moe_status s);

/* Test and diagnosis hooks.  `wait_limit_ns` bounds every device-side wait
 * (0 restores the default of one second).  The bf16 backward runs its four
 * gradient GEMMs as two co-scheduled persistent launches, {D + dSwiGLU, dW2}
 * then {dX, dW13} (no tile waits on another CTA).  Flag
 * MOE_DEBUG_ONE_LAUNCH_BACKWARD runs all four in one persistent cooperative
 * launch instead, where dX / dW13 tiles wait (bounded) on readiness
 * counters bumped by the D tiles; MOE_DEBUG_NEVER_READY (implies it) makes
 * them wait on a counter that is never bumped, so the bounded wait runs out
 * and MOE_ERR_TIMEOUT is reported.  Flag MOE_DEBUG_SINGLE_CTA runs the bf16
 * and MXFP8 GEMMs with single-CTA 128-row tiles instead of 256-row tiles
 * over an SM pair (for A/B comparison).  Flag MOE_DEBUG_SPLIT_BACKWARD runs
 * the four bf16 gradient GEMMs as four consecutive launches (to time each).
 * Process-wide; not thread-safe against concurrent calls. */
enum { MOE_DEBUG_NEVER_READY = 1, MOE_DEBUG_SINGLE_CTA = 2, MOE_DEBUG_SPLIT_BACKWARD = 4,
       MOE_DEBUG_ONE_LAUNCH_BACKWARD = 8 };
void moe_set_debug(int flags, int64_t wait_limit_ns);

/* Diagnosis hook: a bounded side load.  Launches `ctas` thread blocks on
 * `stream`, each holding `smem_bytes` of shared memory (at most 227 KB) for
 * `duration_ns` (at most one second) and then returning, so that a test can
 * run the layer while part of the GPU is busy (the co-scheduled backward
 * must still finish: its launch starts only once all of its CTAs fit).
 * MOE_ERR_INVALID_ARG outside those limits. */
moe_status moe_debug_occupy(int ctas, int smem_bytes, int64_t duration_ns, void* stream);

/* Timing hook for kernel-level measurement.  `start` and `stop` are
 * cudaEvent_t handles (as void*) created by the caller.  The next call of the
 * kind `which` (MOE_WS_FORWARD: the two grouped-GEMM launches of moe_forward;
 * MOE_WS_BACKWARD: the gradient-GEMM launches of moe_backward) records
 * `start` on its stream just before the first of those launches and `stop`
 * just after the last, then forgets the events; in the MXFP8 modes the
 * quantisation passes between the launches fall inside.  NULL events cancel
 * a pending hook.  Process-wide; not thread-safe against concurrent calls. */
void moe_set_gemm_events(int which, void* start, void* stop);

/* Per-launch form of the same hook: the next call of the kind `which`
 * records start[i] just before and stop[i] just after its i-th grouped-GEMM
 * launch, for i < n (n at most 8; launches past n are not timed), then
 * forgets the events.  Each array holds n cudaEvent_t handles (as void*)
 * created by the caller; a NULL array, n <= 0 or a NULL handle cancels a
 * pending hook.  Process-wide; not thread-safe against concurrent calls. */
void moe_set_gemm_launch_events(int which, void* const* start, void* const* stop, int n);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */

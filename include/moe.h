/*
 * moe.h -- C ABI of the GB300 (sm_103a) dropless mixture-of-experts expert
 * layer: training forward and backward on one GPU.
 *
 * The layer (dropless MoE; "NVIDIA lleva el MoE de DeepSeek-V3 de 103 a 1.068
 * TFLOPS", sections on dropless vs capacity MoE, grouped GEMM and expert-
 * parallel dispatch/combine; the Mega MoE kernel description in "Prime
 * Intellect dopisal backward pass do kernela Mega MoE"):
 *   route:    p = softmax(logits_t) over E experts; S_t = the k largest logits
 *             (ties: lower expert index first); w_tj = p_{S_tj} / sum_S p.
 *   dispatch: counts[e] = tokens that chose e; offsets = exclusive prefix;
 *             row(t,j) = offsets[e] + #{t' < t that chose e}  (stable, no
 *             capacity, no dropped token, no padding).
 *   experts:  for every permuted row r of expert e, with x_r = x[token(r)]:
 *             G = x_r W_gate[e], U = x_r W_up[e], A = silu(G) * U,
 *             Y = A W_down[e]                      (SwiGLU MLP, no biases)
 *   combine:  out_t = sum_j w_tj * Y[row(t,j)]      (token order restored)
 *   backward: the same chain transposed -- dyw = w * dy (permuted), dA =
 *             dyw W_down^T, dSwiGLU, dX = dG W_gate^T + dU W_up^T, un-permute
 *             sum into dx, dW_* = grouped X^T-style products over each
 *             expert's rows, and d_logits[t, S_tj] = w_tj (g_tj - sum_i w_ti
 *             g_ti) with g_tj = <dy_t, Y[row(t,j)]>, zero for other experts.
 *
 * Conventions (all calls):
 *   - Memory: the caller owns and allocates every buffer; the library never
 *     allocates, frees or synchronises (only moe_get_device_status waits).
 *     Pointers named "device" are CUDA device pointers; `stream` is a
 *     cudaStream_t passed as void*; every kernel is enqueued on it, so the
 *     calls can be captured into a CUDA graph.
 *   - Counts and offsets stay on the device: no call copies routing results
 *     to the host.
 *   - Layouts are row-major, dense, as given per argument.  bf16 tensors are
 *     IEEE bfloat16 bit patterns.
 *   - Every device pointer must be 16-byte aligned.
 *   - Shapes: T >= 0, H % 64 == 0 and I % 64 == 0 (both >= 64), 1 <= E <= 256,
 *     1 <= k <= min(E, 16), T * k < 2^31; with MOE_PREC_FP8_BWD or
 *     MOE_PREC_MXFP8 also H % 128 == 0 and I % 128 == 0.
 *   - Errors found on the host (null pointer, bad shape, misalignment, a
 *     too-small workspace) return a negative moe_status with nothing launched.
 *     Anomalies found on the device (non-finite logits, a pipeline wait that
 *     ran out of time) set flags in a status word at the start of the call's
 *     scratch buffer; kernels never trap.  Read it with moe_get_device_status.
 *   - The library holds no per-call state; calls on different streams with
 *     disjoint buffers may run concurrently.  Two exceptions, both opt-in:
 *     the per-kernel timing hook (moe_timing_attach, process-wide while
 *     attached) and moe_route_static_scratch's one shared scratch array.
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
  MOE_ERR_INVALID_ARG = -1, /* null pointer, bad shape or precision */
  MOE_ERR_ALIGNMENT = -2,   /* a pointer is not 16-byte aligned */
  MOE_ERR_WORKSPACE = -3,   /* a scratch/saved buffer is smaller than moe_query_workspace says */
  MOE_ERR_UNSUPPORTED = -4, /* no sm_103a device, or a precision this build does not provide */
  MOE_ERR_CUDA = -5,        /* a CUDA runtime/driver call failed */
  MOE_ERR_DEVICE = -6       /* moe_get_device_status: the device reported an anomaly */
} moe_status;

typedef enum {
  MOE_PREC_BF16 = 0,    /* bf16 operands, fp32 accumulation, everywhere */
  MOE_PREC_FP8_BWD = 1, /* bf16 forward; backward grouped GEMMs in MXFP8 (E4M3 values,
                           one UE8M0 scale per 32 elements along each GEMM's K) */
  MOE_PREC_MXFP8 = 2    /* the forward grouped GEMMs in MXFP8 too ("mxfp8" in the Prime
                           Mega MoE write-ups' precision switch): x and W_gate/W_up
                           along H, A (as bf16) and W_down along I; the activations the
                           forward saves stay bf16; the backward is fp8_bwd's */
} moe_precision;

/* Device status flags (moe_get_device_status *host_code). */
#define MOE_DEV_NONFINITE_LOGIT 0x1 /* a logit was NaN or +-Inf; routing outputs unspecified */
#define MOE_DEV_WAIT_TIMEOUT 0x2    /* a pipeline wait exceeded its bound; outputs unspecified */

typedef struct {
  int32_t T;         /* tokens */
  int32_t H;         /* hidden size */
  int32_t I;         /* expert intermediate size */
  int32_t E;         /* experts */
  int32_t k;         /* experts per token */
  int32_t precision; /* moe_precision */
} moe_config;

/* Routing results, written by moe_route, read by moe_forward/moe_backward.
 * All device pointers, caller-owned, M = T*k. */
typedef struct {
  int32_t *topk_idx;    /* [T,k]  chosen experts, ordered by (logit desc, index asc) */
  float *topk_w;        /* [T,k]  renormalised router weights */
  int32_t *counts;      /* [E]    rows per expert */
  int32_t *offsets;     /* [E+1]  exclusive prefix of counts; offsets[E] = M */
  int32_t *row_of_slot; /* [T*k]  permuted row of slot t*k+j */
  int32_t *slot_of_row; /* [M]    inverse: slot t*k+j held by permuted row r */
  float *w_row;         /* [M]    router weight of permuted row r */
} moe_routing;

/* Byte sizes of the caller-provided buffers for a configuration.  The fused
 * kernel of the pages works through preallocated GPU scratch space instead of
 * allocating intermediates per call (the MarkTechPost article in Thai
 * translation, "how the fused kernel works"); here the caller allocates that
 * space once, sized by this call, and passes it to every call:
 *   route_scratch: moe_route's scratch;
 *   saved:        activations moe_forward keeps for moe_backward (layout below);
 *   fwd_scratch:  moe_forward's scratch;  bwd_scratch: moe_backward's scratch.
 * Returns MOE_ERR_INVALID_ARG for an unsupported shape.  Host only. */
moe_status moe_query_workspace(const moe_config *cfg, size_t *route_scratch, size_t *saved,
                               size_t *fwd_scratch, size_t *bwd_scratch);

/* Offsets (bytes) of the saved activations inside `saved`, for inspection:
 * x_perm [M,H], G [M,I], U [M,I], A [M,I], Y [M,H] (unweighted), A_w [M,I]
 * (A times the row's router weight: the weight-gradient operand), all bf16.
 * A_w is written in MOE_PREC_BF16 only: the MXFP8 backwards read w * A
 * quantised along tokens instead (moe_fp8_layout's aw_t, also in `saved`).
 * x_perm is not written in MOE_PREC_MXFP8, whose GEMMs read x's codes and whose
 * backward reads x itself. */
typedef struct {
  size_t x_perm, G, U, A, Y, A_w;
} moe_saved_layout;
moe_status moe_saved_offsets(const moe_config *cfg, moe_saved_layout *layout);

/* MOE_PREC_FP8_BWD and MOE_PREC_MXFP8: byte offsets of the backward GEMMs' MXFP8
 * operands, for inspection after the call: inside moe_backward's scratch, except
 * the ones the forward writes (inside `saved`, listed below).  m_pad is the padded
 * token capacity (a multiple of 128): expert e's rows start at padded row
 * pad_offsets[e] = sum over e' < e of ceil(count/128)*128 (int32 [E+1]); rows
 * past an expert's count are zero codes with zero scale codes; padded rows at
 * and past pad_offsets[E] are left unwritten.
 *   *_q     E4M3 codes, K-major: dy_q [m_pad,H] (padded rows), wd_q [E*I,H],
 *           dg_q/du_q [m_pad,I], wg_q/wu_q [E*H,I];
 *   *_t     token-axis operands transposed, tokens contiguous: aw_t (w*A) and
 *           dg_t/du_t [I,m_pad], dy_t and x_t [H,m_pad];
 *   written by the forward (moe_forward and moe_forward_recompute), so their
 *   offsets are inside `saved`, not the scratch: aw_t (the gate/up epilogue), x_t
 *   (in MOE_PREC_FP8_BWD by the forward's permute, which gathers x into x_perm
 *   and quantises it along tokens in one pass) and the weights' wd_q, wg_q, wu_q
 *   with their scales (in MOE_PREC_FP8_BWD the two bf16 GEMMs quantise each
 *   weight tile as it passes through them, so only the experts that received
 *   rows are written -- no backward GEMM reads the others; in MOE_PREC_MXFP8 the
 *   forward's weight passes write every expert);
 *   *_sf    their UE8M0 scale codes (2^(code-127)), one per 32 elements along
 *           K, in 512-byte atoms of 128 rows x 128 K, the order the tensor core
 *           reads them: row w of atom row-block rb, K-block b, sits at byte
 *           (rb*(K/128) + b/4)*512 + (w%32)*16 + (w/32)*4 + b%4.  For dy_q,
 *           dg_q, du_q, aw_t and x_t (the GEMMs' M side) row r is row r%128 of
 *           block r/128.  For wd_q, wg_q, wu_q, dy_t, dg_t and du_t (the N side,
 *           read in 192-row tiles) rows are cut into segments of S rows (S = I
 *           for wd_q, H for wg_q/wu_q, all rows for the transposed ones), each
 *           segment into groups of 192 rows, each group into two blocks: row r
 *           with s = r/S, g = (r%S)/192, j = (r%S)%192 is row j%128 of block
 *           (s*ceil(S/192) + g)*2 + j/128.  Scale bytes of groups' rows past a
 *           segment's end are left unwritten.
 * Returns MOE_ERR_INVALID_ARG for other precisions or unsupported shapes. */
typedef struct {
  size_t m_pad, pad_offsets;
  size_t dy_q, dy_sf, wd_q, wd_sf, dg_q, dg_sf, du_q, du_sf, wg_q, wg_sf, wu_q, wu_sf;
  size_t aw_t, aw_t_sf, dy_t, dy_t_sf, x_t, x_t_sf, dg_t, dg_t_sf, du_t, du_t_sf;
} moe_fp8_layout;
moe_status moe_fp8_scratch_offsets(const moe_config *cfg, moe_fp8_layout *layout);

/* MOE_PREC_MXFP8 only: byte offsets, inside moe_forward's scratch, of the MXFP8
 * operands of the two forward GEMMs, for inspection after the call (padded row
 * space, pad_offsets, codes and 512-byte scale atoms as in moe_fp8_layout):
 *   x_q   [m_pad,H]  the permuted x along H (M side: row r in block r/128);
 *   a_q   [m_pad,I]  A along I, from its bf16 value (M side);
 *   wgu_q [E*2I,H]   W_gate and W_up along H, transposed and interleaved by 32:
 *                    row e*2I + (i/32)*64 + i%32 holds W_gate[e][:, i] and the
 *                    row 32 after it W_up[e][:, i] (N side, segments of 2I rows);
 *   wdt_q [E*H,I]    W_down along I, transposed: row e*H + h holds W_down[e][:, h]
 *                    (N side, segments of H rows).
 * The same passes over the weights also write the backward GEMMs' weight
 * operands, which live in `saved` (moe_backward does not quantise the weights
 * again; moe_fp8_scratch_offsets reports the same offsets):
 *   bwd_wd_q [E*I,H], bwd_wg_q and bwd_wu_q [E*H,I] and their scales, laid
 *   out as moe_fp8_layout's wd_q, wg_q, wu_q (offsets inside `saved`).
 * Returns MOE_ERR_INVALID_ARG for other precisions or unsupported shapes. */
typedef struct {
  size_t m_pad, pad_offsets, x_q, x_sf, a_q, a_sf, wgu_q, wgu_sf, wdt_q, wdt_sf;
  size_t bwd_wd_q, bwd_wd_sf, bwd_wg_q, bwd_wg_sf, bwd_wu_q, bwd_wu_sf;
} moe_mxfp8_fwd_layout;
moe_status moe_mxfp8_forward_offsets(const moe_config *cfg, moe_mxfp8_fwd_layout *layout);

/* Router and dispatch indices.  logits: device fp32 [T,E].  Writes every field
 * of *routing.  Dropless routing gives per-expert group sizes that change
 * every step; they stay on the device and the grouped GEMMs read them there,
 * so no host copy breaks CUDA-graph capture (NVIDIA article "DeepSeek-V3 MoE
 * from 103 to 1,068 TFLOPS", "optimisations dropless needs" and "grouped
 * GEMM").  Two kernels: the first reads the logits once and writes the top k,
 * the per-block expert histograms and every slot's rank, and its last blocks
 * to finish scan the histograms (counts, offsets, per-block bases); the second
 * writes every slot's row.  Work and scratch grow linearly with T.
 * Non-finite logits set MOE_DEV_NONFINITE_LOGIT; the indices written are still
 * in range. */
moe_status moe_route(const moe_config *cfg, const float *logits, const moe_routing *routing,
                     void *scratch, size_t scratch_bytes, void *stream);

/* Forward.  x: device bf16 [T,H]; W_gate, W_up: device bf16 [E,H,I];
 * W_down: device bf16 [E,I,H]; out: device bf16 [T,H].
 * saved: device, at least moe_query_workspace's `saved` bytes; moe_backward
 * reads it, so keep it unchanged between the two calls. */
moe_status moe_forward(const moe_config *cfg, const void *x, const moe_routing *routing,
                       const void *W_gate, const void *W_up, const void *W_down, void *out,
                       void *saved, size_t saved_bytes, void *scratch, size_t scratch_bytes,
                       void *stream);

/* Activation checkpointing (the pages' "2 fwd + bwd" layer step: the forward
 * runs once without keeping its activations and again just before the
 * backward).  Same arguments and errors as moe_forward.
 * moe_forward_nosave writes out like moe_forward but skips what only the
 * backward reads (bf16 and fp8_bwd: GEMM1's G, U and w*A are not written;
 * mxfp8: GEMM1 writes only A's codes, not the bf16 A, G, U, w*A, and the
 * weights are quantised for the forward GEMMs only); `saved` is used as
 * scratch and is not
 * valid for moe_backward afterwards.  out is bit-identical to moe_forward's.
 * moe_forward_recompute writes everything moe_backward reads into `saved`,
 * and not out (bf16: the permute and GEMM1 only -- the bf16 backward never
 * reads Y; the fp8 modes: GEMM2's Y too, no combine).  moe_backward after it
 * gives results bit-identical to moe_backward after moe_forward. */
moe_status moe_forward_nosave(const moe_config *cfg, const void *x, const moe_routing *routing,
                              const void *W_gate, const void *W_up, const void *W_down, void *out,
                              void *saved, size_t saved_bytes, void *scratch, size_t scratch_bytes,
                              void *stream);
moe_status moe_forward_recompute(const moe_config *cfg, const void *x, const moe_routing *routing,
                                 const void *W_gate, const void *W_up, const void *W_down, void *saved,
                                 size_t saved_bytes, void *scratch, size_t scratch_bytes, void *stream);

/* Backward.  dy: device bf16 [T,H] (gradient of out); x: the forward's input
 * (must be unchanged); routing and saved as left by moe_route/moe_forward.
 * Outputs (device): dx bf16 [T,H]; dW_gate, dW_up bf16 [E,H,I]; dW_down bf16
 * [E,I,H] (overwritten, not accumulated; experts with no token get zeros);
 * d_logits fp32 [T,E]; d_topk_w fp32 [T,k] = g_tj (may be NULL). */
moe_status moe_backward(const moe_config *cfg, const void *dy, const void *x,
                        const moe_routing *routing, const void *W_gate, const void *W_up,
                        const void *W_down, const void *saved, size_t saved_bytes, void *dx,
                        void *dW_gate, void *dW_up, void *dW_down, float *d_logits,
                        float *d_topk_w, void *scratch, size_t scratch_bytes, void *stream);

/* Router projection: the learned router's linear layer in front of moe_route,
 *   logits [T,E] fp32 = x [T,H] bf16 . W_r [H,E] bf16   (fp32 accumulation),
 * and its backward for the d_logits moe_backward returns,
 *   dW_r [H,E] fp32 = x^T . d_logits,   dx [T,H] bf16 += d_logits . W_r^T
 * (dx is updated in place: pass the dx moe_backward wrote to get the layer
 * input's full gradient).  d_logits enters both products rounded to bf16 (the
 * tensor cores' operand type); accumulation is fp32.  cfg->k and cfg->I are not
 * used; requires E % 8 == 0 (8 <= E <= 256) and H % 64 == 0.  Scratch sizes from
 * moe_router_workspace; a status header at the start of the scratch as for the
 * other calls.  With T == 0, logits is untouched and dW_r is zeroed. */
moe_status moe_router_workspace(const moe_config *cfg, size_t *fwd_scratch, size_t *bwd_scratch);
moe_status moe_router_forward(const moe_config *cfg, const void *x, const void *W_r, float *logits,
                              void *scratch, size_t scratch_bytes, void *stream);
moe_status moe_router_backward(const moe_config *cfg, const void *x, const void *W_r,
                               const float *d_logits, void *dx, float *dW_r, void *scratch,
                               size_t scratch_bytes, void *stream);

/* Routing without a caller-provided scratch buffer.  The paper has no
 * counterpart: it exists for callers that cannot allocate device memory --
 * code running while a CUDA graph is captured (cudaMalloc is not allowed
 * there), code inside a framework whose allocator already owns the device
 * memory, or a serving loop that must not allocate on its hot path.
 * Same arguments, results and errors as moe_route, except that the scratch is a
 * fixed 2.5 MiB + 4 KiB array inside this library's device memory (every GPU
 * that loads the library keeps it until the process exits).  It fits every
 * configuration with T <= 32768, and any other whose moe_query_workspace
 * route_scratch is at most that size; for the rest it returns MOE_ERR_WORKSPACE
 * and launches nothing.  Allocates nothing (no cudaMalloc/cudaFree, no
 * allocating library call).
 * device_status: optional device int32 that receives the call's MOE_DEV_* flags
 * (copied on `stream` after the routing kernels); NULL to skip.
 * The first call on a device looks up the array's device address (with that
 * device current) and keeps it for the process; make that first call before
 * any stream capture.  If the lookup fails the call returns MOE_ERR_CUDA with
 * nothing launched and no CUDA error left pending, and the next call on that
 * device looks the address up again.  All calls share the one array and it keeps the last call's
 * contents: calls that overlap on the GPU (for example on two streams) race,
 * so serialise them. */
moe_status moe_route_static_scratch(const moe_config *cfg, const float *logits,
                                    const moe_routing *routing, int32_t *device_status,
                                    void *stream);

/* Diagnostic with no counterpart in the paper: launches one kernel that waits,
 * through the same bounded wait every pipeline stage of the library uses, on
 * an mbarrier nothing arrives at.  The wait gives up after about two seconds
 * of SM clock and the kernel sets MOE_DEV_WAIT_TIMEOUT in *device_status
 * (device int32, 4-byte aligned, zeroed on `stream` first).  It shows that a
 * lost arrival is reported as a status instead of hanging the GPU, and that
 * the context stays usable afterwards.  Returns MOE_ERR_INVALID_ARG for a
 * NULL pointer; asynchronous on `stream`. */
moe_status moe_selftest_wait_timeout(int32_t *device_status, void *stream);

/* Waits for `stream`, then reads the status word at the start of `scratch` (a
 * scratch buffer previously passed to moe_route, moe_forward or moe_backward).
 * *host_code receives the MOE_DEV_* flags; returns MOE_OK when they are zero,
 * MOE_ERR_DEVICE otherwise.  The only call that synchronises. */
moe_status moe_get_device_status(const void *scratch, void *stream, int32_t *host_code);

/* Static description of a status code. */
const char *moe_status_string(moe_status status);

/* Optional per-kernel timing for profiling.  When `events` is non-NULL, every
 * later library call records events[2i] and events[2i+1] (cudaEvent_t as
 * void*) on its stream around the i-th kernel it launches, counting from the
 * attach, up to `capacity` kernels; moe_timing_count returns how many were
 * recorded.  Process-wide, not thread-safe; pass NULL to detach. */
moe_status moe_timing_attach(void *const *events, int32_t capacity);
int32_t moe_timing_count(void);
/* Name of the i-th timed kernel (static string; NULL when out of range). */
const char *moe_timing_label(int32_t i);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */

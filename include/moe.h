/*
 * moe.h - C ABI of the B300 (sm_103a) library for the forward pass of one
 * top-k routed Mixture-of-Experts FFN layer.
 *
 * The method (pages cited by title and section):
 *   [MoE-math]     kwkr.cn, "MoE sparse activation: from the math to the code"
 *                  (title lost in extraction), sections 2.1-2.3 and 3.1-3.2.
 *   [MoE-tutorial] intelliparadigm.com, "MoE模型：动态计算架构解析与实践指南",
 *                  sections 2.1 and 2.3.
 *   [MoE-guide]    lpnh.cn, "Mixture of Experts（MoE）原理与工程落地全指南",
 *                  sections 2.2, 3.2 and 3.3.
 *
 *   logits  l = (x W_g^T + b + g) / tau                 [MoE-math] 2.1, [MoE-guide] 3.3
 *   probs   p = softmax(l)                               [MoE-math] 2.1
 *   K(x)    = top-k of l, descending, ties -> lower expert index   [MoE-math] 2.1
 *   gates   g_j = p_{K_j} / sum_m p_{K_m}               [MoE-math] 2.1
 *   C       = ceil(c k T / E); a slot is kept iff fewer than C earlier tokens
 *             chose the same expert (token order)       [MoE-math] 2.3, 3.2
 *   expert  GELU:   W2 gelu(W1 x + b1) + b2              [MoE-math] 3.1
 *           SwiGLU: W2 (silu(W1 x) * (W3 x))             ([MoE-guide] 3.2 shapes)
 *   y_t     = sum_{kept j} g_j E_{K_j}(x_t)  (0 if every slot dropped)
 *   f_i = count_i/(kT), P_i = mean_t p_{t,i}, L_balance = E sum_i f_i P_i
 *                                                         [MoE-math] 2.2
 *
 * Conventions for every call:
 *   - Pointers are DEVICE pointers unless the name ends in _host.
 *   - Row-major, densely packed. Weights use the nn.Linear storage [out, in]:
 *     Wg [E, d], W1 and W3 [E, H, d], W2 [E, d, H]; expert biases b1 [E, H],
 *     b2 [E, d]. Activations x [T, d], y [T, d].
 *   - dtype MOE_BF16: x, weights, expert biases, xd, Y, y are bf16; MOE_F32:
 *     all fp32. Router bias, noise, logits, gates and statistics are fp32;
 *     ids and offsets int32.
 *   - Every device-side call only enqueues work on `stream` (a cudaStream_t)
 *     and returns. The library never allocates, frees or synchronises, except
 *     moe_device_status, which synchronises `stream`. The caller owns every
 *     buffer and keeps it alive until the stream has run the work.
 *   - Arguments are validated on the host first; on failure nothing is
 *     enqueued and a status is returned. A failed kernel launch returns
 *     MOE_ERR_CUDA.
 *   - The workspace `ws` (size from moe_workspace_size, 256-byte aligned) holds
 *     intermediates and a status header. Zero it once with moe_workspace_init
 *     before first use; afterwards calls leave the header ready for the next
 *     call. Calls sharing one workspace must be ordered (same stream).
 *   - Device-detected errors are recorded in the workspace header and read
 *     with moe_device_status: a bounded wait that ran out
 *     (MOE_ERR_DEVICE_TIMEOUT), or a device-resident input of moe_dispatch or
 *     moe_expert_ffn out of range (MOE_ERR_INVALID_ARG; the host cannot check
 *     those without a synchronisation).
 *   - Checked build (libmoe_b300_check.so, compiled with MOE_CHECK): every
 *     kernel that indexes with rows, slots or tokens another kernel wrote
 *     (the dispatch's row positions, the gather's tokens, the combine's and
 *     the backward's slots) tests each index against its bound, skips the
 *     access if it fails and records MOE_ERR_DEVICE_CHECK (where = 51..56).
 *     The same calls, the same results; a debugging aid where no memory
 *     checker can run.
 *   - Limits: 1 <= k <= 8, k <= E <= 256, T >= 1, T*k < 2^31, capacity >= 1;
 *     d and H multiples of 8 (bf16) or 4 (fp32); activations must be finite.
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#if defined(MOE_BUILD_SO)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *moe_stream_t; /* the same handle as cudaStream_t */
typedef struct CUevent_st *moe_event_t;   /* the same handle as cudaEvent_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,    /* null required pointer, bad shape or limit      */
  MOE_ERR_UNSUPPORTED = 2,    /* valid but outside this build (e.g. k > 8)      */
  MOE_ERR_WORKSPACE = 3,      /* ws too small or misaligned                     */
  MOE_ERR_CUDA = 4,           /* a CUDA runtime call or kernel launch failed    */
  MOE_ERR_DEVICE_TIMEOUT = 5, /* a bounded device-side wait ran out             */
  MOE_ERR_DEVICE_CHECK = 6    /* checked build: an index out of its bounds       */
} moe_status_t;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype_t;
typedef enum { MOE_ACT_GELU = 0, MOE_ACT_SWIGLU = 1 } moe_act_t;

/* Layer shape. capacity is C (see moe_capacity). tau is the router
 * temperature (logits are divided by it; 1.0 = none). dtype and act hold a
 * moe_dtype_t and a moe_act_t.
 * noise_scale sets how the router noise input (where one is passed) enters
 * the logits: 0 adds it as given (a fixed-strength noise, or Gumbel noise:
 * the lpnh.cn MoE guide, section 3.3); s > 0 scales it by s times the
 * token's standard deviation over its E logits before the noise (bias
 * included; population form), so that the noise strength follows the
 * logits' scale (the kwkr.cn MoE article, section 3.3):
 *   l[t,i] = (z[t,i] + s * std_t(z) * noise[t,i]) / tau.
 * Must be finite and >= 0. */
typedef struct {
  int32_t T, d, E, k, H;
  int32_t capacity;
  int32_t dtype;
  int32_t act;
  float tau;
  float noise_scale;
  int32_t flags; /* MOE_FLAG_* bits; 0 for none */
} moe_config_t;

/* flags: moe_layer_forward[_shared] also keeps the experts' pre-activations
 * (xd W1^T + b1 for GELU; gate xd W1^T and up xd W3^T for SwiGLU, bf16) in
 * its workspace, and moe_layer_backward[_shared] reads them there instead of
 * recomputing them (one GEMM1-sized product fewer per backward, and a
 * smaller backward workspace). The forward workspace grows by
 * min(T*k, E*C) * H * 2 bytes (GELU) or twice that (SwiGLU). Training only:
 * the forward's outputs are the same either way. bf16 only
 * (MOE_ERR_UNSUPPORTED for fp32). */
#define MOE_FLAG_KEEP_PREACT 1

/* Version of this ABI (major * 100 + minor). */
MOE_API int32_t moe_abi_version(void);

/* Human-readable name of a status code; never NULL. */
MOE_API const char *moe_status_string(int32_t status);

/* C = ceil(c k T / E) with c = c_num / c_den, in exact integer arithmetic
 * ([MoE-math] 2.3). Host only. Returns -1 if any argument is < 1 or the
 * result does not fit in int32. */
MOE_API int32_t moe_capacity(int64_t c_num, int64_t c_den, int32_t k, int32_t T, int32_t E);

/* Bytes of workspace every call below needs for this shape (the maximum
 * over calls, so one workspace serves all). Host only. */
MOE_API moe_status_t moe_workspace_size(const moe_config_t *cfg, size_t *bytes);

/* Zero the workspace status header (enqueued on stream). Call once after
 * allocating a workspace, and again after a call reported an error. */
MOE_API moe_status_t moe_workspace_init(void *ws, size_t ws_bytes, moe_stream_t stream);

/* Read and clear the device status word in ws. Synchronises `stream`.
 * *code is MOE_OK, or the first status a kernel recorded since the last read
 * (MOE_ERR_DEVICE_TIMEOUT, MOE_ERR_INVALID_ARG or MOE_ERR_DEVICE_CHECK).
 * *where says which kernel
 * recorded it (0 if none): 1..6 a wait of the grouped GEMM (roles: producer,
 * MMA issuer, epilogue), 41 an expert id outside [0, E) in moe_dispatch, 42 /
 * 43 bad expert offsets in moe_expert_ffn (bf16 / fp32 kernel), 11..14 a
 * wait of the tensor-core router, 21..27 a wait of the weight-gradient GEMM;
 * checked builds: 51 a gathered token, 52 a combined slot, 53 a dispatched
 * row, 55 / 56 a slot in the backward's combine / dx sum. */
MOE_API moe_status_t moe_device_status(void *ws, int32_t *code, int32_t *where,
                               moe_stream_t stream);

/* Router, softmax, top-k, renormalised gates ([MoE-math] 2.1, 3.2), one
 * fused kernel.
 *   x          [T, d]   input tokens (dtype)
 *   Wg         [E, d]   router weight (dtype), nn.Linear storage
 *   bias       [E]      fp32 router bias, or NULL
 *   noise      [T, E]   fp32 noise added to the logits (e.g. Gumbel), or NULL
 *   logits     [T, E]   fp32 out: the selection keys l, or NULL
 *   topk_idx   [T, k]   int32 out: chosen experts, descending l, ties to lower id
 *   topk_gate  [T, k]   fp32 out: renormalised gates (sum to 1 per token)
 *   prob_sum   [E]      fp32 out: sum over tokens of p[t, e] (deterministic) */
MOE_API moe_status_t moe_router_topk(const moe_config_t *cfg, const void *x, const void *Wg,
                             const float *bias, const float *noise, float *logits,
                             int32_t *topk_idx, float *topk_gate, float *prob_sum,
                             void *ws, size_t ws_bytes, moe_stream_t stream);

/* Capacity-limited dispatch ([MoE-math] 2.3, 3.2): per-expert counts, a
 * token-order position for every slot, drops beyond C, and the gather of
 * kept rows into an expert-contiguous buffer.
 *   topk_idx      [T, k]   int32 in
 *   x             [T, d]   in (dtype)
 *   expert_count  [E]      int32 out: selections per expert before drops
 *   expert_offset [E+1]    int32 out: offset_e = sum_{e'<e} min(count_e', C)
 *   slot_of       [T, k]   int32 out: packed row of slot (t, j), or -1 if dropped
 *   token_of_row  [T*k]    int32 out: token of each packed row; the first
 *                          expert_offset[E] entries are written
 *   xd            [T*k, d] out (dtype): xd[slot_of[t,j]] = x[t]; first
 *                          expert_offset[E] rows written
 * An id outside [0, E) in topk_idx is counted for no expert, its slot gets
 * slot_of = -1, the other slots are dispatched as if it were absent, and the
 * workspace header records MOE_ERR_INVALID_ARG (where = 41). */
MOE_API moe_status_t moe_dispatch(const moe_config_t *cfg, const int32_t *topk_idx, const void *x,
                          int32_t *expert_count, int32_t *expert_offset, int32_t *slot_of,
                          int32_t *token_of_row, void *xd, void *ws, size_t ws_bytes,
                          moe_stream_t stream);

/* moe_dispatch without a workspace, for callers that cannot allocate device
 * memory: a plugin or custom-op interface that passes only the op's own
 * tensors, or a runtime that forbids cudaMalloc after start-up. The pages
 * have no counterpart; this is a deployment variant of moe_dispatch with the
 * same arguments and results, minus ws.
 *   Scratch: a fixed 512 KiB array in the library's device memory (two int32
 *   arrays of 65536 entries), held on every device that loaded the library
 *   until the process exits. Returns MOE_ERR_UNSUPPORTED when
 *   ceil(T*k / 1024) * E > 65536 (e.g. T*k > 1048576 slots at E = 64).
 *   Allocates nothing (no cudaMalloc, no cudaFree).
 *   The first call on a device (with that device current) looks up the
 *   array's device address; make that first call before any stream capture.
 *   All calls share the one array: calls that overlap on the GPU (different
 *   streams, or several host threads) race and corrupt each other's results;
 *   order them on one stream. Each call rewrites all the scratch it reads, so
 *   leftovers of earlier calls never matter.
 *   An id outside [0, E) is left out as in moe_dispatch but, with no
 *   workspace header, not reported. */
MOE_API moe_status_t moe_dispatch_static_scratch(const moe_config_t *cfg, const int32_t *topk_idx,
                                                 const void *x, int32_t *expert_count,
                                                 int32_t *expert_offset, int32_t *slot_of,
                                                 int32_t *token_of_row, void *xd,
                                                 moe_stream_t stream);

/* Grouped expert FFN over the packed rows ([MoE-math] 3.1; SwiGLU for
 * act = MOE_ACT_SWIGLU). Rows [offset_e, offset_{e+1}) of xd go through expert e.
 *   xd            [T*k, d] in (dtype), first expert_offset[E] rows used
 *   expert_offset [E+1]    int32 in (device; read on the device, no host sync)
 *   W1 [E,H,d], W3 [E,H,d] (SwiGLU only, else NULL), W2 [E,d,H]   (dtype)
 *   b1 [E,H], b2 [E,d]     GELU only, may be NULL (dtype)
 *   Y             [T*k, d] out (dtype), first expert_offset[E] rows written.
 * bf16 runs on the tcgen05 tensor cores with fp32 accumulation; the hidden
 * activation h is rounded to bf16 between the two GEMMs. fp32 runs on fp32
 * FMA.
 * The offsets must satisfy expert_offset[0] = 0 <= expert_offset[1] <= ... <=
 * expert_offset[E] <= min(T*k, E*C); otherwise no row is computed (Y is left
 * as it was) and the workspace header records MOE_ERR_INVALID_ARG (where = 42
 * for bf16, 43 for fp32). */
MOE_API moe_status_t moe_expert_ffn(const moe_config_t *cfg, const void *xd,
                            const int32_t *expert_offset, const void *W1, const void *W3,
                            const void *W2, const void *b1, const void *b2, void *Y,
                            void *ws, size_t ws_bytes, moe_stream_t stream);

/* Gate-weighted combine ([MoE-math] 2.1, 3.2): y_t = sum over j = 0..k-1 with
 * slot_of[t,j] >= 0 of topk_gate[t,j] * Y[slot_of[t,j]], summed in fp32 in
 * slot order (deterministic, no atomics); y_t = 0 if every slot was dropped.
 *   Y [T*k, d] (dtype) in, slot_of [T,k], topk_gate [T,k] in, y [T, d] out. */
MOE_API moe_status_t moe_combine(const moe_config_t *cfg, const void *Y, const int32_t *slot_of,
                         const float *topk_gate, void *y, moe_stream_t stream);

/* Load-balance statistics ([MoE-math] 2.2, drop count per 6.2):
 *   f[e] = expert_count[e] / (k T)   (before drops)
 *   P[e] = prob_sum[e] / T
 *   L_balance[0] = E * sum_e f[e] P[e]
 *   dropped[0] = k T - sum_e min(expert_count[e], C) */
MOE_API moe_status_t moe_aux_stats(const moe_config_t *cfg, const int32_t *expert_count,
                           const float *prob_sum, float *f, float *P, float *L_balance,
                           int32_t *dropped, moe_stream_t stream);

/* Inputs of the fused layer call. Optional pointers may be NULL. */
typedef struct {
  const void *x;      /* [T, d]            */
  const void *Wg;     /* [E, d]            */
  const float *bias;  /* [E] or NULL       */
  const float *noise; /* [T, E] or NULL    */
  const void *W1;     /* [E, H, d]         */
  const void *W3;     /* [E, H, d] or NULL */
  const void *W2;     /* [E, d, H]         */
  const void *b1;     /* [E, H] or NULL    */
  const void *b2;     /* [E, d] or NULL    */
} moe_layer_inputs_t;

/* Outputs of the fused layer call. Required: y. Others may be NULL. */
typedef struct {
  void *y;               /* [T, d]  */
  float *logits;         /* [T, E]  */
  int32_t *topk_idx;     /* [T, k]  */
  float *topk_gate;      /* [T, k]  */
  int32_t *slot_of;      /* [T, k]  */
  int32_t *expert_count; /* [E]     */
  int32_t *expert_offset;/* [E+1]   */
  float *f;              /* [E]     */
  float *P;              /* [E]     */
  float *L_balance;      /* [1]     */
  int32_t *dropped;      /* [1]     */
} moe_layer_outputs_t;

/* The whole layer: router -> dispatch -> expert FFN -> combine -> statistics,
 * enqueued on one stream with no host synchronisation. Intermediates (and any
 * output passed as NULL) live in ws. */
MOE_API moe_status_t moe_layer_forward(const moe_config_t *cfg, const moe_layer_inputs_t *in,
                               const moe_layer_outputs_t *out, void *ws, size_t ws_bytes,
                               moe_stream_t stream);

/* A shared expert: an expert of the layer's FFN form (act) that every token
 * passes through with weight 1, its output added to the routed sum (the
 * lpnh.cn guide, section 4.10, routes tokens to such an expert). It is not
 * subject to capacity or drops. Weights [out, in] in the layer dtype. */
typedef struct {
  int32_t H;          /* hidden size of the shared expert (multiple of 8 bf16 / 4 fp32) */
  const void *W1;     /* [H, d]                         */
  const void *W3;     /* [H, d] for SwiGLU, else NULL   */
  const void *W2;     /* [d, H]                         */
  const void *b1;     /* [H] GELU only, may be NULL     */
  const void *b2;     /* [d] GELU only, may be NULL     */
} moe_shared_expert_t;

/* Workspace bytes for moe_layer_forward_shared (the layer's plus the shared
 * expert's hidden and output rows). */
MOE_API moe_status_t moe_workspace_size_shared(const moe_config_t *cfg, int32_t H_shared,
                                               size_t *bytes);

/* moe_layer_forward plus a shared expert: y_t = E_shared(x_t) + sum over kept
 * slots of g_j E_{K_j}(x_t). Same conventions and outputs as
 * moe_layer_forward; ws must hold moe_workspace_size_shared bytes. */
MOE_API moe_status_t moe_layer_forward_shared(const moe_config_t *cfg,
                                              const moe_layer_inputs_t *in,
                                              const moe_shared_expert_t *shared,
                                              const moe_layer_outputs_t *out, void *ws,
                                              size_t ws_bytes, moe_stream_t stream);

/* moe_layer_forward with timing marks: stage_events points to six
 * cudaEvent_t handles (created by the caller, timing enabled) that are
 * recorded on `stream` before the router, after the router, after the
 * dispatch, after GEMM1 (the hidden activation), after GEMM2 and after the
 * combine and statistics. Where a path has no boundary between two marks
 * (the fp32 path runs both GEMMs in one call) both are recorded at the same
 * point. Results are identical to moe_layer_forward. Called while `stream`
 * is being captured into a CUDA graph, the marks become event-record nodes
 * of the graph (cudaEventRecordExternal), recorded at every replay. */
MOE_API moe_status_t moe_layer_forward_profiled(const moe_config_t *cfg,
                                                const moe_layer_inputs_t *in,
                                                const moe_layer_outputs_t *out, void *ws,
                                                size_t ws_bytes, moe_stream_t stream,
                                                void *const *stage_events);

/* ------------------------------------------------------------------ backward
 * Gradients of loss = sum_t <dy_t, y_t> + alpha * L_balance through the layer
 * computed by moe_layer_forward (the pages train the layer with the balance
 * statistic added to the task loss: the kwkr.cn MoE article, section 2.2;
 * the router is trained with it, section 3.3). The chain rule runs through
 * the combine, the renormalised gates, the balance term (f is piecewise
 * constant, P_i carries the gradient), the softmax, the router GEMM, the
 * experts and the dispatch; selection, capacity and drops get no gradient.
 * Weight gradients are fp32; dx has the layer dtype. */
typedef struct {
  void *dx;       /* [T, d] layer dtype, required                          */
  float *dWg;     /* [E, d] required                                       */
  float *dbias;   /* [E]    required iff in->bias, else NULL               */
  float *dW1;     /* [E, H, d] required                                    */
  float *dW3;     /* [E, H, d] SwiGLU (required), else NULL                */
  float *dW2;     /* [E, d, H] required                                    */
  float *db1;     /* [E, H] GELU: required iff in->b1, else NULL           */
  float *db2;     /* [E, d] GELU: required iff in->b2, else NULL           */
} moe_layer_grads_t;

/* Bytes of the backward workspace (its own buffer, 256-byte aligned; zero its
 * header once with moe_workspace_init; moe_device_status reads it). Host only.
 * MOE_ERR_UNSUPPORTED for shapes the backward does not cover. */
MOE_API moe_status_t moe_workspace_size_backward(const moe_config_t *cfg, size_t *bytes);

/* Backward of one moe_layer_forward call. Enqueue it on the forward's stream
 * after the forward, with the same cfg, in, ws and outputs `fwd`, before
 * anything else reuses ws: it reads the forward's routing (fwd->logits,
 * topk_idx, topk_gate, slot_of, expert_offset and f must all be non-NULL),
 * the gathered rows, the expert hidden activations h and, for k > 1, the
 * expert outputs kept in ws. dy [T, d] is the upstream gradient of y (layer
 * dtype); alpha the weight of L_balance. The expert pre-activations are
 * recomputed (for the activation's derivative). Every sum is taken in
 * a fixed order (results are run-to-run identical). Covered: bf16 on the
 * tensor cores and fp32 on fp32 FMA (any E); with fp32 the pre-activations are
 * always recomputed. A layer with a shared expert uses
 * moe_layer_backward_shared. Nothing is enqueued on a validation failure. */
MOE_API moe_status_t moe_layer_backward(const moe_config_t *cfg, const moe_layer_inputs_t *in,
                                        const moe_layer_outputs_t *fwd, const void *dy,
                                        float alpha, const moe_layer_grads_t *grads,
                                        const void *ws, size_t ws_bytes, void *bwd_ws,
                                        size_t bwd_ws_bytes, moe_stream_t stream);

/* Gradients of the shared expert's weights (fp32), the layout of the
 * moe_shared_expert_t weights. */
typedef struct {
  float *dW1;     /* [Hs, d] required                                      */
  float *dW3;     /* [Hs, d] SwiGLU (required), else NULL                  */
  float *dW2;     /* [d, Hs] required                                      */
  float *db1;     /* [Hs] GELU: required iff shared->b1, else NULL         */
  float *db2;     /* [d]  GELU: required iff shared->b2, else NULL         */
} moe_shared_grads_t;

/* Bytes of the backward workspace of a layer with a shared expert of hidden
 * size H_shared (a multiple of 8). Host only. */
MOE_API moe_status_t moe_workspace_size_backward_shared(const moe_config_t *cfg,
                                                        int32_t H_shared, size_t *bytes);

/* Backward of one moe_layer_forward_shared call (the shared expert of the
 * lpnh.cn MoE guide, section 4.10: an always-on expert added with weight 1 to
 * every token's output). As moe_layer_backward, with the same shared expert
 * and the forward's workspace ws (moe_workspace_size_shared bytes; it holds
 * the shared expert's hidden activations); bwd_ws holds
 * moe_workspace_size_backward_shared bytes. The shared expert's output
 * gradient is dy itself: its weight gradients go to shared_grads and its
 * input gradient is added into grads->dx in the same fixed-order sum as the
 * routed and router terms. */
MOE_API moe_status_t moe_layer_backward_shared(const moe_config_t *cfg,
                                               const moe_layer_inputs_t *in,
                                               const moe_shared_expert_t *shared,
                                               const moe_layer_outputs_t *fwd, const void *dy,
                                               float alpha, const moe_layer_grads_t *grads,
                                               const moe_shared_grads_t *shared_grads,
                                               const void *ws, size_t ws_bytes, void *bwd_ws,
                                               size_t bwd_ws_bytes, moe_stream_t stream);

/* Number of kernels one moe_layer_forward call launches for this shape
 * (0 if cfg is invalid). Host only. */
MOE_API int32_t moe_layer_forward_launch_count(const moe_config_t *cfg);

/* As moe_layer_forward, but x_host [T, d] and y_host [T, d] are HOST buffers
 * (page-locked for asynchronous copies); the weights in `in` stay on the device
 * (in->x is ignored). The copies in and out run on `stream` inside the call's
 * work; the caller synchronises the stream before reading y_host. If
 * L_balance_host is not NULL the statistic is copied back too. Needs
 * moe_workspace_size_host bytes of workspace. */
MOE_API moe_status_t moe_workspace_size_host(const moe_config_t *cfg, size_t *bytes);
MOE_API moe_status_t moe_layer_forward_host(const moe_config_t *cfg, const void *x_host,
                                    const moe_layer_inputs_t *in, void *y_host,
                                    float *L_balance_host, void *ws, size_t ws_bytes,
                                    moe_stream_t stream);

/* moe_layer_forward_host for a stream of calls (a serving loop): the copy in
 * runs on copy_in, the layer on compute, the copies out on copy_out, so that
 * one call's copies overlap other calls' layers while the layers themselves
 * run one after another on compute. ev[3] are three events the caller
 * created for this workspace and passes to every call with it; they order
 * the calls that share the workspace (its staging buffers): a call's copy in
 * waits until the previous call with this ws has finished its layer (ev[1]),
 * and its layer waits for its copy in (ev[0]) and for the previous call's
 * copy out (ev[2]). Alternate two workspaces (each with its own events) to
 * overlap consecutive calls. The caller synchronises copy_out (or waits on
 * ev[2]) before reading y_host. Same workspace size as
 * moe_layer_forward_host. */
MOE_API moe_status_t moe_layer_forward_host_pipelined(
    const moe_config_t *cfg, const void *x_host, const moe_layer_inputs_t *in, void *y_host,
    float *L_balance_host, void *ws, size_t ws_bytes, moe_stream_t copy_in, moe_stream_t compute,
    moe_stream_t copy_out, const moe_event_t *ev);

#ifdef __cplusplus
}
#endif
#endif /* MOE_B300_H */

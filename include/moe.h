/*
 * moe.h -- C ABI of a single-GPU Mixture-of-Experts expert layer for GB300 (sm_103a).
 *
 * One GPU holds all E experts.  A training step of the layer is three calls on
 * one CUDA stream:
 *
 *   moe_plan      router logits -> top-k experts and gate weights, per-expert
 *                 counts, exclusive offsets and the stable token -> row table;
 *   moe_forward   dispatch (row gather), GroupGEMM -> SwiGLU -> GroupGEMM, gated combine;
 *   moe_backward  combine backward, dgrad GroupGEMMs, weight-gradient Transposed
 *                 GroupGEMM, dispatch backward.
 *
 * Sources (by page title and section):
 *   [UniEP]  "UniEP: Unified Expert-Parallel MoE MegaKernel for LLM Training"
 *   [MoonEP] "MoonEP: Balanced Expert Parallelism for MoE Training via Dynamic Redundant Experts"
 *
 * Conventions for every entry point
 *   - Dimensions: T tokens, H hidden, F per-expert FFN width, E experts, k
 *     experts per token, R = moe_rows(d) grouped rows (T*k without padding).
 *   - Every pointer argument is a DEVICE pointer owned by the caller, except
 *     the structs passed by address (host memory) and the host outputs of
 *     moe_get_status.  The library never allocates or frees memory and never
 *     synchronises, except moe_get_status, which synchronises the stream.
 *   - Tensors are dense row-major.  bf16 tensors are passed as void* (IEEE
 *     bfloat16 bit patterns).  Every device pointer must be 16-byte aligned.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy stream).
 *   - Return value: 0 on success, a negative MOE_ERR_* code when the host
 *     rejected the call (nothing was launched), or MOE_ERR_LAUNCH.  Errors the
 *     GPU detects are recorded in the workspace status word and read back with
 *     moe_get_status.
 *   - Results are bitwise reproducible: the same inputs give the same bits on
 *     every call and for every grid size.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

/* ---- error codes ---------------------------------------------------------- */
#define MOE_OK 0
#define MOE_ERR_ARG (-1)     /* null pointer, non-positive dimension, k > E, k > 32, pad outside [0, 4096], R >= 2^31 */
#define MOE_ERR_ALIGN (-2)   /* a pointer is not 16-byte aligned */
#define MOE_ERR_WS (-3)      /* workspace smaller than moe_workspace_bytes() */
#define MOE_ERR_LAUNCH (-4)  /* a CUDA launch or API call failed */
#define MOE_ERR_SHAPE (-5)   /* H or F not a multiple of 128, or E > 1024 */
#define MOE_ERR_DEVICE (-6)  /* current device is not compute capability 10.3 */
/* recorded by the GPU in the workspace status word */
#define MOE_ERR_TIMEOUT 1    /* a bounded wait inside a kernel expired; the kernel returned */
#define MOE_ERR_NONFINITE 2  /* a router logit was NaN or infinite */
#define MOE_ERR_BOUNDS 3     /* an index computed on the GPU fell outside its buffer; the access was skipped */

/* ---- shapes and tables ------------------------------------------------------ */
typedef struct {
  int32_t T, H, F, E, k;
  int32_t pad; /* token padding granule P.  0 or 1 (default): padding-free, the grouped
                  buffers hold exactly R = T*k rows ([UniEP] section 3, padding-free
                  GroupGEMM).  P >= 2: static-shape variant ([MoonEP] "The Buffer API",
                  token_padding): every expert's rows are rounded up to a multiple of P with
                  padding rows (row_src = -1, row_slot = 255, zero in Xp, GU, h, Y, dY, dGU,
                  dXp), and the buffers hold R = T*k + min(E, T*k)*(P-1) rows, a bound that
                  does not depend on the routing.  Results are the same bits as without
                  padding.  Pass the same dims to every call of a step. */
} moe_dims;

/* Routing state of one step.  Filled by moe_plan, read unchanged by
 * moe_forward and moe_backward of the same step (the plan object of the
 * MoonEP Buffer API: "The Buffer API: Dispatch, Combine, Prefetch, and Reduce").
 * All device buffers, caller-allocated. */
typedef struct {
  int32_t *topk_ids; /* [T,k]  expert of slot j of token t; descending logit, ties to the lower id */
  float *topk_w;     /* [T,k]  renormalised gate weight of that slot (fp32) */
  int32_t *counts;   /* [E]    rows per expert n_e (tokens routed to e; padding not counted) */
  int32_t *offsets;  /* [E+1]  first row of each expert's segment: exclusive prefix of the counts
                                (of the counts rounded up to P with padding); offsets[E] = rows in use */
  int32_t *dest;     /* [T,k]  grouped row of slot (t,j): offsets[e] + #{t' < t routed to e} */
  int32_t *row_src;  /* [R]    token of each grouped row (inverse of dest); -1 on padding rows */
  uint8_t *row_slot; /* [R]    slot j of each grouped row; 255 on padding rows */
  int32_t *tiles;    /* [moe_plan_tiles_elems(d)]  128-row GEMM tiles of the grouped buffer (internal) */
} moe_plan_t;

/* Tensors the forward stores for the backward (caller-allocated, bf16). */
typedef struct {
  void *Xp; /* [R,H]   dispatched rows, grouped by expert */
  void *GU; /* [R,2F]  G = Xp W1 in columns [0,F), U = Xp W3 in columns [F,2F) (bf16 of fp32 accumulators) */
  void *h;  /* [R,F]   silu(G) * U */
  void *Y;  /* [R,H]   expert outputs h W2, one row per (token, slot) */
} moe_saved_t;

/* Row gradients the backward produces on its way (caller-allocated, bf16). */
typedef struct {
  void *dY;  /* [R,H]   w[t,j] * dout[t] on the grouped row of (t,j) */
  void *dGU; /* [R,2F]  dG in columns [0,F), dU in columns [F,2F) */
  void *dXp; /* [R,H]   gradient of the dispatched rows */
} moe_grads_t;

/* The router's backward, requested from moe_backward (NULL: routing is held
 * fixed and only dgate is returned, as the pages time the layer).  With it, the
 * gradient flows on through the renormalised top-k softmax, routing held fixed
 * (the selection is piecewise constant in the logits):
 *   dl[t,m] = w[t,m] (dgate[t,m] - sum_j w[t,j] dgate[t,j]) for the k chosen m, 0 otherwise,
 *   dWr = x^T dl (fp32; dl rounded to bf16 for the tensor cores; a fixed number
 *   of token splits reduced in a fixed order, so bitwise reproducible),
 *   and dx gains sum_j dl[t,j] Wr[:, ids[t,j]] (one bf16 rounding of the sum
 *   of both shares).  E must be a multiple of 8. */
typedef struct {
  const void *x;  /* [T,H] bf16: the layer input (the router's input) */
  const void *Wr; /* [H,E] bf16: router weight */
  float *dlogits; /* [T,E] out: dL/dlogits, zero outside each token's k experts */
  float *dWr;     /* [H,E] out */
} moe_router_t;

/* Options (may be NULL for defaults). */
typedef struct {
  int32_t grid;     /* CTAs of the persistent kernels; 0 = one per SM.  Results do not depend on it. */
  int32_t schedule; /* 0 (default): one persistent launch per phase in both passes (gather,
                       GEMM1, GEMM2; the backward's four GEMMs), the fastest measured on GB300.
                       1: the forward's gather, GEMM1 and GEMM2 run as one persistent kernel with
                       a task cursor and per-tile readiness counters (tile shape per cta_pair).
                       2: as 1, and the backward's four GEMMs also run as one persistent kernel
                       (single-CTA tiles).
                       All three give the same bits. */
  void **events;    /* optional: 2*n_events cudaEvent_t recorded around each kernel of the call */
  int32_t n_events; /* capacity of events/2; kernels beyond it are not timed */
  int32_t cta_pair; /* tile shape of the grouped GEMMs that run as their own kernels:
                       1: one CTA per 128 x 256 tile (tcgen05 cta_group::1);
                       2: a cluster of two CTAs per 256 x 256 tile (cta_group::2, each SM holding
                       its 128 rows of A and half of B);
                       0 (default): 2 for every GEMM but the dgrad GEMM with the SwiGLU backward
                       epilogue, which measured faster with 1 unless the experts average at least
                       2048 rows (T*k >= 2048*E).  Both shapes give the same bits.
                       Other values: MOE_ERR_ARG.
                       The fused forward (schedules 1, 2) takes pair tiles unless cta_pair = 1;
                       the fused backward (schedule 2) always uses single-CTA tiles. */
  int32_t combine;  /* schedule 0 only.  0 (default): a separate gated-combine kernel.
                       1: the combine runs in GEMM2's epilogue (per-token arrival counters; the
                       warp that completes a token's k rows sums them, in slot order).  Same
                       bits; measured slower on GB300 (the fence and the combine work in the
                       epilogue hold the accumulator and stall the tensor pipe). */
  int32_t debug_drop_task; /* failure injection, for tests of the bounded waits: with schedule 1
                       or 2, the fused forward withholds the completion signal of its gather task
                       number debug_drop_task - 1, so the GEMM tile that needs those rows waits
                       out its bound (2 s), the kernel records MOE_ERR_TIMEOUT in the status word
                       and returns; the outputs are then undefined.  0 (default): off. */
  int32_t dispatch; /* schedule 0: where the row dispatch Xp = x[row_src] runs.  0 (default) or
                       1: its own kernel (gather by row, or scatter by token when x is large).
                       2: inside GEMM1's A-operand load: the producer warp copies the tile's
                       rows of x into the swizzled stage with 16-byte cp.async copies, and the
                       first N tile of each row block stores the gathered rows to Xp for the
                       backward ([UniEP] section 3: the dispatch workers write the GEMM's
                       operand rows).  Needs pair tiles for GEMM1 and the padding-free layout;
                       otherwise 1 is used.  Same bits. */
  int32_t wgrad_subbatches; /* reduction order of the weight gradients ([UniEP] section 6,
                       Performance Cost of Bitwise Reproducibility).  0 or 1 (default): one
                       accumulation chain over each expert's rows in ascending row order, the
                       bitwise-reproducible (BW) variant.  2: the non-bitwise (NB) variant: the
                       tokens form two sub-batches, [0, ceil(T/2)) and the rest; each weight
                       gradient is the sum of the two sub-batches' own reductions, the second
                       added onto the first by a float32 reduction in the L2 (dW = fl32(dW_0 +
                       dW_1); such reductions may flush subnormal values to zero).  NB results are
                       reproducible from run to run but differ in the last bits from BW; every
                       other output is identical.  Not with schedule 2 (MOE_ERR_ARG). */
} moe_opts;

/* ---- sizes ------------------------------------------------------------------ */

/* Bytes of the scratch workspace every call of one step needs (status word,
 * per-chunk counts and bitmaps of the routing, task cursor and per-tile
 * readiness counters of the persistent kernels, and the router backward's
 * Wr^T, per-slot and bf16 logit gradients and token-split partials of dWr).  Caller-allocated;
 * pass the same workspace to moe_plan, moe_forward and moe_backward of a step.
 * Returns 0 for invalid dims. */
MOE_API size_t moe_workspace_bytes(moe_dims d);

/* int32 elements of moe_plan_t.tiles.  Returns 0 for invalid dims. */
MOE_API size_t moe_plan_tiles_elems(moe_dims d);

/* R: rows of every grouped buffer (row_src, row_slot, Xp, GU, h, Y, dY, dGU, dXp):
 * T*k, or T*k + min(E, T*k)*(P-1) with a padding granule P = d.pad >= 2.
 * Returns 0 for invalid dims. */
MOE_API size_t moe_rows(moe_dims d);

/* ---- the layer -------------------------------------------------------------- */

/* Gating and the deterministic token -> row table.
 * [UniEP] background, Forward Propagation (top-k routing; stable sort keeping
 * the original token order) and section 3.1 Deterministic Token Mapping,
 * Algorithm 1 (counts per source, exclusive prefix over sources, base + local
 * stable index).  Here the sources are 256-token chunks of one GPU.
 *   logits  [T,E] fp32, device.  plan: every field allocated by the caller.
 *   T = 0 is a no-op.  NaN/inf logits set MOE_ERR_NONFINITE in the status word. */
MOE_API int moe_plan(moe_dims d, const float *logits, const moe_plan_t *plan, void *ws, size_t ws_bytes, void *stream);

/* Forward pass: Xp = x[row_src]; per expert e on rows [offsets[e], offsets[e+1]):
 * G = Xp W1[e], U = Xp W3[e], h = silu(G) * U, Y = h W2[e]; then
 * out[t] = sum_j w[t,j] * Y[dest[t,j]] (fp32, slots in order, rounded to bf16).
 * [UniEP] Forward Propagation (Figure 1) and section 3, Top-k accumulation
 * constraint; [MoonEP] zero-copy dispatch.
 *   x [T,H], W1 [E,H,F], W3 [E,H,F], W2 [E,F,H], out [T,H]: bf16, device.
 *   saved: filled with Xp, GU, h, Y for the backward. */
MOE_API int moe_forward(moe_dims d, const void *x, const void *W1, const void *W3, const void *W2, const moe_plan_t *plan,
                const moe_saved_t *saved, void *out, void *ws, size_t ws_bytes, const moe_opts *opts, void *stream);

/* Backward pass given dout = dL/dout [T,H] (bf16):
 *   dY[dest[t,j]] = w[t,j] dout[t];  dgate[t,j] = <dout[t], Y[dest[t,j]]>  (fp32)
 *   dH = dY W2[e]^T;  dG = dH U s (1 + G (1 - s)), dU = dH G s with s = sigmoid(G)
 *   dXp = dG W1[e]^T + dU W3[e]^T;  dx[t] = sum_j dXp[dest[t,j]]
 *   dW1[e] = Xp_e^T dG_e, dW3[e] = Xp_e^T dU_e, dW2[e] = h_e^T dY_e  (fp32; n_e = 0 gives zeros)
 * The weight gradients reduce over each expert's rows in ascending row order
 * with one owner per output tile, so they are bitwise reproducible.
 * [UniEP] Backward Propagation and Numerical Stability (Transposed GroupGEMM
 * along the accumulation dimension); [MoonEP] the dispatch gradient is a combine.
 *   dx [T,H] bf16; dW1, dW3 [E,H,F], dW2 [E,F,H], dgate [T,k]: fp32, device. */
MOE_API int moe_backward(moe_dims d, const void *dout, const void *W1, const void *W3, const void *W2, const moe_plan_t *plan,
                 const moe_saved_t *saved, const moe_grads_t *grads, void *dx, float *dW1, float *dW3, float *dW2,
                 float *dgate, void *ws, size_t ws_bytes, const moe_opts *opts, void *stream,
                 const moe_router_t *router);

/* ---- the router (gating) ----------------------------------------------------- */

/* Router logits on the tensor cores: logits[t,e] = sum_h x[t,h] Wr[h,e]
 * (bf16 in, fp32 accumulate and out).  [UniEP] background, Forward Propagation:
 * the router scores each token against every expert; the scores feed moe_plan.
 *   x [T,H] bf16, Wr [H,E] bf16, logits [T,E] fp32: device, caller-owned.
 *   E must be a multiple of 8 (16-byte rows of Wr).  T = 0 is a no-op. */
MOE_API int moe_router_forward(moe_dims d, const void *x, const void *Wr, float *logits, void *ws, size_t ws_bytes,
                               const moe_opts *opts, void *stream);

/* Synchronises `stream`, copies the status word out of the workspace and clears it.
 * device_status: 0 or a positive MOE_ERR_* code; where/detail: which kernel/task
 * and index reported it (may be NULL).  Returns 0 or MOE_ERR_LAUNCH. */
MOE_API int moe_get_status(void *ws, void *stream, int32_t *device_status, int32_t *where, int32_t *detail);

/* Clears the status words (status, where, detail: the first 12 bytes of `ws`),
 * asynchronously on stream.  Safe on a workspace and on moe_plan_noalloc's
 * 4-int32 status buffer. */
MOE_API int moe_clear_status(void *ws, void *stream);

/* ---- routing without a workspace ------------------------------------------------ */

/* Size of the fixed device buffer moe_plan_noalloc uses instead of a workspace. */
#define MOE_NOALLOC_SCRATCH_BYTES (4u << 20)
#define MOE_ERR_TOO_LARGE (-7) /* moe_plan_noalloc: the dims need more scratch than MOE_NOALLOC_SCRATCH_BYTES */

/* Same routing as moe_plan (same kernels, same results), for callers that
 * cannot allocate device memory while they run: code that must not call
 * cudaMalloc because it runs inside an engine or plugin whose memory plan is
 * fixed before execution, on a real-time path where an allocation could block,
 * or in a process without a device allocator of its own.  There is no
 * counterpart on the pages; it is an interface convenience.
 *
 * Its scratch (per-chunk and per-super-chunk counts and bitmaps) lives in one file-scope
 * device array of MOE_NOALLOC_SCRATCH_BYTES inside the library, which every GPU
 * that loads the library holds until the process exits.  The call allocates
 * and frees nothing.
 *   - Limit: dims whose scratch exceeds the buffer (roughly
 *     ceil(T/256) * E * 37 bytes plus alignment) return MOE_ERR_TOO_LARGE
 *     before anything is launched; e.g. T = 131072 with E = 128 fits.
 *   - status: device pointer to 4 int32 (16 bytes, caller-owned, zero before
 *     first use); the first device-detected error is recorded in its first
 *     three words as in a workspace.  moe_get_status(status, ...) reads and
 *     clears it and moe_clear_status(status, ...) clears it; both touch only
 *     those three words.
 *   - Set-up: the first call in each CUDA context (per device, and again after
 *     cudaDeviceReset or in another context of the same device) looks up the
 *     array's device address with that context current and caches it, keyed
 *     on the context's unique id; make that first call before any stream
 *     capture.
 *   - Every call uses the same array and leaves its contents behind; each
 *     call clears the words that must start at zero (the per-chunk counts)
 *     with an asynchronous memset on `stream` before its kernels run.  Calls
 *     that overlap on the GPU (on different streams, or from different
 *     threads) race on the array: serialise them.
 * Other arguments and errors as moe_plan. */
MOE_API int moe_plan_noalloc(moe_dims d, const float *logits, const moe_plan_t *plan, int32_t *status, void *stream);

/* ---- introspection ---------------------------------------------------------- */
MOE_API const char *moe_strerror(int code);
MOE_API int32_t moe_version(void);
/* Number of kernels this library has launched in this process. */
MOE_API uint64_t moe_launch_count(void);
/* Name of the i-th kernel a call launches (call: 0 plan, 1 forward, 2 backward, 3 forward with
 * schedule 1 or 2, 4 backward with schedule = 2, 5 backward with the router (schedule 0 or 1),
 * 6 moe_router_forward, 7 forward with schedule 0 and combine = 1 (combine in GEMM2's epilogue),
 * 8 backward with wgrad_subbatches = 2, 9 the same with the router, 10 forward with dispatch = 2,
 * 11 forward with dispatch = 2 and combine = 1); NULL past the end. */
MOE_API const char *moe_kernel_name(int32_t call, int32_t i);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */

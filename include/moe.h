/*
 * moe.h — C ABI of the GB300 (sm_103a) MoE expert layer.
 *
 * The layer (kernel-records pages "Sparse expert dispatch and combine",
 * "MoE training token repeat and expert computation", "MoE expert parallel
 * execution backward", each page's description):
 *
 *   given hidden states x[T,H], per token k expert ids idx[T,k] and routing
 *   weights w[T,k], expert weights Wgu[E,H,2I] (gate = columns [0,I),
 *   up = columns [I,2I)) and Wd[E,I,H],
 *
 *     y[t] = sum_j w[t,j] * ( act(x[t] Wgu[e] [:, :I], x[t] Wgu[e] [:, I:]) Wd[e] ),
 *            e = idx[t,j],
 *
 *   with act = SwiGLU  (a = silu(g) * u)  or the clamped GLU
 *   (a = (clamp(u,-L,L) + 1) * min(g,L) * sigmoid(alpha * min(g,L))).
 *   The backward returns dx, d(topk weights), dWgu (d_gate = [:,:,:I],
 *   d_up = [:,:,I:]) and dWd, the gradients of <dy, y>.
 *
 * General conventions
 *   - Every pointer argument is a DEVICE pointer (cudaMalloc / torch), except
 *     the `moe_shape` and `moe_plan_t` structs themselves, which live in host
 *     memory.  Tensors are dense row-major; the caller owns all memory.  The
 *     library never allocates device memory and keeps no state other than a
 *     per-device cache of kernel attributes.
 *   - Calls are asynchronous on `stream` (0 = legacy default stream).  The
 *     return value reports host-side validation and launch failures.  Errors
 *     found on the device (an expert id outside [0,E), a pipeline wait that
 *     timed out) are recorded in a word inside the workspace and read with
 *     moe_get_device_error(); outputs of such a call are undefined.
 *   - Outputs are overwritten, never accumulated into.
 *   - dtype MOE_BF16: x, y, dy, dx, Wgu, Wd are bfloat16; matrix products run
 *     on the tensor cores with fp32 accumulation.  dtype MOE_FP32: those
 *     tensors are float32 and the products run as TF32 with fp32
 *     accumulation.  topk weights, d(topk weights) and the weight gradients
 *     are always float32; expert ids are int32.  The fp32 path is meant for
 *     small correctness cases: every call copies both weight tensors into
 *     its workspace (transposed for the forward, rounded to TF32 for the
 *     backward's dgrads) and transposes the gathered rows for the weight
 *     gradients, so its workspace and traffic grow with E*H*I per call.
 *   - Requirements: T >= 0, 1 <= k <= E <= 1024, T*k < 2^31, H and I
 *     multiples of 8 (16-byte rows for the tensor-memory-access unit),
 *     16-byte aligned pointers.  T = 0 is allowed: outputs with a T extent
 *     are empty, the weight gradients are zero-filled.
 *   - Workspace: `ws` of at least moe_workspace_size(shape, which) bytes,
 *     256-byte aligned, zero-filled by the caller before its FIRST use (the
 *     device error word lives in it).  One workspace must not be used by two
 *     calls that may run concurrently.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t;   /* same type as cudaStream_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,   /* a null pointer, a bad dimension, misalignment */
  MOE_ERR_UNSUPPORTED = 2,   /* no sm_103a device, or a case not built */
  MOE_ERR_WORKSPACE = 3,     /* ws_bytes below moe_workspace_size() */
  MOE_ERR_BAD_INDEX = 4,     /* device: an expert id outside [0, E) */
  MOE_ERR_TIMEOUT = 5,       /* device: a pipeline wait ran out of time */
  MOE_ERR_CUDA = 6           /* a CUDA runtime / driver call failed */
} moe_status;

typedef enum { MOE_ACT_SWIGLU = 0, MOE_ACT_CLAMPED_GLU = 1 } moe_act;
typedef enum { MOE_BF16 = 0, MOE_FP32 = 1 } moe_dtype;
/* Column layout of the fused gate_up weight w_gate_up[e] [H, 2I]: the
 * pages name a fused gate_up projection without fixing its columns.
 * CONCAT: gate = columns [0, I), up = [I, 2I).  INTERLEAVED: gate = the even
 * columns, up = the odd ones (column 2i and 2i+1 belong to output i).
 * dw_gate_up comes back in the same layout. */
typedef enum { MOE_GATE_UP_CONCAT = 0, MOE_GATE_UP_INTERLEAVED = 1 } moe_gate_up_layout;

/* Problem description (model dimensions named on the pages' workload lines:
 * hidden_size H, intermediate size I, number of experts E,
 * num_experts_per_tok k).  clamp_limit / alpha are used by the clamped GLU
 * only (7.0 / 1.702 in the workloads). */
typedef struct {
  int64_t T;
  int32_t H, I, E, k;
  int32_t act;          /* moe_act */
  float clamp_limit;
  float alpha;
  int32_t dtype;        /* moe_dtype */
  int32_t gate_up_layout;   /* moe_gate_up_layout */
  int32_t out_fp32;     /* 0: y and dx in the storage dtype; 1: in fp32 (for
                         * callers that sum them further, e.g. the combine of
                         * the expert-parallel exchange, so the rows are not
                         * rounded twice) */
} moe_shape;

/* Dispatch plan ("masked indexing" / "sparse token extraction" in the pages'
 * descriptions).  Slot s = t*k + j is token t's j-th choice.  Rows of the
 * expert-grouped order are sorted by expert id, and by slot within an
 * expert, so the plan is unique:
 *   counts[e]   number of slots routed to expert e            [E]
 *   offsets[e]  exclusive prefix sum of counts                [E+1]
 *   perm[r]     slot held by grouped row r                    [T*k]
 *   inv[s]      grouped row of slot s (inv[perm[r]] = r)      [T*k]
 * All four are int32 device arrays owned by the caller. */
typedef struct {
  int32_t* counts;
  int32_t* offsets;
  int32_t* perm;
  int32_t* inv;
} moe_plan_t;

/* Optional per-expert biases.  The pages' layer has none; this variant of
 * the layer adds one bias row per expert to each projection:
 *   h = x Wgu[e] + b_gate_up[e],   o = act(h) Wd[e] + b_down[e],
 *   y[t] = sum_j w[t,j] * o,
 * so d(topk weights) also sees the bias (d_w = <dy, o>) and the gradients of
 * the biases are db_gate_up[e] = sum, over the expert's rows, of dh (the
 * gradient of h) and db_down[e] = sum of w * dy.
 *   b_gate_up  [E,2I] storage dtype, columns in the shape's gate_up_layout
 *   b_down     [E,H]  storage dtype
 *   db_gate_up [E,2I] fp32, written by moe_ffn_bwd when non-NULL (same layout)
 *   db_down    [E,H]  fp32, written by moe_ffn_bwd when non-NULL
 * Every pointer may be NULL: a NULL bias is no bias (zero), a NULL gradient
 * is not computed (a frozen bias).  A NULL moe_bias_t* means all four NULL.
 * The backward must see the biases the forward used (the saved context
 * holds h with b_gate_up added; b_down enters d(topk weights)).  Experts with
 * no routed token get zero bias gradients; the sums run in a fixed row order. */
typedef struct {
  const void* b_gate_up;
  const void* b_down;
  float* db_gate_up;
  float* db_down;
} moe_bias_t;

/* Bytes of workspace needed by one call: which = 0 moe_plan (and
 * moe_route with a plan), 1 moe_ffn_fwd, 2 moe_ffn_bwd with a saved
 * context, 3 moe_ffn_bwd without one (it then recomputes the context).
 * Returns 0 for an invalid shape or `which`. */
size_t moe_workspace_size(const moe_shape* shape, int which);

/* Bytes of the context the training forward saves for the backward, in the
 * library's expert-grouped, tile-padded row order: the gathered token rows
 * (storage dtype, so the backward does not gather x again), then, 256-byte
 * aligned, the gate_up pre-activations.  Those are fp32 (the accumulator
 * values, not a bf16 rounding of them), except for the clamped GLU with bf16
 * storage and a clamp limit that fp16 represents exactly (|L| <= 32768, e.g.
 * 7.0): there they are fp16 (11 significant bits), values past the clamp are
 * kept as infinite markers and values inside round to fp16 values inside,
 * so the clamp masks of the backward are exact.
 * Returns 0 for an invalid shape. */
size_t moe_saved_size(const moe_shape* shape);

/* Build the dispatch plan of topk_idx [T,k] (int32, device).
 * Writes plan->counts/offsets/perm/inv.  An id outside [0,E) records
 * MOE_ERR_BAD_INDEX in the workspace; the plan is then undefined. */
moe_status moe_plan(const moe_shape* shape, const int32_t* topk_idx,
                    const moe_plan_t* plan, void* ws, size_t ws_bytes,
                    moe_stream_t stream);

/* Top-k routing, the step before the layer: the layer's inputs topk_idx and
 * topk_w from router logits.  The pages take the routing as given; the
 * workload descriptions that accompany them route each token to the k
 * experts with the largest logits, weighted by the softmax over those k
 * logits (equivalently, the top-k of the full softmax renormalised to one).
 *   logits [T,E] fp32 (device, finite); E <= 1024, k <= 32.
 *   topk_idx [T,k] int32: the chosen ids by descending logit; equal logits
 *     are taken in ascending expert id, so the choice is unique.
 *   topk_w [T,k] fp32: softmax over the chosen logits (each row sums to 1).
 *   plan: NULL, or plan arrays that also receive the dispatch plan of
 *     topk_idx, exactly as moe_plan builds it (ws: moe_workspace_size(shape,
 *     0) bytes, required only with a plan).
 * Outputs are overwritten; T = 0 is a no-op. */
moe_status moe_route(const moe_shape* shape, const float* logits, int32_t* topk_idx,
                     float* topk_w, const moe_plan_t* plan, void* ws, size_t ws_bytes,
                     moe_stream_t stream);

/* Forward pass (dispatch -> gate_up GEMM + activation -> down GEMM with the
 * routing-weight scale -> deterministic k-way combine).
 *   x [T,H], topk_idx [T,k] int32, topk_w [T,k] fp32, w_gate_up [E,H,2I],
 *   w_down [E,I,H]  -> y [T,H].
 *   bias: NULL, or the optional per-expert biases (moe_bias_t above; the
 *         forward reads b_gate_up and b_down only).
 *   plan: a plan built by moe_plan for this topk_idx, or NULL to build one
 *         inside the workspace.
 *   saved: NULL (inference) or a buffer of moe_saved_size() bytes that
 *          receives the context moe_ffn_bwd needs (training).
 * The combine sums each token's k expert outputs in fp32 in the order
 * j = 0..k-1 (no atomics): results are bitwise reproducible. */
moe_status moe_ffn_fwd(const moe_shape* shape, const void* x,
                       const int32_t* topk_idx, const float* topk_w,
                       const void* w_gate_up, const void* w_down,
                       const moe_bias_t* bias,
                       const moe_plan_t* plan, void* y, void* saved,
                       void* ws, size_t ws_bytes, moe_stream_t stream);

/* Backward pass of <dy, y>.
 *   dy [T,H]; x, topk_idx, topk_w, w_gate_up, w_down, bias as given to the
 *   forward (bias also names the bias-gradient outputs); plan: the plan of
 *   topk_idx (required).
 *   saved: the context the training forward wrote, or NULL.  With NULL the
 *   backward recomputes the context (the forward's gather of x and its
 *   gate_up GEMM, one third of the forward's FLOPs) into a workspace of
 *   moe_workspace_size(shape, 3) bytes; the results are bit-identical to
 *   those with the saved context, which needs moe_saved_size() bytes of
 *   caller memory between the two calls instead.
 *   Outputs: dx [T,H]; d_topk_w [T,k] fp32; dw_gate_up [E,H,2I] fp32
 *   (the gate and up columns as in the shape's gate_up_layout); dw_down [E,I,H] fp32.  Experts
 *   with no routed token get zero weight gradients.  All reductions run in
 *   a fixed order (no float atomics). */
moe_status moe_ffn_bwd(const moe_shape* shape, const void* dy, const void* x,
                       const int32_t* topk_idx, const float* topk_w,
                       const void* w_gate_up, const void* w_down,
                       const moe_bias_t* bias,
                       const moe_plan_t* plan, const void* saved,
                       void* dx, float* d_topk_w, float* dw_gate_up,
                       float* dw_down, void* ws, size_t ws_bytes,
                       moe_stream_t stream);

/* ---- expert-parallel exchange primitives ("MoE expert parallel execution
 * backward", title: experts spread over devices).  A rank that owns a
 * contiguous range of experts receives, from every rank, the rows of its
 * experts: the plan's expert-grouped order makes each destination's rows one
 * contiguous segment, so the dispatch is one gather into that order and one
 * all-to-all of the segments (by the caller's communication library), and
 * the combine is the mirrored all-to-all followed by moe_combine_rows.  Both
 * calls are plain device kernels on `stream`; neither allocates. ---- */

/* Row gather: dst[r] = src[index[r] / div] for r < n.
 *   index [n] int32 (device); div >= 1: with index = plan->perm, div = k
 *     gathers token rows into the expert-grouped order (dispatch of x or dy),
 *     div = 1 gathers per-slot values (routing weights); with index =
 *     plan->inv, div = 1 brings per-row values back to slot order.
 *   src [src_rows, row_bytes] and dst [n, row_bytes]: row-major device
 *     arrays; row_bytes > 0 and a multiple of 4 (16-byte accesses when it is
 *     a multiple of 16 and both pointers are 16-byte aligned).
 * An index outside [0, src_rows * div) yields a zero row (no fault, no
 * error).  n = 0 is a no-op.  Returns MOE_ERR_INVALID_ARG for null pointers
 * (with n > 0), div < 1 or a bad row_bytes. */
moe_status moe_gather_rows(const int32_t* index, int64_t n, int32_t div, const void* src,
                           int64_t src_rows, int64_t row_bytes, void* dst,
                           moe_stream_t stream);

/* Combine of rows in the plan's dense expert-grouped order back to tokens:
 *   dst[t] = sum_{j=0..k-1} (topk_w ? topk_w[t,j] : 1) * src[inv[t*k + j]],
 * summed in fp32 in the order j = 0..k-1 (no atomics; bitwise
 * reproducible).  shape gives T, H, k, the storage dtype and out_fp32.
 *   inv [T*k] int32: plan->inv of the plan that ordered the rows.
 *   src [T*k, H]: fp32 when src_fp32, else the storage dtype.
 *   dst [T, H]: fp32 when shape->out_fp32, else the storage dtype.
 * A slot whose inv lies outside [0, T*k) contributes nothing.  16-byte
 * aligned src and dst; T = 0 is a no-op. */
moe_status moe_combine_rows(const moe_shape* shape, const int32_t* inv, const float* topk_w,
                            const void* src, int32_t src_fp32, void* dst,
                            moe_stream_t stream);

/* Synchronise `stream`, return the first device-side error recorded in the
 * workspace since the last call (MOE_OK if none) and clear it. */
moe_status moe_get_device_error(void* ws, moe_stream_t stream);

/* Upper bound, in nanoseconds, on any single pipeline wait inside the GEMM
 * kernels before they give up and record MOE_ERR_TIMEOUT (default 2 s).
 * Process-wide; returns the previous value. */
uint64_t moe_set_wait_timeout_ns(uint64_t ns);

/* Static description of a status code. */
const char* moe_status_string(moe_status status);

/* moe_plan without a workspace.  The pages have no counterpart to this
 * entry point; it exists for callers that cannot allocate device memory at
 * the point where they need a dispatch plan: code running inside an
 * allocator-free region (a memory pool that is already carved up, a
 * latency-critical path where cudaMalloc's implicit synchronisation is not
 * acceptable, a host runtime that owns all device memory and only hands out
 * the tensors it manages).  The plan kernels' scratch (per-chunk expert
 * histograms, tile-padded offsets, an error word) then lives in a fixed
 * 1 MiB array inside this library's device image, present on every GPU that
 * loads the library until the process exits.  This call allocates nothing.
 *   - Arguments and outputs are those of moe_plan, minus the workspace; the
 *     result is identical to moe_plan's.
 *   - Size limit: ceil(T*k / 1024) * E <= 259968 (e.g. T*k <= 1,039,360 for
 *     E = 256, T*k <= 259,072 for E = 1024); larger problems return
 *     MOE_ERR_WORKSPACE without launching anything.
 *   - The first call on a device resolves the device address of the array
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.  The address is kept per device context: a
 *     call that finds a different context current (for instance after
 *     cudaDeviceReset, which unloads the array) resolves it again, so such a
 *     call, too, should come before any stream capture.
 *   - Launches (three plan kernels and one memset of the error word) count in
 *     moe_kernel_launch_count() and the event timer like moe_plan's.
 *   - Every call on a device shares the one array and leaves its contents
 *     behind; the call clears what must start at zero.  Calls whose kernels
 *     may overlap on the GPU (different streams, or different host threads)
 *     race on the array and corrupt each other's plans: serialise them.
 *   - An expert id outside [0, E) is left out of the counts; with no error
 *     word to read, a caller detects it as offsets[E] < T*k. */
moe_status moe_plan_noalloc(const moe_shape* shape, const int32_t* topk_idx,
                            const moe_plan_t* plan, moe_stream_t stream);

/* ---- measurement helpers (no counterpart in the pages; they serve the
 * roofline accounting of the benchmark) ---- */

/* Number of kernels (and memsets) this library has launched in this
 * process, across all entry points and devices. */
uint64_t moe_kernel_launch_count(void);

/* Turn the per-kernel event timer on (on != 0) or off; returns the previous
 * setting.  While on, each entry point records a pair of CUDA events on the
 * caller's stream around every kernel it launches (host-side event objects
 * only, no device memory).  Off by default. */
int moe_profile_enable(int on);

/* Wait for the recorded events, add up the elapsed time per kernel kind since
 * the last read, write up to `n` kinds into total_ms[] / launches[] (either
 * may be NULL), reset the sums and return the number of kinds. */
int moe_profile_read(double* total_ms, uint64_t* launches, int n);

/* Name of kernel kind `kind` (NULL if out of range). */
const char* moe_profile_kernel_name(int kind);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */

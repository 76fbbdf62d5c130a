/*
 * moe.h -- C ABI of the GB300 (sm_103a) mixture-of-experts layer step.
 *
 * One MoE layer step on one GPU: router scoring, top-k with a capacity factor
 * and overflow drop, permutation into contiguous per-expert buffers, the
 * experts' SwiGLU FFN as grouped GEMMs, the inverse permutation with a
 * gate-weighted combine, and the matching backward.  The sequence follows
 * "The step timeline: dispatch, expert GEMM, combine" on the
 * gpu_expert_parallel page: with every expert local, the dispatch and combine
 * all-to-alls reduce to the permute and the unpermute.
 *
 * Conventions shared by every call
 * --------------------------------
 * - All pointers are device pointers on the calling thread's current CUDA
 *   device unless a parameter says otherwise.  The library never allocates,
 *   frees or keeps caller memory; the caller owns every buffer.
 * - Every call that takes a stream is asynchronous on that stream (NULL = the
 *   legacy default stream) and never synchronises with the host, except
 *   moe_get_device_error and moe_profiler_read.
 * - Tensors are dense and row-major.  Activations and expert weights use
 *   cfg->dtype (MOE_F32 or MOE_BF16); router weights, router bias, gates,
 *   probabilities and every gradient buffer except dx are float32; index
 *   tensors are int32.
 * - Activation and weight pointers must be 16-byte aligned.
 * - MOE_BF16 needs d_model and d_ff to be multiples of 256 (the grouped GEMM
 *   tiles); MOE_F32 needs them to be multiples of 4.  1 <= k <= min(E, 8),
 *   1 <= E <= 128.
 * - Argument, shape and alignment errors are detected on the host before any
 *   work is queued and are returned as a status.  Launch failures return
 *   MOE_ERR_CUDA.  Problems found by the kernels (a corrupt routing state, an
 *   out-of-range row, a pipeline wait that exceeded its time limit) are
 *   recorded in a per-device error word and reported by
 *   moe_get_device_error; the offending access is skipped, never performed.
 *
 * Shapes (T tokens, d = d_model, f = d_ff, E experts, k picks per token)
 * -------------------------------------------------------------------------
 *   x, y, dy, dx          [T, d]           dtype
 *   W_r                   [d, E]           float32   router weight
 *   bias                  [E]              float32   fixed router bias (optional)
 *   W1, W3                [E, d, f]        dtype     x W1 -> gate path, x W3 -> up path
 *   W2                    [E, f, d]        dtype
 *   ids, slot, row_of     [T, k]           int32
 *   gates                 [T, k]           float32
 *   probs                 [T, E]           float32
 *   counts                [E]              int32     kept assignments per expert
 *   offsets               [E + 1]          int32     first row of each expert
 *   src_token             [max_rows]       int32     token of each row, -1 on pad rows
 *   x_perm, y_perm, dy_perm, dx_perm [max_rows, d]  dtype
 *   a, b, h, da, db       [max_rows, f]    dtype
 *   dW1, dW3              [E, d, f]        float32
 *   dW2                   [E, f, d]        float32
 *   dW_r                  [d, E]           float32
 *
 * Permutation map layout: the rows of expert e are
 * [offsets[e], offsets[e] + counts[e]), in slot order, followed by zero pad
 * rows up to offsets[e+1]; offsets[e] is a multiple of 128, offsets[0] = 0.
 * max_rows (moe_max_rows) bounds offsets[E] for every routing outcome.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; declared here so the header needs no CUDA headers. */
typedef struct CUstream_st* moe_stream_t;

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,  /* NULL where a pointer is required, bad flag value */
  MOE_ERR_SHAPE = 2,        /* sizes outside the supported range */
  MOE_ERR_DTYPE = 3,        /* unknown dtype */
  MOE_ERR_ALIGNMENT = 4,    /* a pointer is not 16-byte aligned */
  MOE_ERR_WORKSPACE = 5,    /* workspace missing or smaller than moe_workspace_size */
  MOE_ERR_CUDA = 6,         /* a CUDA runtime call or kernel launch failed */
  MOE_ERR_DEVICE_CHECK = 7, /* a kernel found an invalid index (see moe_get_device_error) */
  MOE_ERR_TIMEOUT = 8,      /* a kernel pipeline wait exceeded its time limit */
  MOE_ERR_UNSUPPORTED = 9   /* the device is not sm_103 */
} moe_status;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;

typedef struct {
  int32_t T;                /* tokens in this (micro-)batch, >= 0 */
  int32_t d_model;          /* d */
  int32_t d_ff;             /* f */
  int32_t E;                /* experts */
  int32_t k;                /* experts per token (top-k) */
  float capacity_factor;    /* C = ceil(cf * T * k / E); <= 0 means dropless */
  int32_t capacity;         /* >= 0: use this exact capacity instead of the factor; < 0: use the factor */
  int32_t dtype;            /* moe_dtype of activations and expert weights */
  float aux_loss_coeff;     /* >= 0; > 0 adds the auxiliary load-balancing loss to the backward (moe_aux_loss) */
} moe_config;

/* Expert and router parameters (device pointers, read only). */
typedef struct {
  const float* W_r;   /* [d, E] */
  const float* bias;  /* [E] or NULL */
  const void* W1;     /* [E, d, f] */
  const void* W3;     /* [E, d, f] */
  const void* W2;     /* [E, f, d] */
} moe_weights;

/* Routing state and activations that the forward keeps for the backward.
 * Keeping the assignment indices and the permutation map lets the backward
 * reuse the routing instead of recomputing it ("Recomputation re-runs the
 * dispatch unless you save the permutation", gpu_expert_parallel page).
 * Sizes are in the shape table above.  Recompute variant: with a, b and h all
 * NULL the forward keeps only the routing state, x_perm and y_perm, and the
 * backward recomputes a, b and h with the same up product (bit for bit the
 * forward's); the workspace is then moe_workspace_size(cfg, 2) for both calls. */
typedef struct {
  int32_t* ids;
  float* gates;
  int32_t* slot;
  int32_t* row_of;
  int32_t* src_token;
  int32_t* counts;
  int32_t* offsets;
  float* probs;
  void* x_perm;
  void* a;
  void* b;
  void* h;
  void* y_perm;
} moe_saved;

/* float32 gradient buffers of the parameters (accumulated across calls when
 * accumulate != 0, overwritten otherwise). */
typedef struct {
  float* dW_r;
  float* dW1;
  float* dW3;
  float* dW2;
  float* aux_loss;  /* device fp32 scalar that receives the auxiliary loss, or NULL */
} moe_grads;

/* Human-readable name of a status code (static storage). */
const char* moe_status_string(moe_status s);

/* Expert capacity: *C = ceil(cf * T * k / E) computed in double from the
 * float capacity factor, or cfg->capacity when that is >= 0, or -1 when the
 * layer is dropless.  Capacity-factor passage, "The Capacity Factor: A Dial
 * Between Imbalance and Dropping" (distributed-training tutorial, Expert
 * Parallelism section).  Host only. */
moe_status moe_capacity(const moe_config* cfg, int32_t* C);

/* Upper bound on offsets[E] (rows of the per-expert buffers), a multiple of
 * 128: min(T*k + 127*E, E * roundup128(C)) rounded up to 128.  Host only. */
moe_status moe_max_rows(const moe_config* cfg, int64_t* rows);

/* Bytes of workspace that moe_layer_fwd (training = 0) or moe_layer_fwd and
 * moe_layer_bwd (training = 1; 2 with a, b, h recomputed, see moe_saved) need.  The workspace holds the routing
 * histograms, the forward intermediates when no moe_saved is given, and the
 * backward scratch.  Host only; for bf16 layers the router-weight gradient's
 * partial sums scale with the SM count of the current device, so ask with the
 * device that will run the layer current. */
moe_status moe_workspace_size(const moe_config* cfg, int training, size_t* bytes);

/* Router scoring, softmax, top-k and capacity slotting (steps "the router
 * scores every token" and the capacity dial).
 *   logits l = x W_r + bias in fp32; probs = softmax(l) in fp32;
 *   ids[t, 0..k-1] = experts of the k largest logits, descending, ties to the
 *   lower index; gates: k = 1 -> probs[t, ids[t,0]]; k > 1 -> the picked
 *   probabilities renormalised over the picks;
 *   slot: assignments are visited choice-major then in token order; each
 *   expert hands out slots 0, 1, ...; an assignment at slot >= C is dropped
 *   (slot = -1, row_of = -1);  counts[e] = kept assignments of expert e;
 *   offsets, row_of, src_token as described at the top of this file.
 * probs may be NULL.  Deterministic.  ws must hold moe_workspace_size(cfg, 0). */
moe_status moe_router_topk(const moe_config* cfg, const void* x, const float* W_r, const float* bias,
                           int32_t* ids, float* gates, float* probs, int32_t* slot, int32_t* row_of,
                           int32_t* src_token, int32_t* counts, int32_t* offsets, void* ws, size_t ws_bytes,
                           moe_stream_t stream);

/* Permute tokens into the per-expert buffers ("tokens are permuted into
 * contiguous per-destination buffers"): x_perm[row_of[t,j]] = x[t] for every
 * kept assignment; pad rows [offsets[e] + counts[e], offsets[e+1]) are zeroed.
 * Rows at or beyond offsets[E] are not touched. */
moe_status moe_permute(const moe_config* cfg, const void* x, const int32_t* row_of, const int32_t* counts,
                       const int32_t* offsets, void* x_perm, moe_stream_t stream);

/* The experts' feed-forward as grouped GEMMs over the ragged row segments
 * ("Sorting tokens by destination is what lets the expert computation become
 * a batched or grouped matrix multiply"):
 *   a = X_e W1_e, b = X_e W3_e, h = silu(a) * b, y_perm = h W2_e
 * with fp32 accumulation; silu(z) = z / (1 + exp(-z)).  h is required; a and b
 * may be NULL (they are stored only for the backward).  Pad rows give zero. */
moe_status moe_grouped_ffn(const moe_config* cfg, const void* x_perm, const int32_t* counts,
                           const int32_t* offsets, const void* W1, const void* W3, const void* W2, void* h,
                           void* y_perm, void* a, void* b, moe_stream_t stream);

/* Inverse permutation with the gate-weighted combine ("the inverse permutation
 * restores the original token order"): y[t] = sum over kept j of
 * gates[t,j] * y_perm[row_of[t,j]], summed in fp32 in j order; a token whose
 * assignments were all dropped gets 0. */
moe_status moe_unpermute_combine(const moe_config* cfg, const void* y_perm, const int32_t* row_of,
                                 const float* gates, void* y, moe_stream_t stream);

/* Whole forward: moe_router_topk, moe_permute, moe_grouped_ffn,
 * moe_unpermute_combine.  With saved == NULL the intermediates live in ws;
 * with saved != NULL every field of *saved must be set and receives the state
 * moe_layer_bwd needs. */
moe_status moe_layer_fwd(const moe_config* cfg, const moe_weights* w, const void* x, void* y,
                         const moe_saved* saved, void* ws, size_t ws_bytes, moe_stream_t stream);

/* Backward of the combine (token-gradient routing, the reverse of the combine
 * all-to-all in "Backward walks the same path in reverse"):
 *   dy_perm[row_of[t,j]] = gates[t,j] * dy[t];  dg[t,j] = <dy[t], y_perm[row_of[t,j]]>
 * (0 for dropped assignments); pad rows of dy_perm are zeroed; and the logit
 * gradient dl [T, E] (float32): k > 1 -> dl[t, ids_j] = g_j (dg_j - sum_i g_i dg_i)
 * and 0 elsewhere; k = 1 -> dl[t, :] = g dg (onehot(ids_0) - probs[t, :]).
 * probs may be NULL when k > 1. */
moe_status moe_combine_bwd(const moe_config* cfg, const void* dy, const void* y_perm, const int32_t* ids,
                           const int32_t* row_of, const float* gates, const float* probs,
                           const int32_t* counts, const int32_t* offsets, void* dy_perm, float* dg, float* dl,
                           moe_stream_t stream);

/* Expert backward as grouped GEMMs (dgrad and wgrad):
 *   dH = dY_e W2_e^T;  da = dH * b * s * (1 + a (1 - s)), s = sigmoid(a);  db = dH * silu(a)
 *   dx_perm = da W1_e^T + db W3_e^T
 *   dW1_e (+)= X_e^T da;  dW3_e (+)= X_e^T db;  dW2_e (+)= H_e^T dY_e     (float32)
 * accumulate = 0 overwrites dW1/dW3/dW2, 1 adds to them (gradient
 * accumulation over micro-batches).  da and db are caller scratch of shape
 * [max_rows, f]. */
moe_status moe_grouped_ffn_bwd(const moe_config* cfg, const void* x_perm, const void* a, const void* b,
                               const void* h, const void* dy_perm, const int32_t* counts, const int32_t* offsets,
                               const void* W1, const void* W3, const void* W2, void* da, void* db, void* dx_perm,
                               float* dW1, float* dW3, float* dW2, int accumulate, moe_stream_t stream);

/* Auxiliary load-balancing loss of the router and its logit gradient.  The
 * tutorial's MoE configuration example names an "aux_loss" coefficient
 * (distributed-training tutorial, "The Conflict Between EP and TP") without a
 * formula; the usual expert-balance form is taken:
 *   f_e = (assignments (t, j) with ids[t,j] = e, before the capacity drop) / (T k)
 *   P_e = (1/T) sum_t probs[t,e]
 *   L   = c * E * sum_e f_e P_e,          c = cfg->aux_loss_coeff
 * f is a count and carries no gradient, so
 *   dl[t,e'] += c * E / T * probs[t,e'] * (f_e' - sum_e f_e probs[t,e]).
 * probs [T, E] fp32 and ids [T, k] int32 as moe_router_topk writes them; dl
 * [T, E] fp32 is updated in place (moe_combine_bwd's output); *loss (device
 * fp32, may be NULL) receives L.  Sums run in a fixed order (bitwise
 * reproducible).  ws must hold moe_workspace_size(cfg, 1).  When the
 * coefficient is 0 (or T = 0) dl is left as it is and *loss, if given, is set
 * to 0. */
moe_status moe_aux_loss(const moe_config* cfg, const float* probs, const int32_t* ids, float* loss, float* dl,
                        void* ws, size_t ws_bytes, moe_stream_t stream);

/* Inverse permutation of the token gradient plus the router backward ("Its
 * gradient behaves like any other shared parameter", gpu_expert_parallel page):
 *   dx[t] = sum over kept j of dx_perm[row_of[t,j]] + dl[t] W_r^T
 *   dW_r (+)= x^T dl        (float32, fixed summation order; no bias gradient)
 * ws must hold moe_workspace_size(cfg, 1). */
moe_status moe_unpermute_dx_router_bwd(const moe_config* cfg, const void* x, const void* dx_perm,
                                       const int32_t* row_of, const float* dl, const float* W_r, void* dx,
                                       float* dW_r, int accumulate, void* ws, size_t ws_bytes,
                                       moe_stream_t stream);

/* Whole backward from the state saved by moe_layer_fwd (no re-routing):
 * moe_combine_bwd, moe_aux_loss (when cfg->aux_loss_coeff > 0; saved->probs is
 * then required for every k and grads->aux_loss may receive the loss),
 * moe_grouped_ffn_bwd, moe_unpermute_dx_router_bwd.
 * grads receives dW_r, dW1, dW3, dW2 (accumulate as above); dx [T, d] in dtype. */
moe_status moe_layer_bwd(const moe_config* cfg, const moe_weights* w, const void* x, const void* dy,
                         const moe_saved* saved, void* dx, const moe_grads* grads, int accumulate, void* ws,
                         size_t ws_bytes, moe_stream_t stream);

/* Bytes of device memory the library reserves, on every GPU that loads it and
 * until the process exits, for moe_router_topk_noalloc. */
#define MOE_NOALLOC_SCRATCH_BYTES (4u << 20)

/* moe_router_topk for callers that cannot allocate device memory: a plugin
 * hosted by a program that owns every allocation, a path whose memory budget
 * is fixed at start-up, or a latency-critical loop that cannot afford the
 * implicit device synchronisation of cudaMalloc/cudaFree.  No workspace is
 * passed; the routing histograms, their scan and (bf16 layers of at least
 * 128 tokens) the three bf16 parts of W_r live in a static device array of
 * MOE_NOALLOC_SCRATCH_BYTES owned by the library (the pages have no
 * counterpart of this entry point; it is a deployment convenience).
 * It runs the same kernels as moe_router_topk for the same layer, so
 * arguments, results (bit for bit) and errors are those of moe_router_topk,
 * plus MOE_ERR_WORKSPACE, returned before anything is queued, when the layer
 * needs more than MOE_NOALLOC_SCRATCH_BYTES of scratch:
 * 2 * E * k * ceil(T/64) * 4 bytes of histograms and scan, plus
 * 3 * E_pad * d * 2 bytes of W_r parts for bf16 layers with T >= 128
 * (E_pad = E rounded up to 16, 32, 64 or 128), plus under 2 KB of alignment
 * (E = 32, k = 4, d = 4096 fits up to about 210,000 tokens).  The call
 * allocates nothing.
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  Every call on a device shares the one array and
 * it keeps the previous call's contents (the kernels rewrite or clear all of
 * it they read), so calls that overlap on the GPU -- on two streams, or from
 * two host threads -- race and must be serialised by the caller. */
moe_status moe_router_topk_noalloc(const moe_config* cfg, const void* x, const float* W_r, const float* bias,
                                   int32_t* ids, float* gates, float* probs, int32_t* slot, int32_t* row_of,
                                   int32_t* src_token, int32_t* counts, int32_t* offsets, moe_stream_t stream);

/* Waits for the current device to finish, then reads the device error word:
 * *code is MOE_OK, MOE_ERR_DEVICE_CHECK or MOE_ERR_TIMEOUT, *detail says which
 * kernel and check; clear != 0 resets the word.  Either output may be NULL. */
moe_status moe_get_device_error(int32_t* code, int32_t* detail, int clear);

/* Self-test of failure detection (the pages have no counterpart; it checks
 * this library's own safeguard).  Every mbarrier wait in the tensor-core
 * kernels gives up after a time limit, records MOE_ERR_TIMEOUT in the device
 * error word, drains and exits, so a stalled pipeline is reported rather than
 * hanging the GPU.  This launches one thread that waits with that same helper
 * on a barrier nothing arrives at (arrive = 0) or one that another warp
 * arrives at (arrive = 1, the control), giving up after limit_ns nanoseconds
 * (1e6 <= limit_ns <= 2e9).  Afterwards moe_get_device_error reports
 * MOE_ERR_TIMEOUT (arrive = 0) or MOE_OK (arrive = 1); the GPU stays usable. */
moe_status moe_selftest_bounded_wait(int64_t limit_ns, int arrive, moe_stream_t stream);

/* Kernel launches the library has issued in this process (all devices). */
uint64_t moe_launch_count(void);

/* Optional per-kernel timing with CUDA events recorded on the launch stream
 * around every kernel.  moe_profiler_enable(1) clears earlier records and
 * starts recording; moe_profiler_enable(0) stops.  moe_profiler_read
 * synchronises on the recorded events and fills, for kernel id 0 <= id <
 * moe_kernel_kinds(), the launches and total milliseconds. */
moe_status moe_profiler_enable(int on);
int32_t moe_kernel_kinds(void);
/* Restricts the profiler to launches of kernel kind id (0 <= id <
 * moe_kernel_kinds()), or to every kind when id < 0 (the default).  Applies to
 * launches issued after the call; records already taken are kept. */
moe_status moe_profiler_filter(int32_t id);
const char* moe_kernel_name(int32_t id);
/* NVTX ranges for timeline tools (off by default; the pages have no
 * counterpart).  While on, every kernel launch is bracketed by an NVTX range
 * named after its kernel kind (moe_kernel_name) and every moe_layer_fwd /
 * moe_layer_bwd call by a range of that name, pushed and popped on the
 * calling host thread, so an nsys or ncu timeline can be cut by layer step and
 * kernel.  Without a tool attached a range costs a few nanoseconds.  Host only. */
moe_status moe_nvtx_enable(int on);
moe_status moe_profiler_read(int32_t id, int64_t* launches, double* total_ms);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */

/*
 * moe.h -- C ABI of the GB300 (sm_103a) sparse Mixture-of-Experts forward.
 *
 * The layer (after "Distributed Training Part 4: Tensor Parallelism, Hybrid Parallelism,
 * MoE + Expert Parallelism", jesamkim ai-tech-blog, §3 Mixture of Experts and §4 Expert
 * Parallelism):
 *
 *   z[t,e]    = (x[t] . W_r[e] + b_e) / tau                 router linear      (§3 Structure)
 *   p[t,:]    = softmax(z[t,:])                              router softmax     (§3 Structure)
 *   idx[t,:]  = the k largest z[t,e], descending, ties to the lower e           (§3 TopK)
 *   gate[t,j] = p[t, idx[t,j]]   (not renormalised; MOE_FLAG_RENORM_GATES: / sum_j) (§3 G(x)_i)
 *   dispatch  = rows (t,j) in expert-contiguous order, stable in token order     (§4 Dispatch)
 *   E_e(v)    = W2_e (SiLU(W1_e v) * (W3_e v))             SwiGLU expert FFN  (§3 "FFN")
 *   y[t]      = sum_j gate[t,j] * E_{idx[t,j]}(x[t])         combine            (§3 output, §4 Combine)
 *   aux       = E * sum_e f_e P_e,  f_e = count_e/(T k),  P_e = mean_t p[t,e]  (§3 Load-Balancing Loss)
 *
 * Conventions for every call:
 *   - All tensor pointers are DEVICE pointers unless the name ends in _host.  All are
 *     row-major and contiguous: x [T,d]; W_r [E,d]; router bias [E] fp32; W1, W3 [E,F,d]
 *     (row f of expert e is the weight vector of hidden unit f); W2 [E,d,F]; y [T,d].
 *     x, W_r, W1, W3, W2 have the plan's act_dtype; y has its out_dtype.
 *   - Device pointers must be 16-byte aligned, the workspace 256-byte aligned;
 *     otherwise MOE_ERR_INVALID_ARG.
 *   - The caller owns all device memory, the workspace included.  The library owns only
 *     the host-side plan object; a plan holds no device memory and may be used from one
 *     thread at a time.
 *   - Every call that takes a stream (a cudaStream_t passed as void*, NULL = legacy default
 *     stream) only enqueues work on it: no allocation, no synchronisation, unless its
 *     comment says otherwise.  Workspace contents are defined once the stream reaches the
 *     point after the call.
 *   - Errors are returned as moe_status; nothing is thrown across the ABI.  A CUDA error
 *     from an enqueue maps to MOE_ERR_CUDA; moe_last_error() then describes it.
 *   - Device-side waits are bounded: a kernel that waits longer than the plan's
 *     wait_timeout_ns records MOE_ERR_TIMEOUT in the workspace's status word and returns;
 *     moe_get_device_status() reports it.  No kernel traps.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* bad pointer, size, alignment or config value */
  MOE_ERR_UNSUPPORTED = 2, /* valid config this build does not handle (e.g. bf16 with d % 64 != 0) */
  MOE_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed */
  MOE_ERR_TIMEOUT = 4,     /* a device-side wait ran out (reported by moe_get_device_status) */
  MOE_ERR_INTERNAL = 5     /* a device-side consistency check failed */
} moe_status;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;

/* Which kernels run the router and the expert GEMMs.
 *   MOE_PATH_AUTO:   bf16 -> tcgen05/TMEM/TMA kernels, expert GEMMs on CTA pairs (2-SM MMA);
 *                    fp32 -> fp32 SIMT kernels (true fp32).
 *   MOE_PATH_SIMT:   SIMT kernels for every dtype (fp32 FMA, a cross-check of the tensor path).
 *   MOE_PATH_TC_1SM: bf16 only: as AUTO but the expert GEMMs run one CTA per tile (1-SM MMA). */
typedef enum { MOE_PATH_AUTO = 0, MOE_PATH_SIMT = 1, MOE_PATH_TC_1SM = 2 } moe_path;

/* flags */
#define MOE_FLAG_KEEP_LOGITS 1u /* the router also stores its fp32 logits z [T,E] in the workspace */
#define MOE_FLAG_TEST_STALL 2u  /* test hook: the expert-GEMM producer withholds its first stage,
                                   so its consumers' bounded waits run out (MOE_ERR_TIMEOUT) */
#define MOE_FLAG_TRAINING 8u     /* the forward also keeps what moe_backward needs (the two
                                    pre-activations of every routed row and the router softmax);
                                    bf16 tensor-core plans with bf16 output */
#define MOE_FLAG_RENORM_GATES 4u /* variant: gates renormalised over the k chosen experts
                                    (gate[t,j] = p[t,idx[t,j]] / sum_j' p[t,idx[t,j']]) */

typedef struct {
  int64_t T;                /* tokens, >= 1 */
  int32_t d_model;          /* d, >= 1 */
  int32_t n_experts;        /* E, 1..256 */
  int32_t top_k;            /* k, 1..min(E, 16) */
  int32_t d_expert;         /* F, >= 1 */
  int32_t act_dtype;        /* moe_dtype of x, W_r, W1, W3, W2 */
  int32_t out_dtype;        /* moe_dtype of y */
  float router_temperature; /* tau > 0 */
  int32_t has_router_bias;  /* 0/1: moe_forward reads a bias [E] (fp32) */
  int32_t path;             /* moe_path */
  uint32_t flags;           /* MOE_FLAG_* */
  int64_t wait_timeout_ns;  /* bound on any device-side wait; <= 0 selects 2 s */
} moe_config;

typedef struct moe_plan_s* moe_plan_t;

/* Device pointers into a workspace, for inspecting the intermediates of the last forward
 * run on it.  N = T*k routed rows; "row p" is the p-th row in expert-contiguous order. */
typedef struct {
  uint32_t* status;        /* status word: 0 or a moe_status recorded by a kernel */
  float* aux;              /* balancing scalar (fp32) */
  int32_t* topk_idx;       /* [T,k] chosen experts, descending logit */
  float* topk_gate;        /* [T,k] gates = softmax entries at topk_idx */
  int32_t* expert_counts;  /* [E] rows per expert */
  int32_t* expert_offsets; /* [E+1] exclusive scan of expert_counts */
  int32_t* perm_src;       /* [N] token of row p */
  int32_t* perm_slot;      /* [N] slot t*k+j of row p */
  float* gate_perm;        /* [N] gate of row p */
  int32_t* slot_pos;       /* [N] row p of slot t*k+j */
  float* logits;           /* [T,E] router logits, or NULL unless MOE_FLAG_KEEP_LOGITS */
  void* xp;                /* [N,d] act dtype: x rows in dispatch order */
  void* h;                 /* [N,F] act dtype: SwiGLU hidden rows */
  void* yp;                /* [N,d] act dtype: row p = gate * expert output of row p (expert order) */
  float* expert_psum;      /* [E] sum over the layer's tokens of the softmax p[t,e] (the numerator of
                              the mean P_e of the balancing scalar) */
} moe_views;

/* Build a plan for one layer shape (host only; no device work).  Validates the config
 * (MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED), chooses kernels and tile shapes, and
 * returns in *workspace_bytes the size of the device workspace every forward needs. */
moe_status moe_plan(const moe_config* cfg, moe_plan_t* plan, size_t* workspace_bytes);

/* Release a plan (NULL is ignored). */
void moe_plan_destroy(moe_plan_t plan);

/* The whole forward on `stream`: router, top-k, histogram/scan, dispatch, grouped
 * SwiGLU GEMM, grouped down-projection with gate and un-permute, combine, and the
 * balancing scalar (left in the workspace).  router_bias may be NULL only when the plan
 * has has_router_bias = 0.  y is written completely.  Asynchronous. */
moe_status moe_forward(moe_plan_t plan, const void* x, const void* w_router, const float* router_bias,
                       const void* w1, const void* w3, const void* w2, void* y, void* workspace,
                       size_t workspace_bytes, void* stream);

/* Number of kernel stages moe_forward enqueues, and their names: "route" (router, top-k,
 * per-block counts; its last CTA also runs the scan: per-expert counts, offsets, dispatch
 * bases, tile table, balancing scalar), "permute", "gemm1_swiglu", "gemm2_gate", "combine".
 * An expert-stage plan has none. */
int32_t moe_stage_count(moe_plan_t plan);
const char* moe_stage_name(moe_plan_t plan, int32_t stage);

/* Enqueue only stage `stage` (0 <= stage < moe_stage_count) of moe_forward, with the same
 * arguments.  Running stages 0..n-1 in order on one stream is exactly moe_forward; this
 * lets a caller place timing events between the kernels. */
moe_status moe_forward_stage(moe_plan_t plan, int32_t stage, const void* x, const void* w_router,
                             const float* router_bias, const void* w1, const void* w3, const void* w2,
                             void* y, void* workspace, size_t workspace_bytes, void* stream);

/* The forward with host activations: copies x_host -> x_dev, runs moe_forward(x_dev ... y_dev),
 * copies y_dev -> y_host, all on `stream` (cudaMemcpyAsync; pinned host buffers make the
 * copies asynchronous).  The weights stay device-resident.  The caller synchronises the
 * stream before reading y_host. */
moe_status moe_forward_host(moe_plan_t plan, const void* x_host, void* x_dev, const void* w_router,
                            const float* router_bias, const void* w1, const void* w3, const void* w2,
                            void* y_dev, void* y_host, void* workspace, size_t workspace_bytes,
                            void* stream);

/* Backward of the layer for the loss  L = sum_t dy[t] . y[t] + aux_weight * aux  (the page's
 * training setting, §3 Load-Balancing Loss: the balancing loss is added to the training loss
 * and reaches mainly the router).  Needs a plan made with MOE_FLAG_TRAINING and the workspace
 * of the last moe_forward of that plan on the same x and weights.  The routing (top-k
 * choice, counts) is piecewise constant and passes no gradient; the router receives it
 * through the gate values and through the softmax mean P_e.
 *   dy [T,d]: in the plan's out_dtype.
 *   outputs (fp32, device): dx [T,d]; dw_router [E,d]; dbias [E] (only if the plan has a
 *   bias, may be NULL otherwise); dw1, dw3 [E,F,d]; dw2 [E,d,F].  Every output is written
 *   completely (experts with no routed rows get zero weight gradients).
 * Asynchronous on `stream`; device-side waits are bounded as for moe_forward. */
moe_status moe_backward(moe_plan_t plan, const void* x, const void* w_router, const float* router_bias,
                        const void* w1, const void* w3, const void* w2, const void* dy, float aux_weight, float* dx,
                        float* dw_router, float* dbias, float* dw1, float* dw3, float* dw2, void* workspace,
                        size_t workspace_bytes, void* stream);

/* Number and names of the kernel stages moe_backward enqueues, and one stage alone (same
 * arguments; stages 0..n-1 in order on one stream are exactly moe_backward). */
int32_t moe_backward_stage_count(moe_plan_t plan);
const char* moe_backward_stage_name(moe_plan_t plan, int32_t stage);
moe_status moe_backward_stage(moe_plan_t plan, int32_t stage, const void* x, const void* w_router,
                              const float* router_bias, const void* w1, const void* w3, const void* w2, const void* dy,
                              float aux_weight, float* dx, float* dw_router, float* dbias, float* dw1, float* dw3,
                              float* dw2, void* workspace, size_t workspace_bytes, void* stream);

/* Copy the balancing scalar aux = E * sum_e f_e P_e of the last forward on `workspace`
 * to the device float *aux_out (stream-ordered, asynchronous).  (§3 Load-Balancing Loss) */
moe_status moe_aux_loss(moe_plan_t plan, const void* workspace, float* aux_out, void* stream);

/* Fill *views with pointers into `workspace` (host only, no device access). */
moe_status moe_workspace_views(moe_plan_t plan, void* workspace, moe_views* views);

/* SYNCHRONISES `stream`, then reads the workspace's status word: MOE_OK, or the error a
 * kernel of the last forward recorded (MOE_ERR_TIMEOUT, MOE_ERR_INTERNAL), or MOE_ERR_CUDA
 * if the synchronisation itself failed.  Each moe_forward clears the word first. */
moe_status moe_get_device_status(moe_plan_t plan, const void* workspace, void* stream);

/* ---------------------------------------------------------------------------------------
 * Expert parallelism (§4 Expert Parallelism: experts spread over GPUs; Dispatch sends every
 * routed row to the GPU that holds its expert, Combine sends the outputs back).
 *
 * W ranks; rank r holds its own tokens, the whole router, and the weights of E_l = E / W
 * experts, r*E_l .. (r+1)*E_l - 1.  A step on rank r, with the exchanges done by the caller's
 * collectives (the library moves no data between GPUs):
 *   1. moe_forward_stage "route" and "permute" with a moe_plan over all E experts: the rank's
 *      rows Xp in expert order -- which is destination-rank order -- with expert_counts and
 *      gate_perm (moe_workspace_views);
 *   2. all-to-all of expert_counts viewed [W, E_l]: rank r receives seg_counts [W, E_l];
 *   3. all-to-all of the rows of Xp and of gate_perm, rank-major as they lie: the received
 *      rows form W*E_l segments, source-major (segment s: the rows source s/E_l sent to local
 *      expert s%E_l);
 *   4. moe_expert_forward over the received rows, in place: gate * E_e(row) in the same order;
 *   5. the reverse all-to-all of those rows into the rank's Yp (moe_workspace_views);
 *   6. moe_forward_stage "combine";
 *   7. optionally the balancing scalar over all ranks: all-reduce of expert_counts and
 *      expert_psum, then moe_aux_from_totals with the total token count.
 * ------------------------------------------------------------------------------------- */

typedef struct {
  int64_t max_rows;        /* R: capacity of the received-row buffers, >= 1 (dropless: at most
                              W * T_local * min(k, E_l) rows can arrive) */
  int32_t d_model;         /* d */
  int32_t n_local_experts; /* E_l: the experts whose weights this rank holds, >= 1 */
  int32_t n_sources;       /* W: ranks the rows come from; W * E_l <= 256 */
  int32_t d_expert;        /* F */
  int32_t act_dtype;       /* moe_dtype of the rows, the weights and the output rows */
  int32_t path;            /* moe_path */
  int64_t wait_timeout_ns; /* bound on any device-side wait; <= 0 selects 2 s */
} moe_expert_config;

/* Plan of the expert stage (host only).  Validates as moe_plan does and returns the workspace
 * size (status header, per-segment table, tile descriptors, the hidden rows H [R, F]). */
moe_status moe_expert_plan(const moe_expert_config* cfg, moe_plan_t* plan, size_t* workspace_bytes);

/* The local experts on received rows:  y_rows[p] = gates[p] * E_e(x_rows[p]),
 *   E_e(v) = W2_e (SiLU(W1_e v) * (W3_e v)),  e = the local expert of p's segment.
 *   seg_counts [W*E_l] int32 (device): rows per segment, source-major; the rows of segment s
 *     are x_rows[off_s .. off_s + seg_counts[s]), off_s the sum of the earlier counts.  A
 *     negative count or a sum above max_rows is recorded as MOE_ERR_INTERNAL
 *     (moe_get_device_status) and no row is computed.
 *   x_rows [R,d], gates [R] fp32, y_rows [R,d]: device buffers of max_rows rows; rows past the
 *     sum of the counts are not written.  w1, w3 [E_l,F,d], w2 [E_l,d,F]: the local experts.
 * Asynchronous on `stream`; device-side waits are bounded as for moe_forward. */
moe_status moe_expert_forward(moe_plan_t plan, const int32_t* seg_counts, const void* x_rows, const float* gates,
                              const void* w1, const void* w3, const void* w2, void* y_rows, void* workspace,
                              size_t workspace_bytes, void* stream);

/* The balancing scalar from per-expert totals (§3 Load-Balancing Loss):
 *   aux = E * sum_e (counts[e] / (n_tokens k)) * (psum[e] / n_tokens)
 * counts [E] int32 and psum [E] fp32 on the device (e.g. expert_counts and expert_psum summed
 * over ranks), aux_out one fp32 on the device.  Asynchronous on `stream`. */
moe_status moe_aux_from_totals(int32_t n_experts, int32_t top_k, int64_t n_tokens, const int32_t* counts,
                               const float* psum, float* aux_out, void* stream);

/* Size in bytes of the static device buffer moe_route_noalloc() works in. */
#define MOE_NOALLOC_SCRATCH_BYTES (4u << 20)

/* Routing for callers that cannot allocate device memory.  The paper has no counterpart:
 * this is a service of this library.  Some callers cannot call cudaMalloc at all (their
 * memory budget is fixed in advance, or another runtime owns every device allocation, or
 * the step must not risk an allocation failure part-way), so they cannot provide the
 * workspace moe_forward needs.  This call runs only the router part of the forward --
 * logits, softmax, top-k, gates, per-expert counts and the balancing scalar -- and keeps
 * all of its scratch in one static device array of MOE_NOALLOC_SCRATCH_BYTES that the
 * library holds on every GPU that loads it until the process exits.  Neither the caller
 * nor the library allocates anything; the caller passes only inputs and outputs.
 *   plan: any plan; only its routing is used (flags that make moe_forward keep more, such
 *     as MOE_FLAG_KEEP_LOGITS or MOE_FLAG_TRAINING, do not apply here).
 *   x, w_router, router_bias: as for moe_forward (router_bias may be NULL only when the
 *     plan has no bias).
 *   topk_idx [T,k] int32, topk_gate [T,k] fp32, expert_counts [E] int32, aux (one fp32):
 *     device outputs, the same values moe_forward leaves in its workspace for this plan,
 *     up to the rounding differences between its router kernels (the logits here are fp32
 *     FMA sums).
 *   device_status (one uint32, device): written when the work completes: 0, or the
 *     moe_status a kernel recorded (MOE_ERR_INTERNAL when a logit is NaN; the other
 *     outputs are then unspecified).  Read it after synchronising the stream.
 * Every pointer must be 16-byte aligned (MOE_ERR_INVALID_ARG otherwise); all arguments are
 * checked before any CUDA call.  Returns MOE_ERR_UNSUPPORTED, with the sizes in
 * moe_last_error(), when the plan needs more scratch than MOE_NOALLOC_SCRATCH_BYTES
 * (512 + 4*T*k + 8*ceil(T/128)*E bytes, each part rounded up to 256).  The first call on
 * each device looks up the array's device address with that device current; make that
 * first call before any stream capture.  All calls share the one array and leave their
 * contents in it (each call clears the status words and the completion ticket it starts
 * from): calls whose work overlaps on the GPU (other streams, other host threads) race and
 * must be serialised by the caller.  Asynchronous on `stream`. */
moe_status moe_route_noalloc(moe_plan_t plan, const void* x, const void* w_router, const float* router_bias,
                             int32_t* topk_idx, float* topk_gate, int32_t* expert_counts, float* aux,
                             uint32_t* device_status, void* stream);

/* Text of a status code, and a description of the last error on this thread. */
const char* moe_status_string(moe_status s);
const char* moe_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H */

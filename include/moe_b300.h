/*
 * moe_b300.h -- C ABI of the DeepSeekMoE layer (forward, and its backward) for one
 * B300 GPU (sm_103a).
 *
 * The layer (DeepSeekMoE, Chinese translation on gitcode.csdn.net, section 3.2,
 * eqs (9)-(11)):
 *
 *   s_t   = Softmax(u_t . W_g)                       over the N_r routed experts
 *   g_t   = s_t on Topk(s_t, k), 0 elsewhere           (optionally renormalised)
 *   y_t   = sum_{i<K_s} FFN_i(u_t) + sum_{i routed} g_{i,t} FFN_i(u_t)
 *   FFN_i(u) = W2_i (silu(W1_i u) * (W3_i u))          (SwiGLU expert)
 *
 * y_t excludes the residual +u_t of eq (9); the caller adds it. Two gate
 * variants are supported: the noisy top-k gate of "Outrageously Large Neural
 * Networks" ("Mixture of Experts" notes on blog.carolineworld.cn, section 2,
 * Noisy Top-K Gating) and the auxiliary-loss-free per-expert selection bias
 * ("DeepSeek MoE" article on cloud.tencent.com, load-balancing section).
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     never allocates, frees or keeps them after the call returns.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream). No entry point synchronises the stream except
 *     moe_device_status().
 *   - Layouts are row-major and dense. Expert weights are stacked shared
 *     experts first, then routed (eq (9)'s numbering): routed expert r is
 *     expert K_s + r. W1, W3: [K_s+N_r, I, d]; W2: [K_s+N_r, d, I].
 *   - act_dtype selects the element type of x, x_perm, expert weights and y:
 *     MOE_DT_BF16 (bf16, tensor-core path) or MOE_DT_F32 (fp32 CUDA-core path).
 *     Router weights, noise, bias, gates and logits are always fp32; index
 *     arrays are int32.
 *   - Errors are returned as moe_status; nothing is thrown across the ABI.
 *     Invalid arguments are rejected on the host before anything is enqueued.
 *     Faults found on the device (an expert id out of range, a pipeline wait
 *     that exceeded its time limit) set a sticky per-device flag that
 *     moe_device_status() reports; the kernels skip the offending access.
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,    /* null pointer, bad size, misaligned pointer      */
  MOE_ERR_UNSUPPORTED = 2,    /* valid but outside what the kernels implement    */
  MOE_ERR_WORKSPACE = 3,      /* workspace smaller than the *_workspace_size()   */
  MOE_ERR_CUDA = 4,           /* a CUDA runtime/driver call failed               */
  MOE_ERR_DEVICE_TIMEOUT = 5, /* a kernel's bounded wait expired (pipeline fault)*/
  MOE_ERR_DEVICE_INDEX = 6,   /* a kernel met an out-of-range expert id          */
  MOE_ERR_STATIC_LIMIT = 7    /* too large for moe_permute_static's fixed scratch */
} moe_status;

typedef enum { MOE_DT_F32 = 0, MOE_DT_BF16 = 1 } moe_dtype;

typedef enum {
  MOE_GATE_SOFTMAX = 0,       /* s = Softmax(x W_g); key s (+ bias); gate s      */
  MOE_GATE_NOISY = 1          /* H = x W_g + eps * softplus(x W_noise); key H;
                                 gate = softmax of H over the kept top-k          */
} moe_gate;

/* Shape and mode of one MoE layer. Fixed-width fields only (stable ABI). */
typedef struct {
  int64_t T;           /* tokens (rows of x), >= 0                               */
  int32_t d;           /* model width, multiple of 8                             */
  int32_t n_routed;    /* N_r routed experts, 1..256 (2*N_r <= 256 when noisy)   */
  int32_t n_shared;    /* K_s shared experts, always active, 0..64               */
  int32_t top_k;       /* k routed experts per token, 1..min(N_r, 32)            */
  int32_t d_ff;        /* I, intermediate width of every expert, multiple of 8   */
  int32_t renormalize; /* 1: gates divided by their sum over the selected set    */
  int32_t gate;        /* moe_gate                                               */
  int32_t act_dtype;   /* moe_dtype                                              */
  int32_t capacity;    /* max assignments an expert accepts, 0 = no limit        */
  int32_t expert_act;  /* moe_expert_act                                         */
  int32_t combine;     /* moe_combine_mode (bf16 layers; fp32 layers scatter-add) */
} moe_config;

typedef enum {
  MOE_ACT_SWIGLU = 0,  /* FFN(u) = W2 (silu(W1 u) * (W3 u))                       */
  MOE_ACT_RELU = 1     /* FFN(u) = W2 ReLU(W1 u) (GShard's wo.ReLU(wi.x)); W3 unused */
} moe_expert_act;

/*
 * How moe_forward forms y_t = sum_shared FFN_i(u_t) + sum_j g_{t,j} FFN_j(u_t)
 * (DeepSeekMoE translation on gitcode.csdn.net, section 3.2, eq (9)) in bf16
 * layers. Both sum in fp32 and round y once to bf16; they differ in where the
 * expert rows meet:
 *   MOE_COMBINE_ROWS: the down GEMM stores every expert row FFN_e(u_t) as bf16
 *     (the K_s shared experts summed into one row per token), and a combine
 *     kernel adds each token's rows with their gates in a fixed order.
 *     Deterministic; each row is rounded to bf16 before the sum.
 *   MOE_COMBINE_SCATTER_ADD: the down GEMM's epilogue adds g * FFN_e(u_t) into
 *     an fp32 accumulator with fp32 atomics (shared experts at gate 1), cast to
 *     y at the end. The rows stay fp32; the atomics' order varies run to run.
 * fp32 layers always add straight into y (the scatter-add form).
 */
typedef enum {
  MOE_COMBINE_ROWS = 0,
  MOE_COMBINE_SCATTER_ADD = 1
} moe_combine_mode;

/*
 * Expert capacity ("Mixture of Experts" notes, section 3, GShard expert
 * capacity; section 4, Switch capacity factor): when capacity > 0, expert e
 * accepts the first `capacity` assignments that select it, in ascending flat
 * assignment index t*k + j (a running counter c_e per expert); later ones are
 * dropped: they take no row, their dest is -1, and they add nothing to y (the
 * token's other experts, the shared experts and the caller's residual still
 * do). The gate values in topk_w are not changed. A Switch-style capacity
 * factor f gives capacity = ceil(f * T * k / N_r), computed by the caller.
 * The DeepSeekMoE layer itself is dropless (capacity = 0).
 */

/* Optional per-call router statistics (moe_route); NULL members are skipped.
 * Balance losses are formed from them by the caller:
 *   z-loss ("Mixture of Experts" notes, section 5, ST-MoE) = mean_t lse[t]^2;
 *   P_i (DeepSeekMoE translation, section 3.3, eq (14)) = prob_sum[i] / T;
 *   Importance_i ("Mixture of Experts" notes, section 2) = gate_sum[i];
 *   f_i (eq (13)) from the per-expert counts of moe_permute. */
typedef struct {
  float* lse;          /* [T]   log sum_i exp(x W_g)_i over the routed experts      */
  float* prob_sum;     /* [N_r] sum over tokens of the softmax probabilities s_i   */
  float* gate_sum;     /* [N_r] sum over tokens of the gate values g_i (0 if not selected) */
} moe_router_stats;

/* Human-readable name of a status code (static string). */
const char* moe_status_string(int status);

/* Library ABI version: (major << 16) | minor. */
int moe_version(void);

/* Bytes of scratch moe_route needs (0 only for T = 0): the router's fp32
 * logits rows, which a second kernel turns into softmax, keys, top-k and
 * gates. Tensor-core router (bf16 tokens, <= 128 router columns, T >= 4096):
 * the three bf16 planes of the router weights, then one logits row per token.
 * CUDA-core router: for T <= 512 the partial logits tiles of the split of the
 * reduction over d among more SMs, else one logits row per token. Everything
 * is written before it is read: the scratch needs no initialisation. */
size_t moe_route_workspace_size(const moe_config* cfg);

/*
 * moe_route -- the gate: router GEMM, softmax, top-k and gate values.
 * DeepSeekMoE translation, section 3.2, eqs (10)-(11); noisy variant per the
 * Noisy Top-K Gating passage of the "Mixture of Experts" notes, section 2;
 * bias per the cloud.tencent.com article's auxiliary-loss-free section.
 *
 *   x        [T, d]   act_dtype      token activations u_t
 *   W_g      [d, N_r] fp32           expert centroids as columns
 *   W_noise  [d, N_r] fp32           noise projection; required iff gate = NOISY
 *   eps      [T, N_r] fp32           the StandardNormal() draws; iff gate = NOISY
 *   bias     [N_r]    fp32 or NULL   added to s for selection only (SOFTMAX gate)
 *   topk_ids [T, k]   int32  (out)   selected routed experts, descending key,
 *                                    ties to the lowest index
 *   topk_w   [T, k]   fp32   (out)   gate values g_{i,t} of those experts
 *   logits   [T, N_r] fp32 or NULL (out) the plain logits x W_g
 *   stats    moe_router_stats or NULL (out) per-token logsumexp and per-expert
 *                                    sums of s and g (summed with fp32 atomics)
 *   workspace, ws_bytes              scratch, >= moe_route_workspace_size()
 *                                    (may be NULL when that is 0)
 * The logits are an fp32-accurate dot product of the stored inputs. bf16
 * tokens with at most 128 router columns (N_r, or 2 N_r when noisy) and
 * T >= 4096 run on the tensor cores: W is split exactly into three bf16
 * planes, every product is exact, and the accumulation is fp32. Otherwise a
 * CUDA-core fp32 FMA kernel runs. Softmax, keys and gates are fp32.
 */
moe_status moe_route(const moe_config* cfg, const void* x, const float* W_g,
                     const float* W_noise, const float* eps, const float* bias,
                     int32_t* topk_ids, float* topk_w, float* logits,
                     const moe_router_stats* stats,
                     void* workspace, size_t ws_bytes, void* stream);

/* Bytes of scratch moe_permute needs (per-block histograms and ranks). */
size_t moe_permute_workspace_size(const moe_config* cfg);

/*
 * moe_permute -- token dispatch: group the T*k assignments by expert.
 * The pages say each token goes to its selected experts (DeepSeekMoE
 * translation, section 2) and that the gate keeps a running per-expert
 * counter c_e ("Mixture of Experts" notes, section 3, GShard expert capacity).
 * Rows of expert e occupy [offsets[e], offsets[e+1]) in ascending flat
 * assignment index a = t*k + j (stable by token).
 *
 *   x         [T, d]       act_dtype   activations
 *   topk_ids  [T, k]       int32       routed expert of each assignment
 *   workspace, ws_bytes                scratch, >= moe_permute_workspace_size()
 *   counts    [N_r]        int32 (out) assignments per expert (c_e)
 *   offsets   [N_r + 1]    int32 (out) exclusive prefix sum of counts
 *   dest      [T, k]       int32 (out) grouped row of each assignment
 *   perm_src  [T*k]        int32 (out) flat assignment index of each grouped row
 *   x_perm    [T*k, d]     act_dtype (out) x_perm[dest[t,j]] = x[t]
 * Ids outside [0, N_r) are skipped and raise MOE_ERR_DEVICE_INDEX. With
 * cfg->capacity > 0, counts are the accepted counts and dropped assignments
 * get dest = -1 and no row.
 */
moe_status moe_permute(const moe_config* cfg, const void* x, const int32_t* topk_ids,
                       void* workspace, size_t ws_bytes, int32_t* counts, int32_t* offsets,
                       int32_t* dest, int32_t* perm_src, void* x_perm, void* stream);

/* Largest T*k that moe_permute_static accepts (its fixed scratch holds this many). */
#define MOE_PERMUTE_STATIC_MAX_ASSIGN (1 << 19)

/*
 * moe_permute_static -- moe_permute without a caller workspace. The paper has
 * no counterpart: this entry point exists for callers that cannot allocate
 * device memory for scratch, such as code running under a host framework that
 * owns the whole device-memory budget and forbids allocation after start-up,
 * or a serving loop that must never enter an allocator (cudaMalloc/cudaFree
 * can synchronise the device).
 *
 * The scratch (per-block histograms and ranks) is a file-scope device array
 * of 2.5 MiB in the library, sized for T*k <= MOE_PERMUTE_STATIC_MAX_ASSIGN
 * (524,288 assignments) and N_r <= 256. Every GPU that loads the library holds
 * that array until the process exits. Larger problems are rejected with
 * MOE_ERR_STATIC_LIMIT before anything is enqueued. The call allocates
 * nothing: no cudaMalloc, no cudaFree, no allocating library routine.
 *
 * Set-up: the first call on a device, with that device current, looks up the
 * array's device address (cudaGetSymbolAddress) and caches it; make that first
 * call before any stream capture on that device.
 *
 * Sharing: all calls on a device use the same array and it keeps the last
 * call's contents (the kernels overwrite every entry they read, so nothing has
 * to start at zero). Calls that overlap on the GPU (different streams, or
 * different host threads without ordering) race on the array; order them on
 * one stream. Arguments, outputs and errors are those of moe_permute.
 */
moe_status moe_permute_static(const moe_config* cfg, const void* x, const int32_t* topk_ids,
                              int32_t* counts, int32_t* offsets, int32_t* dest,
                              int32_t* perm_src, void* x_perm, void* stream);

/* Bytes of scratch moe_expert_ffn needs (group plan and the SwiGLU activations). */
size_t moe_expert_ffn_workspace_size(const moe_config* cfg);

/*
 * moe_expert_ffn -- every active expert FFN on its rows, unweighted.
 * Expert FFN: W2 (silu(W1 x) * (W3 x)); each expert is a standard FFN
 * (DeepSeekMoE translation, section 2), evaluated only on the tokens routed
 * to it (sparse evaluation, "Mixture of Experts" notes, section 2).
 *
 *   x         [T, d]        act_dtype  activations (the rows of shared experts)
 *   x_perm    [T*k, d]      act_dtype  grouped rows from moe_permute
 *   offsets   [N_r + 1]     int32      group bounds from moe_permute
 *   W1, W3    [K_s+N_r, I, d] act_dtype; W2 [K_s+N_r, d, I] act_dtype
 *             (W3 may be NULL when cfg->expert_act = MOE_ACT_RELU)
 *   workspace, ws_bytes                scratch, >= moe_expert_ffn_workspace_size()
 *   out_rows  [K_s*T + T*k, d] fp32 (out): row i*T + t = FFN_i(x_t) for shared
 *             expert i; row K_s*T + r = FFN_{K_s+e}(x_perm[r]) for r in group e.
 * bf16: tcgen05 tensor-core GEMMs, fp32 accumulation, SwiGLU activations
 * rounded to bf16 between the two GEMMs. fp32: CUDA-core FMA throughout.
 */
moe_status moe_expert_ffn(const moe_config* cfg, const void* x, const void* x_perm,
                          const int32_t* offsets, const void* W1, const void* W3,
                          const void* W2, void* workspace, size_t ws_bytes,
                          float* out_rows, void* stream);

/*
 * moe_combine -- gate-weighted combine back to token order (eq (9) without
 * the residual; "Mixture of Experts" notes, section 3, y_s = sum_e G_{s,e} FFN_e(x_s)):
 *   y_t = sum_{i<K_s} out_rows[i*T + t] + sum_j topk_w[t,j] out_rows[K_s*T + dest[t,j]]
 *   (terms with dest[t,j] = -1, dropped by an expert's capacity, are skipped)
 *   out_rows [K_s*T + T*k, d] fp32; dest [T, k] int32; topk_w [T, k] fp32;
 *   y [T, d] act_dtype (out). Summed in fp32 in a fixed order (deterministic).
 */
moe_status moe_combine(const moe_config* cfg, const float* out_rows, const int32_t* dest,
                       const float* topk_w, void* y, void* stream);

/* Bytes of scratch moe_forward needs. */
size_t moe_workspace_size(const moe_config* cfg);

/*
 * moe_forward -- the whole layer: route, dispatch, grouped SwiGLU experts and
 * the gate-weighted combine (DeepSeekMoE translation on gitcode.csdn.net,
 * section 3.2, eq (9)), fused as: router -> histogram/scan/plan -> gather ->
 * gate-up GEMM with SiLU*up fused -> down GEMM -> combine, the last two as
 * cfg->combine selects (moe_combine_mode). Arguments as in moe_route /
 * moe_expert_ffn.
 *   y            [T, d]  act_dtype (out)
 *   topk_ids_out [T, k]  int32 or NULL (out) routing decisions
 *   topk_w_out   [T, k]  fp32  or NULL (out) gate values
 *   counts_out   [N_r]   int32 or NULL (out) tokens per routed expert
 * MOE_COMBINE_ROWS gives the same y on every run; with the scatter-add (and
 * in fp32 layers) the atomics' summation order of a token's k + K_s
 * contributions (not the result's tolerance) varies run to run.
 */
moe_status moe_forward(const moe_config* cfg, const void* x, const float* W_g,
                       const float* W_noise, const float* eps, const float* bias,
                       const void* W1, const void* W3, const void* W2,
                       void* workspace, size_t ws_bytes, void* y,
                       int32_t* topk_ids_out, float* topk_w_out, int32_t* counts_out,
                       void* stream);

/* Number of events moe_forward_profiled records per call. */
#define MOE_PROFILE_EVENTS 6

/*
 * moe_forward_profiled -- moe_forward, plus cudaEventRecord of caller-created
 * events on `stream` at the stage boundaries, so a caller can time each
 * kernel of the layer on the stream it runs on. stage_events holds
 * MOE_PROFILE_EVENTS cudaEvent_t handles (or is NULL, which makes the call
 * identical to moe_forward): [0] before the router, [1] after the router,
 * [2] after dispatch (count, scan+plan, gather), [3] after the gate-up GEMM,
 * [4] after the down GEMM, [5] after the combine kernel or the cast to y
 * (bf16 layers; for fp32 layers the down GEMM's scatter-add already formed y).
 */
moe_status moe_forward_profiled(const moe_config* cfg, const void* x, const float* W_g,
                                const float* W_noise, const float* eps, const float* bias,
                                const void* W1, const void* W3, const void* W2,
                                void* workspace, size_t ws_bytes, void* y,
                                int32_t* topk_ids_out, float* topk_w_out, int32_t* counts_out,
                                void* stream, void* const* stage_events);

/* Bytes of scratch moe_backward needs. */
size_t moe_backward_workspace_size(const moe_config* cfg);

/*
 * moe_backward -- gradients of the layer for an upstream gradient dy = dL/dy:
 * dL/dx, dL/dW_g, dL/dW_noise, dL/dW1, dL/dW3, dL/dW2.
 * The pages define the forward only (DeepSeekMoE translation on
 * gitcode.csdn.net, section 3.2, eqs (9)-(11); the noisy gate of the
 * "Mixture of Experts" notes, section 2; GShard's ReLU expert and the expert
 * capacity, sections 3-4). This is the derivative of that forward with the
 * top-k selection, and an expert capacity's keep/drop decisions, held fixed
 * (both are piecewise constant in the inputs): gradients flow through the
 * selected gates and the kept experts only; a dropped assignment and the
 * selection bias receive none.
 *   gate:  dg_{t,j} = <dy_t, FFN_e(u_t)>; renormalised gates pass
 *          (dg_j - <dg, g>) / sum_sel s to the scores; the softmax of eq (11)
 *          gives dlogit = s (ds - <ds, s>); the noisy gate gives dH = g (dg -
 *          <dg, g>) on the kept entries, dlogit = dH, dnoise = dH eps
 *          sigmoid(x W_noise); dW_g = x^T dlogit, dx += dlogit W_g^T.
 *   expert (rows X, gate g, a = X W1^T, b = X W3^T, h = silu(a) b):
 *          dh = dy W2; da = g dh b silu'(a); db = g dh silu(a);
 *          dX = da W1 + db W3; dW1 = da^T X; dW3 = db^T X; dW2 = (g dy)^T h.
 *
 * Arguments are those of moe_forward (the same layer and inputs) plus
 *   dy        [T, d]          act_dtype   upstream gradient of y
 *   workspace, ws_bytes                   scratch, >= moe_backward_workspace_size()
 *   dx        [T, d]          act_dtype (out)
 *   dW_g      [d, N_r]        fp32 (out)
 *   dW_noise  [d, N_r]        fp32 (out), required iff gate = NOISY (else ignored)
 *   dW1, dW3  [K_s+N_r, I, d] fp32 (out) (dW3 may be NULL for ReLU experts)
 *   dW2       [K_s+N_r, d, I] fp32 (out)
 * Every output is overwritten (not accumulated into). The call is
 * self-contained: it recomputes the forward's routing, dispatch and SwiGLU
 * pre-activations from x (the workspace need not hold a forward's state).
 * bf16 layers run the expert GEMMs on the tensor cores (bf16 operands: the
 * saved a, b, g h and the gradient rows da, db, dX are rounded to bf16; fp32
 * accumulation); fp32 layers run fp32 FMA throughout. The router-weight
 * gradients are fp32 sums over token chunks combined with fp32 atomics, so
 * their last bits can vary run to run.
 */
moe_status moe_backward(const moe_config* cfg, const void* x, const float* W_g,
                        const float* W_noise, const float* eps, const float* bias,
                        const void* W1, const void* W3, const void* W2, const void* dy,
                        void* workspace, size_t ws_bytes, void* dx, float* dW_g,
                        float* dW_noise, float* dW1, float* dW3, float* dW2, void* stream);

/* Number of events moe_backward_profiled records per call. */
#define MOE_BWD_PROFILE_EVENTS 8

/*
 * moe_backward_profiled -- moe_backward, plus cudaEventRecord of caller-created
 * events on `stream` at its stage boundaries (stage_events holds
 * MOE_BWD_PROFILE_EVENTS cudaEvent_t handles, or is NULL: then the call is
 * moe_backward): [0] start, [1] after the recomputed routing, dispatch and the
 * gather of dy, [2] after the recomputed a, b, g h, [3] after dh and da, db,
 * [4] after the router's softmax backward, [5] after the dX rows, [6] after the
 * router-weight gradient, the router's dx term and the per-token sum, [7] after
 * the expert weight gradients. With T = 0 no event is recorded.
 */
moe_status moe_backward_profiled(const moe_config* cfg, const void* x, const float* W_g,
                                 const float* W_noise, const float* eps, const float* bias,
                                 const void* W1, const void* W3, const void* W2, const void* dy,
                                 void* workspace, size_t ws_bytes, void* dx, float* dW_g,
                                 float* dW_noise, float* dW1, float* dW3, float* dW2, void* stream,
                                 void* const* stage_events);

/*
 * moe_forward_train -- the forward of a training step: moe_forward's y (the
 * layer of the DeepSeekMoE translation, section 3.2, eqs (9)-(11)), plus the
 * state the backward needs, left in `workspace` (>=
 * moe_backward_workspace_size()): the routing, the logits (and noise logits),
 * the dispatch and group plan, x_perm, and the expert pre-activations a, b and
 * g * h. y is formed from g * h through W2 and the per-token sum of the rows
 * (the gates ride on g * h), so it is the sum of moe_forward; bf16 layers use
 * the row combine whatever cfg->combine says, fp32 layers the scatter-add.
 * Arguments as in moe_forward. Errors: MOE_ERR_INVALID_ARG for a missing or
 * misaligned pointer, MOE_ERR_WORKSPACE for ws_bytes below
 * moe_backward_workspace_size(); T = 0 does nothing.
 */
moe_status moe_forward_train(const moe_config* cfg, const void* x, const float* W_g,
                             const float* W_noise, const float* eps, const float* bias,
                             const void* W1, const void* W3, const void* W2,
                             void* workspace, size_t ws_bytes, void* y, void* stream);

/*
 * moe_backward_from_forward -- moe_backward (the gradients of the layer of the
 * DeepSeekMoE translation, section 3.2, with the top-k selection held fixed;
 * same arguments, results, precision and errors) on a workspace that
 * moe_forward_train filled for the same cfg,
 * x, router weights, noise, bias and expert weights, with nothing in between
 * that wrote to it: the routing, the dispatch and the recompute of a, b and
 * g * h are skipped. It consumes the state (da and db overwrite the saved a
 * and b in place): call it once per moe_forward_train. stage_events: as in
 * moe_backward_profiled, or NULL.
 */
moe_status moe_backward_from_forward(const moe_config* cfg, const void* x, const float* W_g,
                                     const float* W_noise, const float* eps, const float* bias,
                                     const void* W1, const void* W3, const void* W2, const void* dy,
                                     void* workspace, size_t ws_bytes, void* dx, float* dW_g,
                                     float* dW_noise, float* dW1, float* dW3, float* dW2, void* stream,
                                     void* const* stage_events);

/*
 * moe_device_status -- synchronise `stream`, then read and clear the sticky
 * device fault flag of the current device. Returns MOE_OK,
 * MOE_ERR_DEVICE_TIMEOUT, MOE_ERR_DEVICE_INDEX or MOE_ERR_CUDA. Writes the
 * raw flag word to *raw when raw is not NULL.
 */
moe_status moe_device_status(void* stream, int32_t* raw);

/*
 * moe_debug_wait_timeout -- test hook for the bounded-wait machinery: enqueue
 * one kernel that waits on an mbarrier nothing ever arrives on, with a limit
 * of `limit_us` microseconds (1..2000000). The wait runs out, the kernel sets
 * the MOE_ERR_DEVICE_TIMEOUT flag and returns; the context stays usable.
 */
moe_status moe_debug_wait_timeout(uint32_t limit_us, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_B300_H */

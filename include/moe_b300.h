/*
 * moe_b300.h — C ABI of the single-GPU MoE layer forward for NVIDIA B300 (sm_103a).
 *
 * One MoE layer forward, as the pages derive it:
 *   route:    g = x W_gate; softmax (or sigmoid + selection bias with group limit) scores;
 *             Top-k with renormalisation                 ["MoE 路由数学" §2.1; "Systems for
 *                                                         Mixture-of-Experts Models" §2.1, §5.3]
 *   dispatch: group (token, choice) pairs by expert, capacity C = ceil(cf*k*T/E), overflow
 *             dropped in token order                     ["Systems for MoE Models" §2.2, §2.4]
 *   experts:  SwiGLU FFN (SiLU(x W1) * x W3) W2 per expert, plus always-on shared experts
 *                                                        ["Systems for MoE Models" §5.2;
 *                                                         "MoE 路由数学" §2.2]
 *   combine:  out = shared(x) + sum_{i in S} p~_i Expert_i(x)   ["MoE 路由数学" §2.1]
 *   stats:    f_i, P_i, L_balance = E sum f_i P_i, z-loss  ["MoE 路由数学" §3.2; "Mixture of
 *             Experts 架构" load_balancing_loss / router_z_loss code blocks]
 *
 * Conventions (every entry point):
 *   - Returns 0 (MOE_OK) or a negative MOE_ERR_* status; moe_status_string() gives its text.
 *   - Every pointer argument is DEVICE memory owned by the caller unless stated otherwise.
 *     The library allocates and frees no memory and never synchronises the stream; all work
 *     is enqueued on `stream` (a cudaStream_t; NULL = the legacy default stream), except as
 *     moe_forward states for the shared experts.
 *   - Tensors are row-major and contiguous.  "bf16" tensors hold IEEE bfloat16; with
 *     cfg->dtype == MOE_DTYPE_F32 the same tensors hold float32 instead.
 *   - Arguments are validated on the host before any launch (MOE_ERR_ARG / SHAPE /
 *     UNSUPPORTED / WORKSPACE); a launch failure returns MOE_ERR_CUDA.  Faults found on the
 *     device (a bounded wait that ran out) are written to the status word at the start of the
 *     workspace and returned by moe_sync_status(); kernels never trap.
 *   - `ws` is a caller-allocated device workspace of at least moe_workspace_size() bytes,
 *     256-byte aligned.  Calls that share one workspace must not overlap on the GPU.
 *
 * Layouts:
 *   x       [T, d]        tokens
 *   w_gate  [E, d]        router, row e = expert e's vector (g[t,e] = sum_c x[t,c] w_gate[e,c])
 *   bias    [E] float32   selection-only bias (sigmoid scoring); may be NULL (= zeros)
 *   w13     [E, 2F, d]    rows [0,F) = W1 (gate projection), rows [F,2F) = W3 (up projection)
 *   w2      [E, d, F]     down projection (y[c] = sum_f h[f] w2[c,f])
 *   ws13    [2Fs, d], ws2 [d, Fs]   the shared experts concatenated into one SwiGLU expert of
 *                         width Fs = cfg->d_ff_shared (sum of shared experts == concatenation)
 *   topk_idx [T, k] int32 rank order (descending score; ties -> lower expert index)
 *   topk_w   [T, k] float32
 *   y_perm   [T*k, d] float32 expert outputs in expert order; shared_out [T, d] float32
 *   out      [T, d] in cfg->out_dtype
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  MOE_OK = 0,
  MOE_ERR_ARG = -1,          /* NULL pointer or bad enum value */
  MOE_ERR_SHAPE = -2,        /* sizes out of range or not aligned as required */
  MOE_ERR_UNSUPPORTED = -3,  /* a valid request this library does not implement */
  MOE_ERR_WORKSPACE = -4,    /* workspace NULL, too small or misaligned */
  MOE_ERR_CUDA = -5,         /* a CUDA runtime call failed */
  MOE_ERR_TIMEOUT = -6       /* a bounded device-side wait ran out */
};

enum { MOE_SCORE_SOFTMAX = 0, MOE_SCORE_SIGMOID = 1 };
enum { MOE_ROUTE_TOKEN_CHOICE = 0, MOE_ROUTE_EXPERT_CHOICE = 1 };
enum { MOE_DTYPE_BF16 = 0, MOE_DTYPE_F32 = 1 };

typedef struct moe_config {
  int32_t T;            /* tokens, >= 1 */
  int32_t d_model;      /* d; bf16 path: multiple of 128 */
  int32_t E;            /* routed experts, 1..256 */
  int32_t k;            /* experts per token, 1..min(E, 8); expert choice: C = T*k/E */
  int32_t d_ff;         /* F of one routed expert; bf16 path: multiple of 128 */
  int32_t d_ff_shared;  /* width of the concatenated shared experts, 0 = none */
  int32_t score;        /* MOE_SCORE_* */
  int32_t routing;      /* MOE_ROUTE_* */
  int32_t n_groups;     /* expert groups (sigmoid scoring); 1 = no group limit */
  int32_t topk_groups;  /* groups kept per token; == n_groups = no limit; a limit needs
                           >= 2 experts per group (group score = sum of its top two) */
  int32_t renormalize;  /* 1: w = p_S / sum_S p (default); 0: w = p_S (Switch, k = 1) */
  float route_scale;    /* weights are multiplied by it (1.0; DeepSeek-V3: 2.5) */
  float capacity_factor;/* C = ceil(cf*k*T/E); <= 0: no capacity limit */
  int32_t dtype;        /* MOE_DTYPE_*: x, weights, x_perm and h (bf16: tensor cores) */
  int32_t out_dtype;    /* MOE_DTYPE_*: layer output; F32 keeps the fp32 accumulation as is,
                           BF16 rounds it once (up to 2^-8 relative) */
} moe_config;

/* Text of a status code (static storage). */
const char* moe_status_string(int status);

/* Library version string, e.g. "moe_b300 1.0 sm_103a". */
const char* moe_version(void);

/* Validate cfg.  Returns MOE_OK or the first problem found. */
int moe_check_config(const moe_config* cfg);

/* Expert capacity C = ceil(cf*k*T/E) evaluated in double from the float cf
 * ["Systems for MoE Models" §2.4]; T*k when cf <= 0 (no limit).  Host only. */
int moe_capacity(const moe_config* cfg, int32_t* capacity);

/* Bytes of device workspace that the forward-path calls below need for cfg (host only).  The
 * router backward and the FP8 forward have their own queries
 * (moe_router_backward_workspace_size, moe_fp8_workspace_size). */
int moe_workspace_size(const moe_config* cfg, size_t* bytes);

/* Reads and clears the device status word at the start of `ws` (copies 4 bytes to the host
 * and synchronises `stream`).  Returns MOE_OK, or the first device-side error recorded since
 * the last call, or MOE_ERR_CUDA if the copy itself failed. */
int moe_sync_status(void* ws, void* stream);

/* Router: logits, scores, Top-k and weights for every token ["MoE 路由数学" §2.1 (g, p, S,
 * p~); "Mixture of Experts 架构" loss_free_balancing_routing code block; "Systems for MoE
 * Models" §5.3 (sigmoid gate with groups, bias for selection only, route scale)].
 *   x [T,d] bf16, w_gate [E,d] bf16, bias [E] f32 or NULL;
 *   logits [T,E] f32 output or NULL (then kept in the workspace);
 *   topk_idx [T,k] int32 and topk_w [T,k] f32 outputs.
 * Token choice only (cfg->routing == MOE_ROUTE_TOKEN_CHOICE). */
int moe_router_topk(const moe_config* cfg, const void* x, const void* w_gate, const float* bias,
                    float* logits, int32_t* topk_idx, float* topk_w, void* ws, void* stream);

/* Load-balance statistics from router logits and a selection ["MoE 路由数学" §3.2 (f_i, P_i,
 * L_balance = E sum f_i P_i); "Mixture of Experts 架构" load_balancing_loss and router_z_loss
 * code blocks].  f_i = (selections of expert i)/T before capacity drops (sum f = k);
 * P_i = mean_t softmax(g_t)_i (sigmoid scoring: mean_t s_ti / sum_j s_tj);
 * z = mean_t (logsumexp_i g_ti)^2.
 *   logits [T,E] f32, topk_idx [T,k] int32 -> f [E], P [E], l_balance [1], z_loss [1] (f32).
 * Reductions run in float32 in a fixed order (per token block, or per token when E > 32 and
 * T <= 64, then across blocks): results are bit-identical from run to run, and equal to the
 * statistics moe_forward returns for the same logits and selection. */
int moe_aux_stats(const moe_config* cfg, const float* logits, const int32_t* topk_idx, float* f,
                  float* P, float* l_balance, float* z_loss, void* ws, void* stream);

/* Dispatch: group (token, choice) pairs by expert in token order, apply the capacity and
 * gather token rows into expert order ["Systems for MoE Models" §2.2 steps 2-3, §2.4].
 *   counts[E]   selections per expert (before drops)
 *   kept[E]     min(counts, C)
 *   offsets[E+1] exclusive scan of kept (expert e's rows are [offsets[e], offsets[e+1]))
 *   pos[T,k]    number of earlier tokens that chose the same expert
 *   row_of[T,k] offsets[e] + pos when pos < C, else -1 (dropped)
 *   perm[T*k]   perm[row] = t*k + j for kept pairs, -1 for rows >= offsets[E]
 *   x_perm[T*k, d] bf16: x_perm[row] = x[t]; rows >= offsets[E] are left unwritten
 *   n_dropped[1] pairs dropped by the capacity
 * All outputs are bit-exact and deterministic.  x / x_perm may be NULL to skip the gather. */
int moe_dispatch(const moe_config* cfg, const int32_t* topk_idx, const void* x, int32_t* counts,
                 int32_t* kept, int32_t* offsets, int32_t* pos, int32_t* row_of, int32_t* perm,
                 void* x_perm, int32_t* n_dropped, void* ws, void* stream);

/* moe_dispatch for callers that cannot allocate device memory.  The pages have no
 * counterpart: this entry point exists for integration only.  Some callers may not call
 * cudaMalloc (inside another framework's memory pool, in a plugin host that hands over only
 * the tensors it owns, under a locked-down embedded allocator), so this variant takes no
 * workspace: its scratch is one fixed array inside the library, about 2.3 MB on every GPU that
 * loads it, held until the process exits.
 *   Same inputs and outputs as moe_dispatch, and bit-identical results, plus
 *   status [2] int32 (device): a call that passes its host-side checks clears it on the
 *   stream first, then the kernels write (code, detail) of the first device-side error
 *   (MOE_ERR_ARG for an out-of-range or repeated expert index).  A call refused on the host
 *   (its return value is not MOE_OK) enqueues nothing and leaves these words as they were.
 * Limits: T <= 65536 and E <= 256, else MOE_ERR_SHAPE before any launch.  All calls share the
 * one array and it keeps the last call's contents: calls that overlap on the GPU race, so
 * issue them one after another.  A call outside stream capture looks up the array's device
 * address (with the calling device current) and caches it; a call on a capturing stream uses
 * that cached address, so make one uncaptured call on the device before capturing
 * (MOE_ERR_UNSUPPORTED otherwise).  Allocates nothing. */
int moe_dispatch_noalloc(const moe_config* cfg, const int32_t* topk_idx, const void* x,
                         int32_t* counts, int32_t* kept, int32_t* offsets, int32_t* pos,
                         int32_t* row_of, int32_t* perm, void* x_perm, int32_t* n_dropped,
                         int32_t* status, void* stream);

/* Routed expert FFNs on expert-grouped rows ["Systems for MoE Models" §5.2 SwiGLU]:
 *   y_perm[r] = (SiLU(x_perm[r] W1_e^T) * (x_perm[r] W3_e^T)) W2_e^T for
 *   r in [offsets[e], offsets[e+1]).  x_perm [T*k, d] (activation type), y_perm [T*k, d]
 *   float32 (rows beyond offsets[E] untouched); offsets [E+1] device int32; w13, w2 as in the
 *   layout table.
 * bf16: tcgen05 tensor-core grouped GEMMs with fp32 accumulation; the intermediate h is
 * rounded to bf16 (it is the down GEMM's operand).  f32: CUDA-core fp32 path. */
int moe_expert_ffn(const moe_config* cfg, const void* x_perm, const int32_t* offsets,
                   const void* w13, const void* w2, float* y_perm, void* ws, void* stream);

/* Shared experts on every token ["MoE 路由数学" §2.2]: shared_out = SwiGLU(x; ws13, ws2),
 * x [T,d] -> shared_out [T,d] float32 (kept in fp32 so the combine rounds the layer output
 * only once).  cfg->d_ff_shared must be > 0. */
int moe_shared_ffn(const moe_config* cfg, const void* x, const void* ws13, const void* ws2,
                   float* shared_out, void* ws, void* stream);

/* Weighted combine ["MoE 路由数学" §2.1 Output; "Systems for MoE Models" §2.2 step 4]:
 *   out[t] = shared_out[t] + sum_{j : row_of[t,j] >= 0} topk_w[t,j] * y_perm[row_of[t,j]]
 * in fp32 in the order j = 0..k-1, written in cfg->out_dtype.  Dropped pairs add nothing and
 * the remaining weights are not renormalised.  y_perm float32; shared_out [T,d] float32 or
 * NULL.  No atomics. */
int moe_combine(const moe_config* cfg, const float* y_perm, const int32_t* row_of,
                const float* topk_w, const float* shared_out, void* out, void* stream);

/* Expert-choice routing ["MoE混合专家模型深度解析" §2.2 Expert Choice]: each expert takes the
 * C = T*k/E tokens with the largest logit in its column (ties -> lower token index).
 *   logits [T,E] f32 -> ec_tokens [E,C] int32 (ascending token order), ec_w [E,C] f32 =
 *   softmax(g_t)_e, tok_ptr [T+1] int32, tok_rows [E*C] int32: for token t the rows e*C+i of
 *   the experts that chose it, in ascending expert order (a CSR view used by the combine). */
int moe_expert_choice(const moe_config* cfg, const float* logits, int32_t* ec_tokens, float* ec_w,
                      int32_t* tok_ptr, int32_t* tok_rows, void* ws, void* stream);

/* Whole layer forward: router -> dispatch -> routed experts (+ shared experts) -> combine,
 * plus the statistics.  Every intermediate lives in `ws`.
 *   x [T,d], w_gate [E,d], bias [E] or NULL, w13, w2, ws13/ws2 (NULL when d_ff_shared == 0)
 *   out [T,d] in cfg->out_dtype (required)
 *   optional outputs (NULL to skip): topk_idx [T,k], topk_w [T,k], f [E], P [E],
 *   l_balance [1], z_loss [1], n_dropped [1] (token choice)
 * A bf16 prefill layer with shared experts runs their two GEMMs on a side stream of the
 * library's (one per device and host thread, with two events, created on the first such call
 * and never destroyed): forked from `stream` before the router and joined back into
 * it before the routed GEMMs, so the call still orders like one enqueue on `stream` and can be
 * captured into a CUDA graph.  Calls from one host thread on different streams share the side
 * stream, so their shared-expert GEMMs run in call order.  If they cannot be created, or the
 * first such call comes while `stream` is being captured, the shared experts run on `stream`
 * after the routed GEMMs (same kernels, same results).  The environment variable
 * MOE_B300_SHARED=serial always does so. */
int moe_forward(const moe_config* cfg, const void* x, const void* w_gate, const float* bias,
                const void* w13, const void* w2, const void* ws13, const void* ws2, void* out,
                int32_t* topk_idx, float* topk_w, float* f, float* P, float* l_balance,
                float* z_loss, int32_t* n_dropped, void* ws, void* stream);

/* moe_forward that also records two caller-created CUDA events (cudaEvent_t, timing enabled)
 * on `stream` around the expert GEMM launches on `stream`: the routed experts' grouped GEMMs,
 * followed by the shared experts' GEMMs when those run on `stream` (prefill without the side
 * stream), or the routed and shared experts' decode GEMMs.  With the side stream the shared
 * experts' GEMMs run beside the router, outside the events.  Same kernels and results as
 * moe_forward; for measuring the GEMM share of a forward.  Both events are required. */
int moe_forward_timed(const moe_config* cfg, const void* x, const void* w_gate, const float* bias,
                      const void* w13, const void* w2, const void* ws13, const void* ws2,
                      void* out, int32_t* topk_idx, float* topk_w, float* f, float* P,
                      float* l_balance, float* z_loss, int32_t* n_dropped, void* ws,
                      void* stream, void* ev_expert_begin, void* ev_expert_end);

/* Device addresses of the intermediates moe_forward leaves in `ws` (for inspection and
 * tests): logits [T,E] f32, row_of [T,k] int32, offsets [E+1] int32, x_perm, y_perm (f32 from
 * moe_expert_ffn; after a bf16 prefill moe_forward with a separate combine pass it holds the
 * rows in bf16). */
int moe_workspace_views(const moe_config* cfg, void* ws, float** logits, int32_t** row_of,
                        int32_t** offsets, void** x_perm, float** y_perm);

/* Device addresses of the expert-choice selection an expert-choice moe_forward leaves in `ws`
 * ["MoE混合专家模型深度解析" §2.2 Expert Choice]: ec_tokens [E,C] int32, ec_w [E,C] f32,
 * tok_ptr [T+1] int32, tok_rows [E*C] int32, laid out as moe_expert_choice writes them.
 * MOE_ERR_ARG for a token-choice configuration.  Any output pointer may be NULL. */
int moe_workspace_views_ec(const moe_config* cfg, void* ws, int32_t** ec_tokens, float** ec_w,
                           int32_t** tok_ptr, int32_t** tok_rows);

/* Failure-path self test: launches one tiny kernel whose bounded wait on a flag that nothing
 * sets runs out after about `limit_us` microseconds; it records MOE_ERR_TIMEOUT in the status
 * word of `ws` and returns, leaving the context usable.  Read the result with
 * moe_sync_status().  Exists so tests can exercise the timeout path without a fault. */
int moe_selftest_timeout(void* ws, int32_t limit_us, void* stream);

/* ---------------------------------------------------------------------------------------------
 * Router-side backward.
 *
 * Differentiates  L = alpha * L_balance + beta * z + sum_{t,j} d_topk_w[t,j] * topk_w[t,j]
 * with respect to the router logits, the gate weights and the input, holding the selection
 * and the frequencies f fixed:
 *   - L_balance = E * sum_i f_i P_i.  f_i is a count, so the gradient reaches the router only
 *     through P_i ("MoE 路由数学" §3.4; "Systems for Mixture-of-Experts Models" §3.2).
 *     P_i is the token mean of softmax(g) (softmax scoring) or of s_i / sum_j s_j with
 *     s = sigmoid(g) (sigmoid scoring).
 *   - z = mean over tokens of logsumexp(g_t)^2 (router_z_loss code block of "Mixture of
 *     Experts 架构"), in both scoring modes.
 *   - topk_w are the routing weights as moe_forward computes them (renormalised, times
 *     route_scale); the sigmoid route's bias only enters the selection and gets no gradient
 *     ("Systems for Mixture-of-Experts Models" §3.4).
 *
 * Arguments (device pointers, caller-owned, row-major):
 *   x         [T, d_model] bf16 or fp32 (cfg->dtype), the router input of the forward
 *   w_gate    [E, d_model] same type, the router weight
 *   logits    [T, E] fp32, the forward's logits (moe_router_topk, or moe_workspace_views)
 *   topk_idx  [T, k] int32, the forward's selection.  May be NULL when d_topk_w is NULL.
 *   d_topk_w  [T, k] fp32 upstream gradient of topk_w, or NULL (that term is absent)
 *   f         [E] fp32 frequencies as moe_forward / moe_aux_stats return them (count / T, or
 *             any other normalisation the caller's loss uses).  May be NULL when alpha == 0.
 *   alpha, beta  loss coefficients (finite)
 *   d_logits  [T, E] fp32 out: dL/dg, or NULL
 *   d_w_gate  [E, d_model] fp32 out: dL/dW_gate (required)
 *   d_x       [T, d_model] fp32 out: dL/dx through the router, or NULL
 *   ws        workspace of moe_router_backward_workspace_size bytes, 256-byte aligned.  Its
 *             first bytes hold the device status word that moe_sync_status reads.
 * Precision: dL/dg in fp32; with bf16 activations the two gradient GEMMs take dL/dg rounded
 * once to bf16 as their tensor-core operand (fp32 accumulate), so each product carries a
 * relative error <= 2^-8.  With fp32 activations they run in fp32.  Results are
 * deterministic (fixed summation order).
 * Errors: MOE_ERR_ARG for NULL required pointers, a NULL f with alpha != 0, non-finite
 * coefficients; MOE_ERR_UNSUPPORTED for expert-choice configurations; MOE_ERR_WORKSPACE for
 * a missing or misaligned workspace.  An expert index outside [0, E) in topk_idx is skipped
 * and recorded in the status word as MOE_ERR_ARG (detail = token). */
int moe_router_backward_workspace_size(const moe_config* cfg, size_t* bytes);
int moe_router_backward(const moe_config* cfg, const void* x, const void* w_gate,
                        const float* logits, const int32_t* topk_idx, const float* d_topk_w,
                        const float* f, float alpha, float beta, float* d_logits,
                        float* d_w_gate, float* d_x, void* ws, void* stream);

/* One step of the loss-free balancing bias rule ("Systems for Mixture-of-Experts Models"
 * §3.4; update_bias code block of "Mixture of Experts 架构"): for each expert i, with
 * load_i = f_i * T recovered exactly (f as moe_forward returns it, count / T rounded once to
 * fp32) and the mean load T*k/E,
 *   load_i > mean: bias[i] -= gamma;   load_i < mean: bias[i] += gamma;   equal: unchanged.
 * The load counts selections before capacity drops.  f [E] fp32 and bias [E] fp32 (in/out)
 * are device pointers.  Errors: MOE_ERR_ARG for NULL pointers or a non-finite gamma;
 * MOE_ERR_SHAPE when T*k >= 2^23 (the exact recovery of the load needs T*k < 2^23). */
int moe_bias_update(const moe_config* cfg, const float* f, float* bias, float gamma,
                    void* stream);

/* ---------------------------------------------------------------------------------------------
 * FP8 (E4M3) expert weights for decode.
 *
 * A decode step is bound by reading the touched experts' weights ("Systems for
 * Mixture-of-Experts Models" §1.4, which also notes that DeepSeek-V3 keeps its weights in FP8;
 * "MoE 推理优化深入" §4.2 on quantised experts).  One-byte E4M3 weights halve those bytes.  The
 * tensor cores multiply E4M3 by E4M3, so the activations entering each expert GEMM (the token's
 * x, then its h) are quantised per row the same way on the fly.
 *
 * Quantisation of one row v (float32 decisions):
 *   amax = max |v|;  inv = 448 / amax;  code = e4m3(v * inv);  scale = amax / 448
 * with round to nearest even and saturation at +-448 (the largest finite E4M3 value); a row of
 * zeros gets codes 0 and scale 0.  The row is represented by code * scale.
 *
 * moe_quantize_fp8: rows x cols bf16 (device, row-major, cols a multiple of 16) -> dst
 * [rows, cols] E4M3 codes (one byte each) and scale [rows] fp32.  Use it once per weight
 * tensor: W13 [E*2F, d], W2 [E*d, F], shared WS13 [2Fs, d], WS2 [d, Fs].  Errors: MOE_ERR_ARG
 * (NULL pointer), MOE_ERR_SHAPE (rows < 1, cols < 16 or not a multiple of 16).
 *
 * moe_forward_fp8: the layer of moe_forward with the quantised expert weights (codes and
 * scales as moe_quantize_fp8 writes them, in the layouts of moe_forward's w13/w2/ws13/ws2).
 * Routing, statistics and combine are those of moe_forward (bf16 router); the expert GEMMs
 * run on the decode kernels (weights on the MMA's M side, tokens on N) for every batch size,
 * so the call is meant for decode-sized batches.  Requires cfg->dtype bf16 (activations),
 * token choice and d_model % 256 == 0 (MOE_ERR_UNSUPPORTED / MOE_ERR_SHAPE otherwise).  The
 * workspace is moe_fp8_workspace_size bytes, 256-byte aligned; its status word is read by
 * moe_sync_status.  Other arguments and outputs as in moe_forward. */
int moe_quantize_fp8(int64_t rows, int64_t cols, const void* src, uint8_t* dst, float* scale,
                     void* stream);
int moe_fp8_workspace_size(const moe_config* cfg, size_t* bytes);
int moe_forward_fp8(const moe_config* cfg, const void* x, const void* w_gate, const float* bias,
                    const uint8_t* w13_q, const float* w13_scale, const uint8_t* w2_q,
                    const float* w2_scale, const uint8_t* ws13_q, const float* ws13_scale,
                    const uint8_t* ws2_q, const float* ws2_scale, void* out, int32_t* topk_idx,
                    float* topk_w, float* f, float* P, float* l_balance, float* z_loss,
                    int32_t* n_dropped, void* ws, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_B300_H */

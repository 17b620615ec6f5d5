/*
 * moe_b300.h -- C ABI of the single-GPU sparsely-gated Mixture-of-Experts SwiGLU
 * FFN forward for NVIDIA B300 (sm_103a).
 *
 * The layer (notation: T tokens, d model width, E routed experts, f expert hidden
 * width, k experts per token):
 *
 *   u = x W_r (+ logit_offset)                       router logits        [T, E]
 *   p = softmax(u) | sigmoid(u)                      scores
 *   token choice: top-k of p (+ sel_bias) per token  -> topk_idx, topk_w
 *   expert choice: top-cap of p[:, e] per expert     -> ec_tok, ec_w
 *   capacity drop, permute x rows into expert order  -> off, slot_of, x_perm
 *   per expert e: Y_e = (SiLU(X_e W1_e) * (X_e W3_e)) W2_e
 *   y[t] = sum_j topk_w[t,j] Y[slot_of[t,j]]  (+ sum of shared experts on x_t)
 *
 * Sources (page title, section):
 *   "技术日报 2026-04-14" (jsqmd.com): §3.1 Top-K gating and y = sum_i G(x)_i E_i(x);
 *     §3.2 Switch top-1, capacity factor K_max = floor(C N_tokens / N_experts) and
 *     overflow drop; §3.3 Expert Choice; §3.4 shared experts (DeepSeekMoE);
 *     §3.5 sigmoid gate; §4.3 selection-only bias; §9.1 MoELayer (renormalised
 *     top-k weights, shared experts summed unweighted).
 *   "MoE稀疏架构" (cloud.baidu.com), §4 工作原理: the six-step forward.
 *   lnwmold.com GPT-4 MoE article, §2.2: experts with W1, W2, W3.
 *
 * Conventions for every entry point:
 *   - Pointers named as device buffers are caller-owned device memory; the
 *     library allocates nothing.  Scratch comes from `ws` (`ws_bytes` long, size
 *     from moe_workspace_size for the same stage).
 *   - All work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream).  No call synchronises the host except
 *     moe_check_device_error, which waits for its stream, so a sequence of the
 *     other calls can be captured in a CUDA graph.  The kernels are programmatic
 *     dependent launches: one may start its setup while the previous kernel on
 *     the stream finishes, but it waits on the device for that kernel to complete
 *     before touching memory, so stream order holds against the caller's own work
 *     as well.
 *   - Arguments are checked before anything is launched.  A rejected call returns
 *     a non-zero moe_status and has no side effect.
 *   - Row-major layouts.  Device buffers must be 16-byte aligned; `ws` and the
 *     packed weight buffer 256-byte aligned (any torch CUDA allocation is).
 *   - dtype MOE_BF16: x, W_r, weights, x_perm, Y and y are bf16 (fp32 accumulate);
 *     dtype MOE_F32: all of those are fp32 (no TF32 anywhere);
 *     dtype MOE_BF16_FP8W: as MOE_BF16, except that moe_pack_weights stores the
 *     expert weights as FP8 E4M3 with one fp32 scale per output channel (the
 *     grouped FFN streams half the weight bytes; see moe_pack_weights);
 *     dtype MOE_BF16_FP8UP: as MOE_BF16, except that the up projection (x W1,
 *     x W3) runs on the FP8 tensor cores: its input rows are quantised to E4M3
 *     with one fp32 scale per token row, W1 and W3 with one scale per output
 *     channel (see moe_pack_weights); H, W2 and Y stay bf16.
 *     Scores and gate weights are always fp32; indices are int32.
 *   - Device-side waits are bounded.  A wait that gives up sets a device error
 *     word; moe_check_device_error reports it as MOE_ERR_TIMEOUT.
 *   - On first use of a device the library looks up, and keeps, the device
 *     addresses of its own device variables (the error word; the scratch array of
 *     moe_dispatch_noalloc).  Do not use the library on a device after a
 *     cudaDeviceReset of that device in the same process.
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
    MOE_ERR_INVALID_ARG = 1,   /* bad size, mode or null pointer                      */
    MOE_ERR_UNSUPPORTED = 2,   /* valid but outside this build's limits, or not sm_103 */
    MOE_ERR_MISALIGNED = 3,    /* a pointer is not 16-byte aligned                    */
    MOE_ERR_WORKSPACE = 4,     /* ws_bytes smaller than moe_workspace_size()          */
    MOE_ERR_CUDA = 5,          /* a CUDA runtime call failed                          */
    MOE_ERR_TIMEOUT = 6        /* a bounded device-side wait gave up                  */
} moe_status;

typedef enum { MOE_GATE_SOFTMAX = 0, MOE_GATE_SIGMOID = 1 } moe_gate;
typedef enum { MOE_TOKEN_CHOICE = 0, MOE_EXPERT_CHOICE = 1 } moe_mode;
typedef enum { MOE_F32 = 0, MOE_BF16 = 1, MOE_BF16_FP8W = 2, MOE_BF16_FP8UP = 3 } moe_dtype;
typedef enum { MOE_DROP_TOKEN_ORDER = 0, MOE_DROP_AFFINITY = 1 } moe_drop_policy;
typedef enum {
    MOE_STAGE_ROUTE = 0,
    MOE_STAGE_DISPATCH = 1,
    MOE_STAGE_GROUPED_FFN = 2,
    MOE_STAGE_COMBINE = 3,
    MOE_STAGE_FORWARD = 4
} moe_stage;

/*
 * Problem statement of one layer.
 *   T >= 0 tokens; d model width; E routed experts (1..256); f expert hidden width.
 *   k: experts per token, token choice only (1..min(8, E)).
 *   gate: MOE_GATE_SOFTMAX ("技术日报" §3.2) or MOE_GATE_SIGMOID (§3.5).
 *   mode: MOE_TOKEN_CHOICE (§3.1) or MOE_EXPERT_CHOICE (§3.3, softmax affinity).
 *   renormalize: token choice; 1 divides the k selected scores by their sum (§9.1),
 *     0 keeps the raw score (Switch top-1, §3.2).
 *   capacity_factor: token choice; C > 0 limits every expert to
 *     floor(C * T * k / E) assignments, kept in token order, the rest dropped
 *     (§3.2); C <= 0 means no limit.
 *   ec_capacity: expert choice; tokens each expert takes (1..T).
 *   n_shared, f_shared: always-on shared experts (§3.4), each of hidden width
 *     f_shared; their outputs are added unweighted.
 *   dtype: MOE_BF16, MOE_F32, MOE_BF16_FP8W or MOE_BF16_FP8UP.
 *   drop_policy: token choice with a capacity limit; which assignments an
 *     expert over capacity keeps: MOE_DROP_TOKEN_ORDER the first `cap` in token
 *     order (§3.2), MOE_DROP_AFFINITY the `cap` with the largest gate weights
 *     (DeepSeek-V2, "技术日报" §5.2: tokens dropped by descending affinity).
 * Build limits: MOE_BF16 needs d % 128 == 0, f % 64 == 0, f_shared % 64 == 0;
 * MOE_F32 needs d % 64 == 0, f % 64 == 0, f_shared % 64 == 0;
 * MOE_BF16_FP8W and MOE_BF16_FP8UP need d % 256 == 0, f % 128 == 0,
 * n_shared * f_shared % 128 == 0.
 */
typedef struct moe_config {
    int32_t T, d, E, f, k;
    int32_t gate;
    int32_t mode;
    int32_t renormalize;
    float capacity_factor;
    int32_t ec_capacity;
    int32_t n_shared, f_shared;
    int32_t dtype;
    int32_t drop_policy;   /* moe_drop_policy; see moe_dispatch */
} moe_config;

/* Human-readable name of a status code (static string, never NULL). */
const char *moe_status_string(moe_status s);

/* Checks a configuration against the rules above.  No CUDA call. */
moe_status moe_validate_config(const moe_config *cfg);

/* Capacity of one expert, floor(C*T*k/E) ("技术日报" §3.2), or -1 when
 * unlimited (token choice with C <= 0).  Expert choice: ec_capacity.  No CUDA call. */
moe_status moe_expert_capacity(const moe_config *cfg, int32_t *cap);

/* Rows of the expert-ordered buffers x_perm / Y a caller must provide:
 *   rows_routed = T*k (token choice) or E*ec_capacity (expert choice);
 *   rows_total  = rows_routed + (n_shared > 0 ? T : 0).  No CUDA call. */
moe_status moe_buffer_rows(const moe_config *cfg, int64_t *rows_routed, int64_t *rows_total);

/* Scratch bytes a stage needs in `ws` (MOE_STAGE_FORWARD: the whole layer).  No CUDA call. */
moe_status moe_workspace_size(const moe_config *cfg, moe_stage stage, size_t *bytes);

/* Bytes of the packed expert-weight buffer moe_pack_weights writes.  No CUDA call. */
moe_status moe_packed_weights_size(const moe_config *cfg, size_t *bytes);

/*
 * One-time re-layout of the expert weights into the operand layout of the grouped
 * expert GEMM (not part of the timed forward).
 *   W1, W3: [E][d][f], W2: [E][f][d] (the pages' per-expert x W1, h W2 layout);
 *   W1s, W3s: [n_shared][d][f_shared], W2s: [n_shared][f_shared][d] (NULL when
 *   n_shared == 0).  All in cfg->dtype, device memory, read only.
 *   packed: device buffer of moe_packed_weights_size bytes, written on `stream`.
 * MOE_BF16_FP8W (weights given in bf16): every output channel of every expert
 *   matrix (a hidden column of W1 and of W3, a model column of W2) gets the scale
 *   s = amax / 448 over its K inputs (fp32: amax of |w|, divided by the largest
 *   E4M3 value), and its weights are stored as the E4M3 code of w / s (fp32
 *   division, round to nearest even, saturated to +-448; s = 0 for an all-zero
 *   channel, whose codes are 0).  The GEMMs compute with q * s ("技术日报" §5
 *   lists FP8 expert weights; this is weight-only quantisation, activations stay
 *   bf16).  Several shared experts are packed as one merged expert, so the
 *   scale of a W2 output column covers all shared experts' rows of that column.
 *   The packed buffer is about half the bf16 one.  The grouped FFN expands the
 *   codes to bf16 in shared memory; on B300 this mode runs slower than MOE_BF16
 *   (it saves memory, not time).
 * MOE_BF16_FP8UP (weights given in bf16): W1 and W3 are quantised as above (a
 *   scale per hidden column of each, E4M3 codes in the operand layout of the FP8
 *   MMA); W2 is packed in bf16 as for MOE_BF16.  At run time each row entering the
 *   up projection (a token's x) gets the scale s = amax / 448 over its d values
 *   and the codes E4M3(x / s) by the same rule (all-zero row: s = 0, codes 0);
 *   the up GEMM multiplies codes by codes and scales the fp32 sums by the row and
 *   column scales ("技术日报" §7.4 FP8 for the expert GEMMs).  The packed buffer is
 *   two thirds of the bf16 one.
 */
moe_status moe_pack_weights(const moe_config *cfg, const void *W1, const void *W3, const void *W2,
                            const void *W1s, const void *W3s, const void *W2s, void *packed,
                            size_t packed_bytes, void *stream);

/*
 * Router ("技术日报" §3.1-§3.3, §3.5, §4.3; "MoE稀疏架构" §4 steps 1-2).
 *   x: [T][d], W_r: [d][E] (cfg->dtype).  logit_offset: [E] fp32 added to the
 *   logits before scoring, or NULL.  sel_bias: [E] fp32 added to the scores for
 *   the token-choice selection only (weights use the unbiased score), or NULL.
 * Token choice writes topk_idx[T][k] (int32, slots in descending key order, ties to
 *   the lower expert index) and topk_w[T][k] (fp32).
 * Expert choice writes topk_idx as ec_tok[E][cap] (int32, ascending token ids; ties
 *   to the lower token index) and topk_w as ec_w[E][cap] = softmax score of that
 *   token for that expert.
 * prob_sum: [E] fp32 device buffer or NULL.  When given it is overwritten with the
 *   sum over the T tokens of each expert's router score (softmax probability, or
 *   sigmoid score without the selection bias), the input of moe_load_stats.  The
 *   sum is accumulated with atomics, so its last bits vary from run to run.
 */
moe_status moe_route(const moe_config *cfg, const void *x, const void *W_r, const float *logit_offset,
                     const float *sel_bias, int32_t *topk_idx, float *topk_w, float *prob_sum, void *ws,
                     size_t ws_bytes, void *stream);

/*
 * Capacity-limited dispatch ("技术日报" §3.2; "MoE稀疏架构" §4 step 3).
 * Token choice: topk_idx[T][k] (values in [0, E)).  Assignments are visited in
 *   token order, slots in order; the first `cap` assignments of each expert are
 *   kept.  Writes
 *     cnt_raw[E]   assignments per expert before the drop,
 *     off[E+1]     exclusive prefix sum of the kept counts (off[E] = rows used),
 *     slot_of[T][k] row of the assignment in x_perm, -1 when dropped,
 *     x_perm[rows_routed][d] rows [0, off[E]) = x[token of the row] (rest untouched).
 * MOE_DROP_AFFINITY (capacity limited): an expert with more than `cap` assignments
 *   keeps the `cap` with the largest topk_w[T][k] (fp32 gate weights as moe_route
 *   wrote them), ties to the lower token index; its rows are still in token order.
 *   The experts of one token must be distinct.  topk_w is read only in that case
 *   (NULL otherwise).
 * Expert choice: topk_idx is ec_tok[E][cap]; writes off[e] = e*cap, cnt_raw[e] = cap,
 *   slot_of[T][E] (row e*cap + r when expert e took the token as its r-th pick, else
 *   -1) and x_perm[E*cap][d].
 */
moe_status moe_dispatch(const moe_config *cfg, const int32_t *topk_idx, const float *topk_w, const void *x,
                        int32_t *off, int32_t *cnt_raw, int32_t *slot_of, void *x_perm, void *ws,
                        size_t ws_bytes, void *stream);

/*
 * moe_dispatch for callers that cannot allocate device memory.  (The paper has
 * no counterpart; this is an interface convenience of the library.)
 *
 * Some callers cannot provide a workspace: a plugin inside a host framework that
 * owns all device memory and hands over only the layer's inputs and outputs, or
 * a latency-critical serving loop where a cudaMalloc could synchronise the
 * device.  This call takes the same arguments and writes the same outputs as
 * moe_dispatch, minus `ws`: its scratch is a 512 KiB array compiled into the
 * library, present on every GPU that loads the library until the process exits.
 *   - Token choice: T * k must not exceed MOE_DISPATCH_NOALLOC_MAX_ASSIGNMENTS,
 *     otherwise MOE_ERR_UNSUPPORTED is returned and nothing is launched.  Expert
 *     choice needs no scratch and has no extra limit.
 *   - The first call on a device looks up the array's address on that device;
 *     make that first call before any stream capture.
 *   - The call allocates nothing (no cudaMalloc, cudaFree or allocating library
 *     routine).  All calls share the array and it keeps the last call's
 *     contents; nothing in it needs clearing between calls, but calls whose work
 *     overlaps on the GPU (other streams, other host threads) race on it and
 *     must be serialised by the caller.
 */
#define MOE_DISPATCH_NOALLOC_MAX_ASSIGNMENTS 65536
moe_status moe_dispatch_noalloc(const moe_config *cfg, const int32_t *topk_idx, const void *x, int32_t *off,
                                int32_t *cnt_raw, int32_t *slot_of, void *x_perm, void *stream);

/*
 * Grouped SwiGLU experts over the ragged expert segments of x_perm ("lnwmold"
 * §2.2 W1, W2, W3; SwiGLU: (SiLU(X W1) * (X W3)) W2).
 *   x_perm[rows_routed][d], off[E+1] as written by moe_dispatch (read on the device;
 *   no host synchronisation), packed: moe_pack_weights output, x: [T][d] input of
 *   the shared experts (NULL when n_shared == 0).
 *   Y[rows_total][d]: rows [0, off[E]) = expert outputs in x_perm order; with shared
 *   experts, rows [rows_routed, rows_routed + T) = sum of the shared experts on x.
 */
moe_status moe_grouped_ffn(const moe_config *cfg, const void *x_perm, const int32_t *off,
                           const void *packed, const void *x, void *Y, void *ws, size_t ws_bytes,
                           void *stream);

/*
 * The two halves of moe_grouped_ffn, for callers that keep the hidden activations.
 * moe_grouped_ffn_up:   H[rows_routed][f] rows [0, off[E]) = SiLU(X W1) * (X W3) of
 *   each row's expert; with shared experts Hs[T][n_shared*f_shared] = the merged
 *   shared hidden activations of x (Hs may be NULL when n_shared == 0).
 * moe_grouped_ffn_down: Y rows [0, off[E]) = H W2 of each row's expert; with shared
 *   experts rows [rows_routed, rows_routed + T) = Hs times the merged shared W2.
 * H, Hs in cfg->dtype.  Neither call needs workspace.  MOE_BF16_FP8UP returns
 * MOE_ERR_UNSUPPORTED (its up projection quantises rows into a workspace; use
 * moe_grouped_ffn or moe_forward).
 */
moe_status moe_grouped_ffn_up(const moe_config *cfg, const void *x_perm, const int32_t *off,
                              const void *packed, const void *x, void *H, void *Hs, void *stream);
moe_status moe_grouped_ffn_down(const moe_config *cfg, const void *H, const void *Hs, const int32_t *off,
                                const void *packed, void *Y, void *stream);

/*
 * Gate-weighted combine back to token order ("技术日报" §3.1, §3.4, §9.1).
 * Token choice: y[t] = sum_{j: slot_of[t][j] >= 0} topk_w[t][j] * Y[slot_of[t][j]]
 *   (+ Y[rows_routed + t] with shared experts), slots in order.
 * Expert choice: y[t] = sum_{e: slot_of[t][e] >= 0} ec_w[slot] * Y[slot]
 *   (+ shared), experts in ascending order; `topk_w` is ec_w[E][cap].
 *   y: [T][d] in cfg->dtype, fp32 accumulation.  Dropped or unpicked tokens get
 *   only the shared part (zero without shared experts); the residual is the
 *   caller's.
 */
moe_status moe_combine(const moe_config *cfg, const void *Y, const int32_t *slot_of, const float *topk_w,
                       void *y, void *ws, size_t ws_bytes, void *stream);

/*
 * The whole layer: moe_route -> moe_dispatch -> moe_grouped_ffn -> moe_combine, with
 * every intermediate carved from `ws` (moe_workspace_size(MOE_STAGE_FORWARD)).
 *   x: [T][d]; W_r: [d][E]; logit_offset, sel_bias: as moe_route; packed: as
 *   moe_grouped_ffn; y: [T][d] output.
 */
moe_status moe_forward(const moe_config *cfg, const void *x, const void *W_r, const float *logit_offset,
                       const float *sel_bias, const void *packed, void *y, void *ws, size_t ws_bytes,
                       void *stream);

/*
 * Load statistics of one routing ("技术日报 2026-04-14" §4.4 diagnostics; §4.2
 * Switch auxiliary loss and DeepSeek V1 expert-level balance, both without their
 * alpha).  Inputs (device, read only): topk_idx and cnt_raw as moe_route and
 * moe_dispatch wrote them, prob_sum as moe_route wrote it.  With
 *   f_e  = cnt_raw[e] / sum(cnt_raw)   (assignment share before any capacity drop),
 *   f1_e = share of the T tokens whose slot-0 expert is e (Expert Choice: f_e),
 *   P_e  = prob_sum[e] / T              (mean router score),
 * writes token_fraction[e] = f_e and prob_mean[e] = P_e ([E] fp32 each), and
 * summary (device, 5 doubles) = { E*max f, std(f)/mean(f) (population std),
 * -sum q ln q with q = P/sum(P), E*sum f1*P, E*sum f*P }.  Balanced routing gives
 * {1, 0, ln E, 1, 1} for softmax scores.  One kernel on `stream`; T == 0 writes
 * nothing.
 */
moe_status moe_load_stats(const moe_config *cfg, const int32_t *topk_idx, const int32_t *cnt_raw,
                          const float *prob_sum, float *token_fraction, float *prob_mean, double *summary,
                          void *stream);

/* Number of CUDA kernels one call of `stage` enqueues for this configuration
 * (memsets not counted; MOE_STAGE_FORWARD: the whole layer).  No CUDA call. */
moe_status moe_launch_count(const moe_config *cfg, moe_stage stage, int32_t *kernels);

/*
 * Limit of every bounded device-side wait of the tensor-core kernels, in
 * nanoseconds: a pipeline stage, an accumulator, or (fused expert launch) the up
 * tiles that produce a down tile's rows.  A wait that reaches the limit gives up:
 * the kernel records the timeout in the device error word, drains the copies and
 * MMAs it has issued, frees its tensor memory and ends, so the context stays
 * usable, and moe_check_device_error reports MOE_ERR_TIMEOUT.  The limit is
 * process-wide and read when a call launches its kernels.  0 restores the
 * default of 2 s; values outside [1e3, 6e10] return MOE_ERR_INVALID_ARG.  A limit
 * shorter than the longest legitimate wait (a down tile waits for its up tiles,
 * milliseconds on large layers) makes correct calls report timeouts.  No CUDA call.
 */
moe_status moe_set_wait_limit_ns(uint64_t limit_ns);
moe_status moe_get_wait_limit_ns(uint64_t *limit_ns);

/*
 * Tile order of the tensor-core expert GEMMs (a tuning knob of the library; the
 * pages prescribe no schedule).  Each expert segment's 128-row M tiles are taken
 * in groups of nearly equal size, every N block of a group before the next group,
 * so that a group's activation rows stay in L2 while the group streams the
 * expert's weights once.  A group holds at most as many M tiles as fit `up_bytes`
 * of x_perm rows (up projection: 128 x d x 2 bytes per tile) or `down_bytes` of H
 * rows (down projection: 128 x f x 2 bytes per tile), and at least one.  The
 * order changes which tiles run together, never a result: every output element is
 * computed by one tile with the same k order.  Process-wide, read when a call
 * launches its kernels; 0 restores a default (40 MiB up, 64 MiB down); values
 * above 2^40 return MOE_ERR_INVALID_ARG.  No CUDA call.
 */
moe_status moe_set_tile_group_bytes(uint64_t up_bytes, uint64_t down_bytes);
moe_status moe_get_tile_group_bytes(uint64_t *up_bytes, uint64_t *down_bytes);

/*
 * Probe of the failure path of the bounded waits (the pages define no failure
 * behaviour; this is a diagnostic of the library).  Launches one small kernel on
 * `stream` that runs the two wait routines of the tensor-core kernels with the
 * current limit: first until the device int32 *flag reaches `target` (read with
 * acquire semantics; the caller owns the flag and decides whether anything sets
 * it), then on a shared-memory barrier that completes only if the first wait
 * succeeded.  With the condition met both waits succeed and nothing is recorded;
 * otherwise each gives up after the limit (about twice the limit in all) and the
 * next moe_check_device_error returns MOE_ERR_TIMEOUT.
 */
moe_status moe_wait_probe(const int32_t *flag, int32_t target, void *stream);

/*
 * Waits for `stream`, then reads and clears the device error word.  Returns
 * MOE_ERR_TIMEOUT if a bounded device-side wait gave up since the last check,
 * MOE_ERR_INVALID_ARG if a kernel skipped an expert or token id outside its range
 * (such an assignment is treated as dropped), MOE_OK otherwise.
 */
moe_status moe_check_device_error(void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_B300_H */

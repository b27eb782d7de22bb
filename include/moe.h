/*
 * moe.h -- C ABI of the Sparsely-Gated Mixture-of-Experts layer forward pass
 * on one NVIDIA B300 (sm_103a).
 *
 * The layer (Shazeer et al. 2017, "Outrageously Large Neural Networks: The
 * Sparsely-Gated Mixture-of-Experts Layer"), as the lesson page
 * "MoE:稀疏门控混合专家" states it:
 *   section 三 "门控怎么挑": a gate matrix W_g with one column per expert
 *     scores each token; KeepTopK sets all but the k best scores to -inf; a
 *     softmax turns the survivors into weights G(x) that sum to 1.  With
 *     thousands of experts the choice is two-level (MoE-N-h): pick the best
 *     groups first, then the best experts inside each chosen group.
 *   section 四 "为什么要加噪声": the score is noisy,
 *     H(x)_i = (x.W_g)_i + eps_i * softplus((x.W_noise)_i), eps redrawn each time.
 *   section 二 "一层 MoE 长什么样": each expert E_i is a feed-forward net with
 *     one hidden ReLU layer, and y = sum_i G(x)_i E_i(x); experts with weight 0
 *     are not computed.
 * The ai-papers.xuzou.cn card "Outrageously Large Neural Networks - 中文验证版"
 * (section 瓶颈) adds that each expert sees about k*b/n rows, and (section
 * 方法适配) that an importance loss and a load loss keep the experts balanced;
 * this library returns the importance vector, its CV^2 and the per-expert
 * counts that those terms are built from.
 *
 * Conventions for every call
 *   - All tensor pointers are DEVICE pointers (cudaMalloc'd or torch CUDA
 *     memory of the current device), row-major, 16-byte aligned.  The caller
 *     allocates and owns every buffer, including the workspace; the library
 *     never allocates or frees device memory and keeps no global mutable state
 *     (calls with distinct workspaces may run concurrently on different streams).
 *   - `stream` is a cudaStream_t (passed as void*); NULL is the legacy default
 *     stream.  Calls enqueue work and return without synchronising.
 *   - Host-detectable errors (bad shape, NULL or misaligned pointer, workspace
 *     too small, unsupported size) return a negative moe_status synchronously
 *     and enqueue nothing.  Errors found on the device (an expert index out of
 *     range, a bounded wait that ran out) are recorded in the workspace's error
 *     word; moe_check() reads it.  Nothing crosses the ABI as an exception.
 *   - Results are deterministic: identical inputs give bit-identical outputs
 *     (no floating-point atomics, fixed reduction orders, stable permutation).
 *
 * Layouts (C = n for flat gating, C = G + n for hierarchical gating; S = T*k
 * slots, slot s = t*k + j is the j-th expert choice of token t):
 *   x        [T, d]     dtype (MOE_BF16 or MOE_F32)
 *   Wg, Wn   [d, C]     fp32.  Hierarchical: columns 0..G-1 score the groups,
 *                        then G blocks of m = n/G columns, block g scoring the
 *                        experts g*m .. g*m+m-1 of group g.
 *   bg       [C]        fp32 or NULL; added to the clean score x.W_g
 *   eps      [T, C]     fp32; required (with Wn) when shape.noisy == 1, ignored
 *                        (may be NULL) when shape.noisy == 0
 *   idx      [T, k]     int32, the chosen experts in descending H order
 *                        (hierarchical: group rank major, inner rank minor)
 *   G        [T, k]     fp32, their gate weights (sum to 1 per token)
 *   W1       [n, h, d]  dtype; expert e's first layer, out x in (a = W1[e] x + b1[e])
 *   b1       [n, h]     fp32 or NULL (= zeros)
 *   W2       [n, d, h]  dtype; expert e's second layer, out x in
 *   b2       [n, d]     fp32 or NULL (= zeros)
 *   counts   [n]        int32, slots routed to each expert
 *   offsets  [n+1]      int32, exclusive prefix sum of counts
 *   perm     [S]        int32, expert-ordered row r -> slot (stable: rows of
 *                        one expert are in increasing slot order)
 *   inv_perm [S]        int32, slot -> row
 *   importance [n]      fp32, sum of the gate weights routed to each expert
 *   cv2      [1]        fp32, population variance(importance) / mean^2
 *   Y_slot   [S, d]     dtype, expert output of row r (expert-row order)
 *   y        [T, d]     dtype, the layer output
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t moe_status;
#define MOE_OK 0
#define MOE_ERR_INVALID_ARG (-1) /* bad shape, NULL or misaligned pointer */
#define MOE_ERR_UNSUPPORTED (-2) /* valid but outside this build's limits */
#define MOE_ERR_WORKSPACE (-3)   /* workspace NULL, misaligned or too small */
#define MOE_ERR_CUDA (-4)        /* a CUDA runtime/driver call failed */
#define MOE_ERR_TIMEOUT (-5)     /* a bounded device wait ran out (device-side) */
#define MOE_ERR_DEVICE (-6)      /* bad data found on the device, e.g. idx >= n */

#define MOE_F32 0
#define MOE_BF16 1

/* Limits of this build (MOE_ERR_UNSUPPORTED beyond them). */
#define MOE_MAX_K 16          /* experts per token; also k_groups and k/k_groups */
#define MOE_MAX_COLS 16384    /* gate columns C */
#define MOE_MAX_SLOTS 0x7FFFFFFF

typedef struct moe_shape {
    int64_t T;        /* tokens (0 allowed: outputs are zero-filled, nothing else runs) */
    int32_t d;        /* model width; multiple of 64, <= 8192 */
    int32_t h;        /* expert hidden width; multiple of 64, <= 16384 */
    int32_t n;        /* experts, >= 1 */
    int32_t k;        /* experts per token in total, 1 <= k <= min(n, MOE_MAX_K) */
    int32_t groups;   /* 0: flat gating.  G > 0: hierarchical, n % G == 0 */
    int32_t k_groups; /* hierarchical only: groups kept per token, k % k_groups == 0,
                         k_groups <= G and k / k_groups <= n / G */
    int32_t dtype;    /* MOE_BF16 or MOE_F32: the type of x, W1, W2, Y_slot and y */
    int32_t noisy;    /* 1: add eps * softplus(x.W_noise) to the score; 0: clean score */
} moe_shape;

/* Library version, major*10000 + minor*100 + patch. */
MOE_API int32_t moe_version(void);

/* Static text for a status code. */
MOE_API const char *moe_status_string(moe_status s);

/* The CUDA error code (a cudaError_t value) behind the last MOE_ERR_CUDA that
 * an entry point returned on the calling host thread, 0 if there was none,
 * and the CUDA runtime's static name for such a code.  Host-only; no device
 * work. */
MOE_API int32_t moe_last_cuda_error(void);
MOE_API const char *moe_cuda_error_name(int32_t code);

/* Host-only check of a shape against the rules above.  No device work. */
MOE_API moe_status moe_validate(const moe_shape *shape);

/* Workspace bytes every call below needs for this shape (0 if the shape is
 * invalid).  The pages have no counterpart (their layer ran inside a training
 * framework that owned memory); the workspace holds what the stages pass to
 * each other: the packed gate matrices of section 三/四 of
 * "MoE:稀疏门控混合专家", the routing scratch, and the expert-ordered rows of
 * "Outrageously Large Neural Networks - 中文验证版" section 瓶颈.  One
 * workspace serves all calls of one shape; its first 256 bytes hold the
 * device error word.  The workspace must be 256-byte aligned. */
MOE_API size_t moe_workspace_bytes(const moe_shape *shape);

/* Clears the device error word of a workspace (enqueued on `stream`).  Call it
 * once on a fresh workspace before its first use. */
MOE_API moe_status moe_workspace_init(void *ws, size_t ws_bytes, void *stream);

/*
 * Gate ("MoE:稀疏门控混合专家", sections 三 and 四): for every token the
 * noisy score H = x.W_g (+ bg) + eps * softplus(x.W_noise), KeepTopK and
 * softmax over the k survivors (flat), or the two-level choice (hierarchical:
 * k_groups groups by their noisy group score, then k/k_groups experts in each
 * kept group by that group's own columns; weight = group weight x inner weight).
 * Scores are computed with fp32-faithful accuracy; ties go to the lower index.
 * Writes idx [T,k] and G [T,k].
 */
MOE_API moe_status moe_gate(const moe_shape *shape, const void *x, const float *Wg, const float *Wn,
                    const float *bg, const float *eps, int32_t *idx, float *G, void *ws,
                    size_t ws_bytes, void *stream);

/*
 * Dispatch (routing).  "Outrageously Large Neural Networks - 中文验证版",
 * section 瓶颈: each expert receives only the rows routed to it (about k*b/n
 * of a batch of b), so those rows are gathered together; "MoE:稀疏门控混合专家"
 * section 二: experts with weight 0 are not computed; section 方法适配 of the
 * first page and the wudongming97 note (section 方法怎么做): the importance of
 * an expert is the batch sum of its gate weights.
 * Outputs: per-expert counts, their exclusive scan, the stable
 * permutation of the slots into expert-contiguous rows and its inverse, the
 * importance vector (gate weight summed per expert in a fixed order: slots
 * of a 32-slot group, the groups of a 1024-slot chunk, then the chunks; fp32)
 * and its CV^2.  An idx entry outside [0, n) sets
 * MOE_ERR_DEVICE in the error word; that slot is left out of every output
 * (inv_perm[s] = -1) and the rest stays consistent.
 */
MOE_API moe_status moe_dispatch(const moe_shape *shape, const int32_t *idx, const float *G,
                        int32_t *counts, int32_t *offsets, int32_t *perm, int32_t *inv_perm,
                        float *importance, float *cv2, void *ws, size_t ws_bytes, void *stream);

/*
 * moe_dispatch without a workspace.  The pages have no counterpart to this
 * call: it exists for callers that cannot allocate device memory (code
 * running inside another framework's fixed memory pool, plug-ins whose host
 * owns every allocation, latency-critical paths where an allocation may block
 * or fail).  It computes exactly what moe_dispatch computes, with the same
 * kernels, but keeps their scratch in one array of static device storage
 * inside this library (8 MiB, resident on every device that loads the
 * library until the process exits).  It calls no allocation routine.
 *   - Limit: the scratch needed is 256 B + 4*S + 8*ceil(S/1024)*n + 4*n
 *     bytes (each term rounded up to 256 B); a shape that needs more than
 *     8 MiB returns MOE_ERR_UNSUPPORTED and enqueues nothing.
 *   - Every call looks up the array's device address (cudaGetSymbolAddress)
 *     with the caller's current device, so the address stays right after a
 *     device reset.  The first call on a device may load the library's
 *     module there: make that first call before any stream capture.
 *   - Every call on a device shares the one array, which keeps the previous
 *     call's contents (each call clears the part that must start at zero).
 *     Calls whose work overlaps on the GPU (different streams, or different
 *     host threads) race on it: serialise them.
 *   - An idx entry outside [0, n) is skipped as in moe_dispatch (inv_perm = -1),
 *     but there is no workspace to carry the error word, so it is not reported.
 */
MOE_API moe_status moe_dispatch_noalloc(const moe_shape *shape, const int32_t *idx,
                                        const float *G, int32_t *counts, int32_t *offsets,
                                        int32_t *perm, int32_t *inv_perm, float *importance,
                                        float *cv2, void *stream);

/*
 * Expert FFNs on expert-contiguous rows ("MoE:稀疏门控混合专家", section 二):
 * for every expert e and row r in [offsets[e], offsets[e+1]), with token
 * t = perm[r] / k,  Y_slot[r] = W2[e] . ReLU(W1[e] . x[t] + b1[e]) + b2[e].
 * BF16: bf16 operands, fp32 accumulation on the tensor cores, the hidden
 * activation rounded once to bf16 between the layers, Y_slot rounded once.
 * F32: fp32 throughout.  Unselected experts are not computed.
 */
MOE_API moe_status moe_expert_ffn(const moe_shape *shape, const void *x, const int32_t *perm,
                          const int32_t *offsets, const void *W1, const float *b1, const void *W2,
                          const float *b2, void *Y_slot, void *ws, size_t ws_bytes, void *stream);

/*
 * Combine ("MoE:稀疏门控混合专家", section 二: y = sum_i G(x)_i E_i(x), only
 * the selected experts contributing):
 * y[t] = sum_{j=0..k-1} G[t,j] * Y_slot[inv_perm[t*k+j]], summed in
 * fp32 in that fixed j order and rounded once to the output type.  A slot
 * with inv_perm = -1 contributes nothing; an entry >= S sets MOE_ERR_DEVICE.
 */
MOE_API moe_status moe_combine(const moe_shape *shape, const void *Y_slot, const int32_t *inv_perm,
                       const float *G, void *y, void *ws, size_t ws_bytes, void *stream);

/*
 * The whole forward pass on one stream ("MoE:稀疏门控混合专家", sections 二,
 * 三 and 四: noisy score, KeepTopK, softmax, the selected experts, their
 * weighted sum): gate, dispatch, expert FFNs and combine.  Outputs y [T,d], G [T,k], idx [T,k], importance [n], cv2 [1],
 * counts [n]; the permutation and the expert outputs live in the workspace.
 */
MOE_API moe_status moe_forward(const moe_shape *shape, const void *x, const float *Wg, const float *Wn,
                       const float *bg, const float *eps, const void *W1, const float *b1,
                       const void *W2, const float *b2, void *y, float *G, int32_t *idx,
                       float *importance, float *cv2, int32_t *counts, void *ws,
                       size_t ws_bytes, void *stream);

/*
 * Load estimate of the noisy gate, the smooth per-expert load that the load
 * loss balances ("Outrageously Large Neural Networks - 中文验证版", section
 * 方法适配: an importance loss and a load loss keep the samples spread over
 * the experts; the pages stop before its formula, which is taken from the
 * paper's load-balancing appendix).  For token t and expert i,
 *   P(t, i) = Phi((c_i - thr_i) / softplus(r_i)),  c = x.W_g (+ bg), r = x.W_noise,
 * thr_i = the k-th largest noisy score H of the other experts: the
 * probability that i stays among the k kept when only its own noise is
 * redrawn.  load[i] = sum over tokens of P(t, i) (fp64 sums in token order,
 * rounded to fp32), load_cv2 = population variance(load) / mean^2.
 * The call runs the gate too (idx, G as moe_gate).  Flat, noisy (eps and Wn
 * required), bf16 shapes with k <= 15 only (MOE_ERR_UNSUPPORTED otherwise).
 * lws: a second, caller-owned, 256-byte aligned workspace of
 * moe_load_workspace_bytes(shape) bytes (8*T*n + 8*T + 8*n*ceil(T/64) + 8*n
 * bytes, each region rounded up to 256); `ws` is the ordinary workspace.
 */
MOE_API size_t moe_load_workspace_bytes(const moe_shape *shape);
MOE_API moe_status moe_gate_load(const moe_shape *shape, const void *x, const float *Wg,
                                 const float *Wn, const float *bg, const float *eps, int32_t *idx,
                                 float *G, float *load, float *load_cv2, void *ws,
                                 size_t ws_bytes, void *lws, size_t lws_bytes, void *stream);

/*
 * Backward pass of the layer, flat or hierarchical.  The pages train the
 * layer with noise in the gate ("MoE:稀疏门控混合专家", section 四) and an
 * importance loss beside the task loss ("Outrageously Large Neural Networks —
 * MoE 怎样让模型“很大但不每次全算”", section 方法怎么做); the gradients are the
 * chain rule of the forward pass with the forward's selection idx held
 * fixed, for the loss
 *   L = sum_t <dy[t], y[t]> + w_importance * CV^2(importance).
 * Hierarchical gate (section 三 of the first page): the final weight of slot
 * (q, j) is Gp_q * Gi_qj, the group weight times the in-group weight; the
 * gradient passes through both softmaxes to the kept group columns and the
 * kept expert columns of Wg, Wnoise and bg.
 * Inputs: the forward's inputs (x, W1, W2, dy in the shape's dtype; Wg, Wnoise
 * [d,C], eps [T,C], b1, b2 fp32, with C the gate's score columns: n flat,
 * groups + n hierarchical, the group columns first; bg is not needed), its
 * outputs idx [T,k], G [T,k] and importance [n] (only read when
 * w_importance != 0), and dy [T,d].
 * Outputs, all fp32 and overwritten: dx [T,d], dWg [d,C], dWnoise [d,C] (all
 * zero when noisy == 0; may then be NULL), dbg [C], dW1 [n,h,d], db1 [n,h],
 * dW2 [n,d,h], db2 [n,d]; dbg, db1, db2 may be NULL when not wanted.
 * Every sum runs in a fixed order, so results are bit-reproducible.  bf16
 * shapes whose d and h are multiples of 128 run the contractions on the
 * tensor cores (bf16 operands, fp32
 * accumulation, the recomputed expert outputs and the intermediate gradient
 * rows rounded to bf16, as in the forward's expert stage); all other shapes
 * run in fp32 on the CUDA cores.  ws: a caller-owned, 256-byte aligned
 * workspace of moe_backward_workspace_bytes(shape) bytes (it grows with
 * S*(d + h), S = T*k, and with n*d*h on the tensor-core path, which also
 * holds the experts' weights transposed); its first 256 bytes are the error
 * header that moe_check reads.  An idx or routing entry out of range sets
 * MOE_ERR_DEVICE.
 */
MOE_API size_t moe_backward_workspace_bytes(const moe_shape *shape);
MOE_API moe_status moe_backward(const moe_shape *shape, const void *x, const float *Wg,
                                const float *Wnoise, const float *eps, const void *W1,
                                const float *b1, const void *W2, const float *b2,
                                const int32_t *idx, const float *G, const float *importance,
                                const void *dy, float w_importance, float *dx, float *dWg,
                                float *dWnoise, float *dbg, float *dW1, float *db1, float *dW2,
                                float *db2, void *ws, size_t ws_bytes, void *stream);

/*
 * The layer with balanced routing ("Outrageously Large Neural Networks -
 * 中文验证版", section 方法适配: a per-batch mask gives every expert the same
 * batch size during training; per-expert thresholds approximate it at
 * inference).  Flat gating only (MOE_ERR_UNSUPPORTED otherwise).  H = the flat
 * gate's noisy score, x.Wg (+ bg) + eps * softplus(x.Wnoise), fp32.
 *   thr == NULL  batchwise mask: expert e keeps the m = floor(k*T/n) tokens
 *                with the largest H[:, e] (equal scores: the lower token
 *                index first); rows_cap must be at least n*m.
 *   thr [n]      thresholds: expert e keeps token t iff H[t, e] > thr[e]; a
 *                total above rows_cap drops the rows past it and sets
 *                MOE_ERR_DEVICE.
 * Weights: softmax of H[t, .] over the experts that kept t.  y[t] = sum over
 * those experts, in increasing e, of w * E_e(x_t) (0 when none kept t); fp32
 * accumulation, one rounding to x's dtype.  Outputs: y [T,d], counts [n]
 * (tokens kept per expert, before any capacity cut), W [T,n] fp32 weights (0
 * where not kept; may be NULL).  ws: caller-owned, 256-byte aligned, of
 * moe_balanced_workspace_bytes(shape, rows_cap) bytes; T*n must not exceed
 * MOE_MAX_SLOTS.
 */
MOE_API size_t moe_balanced_workspace_bytes(const moe_shape *shape, int64_t rows_cap);
MOE_API moe_status moe_forward_balanced(const moe_shape *shape, const void *x, const float *Wg,
                                        const float *Wnoise, const float *bg, const float *eps,
                                        const float *thr, int64_t rows_cap, const void *W1,
                                        const float *b1, const void *W2, const float *b2, void *y,
                                        int32_t *counts, float *W, void *ws, size_t ws_bytes,
                                        void *stream);

/*
 * Diagnostic: launches one thread that waits, through the same bounded wait
 * every pipelined kernel of this library uses, on a barrier that nothing
 * arrives at.  After the 2 s limit it records MOE_ERR_TIMEOUT in the
 * workspace's error word and returns; moe_check then reports it.  Nothing
 * faults or traps and the context stays usable.  ws: any workspace of at
 * least 256 bytes, 256-byte aligned.
 */
MOE_API moe_status moe_selftest_timeout(void *ws, size_t ws_bytes, void *stream);

/*
 * Synchronises `stream`, reads the workspace's device error word, clears it
 * and returns it (MOE_OK when no device error was recorded).  Returns
 * MOE_ERR_CUDA if the stream itself failed.  The pages have no counterpart:
 * this is how device-side checks of the steps above (an expert index outside
 * the n experts of "MoE:稀疏门控混合专家" section 三, a routing entry outside
 * the S = T*k slots, a bounded wait that ran out) reach the caller without a
 * fault.
 */
MOE_API moe_status moe_check(void *ws, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_B300_H */

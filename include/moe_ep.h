/*
 * moe_ep.h -- device calls of the expert-parallel MoE layer (libmoe_b300.so).
 *
 * The pages' own system spreads the experts over devices and moves each
 * token's rows to its experts' devices and back by all-to-all
 * ("Outrageously Large Neural Networks - MoE 怎样让模型'很大但不每次全算'",
 * section 方法怎么做); each device keeps a share of the experts and the
 * devices' batches are merged at the MoE layer, so that every expert sees
 * the rows of all devices at once ("Outrageously Large Neural Networks -
 * 中文验证版", sections 计算设置 and 方法适配).
 *
 * Partition used here: P ranks, n % P == 0, rank q owns the n_local = n / P
 * experts [q*n_local, (q+1)*n_local) (a contiguous block).  One layer call on
 * rank r, with its own T_r tokens:
 *   1. moe_gate, moe_dispatch on the local tokens against all n experts
 *      (include/moe.h); the slots bound for rank q are then the contiguous
 *      range [offsets[q*n_local], offsets[(q+1)*n_local]) of the dispatch's
 *      expert order.
 *   2. moe_gather_rows(x, perm, div = k): the x rows in that order (the send
 *      buffer).
 *   3. exchange (the caller's collective): counts [P][n_local] all-to-all,
 *      then the rows all-to-all with per-rank row counts.
 *   4. moe_ep_regroup: the received rows, ordered (source rank, local expert,
 *      source order), into the merged expert-major order.
 *   5. moe_expert_ffn on the merged rows (shape: T = R received rows, k = 1,
 *      n = n_local, perm = perm_local, offsets = offsets_local).
 *   6. moe_gather_rows(Y, inv_local, div = 1): the outputs back in received
 *      order; exchange back (the reverse all-to-all); the rows then arrive in
 *      the rank's own expert order, i.e. as its Y_slot.
 *   7. moe_combine on the local tokens; importance summed over the ranks
 *      (the caller's all-reduce) and moe_importance_cv2 for the batch CV^2.
 *
 * All pointers are device pointers, 16-byte aligned, owned by the caller;
 * calls only enqueue work on `stream` (a cudaStream_t, NULL = legacy default
 * stream).  `err` is an optional device error word (4 int32: code, site,
 * aux, unused), for example the first 16 bytes of a moe workspace; the first
 * device-side error is recorded there (read it with moe_check on that
 * workspace).
 */
#ifndef MOE_B300_EP_H
#define MOE_B300_EP_H

#include "moe.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Merged order of the rows one rank received from P ranks.
 *   recv_counts [P][n_local] int32: rows of local expert e sent by rank q.
 *   The R received rows are ordered by q, then e, then the sender's order.
 * Writes
 *   offsets_local [n_local + 1]: exclusive scan of the per-expert totals
 *     sum over q of recv_counts[q][e]  (offsets_local[n_local] = R);
 *   perm_local [R]: merged row j -> received row.  Within expert e the merged
 *     rows take the received rows of rank 0 first, then rank 1, ..., each in
 *     the sender's order (a stable sort of the received rows by expert);
 *   inv_local [R]: its inverse.
 * Errors: MOE_ERR_INVALID_ARG (P or n_local <= 0, R < 0, NULL or misaligned
 * pointer), MOE_ERR_UNSUPPORTED (P * n_local > 4096); on the device, a
 * negative count or counts that do not sum to R record MOE_ERR_DEVICE in
 * `err` and leave perm_local / inv_local unwritten.
 */
MOE_API moe_status moe_ep_regroup(int32_t P, int32_t n_local, const int32_t *recv_counts,
                                  int64_t R, int32_t *offsets_local, int32_t *perm_local,
                                  int32_t *inv_local, int32_t *err, void *stream);

/*
 * Row gather: dst[i, :] = src[rows[i] / div, :] for i < R; rows of d
 * elements of `dtype` (MOE_BF16 or MOE_F32), copied bit for bit.
 *   src [src_rows, d], rows [R] int32, dst [R, d].
 * With rows = perm and div = k it builds the send buffer of step 2; with
 * rows = inv_local and div = 1 it returns the expert outputs of step 6.
 * Errors: MOE_ERR_INVALID_ARG (negative sizes, div <= 0, bad dtype, NULL or
 * misaligned pointer when R > 0), MOE_ERR_UNSUPPORTED (a row of d elements is
 * not a multiple of 16 bytes); a row index outside [0, src_rows) after the
 * division writes a zero row and records MOE_ERR_DEVICE in `err`.
 */
MOE_API moe_status moe_gather_rows(const void *src, int64_t src_rows, const int32_t *rows,
                                   int32_t div, int64_t R, int32_t d, int32_t dtype, void *dst,
                                   int32_t *err, void *stream);

/*
 * cv2[0] = population variance / mean^2 of importance[0..n) (0 when the mean
 * is 0), with the fixed-order fp32 sums of moe_dispatch's CV^2: the
 * statistic of the importance loss ("Outrageously Large Neural Networks -
 * 中文验证版", section 方法适配) for a batch merged over ranks.
 * Errors: MOE_ERR_INVALID_ARG (n <= 0, NULL or misaligned pointer).
 */
MOE_API moe_status moe_importance_cv2(const float *importance, int32_t n, float *cv2,
                                      void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_B300_EP_H */

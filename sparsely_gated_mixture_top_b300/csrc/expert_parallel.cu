// expert_parallel.cu -- the device side of the expert-parallel layer
// ("Outrageously Large Neural Networks - MoE 怎样让模型'很大但不每次全算'",
// section 方法怎么做: experts live on different devices and tokens reach them
// by all-to-all; "Outrageously Large Neural Networks - 中文验证版", sections
// 计算设置 and 方法适配: each device keeps a share of the experts and the
// devices' batches are merged at the MoE layer).
//
// The exchange itself (NCCL all-to-all) is the caller's; the kernels here do
// the index work and the row copies around it:
//   ep_regroup   rows received from P ranks, ordered (source rank, local
//                expert, source slot order), into the expert-major order of
//                the merged batch: offsets per local expert, perm (merged
//                row -> received row) and its inverse
//   gather_rows  dst[i] = src[rows[i] / div]: packs the rows to send (x rows
//                in the sender's expert order) and returns expert outputs to
//                the received order
//   imp_cv2      CV^2 of an importance vector summed over the ranks
#include "moe_ep.h"
#include "moe_device.cuh"
#include "moe_launch.h"

namespace moe {
namespace {

constexpr int kEpMaxSegs = 4096;      // P * n_local
constexpr int kEpRowsPerBlock = 4096;

// Every block rebuilds the two segment tables from the P x nl count matrix
// (at most 4096 entries) and then places its share of the received rows.
//   src[m], m = q*nl + e: first received row of (source q, expert e)
//   dst[m]:               first merged row of the same segment
//                         = offsets[e] + sum over q' < q of c[q'][e]
__global__ void __launch_bounds__(1024) ep_regroup(int P, int nl, const int32_t *__restrict__ counts,
                                                   int64_t R, int32_t *__restrict__ offsets,
                                                   int32_t *__restrict__ perm,
                                                   int32_t *__restrict__ inv,
                                                   int32_t *__restrict__ err) {
    __shared__ int32_t src[kEpMaxSegs + 1];
    __shared__ int32_t dst[kEpMaxSegs];
    __shared__ int32_t ish[32];
    __shared__ int bad;
    const int M = P * nl;
    const int tid = threadIdx.x;
    if (tid == 0) bad = 0;
    __syncthreads();
    const int per = (M + 1023) / 1024;
    const int i0 = min(M, tid * per), i1 = min(M, i0 + per);
    // source-major order: m = q*nl + e
    int32_t sum = 0;
    for (int m = i0; m < i1; ++m) {
        const int32_t c = __ldg(counts + m);
        if (c < 0) bad = 1;
        sum += c;
    }
    int32_t total;
    int32_t run = block_exclusive_scan_1024(sum, ish, &total);
    for (int m = i0; m < i1; ++m) {
        src[m] = run;
        run += max(__ldg(counts + m), 0);
    }
    if (tid == 0) src[M] = total;
    // expert-major order: m' = e*P + q, the segment (q, e)
    sum = 0;
    for (int mp = i0; mp < i1; ++mp) {
        const int e = mp / P, q = mp - e * P;
        sum += max(__ldg(counts + q * nl + e), 0);
    }
    int32_t total2;
    run = block_exclusive_scan_1024(sum, ish, &total2);
    for (int mp = i0; mp < i1; ++mp) {
        const int e = mp / P, q = mp - e * P;
        dst[q * nl + e] = run;
        if (q == 0 && blockIdx.x == 0) offsets[e] = run;
        run += max(__ldg(counts + q * nl + e), 0);
    }
    __syncthreads();
    if (bad || static_cast<int64_t>(total) != R) {
        if (tid == 0 && blockIdx.x == 0) report(err, MOE_ERR_DEVICE, kSiteEpCounts, total);
        return;
    }
    if (tid == 0 && blockIdx.x == 0) offsets[nl] = total;
    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * kEpRowsPerBlock;
    const int64_t r1 = min(R, r0 + kEpRowsPerBlock);
    for (int64_t i = r0 + tid; i < r1; i += 1024) {
        // last segment whose first row is <= i (it is not empty)
        int lo = 0, hi = M;  // src[lo] <= i < src[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (src[mid] <= i) lo = mid; else hi = mid;
        }
        const int32_t j = dst[lo] + static_cast<int32_t>(i - src[lo]);
        perm[j] = static_cast<int32_t>(i);
        inv[i] = j;
    }
}

// One warp per row, 16-byte copies.  A row index outside [0, src_rows)
// (after the division) writes a zero row and records the error.
__global__ void __launch_bounds__(256) gather_rows(const uint4 *__restrict__ src, int64_t src_rows,
                                                   const int32_t *__restrict__ rows, int32_t div,
                                                   int64_t R, int vec, uint4 *__restrict__ dst,
                                                   int32_t *__restrict__ err) {
    const int64_t i = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (i >= R) return;
    const int32_t r = __ldg(rows + i);
    const int64_t s = r >= 0 ? r / div : -1;
    uint4 *o = dst + i * vec;
    if (s < 0 || s >= src_rows) {
        if (lane == 0) report(err, MOE_ERR_DEVICE, kSiteEpGather, static_cast<int32_t>(i));
        for (int c = lane; c < vec; c += 32) o[c] = make_uint4(0, 0, 0, 0);
        return;
    }
    const uint4 *p = src + s * vec;
    for (int c = lane; c < vec; c += 32) o[c] = __ldg(p + c);
}

// CV^2 = population variance / mean^2 of n values, the same fixed-order fp32
// tree sums as the dispatch's.
__global__ void __launch_bounds__(1024) imp_cv2(const float *__restrict__ imp, int n,
                                                float *__restrict__ cv2) {
    __shared__ float fsh[33];
    const int tid = threadIdx.x;
    float s = 0.0f;
    for (int e = tid; e < n; e += 1024) s += __ldg(imp + e);
    const float mean = block_sum_1024(s, fsh) / static_cast<float>(n);
    float q = 0.0f;
    for (int e = tid; e < n; e += 1024) {
        const float v = __ldg(imp + e) - mean;
        q = fmaf(v, v, q);
    }
    const float var = block_sum_1024(q, fsh) / static_cast<float>(n);
    if (tid == 0) cv2[0] = mean != 0.0f ? var / (mean * mean) : 0.0f;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

moe_status moe_ep_regroup(int32_t P, int32_t n_local, const int32_t *recv_counts, int64_t R,
                          int32_t *offsets_local, int32_t *perm_local, int32_t *inv_local,
                          int32_t *err, void *stream) {
    if (P <= 0 || n_local <= 0 || R < 0 || R > MOE_MAX_SLOTS) return MOE_ERR_INVALID_ARG;
    if (static_cast<int64_t>(P) * n_local > kEpMaxSegs) return MOE_ERR_UNSUPPORTED;
    if (!recv_counts || !offsets_local || !aligned16(recv_counts) || !aligned16(offsets_local))
        return MOE_ERR_INVALID_ARG;
    if (R > 0 && (!perm_local || !inv_local || !aligned16(perm_local) || !aligned16(inv_local)))
        return MOE_ERR_INVALID_ARG;
    const unsigned blocks =
        static_cast<unsigned>(R > 0 ? (R + kEpRowsPerBlock - 1) / kEpRowsPerBlock : 1);
    ep_regroup<<<blocks, 1024, 0, static_cast<cudaStream_t>(stream)>>>(
        P, n_local, recv_counts, R, offsets_local, perm_local, inv_local, err);
    return cuda_to_status(cudaGetLastError());
}

moe_status moe_gather_rows(const void *src, int64_t src_rows, const int32_t *rows, int32_t div,
                           int64_t R, int32_t d, int32_t dtype, void *dst, int32_t *err,
                           void *stream) {
    if (R < 0 || src_rows < 0 || d <= 0 || div <= 0) return MOE_ERR_INVALID_ARG;
    if (dtype != MOE_F32 && dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
    const int64_t row_bytes = static_cast<int64_t>(d) * (dtype == MOE_BF16 ? 2 : 4);
    if (row_bytes % 16 != 0) return MOE_ERR_UNSUPPORTED;
    if (R == 0) return MOE_OK;
    if (!src || !rows || !dst || !aligned16(src) || !aligned16(rows) || !aligned16(dst))
        return MOE_ERR_INVALID_ARG;
    const int64_t threads = R * 32;
    gather_rows<<<static_cast<unsigned>((threads + 255) / 256), 256, 0,
                  static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4 *>(src), src_rows, rows, div, R, static_cast<int>(row_bytes / 16),
        static_cast<uint4 *>(dst), err);
    return cuda_to_status(cudaGetLastError());
}

moe_status moe_importance_cv2(const float *importance, int32_t n, float *cv2, void *stream) {
    if (n <= 0 || !importance || !cv2 || !aligned16(importance) || !aligned16(cv2))
        return MOE_ERR_INVALID_ARG;
    imp_cv2<<<1, 1024, 0, static_cast<cudaStream_t>(stream)>>>(importance, n, cv2);
    return cuda_to_status(cudaGetLastError());
}

}  // extern "C"

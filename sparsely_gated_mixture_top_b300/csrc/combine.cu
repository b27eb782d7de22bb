// combine.cu -- y[t] = sum_j G[t,j] * Y_slot[inv_perm[t*k+j]]
// ("MoE:稀疏门控混合专家", section 二: y = sum_i G(x)_i E_i(x), only the selected
// experts contributing).  One warp per token, 16-byte vector loads of the
// expert rows (eight in flight per lane), fp32 accumulation in the fixed slot
// order j = 0..k-1 and one rounding to the output type.  The warps stride over
// the tokens and look up the next token's rows while summing the current one.
#include <algorithm>

#include "moe_device.cuh"
#include "moe_launch.h"

namespace moe {

namespace {

// 16-byte pieces of a row and their conversion to fp32.
template <typename T>
struct Vec;
template <>
struct Vec<__nv_bfloat16> {
    static constexpr int N = 8;  // elements per 16-byte piece
    __device__ static void to_f(const uint4 &u, float (&v)[8]) {
        const __nv_bfloat162 *b = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(b[i]);
            v[2 * i] = f.x;
            v[2 * i + 1] = f.y;
        }
    }
    __device__ static uint4 from_f(const float (&v)[8]) {
        uint4 u;
        u.x = pack_bf16x2(v[0], v[1]);
        u.y = pack_bf16x2(v[2], v[3]);
        u.z = pack_bf16x2(v[4], v[5]);
        u.w = pack_bf16x2(v[6], v[7]);
        return u;
    }
};
template <>
struct Vec<float> {
    static constexpr int N = 4;
    __device__ static void to_f(const uint4 &u, float (&v)[4]) {
        v[0] = __uint_as_float(u.x);
        v[1] = __uint_as_float(u.y);
        v[2] = __uint_as_float(u.z);
        v[3] = __uint_as_float(u.w);
    }
    __device__ static uint4 from_f(const float (&v)[4]) {
        return make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]),
                          __float_as_uint(v[3]));
    }
};

// A token's expert rows (checked against S) and gate weights.
template <int KM>
__device__ __forceinline__ void combine_meta(int64_t t, int k, int64_t S, int lane,
                                             const int32_t *__restrict__ inv_perm,
                                             const float *__restrict__ G, int32_t *err,
                                             int32_t (&rows)[KM], float (&w)[KM]) {
#pragma unroll
    for (int j = 0; j < KM; ++j) {
        rows[j] = -1;
        w[j] = 0.0f;
        if (j < k) {
            int32_t row = __ldg(inv_perm + t * k + j);
            if (row >= S) {
                if (lane == 0) report(err, MOE_ERR_DEVICE, kSiteCombineRow, static_cast<int32_t>(t));
                row = -1;
            }
            rows[j] = row;
            w[j] = __ldg(G + t * k + j);
        }
    }
}

// Warps stride over the tokens (a grid of a few blocks per SM); a warp reads
// the next token's rows and weights before it sums the current one, so that
// lookup overlaps the current token's row loads.  For every pair of 32-piece
// column spans, all of the (up to four at a time) expert rows' pieces are
// requested before any is summed, so each lane keeps eight 16-byte loads in
// flight; the sum runs in the fixed slot order j = 0..k-1 in fp32 and is
// rounded once.
template <typename T, int KM>
__global__ void __launch_bounds__(256, KM <= 4 ? 3 : 2)
    combine_kernel(const T *__restrict__ Y, const int32_t *__restrict__ inv_perm,
                   const float *__restrict__ G, int64_t T_, int d, int k, int64_t S,
                   T *__restrict__ y, int32_t *err) {
    constexpr int V = Vec<T>::N;
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * 8;
    int64_t t = static_cast<int64_t>(blockIdx.x) * 8 + threadIdx.x / 32;
    if (t >= T_) return;
    int32_t rows[KM];
    float w[KM];
    combine_meta<KM>(t, k, S, lane, inv_perm, G, err, rows, w);
    const int pieces = d / V;  // 16-byte pieces per row
    for (; t < T_; t += nwarps) {
        int32_t nrows[KM];
        float nw[KM];
        if (t + nwarps < T_) combine_meta<KM>(t + nwarps, k, S, lane, inv_perm, G, err, nrows, nw);
        for (int p0 = lane; p0 < pieces; p0 += 64) {
            const int p1 = p0 + 32;
            const bool two = p1 < pieces;
            float acc0[V], acc1[V];
#pragma unroll
            for (int i = 0; i < V; ++i) acc0[i] = acc1[i] = 0.0f;
#pragma unroll
            for (int j0 = 0; j0 < KM; j0 += 4) {
                if (j0 >= k) break;
                uint4 u[4][2];
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const int j = j0 + jj;
                    u[jj][0] = u[jj][1] = make_uint4(0, 0, 0, 0);
                    if (j < k && rows[j] >= 0) {
                        const uint4 *src =
                            reinterpret_cast<const uint4 *>(Y + static_cast<int64_t>(rows[j]) * d);
                        u[jj][0] = __ldg(src + p0);
                        if (two) u[jj][1] = __ldg(src + p1);
                    }
                }
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const int j = j0 + jj;
                    if (j < k && rows[j] >= 0) {
                        float a[V], b[V];
                        Vec<T>::to_f(u[jj][0], a);
                        Vec<T>::to_f(u[jj][1], b);
#pragma unroll
                        for (int i = 0; i < V; ++i) {
                            acc0[i] = fmaf(w[j], a[i], acc0[i]);
                            acc1[i] = fmaf(w[j], b[i], acc1[i]);
                        }
                    }
                }
            }
            uint4 *dst = reinterpret_cast<uint4 *>(y + t * d);
            dst[p0] = Vec<T>::from_f(acc0);
            if (two) dst[p1] = Vec<T>::from_f(acc1);
        }
#pragma unroll
        for (int j = 0; j < KM; ++j) {
            rows[j] = nrows[j];
            w[j] = nw[j];
        }
    }
}

}  // namespace

cudaError_t launch_combine(const moe_shape &s, const void *Y_slot, const int32_t *inv_perm,
                           const float *G, void *y, int32_t *err, cudaStream_t st) {
    if (s.T == 0) return cudaSuccess;
    // Blocks of 8 warps, a few per SM, striding over the tokens.
    const int64_t per_sm = s.k <= 4 ? 3 : 2;
    const int64_t need = (s.T + 7) / 8;
    const unsigned blocks = static_cast<unsigned>(std::min<int64_t>(need, sm_count() * per_sm));
    const int64_t S = slots(s);
    if (s.dtype == MOE_BF16) {
        const auto *Yb = static_cast<const __nv_bfloat16 *>(Y_slot);
        auto *yb = static_cast<__nv_bfloat16 *>(y);
        if (s.k <= 4)
            return launch_pdl(combine_kernel<__nv_bfloat16, 4>, dim3(blocks), dim3(256), 0, st, Yb, inv_perm, G, s.T, s.d, s.k, S, yb, err);
        else
            return launch_pdl(combine_kernel<__nv_bfloat16, MOE_MAX_K>, dim3(blocks), dim3(256), 0, st, Yb, inv_perm, G, s.T, s.d, s.k, S, yb, err);
    } else {
        const auto *Yf = static_cast<const float *>(Y_slot);
        auto *yf = static_cast<float *>(y);
        if (s.k <= 4)
            return launch_pdl(combine_kernel<float, 4>, dim3(blocks), dim3(256), 0, st, Yf, inv_perm, G, s.T, s.d, s.k, S, yf, err);
        else
            return launch_pdl(combine_kernel<float, MOE_MAX_K>, dim3(blocks), dim3(256), 0, st, Yf, inv_perm, G, s.T, s.d, s.k, S, yf, err);
    }
    return cudaGetLastError();
}

}  // namespace moe

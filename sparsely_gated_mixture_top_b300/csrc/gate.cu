// gate.cu -- noisy top-k gating ("MoE:稀疏门控混合专家", sections 三 and 四),
// CUDA-core path for fp32 inputs (bf16 shapes take gate_tc.cu).
//
// Two kernels:
//   gate_scores_simt  H[t,c] = x[t].Wg[:,c] (+ bg[c]) + eps[t,c] * softplus(x[t].Wn[:,c])
//                     a tiled fp32 SIMT GEMM over both gate matrices at once, with the
//                     noise epilogue fused; every product and sum in fp32, sums in
//                     increasing d order.
//   gate_select       one warp per token: register top-k with warp shuffles
//                     (KeepTopK; ties to the lower index; descending order), then the
//                     softmax over the k survivors.  Hierarchical gating runs it twice:
//                     over the G group columns, then over each chosen group's m columns.
#include "moe_device.cuh"
#include "moe_launch.h"

#include <float.h>
#include <limits.h>

namespace moe {

namespace {

constexpr int kBT = 64;  // tokens per tile
constexpr int kBC = 64;  // score columns per tile
constexpr int kBK = 16;  // d per step

template <typename XT>
__global__ void __launch_bounds__(256) gate_scores_simt(const XT *__restrict__ x,
                                                        const float *__restrict__ Wg,
                                                        const float *__restrict__ Wn,
                                                        const float *__restrict__ bg,
                                                        const float *__restrict__ eps, int64_t T,
                                                        int d, int C, int noisy,
                                                        float *__restrict__ H) {
    __shared__ float xs[kBK][kBT + 4];
    __shared__ float gs[kBK][kBC + 4];
    __shared__ float ns[kBK][kBC + 4];
    const int tid = threadIdx.x;
    const int tx = tid % 16, ty = tid / 16;
    const int64_t t0 = static_cast<int64_t>(blockIdx.y) * kBT;
    const int c0 = blockIdx.x * kBC;
    float accg[4][4] = {}, accn[4][4] = {};
    for (int k0 = 0; k0 < d; k0 += kBK) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int e = tid + q * 256;      // 0..1023
            const int r = e / kBK, kk = e % kBK;  // x tile: 64 tokens x 16 d
            const int64_t t = t0 + r;
            xs[kk][r] = (t < T) ? to_f(x[t * d + k0 + kk]) : 0.0f;
            const int wr = e / kBC, wc = e % kBC;  // W tiles: 16 d x 64 columns
            const int c = c0 + wc;
            const int64_t off = static_cast<int64_t>(k0 + wr) * C + c;
            gs[wr][wc] = (c < C) ? Wg[off] : 0.0f;
            ns[wr][wc] = (c < C && noisy) ? Wn[off] : 0.0f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < kBK; ++kk) {
            float xv[4], gv[4], nv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                xv[i] = xs[kk][ty * 4 + i];
                gv[i] = gs[kk][tx * 4 + i];
                nv[i] = ns[kk][tx * 4 + i];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    accg[i][j] = fmaf(xv[i], gv[j], accg[i][j]);
                    accn[i][j] = fmaf(xv[i], nv[j], accn[i][j]);
                }
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t t = t0 + ty * 4 + i;
        if (t >= T) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int c = c0 + tx * 4 + j;
            if (c >= C) continue;
            float clean = accg[i][j] + (bg ? bg[c] : 0.0f);
            float hv = noisy ? clean + eps[t * C + c] * softplus_f(accn[i][j]) : clean;
            H[t * C + c] = hv;
        }
    }
}

// (a, ia) ranks before (b, ib): larger value first, equal values by lower index.
__device__ __forceinline__ bool better(float a, int ia, float b, int ib) {
    return a > b || (a == b && ia < ib);
}

// Top-kk (kk <= KM) of row[0..m) for one warp; result in descending order,
// identical in every lane.
template <int KM>
__device__ __forceinline__ void warp_top_k(const float *__restrict__ row, int m, int kk,
                                           float (&v)[KM], int (&ix)[KM]) {
    const int lane = threadIdx.x & 31;
    float lv[KM];
    int li[KM];
#pragma unroll
    for (int q = 0; q < KM; ++q) {
        lv[q] = -INFINITY;
        li[q] = INT_MAX;
    }
    for (int c = lane; c < m; c += 32) {
        float cv = row[c];
        int ci = c;
#pragma unroll
        for (int p = 0; p < KM; ++p) {
            if (better(cv, ci, lv[p], li[p])) {
                const float tv = lv[p];
                const int ti = li[p];
                lv[p] = cv;
                li[p] = ci;
                cv = tv;
                ci = ti;
            }
        }
    }
#pragma unroll
    for (int r = 0; r < KM; ++r) {
        v[r] = -INFINITY;
        ix[r] = INT_MAX;
        if (r < kk) {
            float bv = lv[0];
            int bi = li[0];
#pragma unroll
            for (int s = 16; s > 0; s >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, s);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, s);
                if (better(ov, oi, bv, bi)) {
                    bv = ov;
                    bi = oi;
                }
            }
            v[r] = bv;
            ix[r] = bi;
            if (li[0] == bi) {  // this lane's head won: pop it
#pragma unroll
                for (int p = 0; p + 1 < KM; ++p) {
                    lv[p] = lv[p + 1];
                    li[p] = li[p + 1];
                }
                lv[KM - 1] = -INFINITY;
                li[KM - 1] = INT_MAX;
            }
        }
    }
}

// Softmax over the kk survivors (the KeepTopK'd entries are e^-inf = 0).
template <int KM>
__device__ __forceinline__ void softmax_k(const float (&v)[KM], int kk, float (&g)[KM]) {
    const float mx = v[0];
    float s = 0.0f;
#pragma unroll
    for (int r = 0; r < KM; ++r) {
        g[r] = 0.0f;
        if (r < kk) {
            g[r] = expf(v[r] - mx);
            s += g[r];
        }
    }
    const float inv = 1.0f / s;
#pragma unroll
    for (int r = 0; r < KM; ++r) g[r] *= inv;
}

template <int KM>
__global__ void __launch_bounds__(256) gate_select(const float *__restrict__ H, int64_t T, int C,
                                                   int n, int k, int groups, int k_groups,
                                                   int32_t *__restrict__ idx,
                                                   float *__restrict__ G) {
    const int64_t t = static_cast<int64_t>(blockIdx.x) * 8 + threadIdx.x / 32;
    if (t >= T) return;
    const int lane = threadIdx.x & 31;
    const float *row = H + t * C;
    if (groups == 0) {
        float v[KM], g[KM];
        int ix[KM];
        warp_top_k<KM>(row, n, k, v, ix);
        softmax_k<KM>(v, k, g);
        if (lane == 0) {
#pragma unroll
            for (int r = 0; r < KM; ++r)
                if (r < k) {
                    idx[t * k + r] = ix[r];
                    G[t * k + r] = g[r];
                }
        }
        return;
    }
    const int m = n / groups;
    const int k_inner = k / k_groups;
    float gv[KM], gp[KM];
    int gi[KM];
    warp_top_k<KM>(row, groups, k_groups, gv, gi);
    softmax_k<KM>(gv, k_groups, gp);
#pragma unroll
    for (int r = 0; r < KM; ++r) {
        if (r >= k_groups) break;
        const int g = gi[r];
        float ev[KM], ew[KM];
        int ei[KM];
        warp_top_k<KM>(row + groups + static_cast<int64_t>(g) * m, m, k_inner, ev, ei);
        softmax_k<KM>(ev, k_inner, ew);
        if (lane == 0) {
#pragma unroll
            for (int q = 0; q < KM; ++q)
                if (q < k_inner) {
                    idx[t * k + r * k_inner + q] = g * m + ei[q];
                    G[t * k + r * k_inner + q] = gp[r] * ew[q];
                }
        }
    }
}

template <int KM>
void launch_select(const float *H, const moe_shape &s, int C, int32_t *idx, float *G,
                   cudaStream_t st) {
    const unsigned blocks = static_cast<unsigned>((s.T + 7) / 8);
    gate_select<KM><<<blocks, 256, 0, st>>>(H, s.T, C, s.n, s.k, s.groups, s.k_groups, idx, G);
}

}  // namespace

cudaError_t launch_gate(const moe_shape &s, const void *x, const float *Wg, const float *Wn,
                        const float *bg, const float *eps, int32_t *idx, float *G, void *ws,
                        const WsLayout &L, cudaStream_t st) {
    if (gate_tc_supported(s)) return launch_gate_tc(s, x, Wg, Wn, bg, eps, idx, G, ws, L, st);
    float *Hbuf = ws_ptr<float>(ws, L.scores);
    const int C = gate_cols(s);
    const int noisy = (s.noisy && eps != nullptr) ? 1 : 0;
    dim3 grid(static_cast<unsigned>((C + kBC - 1) / kBC), static_cast<unsigned>((s.T + kBT - 1) / kBT));
    if (s.dtype == MOE_BF16)
        gate_scores_simt<__nv_bfloat16><<<grid, 256, 0, st>>>(
            static_cast<const __nv_bfloat16 *>(x), Wg, Wn, bg, eps, s.T, s.d, C, noisy, Hbuf);
    else
        gate_scores_simt<float><<<grid, 256, 0, st>>>(static_cast<const float *>(x), Wg, Wn, bg,
                                                      eps, s.T, s.d, C, noisy, Hbuf);
    const int kmax = s.k;  // k_groups and k/k_groups are <= k
    if (kmax <= 1)
        launch_select<1>(Hbuf, s, C, idx, G, st);
    else if (kmax <= 2)
        launch_select<2>(Hbuf, s, C, idx, G, st);
    else if (kmax <= 4)
        launch_select<4>(Hbuf, s, C, idx, G, st);
    else if (kmax <= 8)
        launch_select<8>(Hbuf, s, C, idx, G, st);
    else
        launch_select<16>(Hbuf, s, C, idx, G, st);
    return cudaGetLastError();
}

}  // namespace moe

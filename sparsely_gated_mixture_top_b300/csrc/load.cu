// load.cu -- the load estimate of the flat noisy gate: the smooth per-expert
// load that the load loss balances ("Outrageously Large Neural Networks -
// 中文验证版", section 方法适配: an importance loss and a load loss keep the
// samples spread over the experts; the estimate follows the paper's
// load-balancing appendix, the pages being cut off before its formula).
//
// For token t and expert i, the probability that i stays among the k best
// when only its own noise is redrawn:
//   P(t, i) = Phi((c_i - thr_i) / s_i),  c = x.W_g (+ b_g),  s = softplus(x.W_noise),
//   thr_i = the k-th largest noisy score H of the other experts
//         = H_(k+1) when i is among the k kept, H_(k) otherwise,
// load[i] = sum_t P(t, i) and CV^2 = population variance / mean^2 of load.
// The tensor-core gate (load mode) writes c, s and H_(k), H_(k+1); here
//   load_accumulate  one thread per expert column, the tokens of one
//                    64-token chunk in order: P in fp32 (erfcf), sums in fp64
//   load_colsum      one thread per expert: the chunk sums in chunk order
//   load_cv2         one block: CV^2 of the load vector
// so the same inputs always give the same bits.
#include "moe_device.cuh"
#include "moe_launch.h"

namespace moe {

namespace {

constexpr int kLoadChunk = 64;  // tokens per partial sum

__global__ void __launch_bounds__(256) load_accumulate(const float *__restrict__ c,
                                                       const float *__restrict__ s,
                                                       const float *__restrict__ vk,
                                                       const int32_t *__restrict__ idx, int64_t T,
                                                       int n, int k,
                                                       double *__restrict__ part) {
    const int col = blockIdx.x * 256 + threadIdx.x;
    const int64_t t0 = static_cast<int64_t>(blockIdx.y) * kLoadChunk;
    if (col >= n) return;
    const int64_t t1 = t0 + kLoadChunk < T ? t0 + kLoadChunk : T;
    double acc = 0.0;
    for (int64_t t = t0; t < t1; ++t) {
        bool member = false;
        for (int q = 0; q < k; ++q) member |= idx[t * k + q] == col;
        const float thr = member ? vk[2 * t + 1] : vk[2 * t];
        const float cv = c[t * n + col], sv = s[t * n + col];
        float p;
        if (thr == -INFINITY) {
            p = 1.0f;
        } else if (sv > 0.0f) {
            p = 0.5f * erfcf(-(cv - thr) / (sv * 1.41421356f));
        } else {  // no noise left: the hard decision
            p = cv > thr ? 1.0f : (cv == thr ? 0.5f : 0.0f);
        }
        acc += static_cast<double>(p);
    }
    part[static_cast<int64_t>(blockIdx.y) * n + col] = acc;
}

// Sum over the 256 threads in a fixed order (shuffle tree, then warps in order).
__device__ double block_sum_256(double v, double *sh) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = v;
    __syncthreads();
    double r = 0.0;
#pragma unroll
    for (int w = 0; w < 8; ++w) r += sh[w];
    __syncthreads();
    return r;
}

// One thread per expert: the chunk partials in chunk order.
__global__ void __launch_bounds__(256) load_colsum(const double *__restrict__ part, int chunks,
                                                   int n, double *__restrict__ load64,
                                                   float *__restrict__ load) {
    const int e = blockIdx.x * 256 + threadIdx.x;
    if (e >= n) return;
    double acc = 0.0;
    for (int ch = 0; ch < chunks; ++ch) acc += part[static_cast<int64_t>(ch) * n + e];
    load64[e] = acc;
    load[e] = static_cast<float>(acc);
}

// One block: CV^2 = population variance / mean^2 of the load vector.
__global__ void __launch_bounds__(256) load_cv2(const double *__restrict__ load64, int n,
                                                float *__restrict__ cv2) {
    __shared__ double sh[8];
    double s = 0.0;
    for (int e = threadIdx.x; e < n; e += 256) s += load64[e];
    const double mean = block_sum_256(s, sh) / n;
    double q = 0.0;
    for (int e = threadIdx.x; e < n; e += 256) q += (load64[e] - mean) * (load64[e] - mean);
    const double var = block_sum_256(q, sh) / n;
    if (threadIdx.x == 0) cv2[0] = mean != 0.0 ? static_cast<float>(var / (mean * mean)) : 0.0f;
}

}  // namespace

LoadLayout load_layout(const moe_shape &s) {
    LoadLayout L;
    const size_t T = static_cast<size_t>(s.T), n = static_cast<size_t>(s.n);
    const size_t chunks = (T + kLoadChunk - 1) / kLoadChunk;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = align_up(o + bytes, 256);
        return at;
    };
    L.c = take(T * n * 4);
    L.s = take(T * n * 4);
    L.vk = take(T * 2 * 4);
    L.part = take(chunks * n * 8);
    L.load64 = take(n * 8);
    L.chunks = static_cast<int>(chunks);
    L.total = o;
    return L;
}

cudaError_t launch_load(const moe_shape &s, const int32_t *idx, void *lws, const LoadLayout &L,
                        float *load, float *cv2, cudaStream_t st) {
    if (s.T == 0) {
        cudaMemsetAsync(load, 0, sizeof(float) * s.n, st);
        cudaMemsetAsync(cv2, 0, sizeof(float), st);
        return cudaGetLastError();
    }
    const float *c = ws_ptr<float>(lws, L.c);
    const float *sp = ws_ptr<float>(lws, L.s);
    const float *vk = ws_ptr<float>(lws, L.vk);
    double *part = ws_ptr<double>(lws, L.part);
    load_accumulate<<<dim3((s.n + 255) / 256, L.chunks), 256, 0, st>>>(c, sp, vk, idx, s.T, s.n, s.k,
                                                                      part);
    double *load64 = ws_ptr<double>(lws, L.load64);
    load_colsum<<<(s.n + 255) / 256, 256, 0, st>>>(part, L.chunks, s.n, load64, load);
    load_cv2<<<1, 256, 0, st>>>(load64, s.n, cv2);
    return cudaGetLastError();
}

}  // namespace moe

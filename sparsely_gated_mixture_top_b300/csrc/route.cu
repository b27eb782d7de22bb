// route.cu -- dispatch of the S = T*k slots to expert-contiguous rows.
//
// The pages' conditional computation ("MoE:稀疏门控混合专家", section 二: experts
// with weight 0 are not computed) needs each expert's rows gathered together;
// each expert then sees about k*b/n rows ("Outrageously Large Neural Networks -
// 中文验证版", section 瓶颈).  This is a deterministic counting sort:
//
//   route_rank      per chunk of 1024 slots: the rank of each slot among the
//                   earlier slots of its chunk with the same expert (warp
//                   __match_any + warps taken in order), the chunk's
//                   per-expert counts and gate-weight sums (each warp's group
//                   of <= 32 slots in fp32, the groups in fp64, slot order);
//                   route_rank_warps gives the same for n <= 512 from a
//                   [warp][expert] table instead of 32 barrier rounds
//   route_colscan   per expert, an exclusive scan of the counts down the
//                   chunks (chunk bases), the expert's count and its
//                   importance (chunk partials summed in chunk order)
//   route_finish    one block: exclusive scan of the counts over the experts
//                   (offsets), importance in fp32, population variance /
//                   mean^2 of the importance vector (CV^2)
//   route_scatter   row = offsets[e] + chunk base + local rank: perm, inv_perm
//
// The permutation is stable and every sum has a fixed order, so the same idx
// and G always give the same outputs bit for bit.
#include "moe_device.cuh"
#include "moe_launch.h"

namespace moe {

namespace {

__global__ void __launch_bounds__(1024) route_rank(const int32_t *__restrict__ idx,
                                                   const float *__restrict__ G, int64_t S, int n,
                                                   int32_t *__restrict__ local_rank,
                                                   int32_t *__restrict__ chunk,
                                                   double *__restrict__ chunk_imp, int32_t *err) {
    extern __shared__ __align__(8) unsigned char route_sh[];
    double *imp = reinterpret_cast<double *>(route_sh);              // [n]
    int32_t *cnt = reinterpret_cast<int32_t *>(route_sh + 8 * n);     // [n]
    __shared__ int32_t base_sh[32][32];
    for (int e = threadIdx.x; e < n; e += blockDim.x) {
        cnt[e] = 0;
        imp[e] = 0.0;
    }
    __syncthreads();
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int64_t s = static_cast<int64_t>(blockIdx.x) * kRouteChunk + threadIdx.x;
    int e = -1;
    float g = 0.0f;
    if (s < S) {
        e = idx[s];
        if (e < 0 || e >= n) {
            report(err, MOE_ERR_DEVICE, kSiteRouteIdx, static_cast<int32_t>(s));
            e = -1;
        } else {
            g = G[s];
        }
    }
    const unsigned mask = __match_any_sync(0xffffffffu, e);
    const int leader = __ffs(mask) - 1;
    const int rank_in_warp = __popc(mask & ((1u << lane) - 1u));
    // Gate weight of this lane's expert group (at most 32 slots) summed in
    // lane order in fp32; the groups are then accumulated in fp64.
    float seg = 0.0f;
#pragma unroll
    for (int src = 0; src < 32; ++src) {
        const float v = __shfl_sync(0xffffffffu, g, src);
        if ((mask >> src) & 1u) seg += v;
    }
    // Warps take their turn in slot order, so ranks and importance sums
    // follow slot order.
    for (int w = 0; w < 32; ++w) {
        if (warp == w && lane == leader && e >= 0) {
            base_sh[w][lane] = cnt[e];
            cnt[e] += __popc(mask);
            imp[e] += static_cast<double>(seg);
        }
        __syncthreads();
    }
    if (e >= 0) local_rank[s] = base_sh[warp][leader] + rank_in_warp;
    int32_t *row = chunk + static_cast<int64_t>(blockIdx.x) * n;
    double *irow = chunk_imp + static_cast<int64_t>(blockIdx.x) * n;
    for (int ee = threadIdx.x; ee < n; ee += blockDim.x) {
        row[ee] = cnt[ee];
        irow[ee] = imp[ee];
    }
}

// Block (32 x 32): 32 experts (x) by 32 chunk segments (y).  Chunk counts
// become chunk bases (exclusive scan down the chunks); the expert's count
// and importance (fp64, chunk order) are the column totals.
// route_rank for n <= kRankWarpsMaxN: the same outputs without the 32
// barrier rounds.  Each warp's leaders write their group's count and fp32
// gate-weight sum to a [32 warps][n] table; one thread per expert then walks
// the warps in order (exclusive scan of the counts, fp64 sum of the groups,
// the same order as route_rank) and every slot reads its warp's base.
constexpr int kRankWarpsMaxN = 512;

__global__ void __launch_bounds__(1024) route_rank_warps(const int32_t *__restrict__ idx,
                                                         const float *__restrict__ G, int64_t S,
                                                         int n, int32_t *__restrict__ local_rank,
                                                         int32_t *__restrict__ chunk,
                                                         double *__restrict__ chunk_imp,
                                                         int32_t *err) {
    extern __shared__ __align__(8) unsigned char route_sh[];
    int32_t *wc = reinterpret_cast<int32_t *>(route_sh);           // [32][n] counts, then bases
    float *wsum = reinterpret_cast<float *>(route_sh + 128 * n);    // [32][n] group sums
    for (int i = threadIdx.x; i < 32 * n; i += blockDim.x) {
        wc[i] = 0;
        wsum[i] = 0.0f;
    }
    __syncthreads();
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int64_t s = static_cast<int64_t>(blockIdx.x) * kRouteChunk + threadIdx.x;
    int e = -1;
    float g = 0.0f;
    if (s < S) {
        e = idx[s];
        if (e < 0 || e >= n) {
            report(err, MOE_ERR_DEVICE, kSiteRouteIdx, static_cast<int32_t>(s));
            e = -1;
        } else {
            g = G[s];
        }
    }
    const unsigned mask = __match_any_sync(0xffffffffu, e);
    const int leader = __ffs(mask) - 1;
    const int rank_in_warp = __popc(mask & ((1u << lane) - 1u));
    float seg = 0.0f;
#pragma unroll
    for (int src = 0; src < 32; ++src) {
        const float v = __shfl_sync(0xffffffffu, g, src);
        if ((mask >> src) & 1u) seg += v;
    }
    if (lane == leader && e >= 0) {
        wc[warp * n + e] = __popc(mask);
        wsum[warp * n + e] = seg;
    }
    __syncthreads();
    int32_t *row = chunk + static_cast<int64_t>(blockIdx.x) * n;
    double *irow = chunk_imp + static_cast<int64_t>(blockIdx.x) * n;
    for (int ee = threadIdx.x; ee < n; ee += blockDim.x) {
        int32_t run = 0;
        double imp = 0.0;
        for (int w = 0; w < 32; ++w) {
            const int32_t c = wc[w * n + ee];
            wc[w * n + ee] = run;
            run += c;
            if (c) imp += static_cast<double>(wsum[w * n + ee]);
        }
        row[ee] = run;
        irow[ee] = imp;
    }
    __syncthreads();
    if (e >= 0) local_rank[s] = wc[warp * n + e] + rank_in_warp;
}

__global__ void __launch_bounds__(1024) route_colscan(int32_t *__restrict__ chunk,
                                                      const double *__restrict__ chunk_imp,
                                                      int chunks, int n, int32_t *__restrict__ counts,
                                                      double *__restrict__ imp64) {
    __shared__ int32_t part[32][33];
    __shared__ double ipart[32][33];
    const int tx = threadIdx.x, ty = threadIdx.y;
    const int e = blockIdx.x * 32 + tx;
    const int seg = (chunks + 31) / 32;
    const int b0 = ty * seg, b1 = min(chunks, b0 + seg);
    int32_t sum = 0;
    double isum = 0.0;
    if (e < n)
        for (int b = b0; b < b1; ++b) {
            sum += chunk[static_cast<int64_t>(b) * n + e];
            isum += chunk_imp[static_cast<int64_t>(b) * n + e];
        }
    part[ty][tx] = sum;
    ipart[ty][tx] = isum;
    __syncthreads();
    if (ty == 0) {
        int32_t run = 0;
        double irun = 0.0;
        for (int y = 0; y < 32; ++y) {
            const int32_t v = part[y][tx];
            part[y][tx] = run;
            run += v;
            irun += ipart[y][tx];
        }
        if (e < n) {
            counts[e] = run;
            imp64[e] = irun;
        }
    }
    __syncthreads();
    if (e < n) {
        int32_t run = part[ty][tx];
        for (int b = b0; b < b1; ++b) {
            const int64_t at = static_cast<int64_t>(b) * n + e;
            const int32_t v = chunk[at];
            chunk[at] = run;
            run += v;
        }
    }
}

// Sum over the 256 threads of the block in a fixed order (warp shuffle tree,
// then the 8 warp sums in warp order); every thread gets the result.
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

// One block of 256 threads: offsets = exclusive scan of counts (offsets[n] =
// total), importance in fp32, and CV^2 = population variance / mean^2.
__global__ void __launch_bounds__(256) route_finish(const int32_t *__restrict__ counts,
                                                    const double *__restrict__ imp64, int n,
                                                    int32_t *__restrict__ offsets,
                                                    float *__restrict__ importance,
                                                    float *__restrict__ cv2) {
    __shared__ int32_t wsum[8];
    __shared__ double sh[8];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int per = (n + 255) / 256;
    const int i0 = threadIdx.x * per, i1 = min(n, i0 + per);
    int32_t sum = 0;
    for (int i = i0; i < i1; ++i) sum += counts[i];
    // exclusive scan of the per-thread sums: warp shuffles, then the warps
    int32_t inc = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t v = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += v;
    }
    if (lane == 31) wsum[warp] = inc;
    __syncthreads();
    int32_t base = 0;
    for (int w = 0; w < warp; ++w) base += wsum[w];
    int32_t run = base + inc - sum;
    for (int i = i0; i < i1; ++i) {
        offsets[i] = run;
        run += counts[i];
    }
    if (threadIdx.x == 255) offsets[n] = base + inc;
    double s = 0.0;
    for (int e = threadIdx.x; e < n; e += 256) {
        s += imp64[e];
        importance[e] = static_cast<float>(imp64[e]);
    }
    const double mean = block_sum_256(s, sh) / n;
    double q = 0.0;
    for (int e = threadIdx.x; e < n; e += 256) q += (imp64[e] - mean) * (imp64[e] - mean);
    const double var = block_sum_256(q, sh) / n;
    if (threadIdx.x == 0) cv2[0] = mean != 0.0 ? static_cast<float>(var / (mean * mean)) : 0.0f;
}

__global__ void route_scatter(const int32_t *__restrict__ idx, int64_t S, int n,
                              const int32_t *__restrict__ offsets,
                              const int32_t *__restrict__ chunk,
                              const int32_t *__restrict__ local_rank, int32_t *__restrict__ perm,
                              int32_t *__restrict__ inv_perm) {
    const int64_t s = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (s >= S) return;
    const int e = idx[s];
    if (e < 0 || e >= n) {
        inv_perm[s] = -1;
    } else {
        const int32_t row = offsets[e] + chunk[(s / kRouteChunk) * n + e] + local_rank[s];
        perm[row] = static_cast<int32_t>(s);
        inv_perm[s] = row;
    }
    if (s >= offsets[n]) perm[s] = -1;  // rows left empty by invalid slots
}

}  // namespace

cudaError_t launch_dispatch(const moe_shape &s, const int32_t *idx, const float *G,
                            int32_t *counts, int32_t *offsets, int32_t *perm, int32_t *inv_perm,
                            float *importance, float *cv2, void *ws, const WsLayout &L,
                            cudaStream_t st) {
    const int64_t S = slots(s);
    const int n = s.n;
    int32_t *err = ws_ptr<int32_t>(ws, 0);
    if (S == 0) {
        cudaMemsetAsync(counts, 0, sizeof(int32_t) * n, st);
        cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (n + 1), st);
        cudaMemsetAsync(importance, 0, sizeof(float) * n, st);
        cudaMemsetAsync(cv2, 0, sizeof(float), st);
        return cudaGetLastError();
    }
    const int chunks = static_cast<int>((S + kRouteChunk - 1) / kRouteChunk);
    int32_t *local_rank = ws_ptr<int32_t>(ws, L.local_rank);
    int32_t *chunk = ws_ptr<int32_t>(ws, L.chunk);
    double *chunk_imp = ws_ptr<double>(ws, L.chunk_imp);
    double *imp64 = ws_ptr<double>(ws, L.imp64);
    // Dynamic shared memory above the default 48 KB needs an opt-in, which
    // belongs to the current device's context: it is set before each launch.
    if (n <= kRankWarpsMaxN) {
        const size_t smem = 256 * static_cast<size_t>(n);  // [32][n] counts and sums
        if (smem > 48 * 1024) {
            cudaError_t e = cudaFuncSetAttribute(
                route_rank_warps, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
            if (e != cudaSuccess) return e;
        }
        route_rank_warps<<<chunks, 1024, smem, st>>>(idx, G, S, n, local_rank, chunk, chunk_imp,
                                                     err);
    } else {
        const size_t smem = 12 * static_cast<size_t>(n);  // n doubles and n ints (+4 KB static)
        if (smem + 4096 > 48 * 1024) {
            cudaError_t e = cudaFuncSetAttribute(
                route_rank, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
            if (e != cudaSuccess) return e;
        }
        route_rank<<<chunks, 1024, smem, st>>>(idx, G, S, n, local_rank, chunk, chunk_imp, err);
    }
    route_colscan<<<(n + 31) / 32, dim3(32, 32), 0, st>>>(chunk, chunk_imp, chunks, n, counts, imp64);
    route_finish<<<1, 256, 0, st>>>(counts, imp64, n, offsets, importance, cv2);
    route_scatter<<<static_cast<unsigned>((S + 255) / 256), 256, 0, st>>>(
        idx, S, n, offsets, chunk, local_rank, perm, inv_perm);
    return cudaGetLastError();
}

}  // namespace moe

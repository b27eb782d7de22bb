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
//                   of <= 32 slots, then the groups in warp order; fp32);
//                   route_rank_warps gives the same for n <= 512 from a
//                   [warp][expert] table instead of 32 barrier rounds
//   route_scan      per expert, an exclusive scan of the counts down the
//                   chunks (chunk bases), the expert's count and its
//                   importance (chunk partials summed in chunk order, fp32); the
//                   last block to finish then scans the counts over the
//                   experts (offsets), writes importance in fp32 and the
//                   population variance / mean^2 of the importance vector
//                   (CV^2), and, for the forward pass, the expert stage's
//                   tile schedules
//   route_scatter   row = offsets[e] + chunk base + local rank: perm, inv_perm
//                   (route_scatter_gather also copies each slot's x row to
//                   its expert-order row for the expert stage)
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
                                                   float *__restrict__ chunk_imp, int32_t *err) {
    extern __shared__ __align__(8) unsigned char route_sh[];
    pdl_wait();
    pdl_launch_dependents();
    float *imp = reinterpret_cast<float *>(route_sh);                // [n]
    int32_t *cnt = reinterpret_cast<int32_t *>(route_sh + 4 * n);     // [n]
    __shared__ int32_t base_sh[32][32];
    for (int e = threadIdx.x; e < n; e += blockDim.x) {
        cnt[e] = 0;
        imp[e] = 0.0f;
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
    // lane order in fp32; the groups are then accumulated in fp32 in warp order.
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
            imp[e] += seg;
        }
        __syncthreads();
    }
    if (e >= 0) local_rank[s] = base_sh[warp][leader] + rank_in_warp;
    int32_t *row = chunk + static_cast<int64_t>(blockIdx.x) * n;
    float *irow = chunk_imp + static_cast<int64_t>(blockIdx.x) * n;
    for (int ee = threadIdx.x; ee < n; ee += blockDim.x) {
        row[ee] = cnt[ee];
        irow[ee] = imp[ee];
    }
}

// route_rank for n <= kRankWarpsMaxN: the same outputs without the 32
// barrier rounds.  Each warp's leaders write their group's count and fp32
// gate-weight sum to a [32 warps][n] table; one thread per expert then walks
// the warps in order (exclusive scan of the counts, fp32 sum of the groups,
// the same order as route_rank) and every slot reads its warp's base.
constexpr int kRankWarpsMaxN = 512;

__global__ void __launch_bounds__(1024) route_rank_warps(const int32_t *__restrict__ idx,
                                                         const float *__restrict__ G, int64_t S,
                                                         int n, int32_t *__restrict__ local_rank,
                                                         int32_t *__restrict__ chunk,
                                                         float *__restrict__ chunk_imp,
                                                         int32_t *err) {
    extern __shared__ __align__(8) unsigned char route_sh[];
    pdl_wait();
    pdl_launch_dependents();
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
    float *irow = chunk_imp + static_cast<int64_t>(blockIdx.x) * n;
    for (int ee = threadIdx.x; ee < n; ee += blockDim.x) {
        int32_t run = 0;
        float imp = 0.0f;
        for (int w = 0; w < 32; ++w) {
            const int32_t c = wc[w * n + ee];
            wc[w * n + ee] = run;
            run += c;
            if (c) imp += wsum[w * n + ee];
        }
        row[ee] = run;
        irow[ee] = imp;
    }
    __syncthreads();
    if (e >= 0) local_rank[s] = wc[warp * n + e] + rank_in_warp;
}

struct ScanOut {
    int32_t *counts;
    float *imp;
    int32_t *offsets;
    float *importance;
    float *cv2;
    int32_t *rtiles;    // optional: starts of bm-row tiles per expert
    int bm;
    int32_t *ptiles;    // optional: pair token tiles per expert, and their table
    int4 *plist;
    int pcap;           // rows per pair token tile at most
};

// The serial tail of the dispatch, run by one block of 1024 threads once every
// expert's count and importance are known: offsets = exclusive scan of the
// counts (offsets[n] = total), importance in fp32, CV^2 = population variance
// / mean^2 (fp32 tree sums, fixed order), and the expert stage's schedules.
__device__ void dispatch_finish(int n, const ScanOut &o) {
    __shared__ int32_t ish[32];
    __shared__ float fsh[33];
    const int tid = threadIdx.y * blockDim.x + threadIdx.x;
    const int per = (n + 1023) / 1024;
    const int i0 = min(n, tid * per), i1 = min(n, i0 + per);
    int32_t sum = 0, rt = 0, pt = 0;
    for (int i = i0; i < i1; ++i) {
        const int32_t c = __ldcg(o.counts + i);
        sum += c;
        if (o.rtiles) rt += (c + o.bm - 1) / o.bm;
        if (o.ptiles) {
            int tn, nt;
            token_tiling(c, tn, nt, o.pcap);
            pt += nt;
        }
    }
    int32_t total;
    int32_t run = block_exclusive_scan_1024(sum, ish, &total);
    int32_t rrun = 0, prun = 0, rtotal = 0, ptotal = 0;
    if (o.rtiles) rrun = block_exclusive_scan_1024(rt, ish, &rtotal);
    if (o.ptiles) prun = block_exclusive_scan_1024(pt, ish, &ptotal);
    for (int i = i0; i < i1; ++i) {
        const int32_t c = __ldcg(o.counts + i);
        o.offsets[i] = run;
        if (o.rtiles) {
            o.rtiles[i] = rrun;
            rrun += (c + o.bm - 1) / o.bm;
        }
        if (o.ptiles) {
            o.ptiles[i] = prun;
            int tn, nt;
            token_tiling(c, tn, nt, o.pcap);
            for (int j = 0; j < nt; ++j) {
                const int rows = min(tn, c - j * tn);
                o.plist[prun + j] = make_int4(i, run + j * tn, rows, (rows + 31) & ~31);
            }
            prun += nt;
        }
        run += c;
    }
    if (tid == 0) {
        o.offsets[n] = total;
        if (o.rtiles) o.rtiles[n] = rtotal;
        if (o.ptiles) o.ptiles[n] = ptotal;
    }
    float sacc = 0.0f;
    for (int e = tid; e < n; e += 1024) {
        const float v = __ldcg(o.imp + e);
        sacc += v;
        o.importance[e] = v;
    }
    const float mean = block_sum_1024(sacc, fsh) / static_cast<float>(n);
    float q = 0.0f;
    for (int e = tid; e < n; e += 1024) {
        const float v = __ldcg(o.imp + e) - mean;
        q = fmaf(v, v, q);
    }
    const float var = block_sum_1024(q, fsh) / static_cast<float>(n);
    if (tid == 0) o.cv2[0] = mean != 0.0f ? var / (mean * mean) : 0.0f;
}

// Block (32 x 32): 32 experts (x) by 32 chunk segments (y).  Chunk counts
// become chunk bases (exclusive scan down the chunks); the expert's count
// and importance (fp32, chunk order) are the column totals.  The last block
// to finish (a counter in the workspace header, reset by that block) then
// runs dispatch_finish.
__global__ void __launch_bounds__(1024) route_scan(int32_t *__restrict__ chunk,
                                                   const float *__restrict__ chunk_imp, int chunks,
                                                   int n, ScanOut o, int32_t *done) {
    __shared__ int32_t part[32][33];
    __shared__ float ipart[32][33];
    __shared__ int is_last;
    pdl_wait();
    pdl_launch_dependents();
    const int tx = threadIdx.x, ty = threadIdx.y;
    const int e = blockIdx.x * 32 + tx;
    const int seg = (chunks + 31) / 32;
    const int b0 = ty * seg, b1 = min(chunks, b0 + seg);
    int32_t sum = 0;
    float isum = 0.0f;
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
        float irun = 0.0f;
        for (int y = 0; y < 32; ++y) {
            const int32_t v = part[y][tx];
            part[y][tx] = run;
            run += v;
            irun += ipart[y][tx];
        }
        if (e < n) {
            o.counts[e] = run;
            o.imp[e] = irun;
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
    // Publish this block's results, then count it; the last block sees all.
    __threadfence();
    __syncthreads();
    if (tx == 0 && ty == 0) is_last = atomicAdd(done, 1) == static_cast<int>(gridDim.x) - 1;
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    dispatch_finish(n, o);
    if (tx == 0 && ty == 0) *done = 0;
}

__global__ void route_scatter(const int32_t *__restrict__ idx, int64_t S, int n,
                              const int32_t *__restrict__ offsets,
                              const int32_t *__restrict__ chunk,
                              const int32_t *__restrict__ local_rank, int32_t *__restrict__ perm,
                              int32_t *__restrict__ inv_perm) {
    pdl_wait();
    pdl_launch_dependents();
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

// route_scatter with each token's x row copied to the expert-order rows of
// its k slots (xperm[row] = x[t]): one warp per token, lane j < k handles
// slot t*k + j, and the row is read once (16-byte loads) and stored k times.
constexpr int kScatterTokensPerBlock = 8;

__global__ void __launch_bounds__(256) route_scatter_gather(
    const int32_t *__restrict__ idx, int64_t T, int n, int k, int d,
    const int32_t *__restrict__ offsets, const int32_t *__restrict__ chunk,
    const int32_t *__restrict__ local_rank, int32_t *__restrict__ perm,
    int32_t *__restrict__ inv_perm, const __nv_bfloat16 *__restrict__ x,
    __nv_bfloat16 *__restrict__ xperm) {
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t t = static_cast<int64_t>(blockIdx.x) * kScatterTokensPerBlock + threadIdx.x / 32;
    if (t >= T) return;
    const int total = offsets[n];
    // the x row's first pieces are requested before the routing lookups
    const uint4 *src = reinterpret_cast<const uint4 *>(x + t * static_cast<int64_t>(d));
    const int nv = d / 8;
    uint4 v0 = lane < nv ? __ldg(src + lane) : make_uint4(0, 0, 0, 0);
    uint4 v1 = lane + 32 < nv ? __ldg(src + lane + 32) : make_uint4(0, 0, 0, 0);
    int32_t row = -1;
    if (lane < k) {
        const int64_t s = t * k + lane;
        const int e = idx[s];
        if (e >= 0 && e < n) row = offsets[e] + chunk[(s / kRouteChunk) * n + e] + local_rank[s];
        if (row >= 0) perm[row] = static_cast<int32_t>(s);
        inv_perm[s] = row;
        if (s >= total) perm[s] = -1;  // rows left empty by invalid slots
    }
    for (int j = 0; j < k; ++j) {
        const int32_t r = __shfl_sync(0xffffffffu, row, j);
        if (r < 0) continue;
        uint4 *dst = reinterpret_cast<uint4 *>(xperm + static_cast<int64_t>(r) * d);
        if (lane < nv) dst[lane] = v0;
        if (lane + 32 < nv) dst[lane + 32] = v1;
        for (int c = lane + 64; c < nv; c += 32) dst[c] = __ldg(src + c);
    }
}

}  // namespace

cudaError_t launch_dispatch(const moe_shape &s, const int32_t *idx, const float *G,
                            int32_t *counts, int32_t *offsets, int32_t *perm, int32_t *inv_perm,
                            float *importance, float *cv2, void *ws, const WsLayout &L,
                            cudaStream_t st, const DispatchExtras *ex) {
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
    float *chunk_imp = ws_ptr<float>(ws, L.chunk_imp);
    float *imp_acc = ws_ptr<float>(ws, L.imp_acc);
    // Dynamic shared memory above the default 48 KB needs an opt-in, which
    // belongs to the current device's context: it is set before each launch.
    if (n <= kRankWarpsMaxN) {
        const size_t smem = 256 * static_cast<size_t>(n);  // [32][n] counts and sums
        if (smem > 48 * 1024) {
            cudaError_t e = cudaFuncSetAttribute(
                route_rank_warps, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
            if (e != cudaSuccess) return e;
        }
        cudaError_t e = launch_pdl(route_rank_warps, dim3(chunks), dim3(1024), smem, st, idx, G, S, n,
                                   local_rank, chunk, chunk_imp, err);
        if (e != cudaSuccess) return e;
    } else {
        const size_t smem = 8 * static_cast<size_t>(n);  // n floats and n ints (+4 KB static)
        if (smem + 4096 > 48 * 1024) {
            cudaError_t e = cudaFuncSetAttribute(
                route_rank, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
            if (e != cudaSuccess) return e;
        }
        cudaError_t e = launch_pdl(route_rank, dim3(chunks), dim3(1024), smem, st, idx, G, S, n,
                                   local_rank, chunk, chunk_imp, err);
        if (e != cudaSuccess) return e;
    }
    ScanOut o{counts, imp_acc, offsets, importance, cv2, nullptr, 0, nullptr, nullptr, 256};
    if (ex) {
        o.rtiles = ex->rtiles;
        o.bm = ex->bm;
        o.ptiles = ex->ptiles;
        o.plist = ex->plist;
        o.pcap = ex->pcap;
    }
    int32_t *done = reinterpret_cast<int32_t *>(static_cast<char *>(ws) + kWsDoneCounterOffset);
    cudaError_t e = launch_pdl(route_scan, dim3((n + 31) / 32), dim3(32, 32), 0, st, chunk,
                               chunk_imp, chunks, n, o, done);
    if (e != cudaSuccess) return e;
    if (ex && ex->x) {
        e = launch_pdl(route_scatter_gather,
                       dim3(static_cast<unsigned>((s.T + kScatterTokensPerBlock - 1) /
                                                  kScatterTokensPerBlock)),
                       dim3(256), 0, st, idx, s.T, n, s.k, s.d, offsets, chunk, local_rank, perm,
                       inv_perm, ex->x, ex->xperm);
    } else {
        e = launch_pdl(route_scatter, dim3(static_cast<unsigned>((S + 255) / 256)), dim3(256), 0, st,
                       idx, S, n, offsets, chunk, local_rank, perm, inv_perm);
    }
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace moe

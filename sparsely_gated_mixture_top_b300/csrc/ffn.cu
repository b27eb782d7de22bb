// ffn.cu -- the expert feed-forward stage ("MoE:稀疏门控混合专家", section 二:
// each expert is a one-hidden-layer ReLU network, E(x) = W2 ReLU(W1 x + b1) + b2),
// run only for the rows routed to each expert.
//
//   ffn_tiles      row-tile schedule: tiles[e] = sum over e' < e of ceil(count/BM)
//   ffn_gather     x rows copied into expert order (bf16 path): xperm[r] = x[perm[r]/k]
//   grouped_gemm_simt  fp32 path: the same grouped GEMM on CUDA cores (gathering
//                  x through perm directly), fp32 throughout
// The bf16 path runs the two layers on the tensor cores with the hidden
// activation rounded once to bf16 in between: in one kernel that keeps it on
// chip (ffn_fused.cu) where the widths allow, else as two grouped GEMMs
// (ffn_pair.cu, ffn_tc.cu) through the workspace.
#include "moe_device.cuh"
#include "moe_launch.h"

namespace moe {

cudaError_t launch_grouped_gemm_tc(const moe_shape &s, const __nv_bfloat16 *A, int K,
                                   const __nv_bfloat16 *B, int N, const float *bias, int relu,
                                   const int32_t *offsets, const int32_t *tiles,
                                   __nv_bfloat16 *out, int32_t *err, cudaStream_t st);

namespace {

// One block of 1024 threads.
__global__ void __launch_bounds__(1024) ffn_tiles(const int32_t *__restrict__ offsets, int n,
                                                  int bm, int32_t *__restrict__ tiles) {
    __shared__ int32_t part[1024];
    const int per = (n + 1023) / 1024;
    const int i0 = threadIdx.x * per, i1 = min(n, i0 + per);
    int32_t sum = 0;
    for (int i = i0; i < i1; ++i) sum += (offsets[i + 1] - offsets[i] + bm - 1) / bm;
    part[threadIdx.x] = sum;
    __syncthreads();
    for (int off = 1; off < 1024; off <<= 1) {
        const int32_t v = threadIdx.x >= off ? part[threadIdx.x - off] : 0;
        __syncthreads();
        part[threadIdx.x] += v;
        __syncthreads();
    }
    int32_t run = threadIdx.x ? part[threadIdx.x - 1] : 0;
    for (int i = i0; i < i1; ++i) {
        tiles[i] = run;
        run += (offsets[i + 1] - offsets[i] + bm - 1) / bm;
    }
    if (threadIdx.x == 1023) tiles[n] = part[1023];
}

// Four rows per warp, 16-byte copies: the four rows' indices, then each
// 16-byte column of the four rows loaded before any is stored.
constexpr int kGatherRows = 4;

__global__ void __launch_bounds__(256) ffn_gather(const __nv_bfloat16 *__restrict__ x,
                                                  const int32_t *__restrict__ perm,
                                                  const int32_t *__restrict__ offsets, int n,
                                                  int64_t S, int d, int k,
                                                  __nv_bfloat16 *__restrict__ xperm, int32_t *err) {
    const int lane = threadIdx.x & 31;
    const int64_t r0 = (static_cast<int64_t>(blockIdx.x) * 8 + threadIdx.x / 32) * kGatherRows;
    const int64_t rows = S < offsets[n] ? S : offsets[n];
    if (r0 >= rows) return;
    const uint4 *src[kGatherRows];
    uint4 *dst[kGatherRows];
#pragma unroll
    for (int i = 0; i < kGatherRows; ++i) {
        const int64_t r = r0 + i;
        src[i] = nullptr;
        dst[i] = nullptr;
        if (r < rows) {
            dst[i] = reinterpret_cast<uint4 *>(xperm + r * d);
            const int32_t s = perm[r];
            if (s < 0 || s >= S) {
                if (lane == 0) report(err, MOE_ERR_DEVICE, kSiteFfnPerm, static_cast<int32_t>(r));
            } else {
                src[i] = reinterpret_cast<const uint4 *>(x + static_cast<int64_t>(s / k) * d);
            }
        }
    }
    for (int c = lane; c < d / 8; c += 32) {
        uint4 v[kGatherRows];
#pragma unroll
        for (int i = 0; i < kGatherRows; ++i) v[i] = src[i] ? src[i][c] : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int i = 0; i < kGatherRows; ++i)
            if (dst[i]) dst[i][c] = v[i];
    }
}

constexpr int kSB = 64;  // rows and columns per SIMT tile
constexpr int kSK = 16;

// out[r, c] = act(sum_kk A[row(r), kk] * B[e][c, kk] + bias[e][c]) for the rows
// r of expert e; row(r) = perm[r] / kdiv when perm is given, else r.
__global__ void __launch_bounds__(256) grouped_gemm_simt(
    const float *__restrict__ A, const int32_t *__restrict__ perm, int kdiv, int64_t S,
    const float *__restrict__ B, const float *__restrict__ bias, int K, int N, int relu,
    const int32_t *__restrict__ offsets, const int32_t *__restrict__ tiles, int n,
    float *__restrict__ out, int32_t *err) {
    __shared__ float As[kSK][kSB + 4];
    __shared__ float Bs[kSK][kSB + 4];
    __shared__ int64_t arow[kSB];
    const int rt = blockIdx.x;
    if (rt >= tiles[n]) return;
    int lo = 0, hi = n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tiles[mid] <= rt)
            lo = mid;
        else
            hi = mid - 1;
    }
    const int e = lo;
    const int row0 = offsets[e] + (rt - tiles[e]) * kSB;
    const int rows = min(kSB, offsets[e + 1] - row0);
    const int c0 = blockIdx.y * kSB;
    const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
    if (tid < kSB) {
        int64_t ar = -1;
        if (tid < rows) {
            const int64_t r = row0 + tid;
            if (perm) {
                const int32_t s = perm[r];
                if (s < 0 || s >= S)
                    report(err, MOE_ERR_DEVICE, kSiteFfnPerm, static_cast<int32_t>(r));
                else
                    ar = s / kdiv;
            } else {
                ar = r;
            }
        }
        arow[tid] = ar;
    }
    __syncthreads();
    const float *Be = B + static_cast<int64_t>(e) * N * K;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < K; k0 += kSK) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int idx = tid + q * 256;
            const int r = idx / kSK, kk = idx % kSK;
            const int64_t ar = arow[r];
            As[kk][r] = ar >= 0 ? A[ar * K + k0 + kk] : 0.0f;
            Bs[kk][r] = Be[static_cast<int64_t>(c0 + r) * K + k0 + kk];
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < kSK; ++kk) {
            float av[4], bv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                av[i] = As[kk][ty * 4 + i];
                bv[i] = Bs[kk][tx * 4 + i];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = ty * 4 + i;
        if (r >= rows) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int c = c0 + tx * 4 + j;
            float v = acc[i][j] + (bias ? bias[static_cast<int64_t>(e) * N + c] : 0.0f);
            if (relu) v = fmaxf(v, 0.0f);
            out[static_cast<int64_t>(row0 + r) * N + c] = v;
        }
    }
}

}  // namespace

cudaError_t launch_row_tiles(const int32_t *offsets, int n, int bm, int32_t *tiles,
                             cudaStream_t st) {
    ffn_tiles<<<1, 1024, 0, st>>>(offsets, n, bm, tiles);
    return cudaGetLastError();
}

cudaError_t launch_gather_rows(const __nv_bfloat16 *x, const int32_t *perm, const int32_t *offsets,
                               int n, int64_t S, int d, int k, __nv_bfloat16 *out, int32_t *err,
                               cudaStream_t st) {
    if (S == 0) return cudaSuccess;
    ffn_gather<<<static_cast<unsigned>((S + 8 * kGatherRows - 1) / (8 * kGatherRows)), 256, 0, st>>>(
        x, perm, offsets, n, S, d, k, out, err);
    return cudaGetLastError();
}

DispatchExtras dispatch_extras_for_ffn(const moe_shape &s, const void *x, void *ws,
                                       const WsLayout &L) {
    DispatchExtras ex;
    if (s.dtype == MOE_BF16) {
        const bool pair1 = pair_gemm_supported(s.h), pair2 = pair_gemm_supported(s.d);
        ex.x = static_cast<const __nv_bfloat16 *>(x);
        ex.xperm = ws_ptr<__nv_bfloat16>(ws, L.xperm);
        if (fused_ffn_supported(s)) {
            ex.ptiles = ws_ptr<int32_t>(ws, L.ptiles);
            ex.plist = ws_ptr<int4>(ws, L.plist);
            ex.pcap = 128;
            return ex;
        }
        if (pair1 || pair2) {
            ex.ptiles = ws_ptr<int32_t>(ws, L.ptiles);
            ex.plist = ws_ptr<int4>(ws, L.plist);
        }
        if (!pair1 || !pair2) {
            ex.rtiles = ws_ptr<int32_t>(ws, L.tiles);
            ex.bm = kTcRows;
        }
    } else {
        ex.rtiles = ws_ptr<int32_t>(ws, L.tiles);
        ex.bm = kSimtRows;
    }
    return ex;
}

cudaError_t launch_expert_ffn(const moe_shape &s, const void *x, const int32_t *perm,
                              const int32_t *offsets, const void *W1, const float *b1,
                              const void *W2, const float *b2, void *Y_slot, void *ws,
                              const WsLayout &L, cudaStream_t st, bool prepared,
                              bool keep_hidden) {
    const int64_t S = slots(s);
    if (S == 0) return cudaSuccess;
    int32_t *err = ws_ptr<int32_t>(ws, 0);
    int32_t *tiles = ws_ptr<int32_t>(ws, L.tiles);
    if (s.dtype == MOE_BF16 && !keep_hidden && fused_ffn_supported(s)) {
        // both layers in one kernel, the hidden activations on chip
        int32_t *ptiles = ws_ptr<int32_t>(ws, L.ptiles);
        int4 *plist = ws_ptr<int4>(ws, L.plist);
        __nv_bfloat16 *xperm = ws_ptr<__nv_bfloat16>(ws, L.xperm);
        if (!prepared) {
            cudaError_t e = launch_pair_tiles(offsets, s.n, ptiles, plist, st, 128);
            if (e != cudaSuccess) return e;
            ffn_gather<<<static_cast<unsigned>((S + 8 * kGatherRows - 1) / (8 * kGatherRows)), 256,
                         0, st>>>(static_cast<const __nv_bfloat16 *>(x), perm, offsets, s.n, S, s.d,
                                  s.k, xperm, err);
        }
        return launch_ffn_fused(s, xperm, static_cast<const __nv_bfloat16 *>(W1), b1,
                                static_cast<const __nv_bfloat16 *>(W2), b2, ptiles, plist,
                                static_cast<__nv_bfloat16 *>(Y_slot), err, st);
    }
    if (s.dtype == MOE_BF16) {
        // Each layer runs on a pair of SMs when its output width is a
        // multiple of 256 (ffn_pair.cu), else on the single-SM kernel.
        const bool pair1 = pair_gemm_supported(s.h), pair2 = pair_gemm_supported(s.d);
        int32_t *ptiles = ws_ptr<int32_t>(ws, L.ptiles);
        int4 *plist = ws_ptr<int4>(ws, L.plist);
        __nv_bfloat16 *xperm = ws_ptr<__nv_bfloat16>(ws, L.xperm);
        __nv_bfloat16 *hid = ws_ptr<__nv_bfloat16>(ws, L.hidden);
        if (!prepared) {
            if (pair1 || pair2) {
                cudaError_t e = launch_pair_tiles(offsets, s.n, ptiles, plist, st);
                if (e != cudaSuccess) return e;
            }
            if (!pair1 || !pair2) ffn_tiles<<<1, 1024, 0, st>>>(offsets, s.n, kTcRows, tiles);
            ffn_gather<<<static_cast<unsigned>((S + 8 * kGatherRows - 1) / (8 * kGatherRows)), 256,
                         0, st>>>(static_cast<const __nv_bfloat16 *>(x), perm, offsets, s.n, S, s.d,
                                  s.k, xperm, err);
        }
        const auto *W1b = static_cast<const __nv_bfloat16 *>(W1);
        const auto *W2b = static_cast<const __nv_bfloat16 *>(W2);
        cudaError_t e = pair1 ? launch_grouped_gemm_pair(s, xperm, s.d, W1b, s.h, b1, 1, ptiles,
                                                         plist, hid, err, st)
                              : launch_grouped_gemm_tc(s, xperm, s.d, W1b, s.h, b1, 1, offsets,
                                                       tiles, hid, err, st);
        if (e != cudaSuccess) return e;
        auto *Y = static_cast<__nv_bfloat16 *>(Y_slot);
        return pair2 ? launch_grouped_gemm_pair(s, hid, s.h, W2b, s.d, b2, 0, ptiles, plist, Y,
                                                err, st)
                     : launch_grouped_gemm_tc(s, hid, s.h, W2b, s.d, b2, 0, offsets, tiles, Y, err,
                                              st);
    }
    if (!prepared) ffn_tiles<<<1, 1024, 0, st>>>(offsets, s.n, kSimtRows, tiles);
    float *hid = ws_ptr<float>(ws, L.hidden);
    const unsigned max_rt = static_cast<unsigned>((S + kSB - 1) / kSB + s.n);
    grouped_gemm_simt<<<dim3(max_rt, s.h / kSB), 256, 0, st>>>(
        static_cast<const float *>(x), perm, s.k, S, static_cast<const float *>(W1), b1, s.d, s.h, 1,
        offsets, tiles, s.n, hid, err);
    grouped_gemm_simt<<<dim3(max_rt, s.d / kSB), 256, 0, st>>>(
        hid, nullptr, 1, S, static_cast<const float *>(W2), b2, s.h, s.d, 0, offsets, tiles, s.n,
        static_cast<float *>(Y_slot), err);
    return cudaGetLastError();
}

}  // namespace moe

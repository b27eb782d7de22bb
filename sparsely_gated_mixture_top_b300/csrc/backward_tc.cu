// backward_tc.cu -- tensor-core pieces of the bf16 backward pass: the
// per-expert weight-gradient GEMM and the layout kernels around it.
//
// Weight gradients of an expert are sums over the rows that chose it:
//     dW2[e] = sum_r dE_r a_r^T   ([d, h]),    dW1[e] = sum_r dz_r x_r^T   ([h, d])
// (chain rule of E = W2 ReLU(W1 x + b1) + b2, "MoE:稀疏门控混合专家" section 二).
// The rows are the contraction axis, so both operands are laid out
// transposed: P^T [M, Kcap] and Q^T [N, Kcap], each expert's rows taking
// ceil(rows/64) 64-wide column blocks starting at block kblk[e] (the pad
// columns are zero).  wgrad_gemm_tc then computes, per expert e and 128 x BN
// output tile,
//     out[e][i, j] = sum over k-blocks kblk[e] .. kblk[e+1]-1 of P^T[i, k] Q^T[j, k]
// on the 5th-generation tensor cores (TMA 128-byte-swizzled k-blocks into a
// STAGES-deep ring, one thread issuing tcgen05.mma M = 128, N = BN, K = 16,
// the fp32 accumulator double-buffered in tensor memory, eight epilogue warps
// storing fp32).  An expert without rows gets zeros.  Every wait is bounded;
// on a timeout the kernel records MOE_ERR_TIMEOUT, drains its copies and
// MMAs, frees tensor memory and returns.
#include "backward_tc.h"
#include "moe_device.cuh"

#include <mutex>

namespace moe {
namespace {

constexpr int kWgRows = 128;
constexpr int kWgEpiWarps = 8;
constexpr int kWgThreads = 32 * (2 + kWgEpiWarps);
constexpr int32_t kSiteWgProducer = 30, kSiteWgMma = 31, kSiteWgEpilogue = 32, kSiteWgDrain = 33;
constexpr int32_t kSiteRowsPerm = 34;  // a perm entry out of range while building dE rows

template <int BN, int STAGES>
struct WgCfg {
    static constexpr int kBK = 64;
    static constexpr int kABytes = kWgRows * kBK * 2;
    static constexpr int kBBytes = BN * kBK * 2;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kBarBytes = 8 * (2 * STAGES + 5) + 16;
    // per epilogue warp a 32 x 33 fp32 staging tile (rows 33 words apart)
    static constexpr int kStageOutBytes = kWgEpiWarps * 32 * 33 * 4;
    static constexpr int kSmem = STAGES * kStageBytes + 1024 + kBarBytes + kStageOutBytes;
    static constexpr uint32_t kTmemCols = 2 * BN;
};

__device__ __forceinline__ bool wg_drain(uint32_t bar, uint32_t parity, int32_t *err) {
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_ns() - t0 > kWaitLimitNs) {
            report(err, MOE_ERR_TIMEOUT, kSiteWgDrain);
            return false;
        }
    }
    return true;
}

template <int BN, int STAGES>
__global__ void __launch_bounds__(kWgThreads, 1)
    wgrad_gemm_tc(const __grid_constant__ CUtensorMap mapP, const __grid_constant__ CUtensorMap mapQ,
                  const int32_t *__restrict__ kblk, int n, int M, int N, float *__restrict__ out,
                  int32_t *err) {
    using Cfg = WgCfg<BN, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint8_t *sA = smem;
    uint8_t *sB = smem + STAGES * Cfg::kABytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sB + STAGES * Cfg::kBBytes);
    // bars: full[STAGES], empty[STAGES], tfull[2], tempty[2], drain
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * STAGES + 5);
    volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(tmem_slot + 1);
    float *stage_out = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(bars) + Cfg::kBarBytes);
    auto full = [&](int s) { return smem_u32(bars + s); };
    auto empty = [&](int s) { return smem_u32(bars + STAGES + s); };
    auto tfull = [&](int b) { return smem_u32(bars + 2 * STAGES + b); };
    auto tempty = [&](int b) { return smem_u32(bars + 2 * STAGES + 2 + b); };
    const uint32_t drain_bar = smem_u32(bars + 2 * STAGES + 4);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull(b), 1);
            mbar_init(tempty(b), 32 * kWgEpiWarps);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&mapP);
        tma_prefetch_map(&mapQ);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int mt = M / kWgRows, nt = N / BN;
    const int per_e = mt * nt;
    const int total = n * per_e;

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int64_t issued = 0;
            bool ok = true;
            for (int q = blockIdx.x; q < total && ok; q += gridDim.x) {
                const int e = q / per_e, rem = q - e * per_e;
                const int mi = rem / nt, ni = rem - mi * nt;
                const int kb0 = kblk[e], kb1 = kblk[e + 1];
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait_bounded(empty(stage), phase ^ 1u, abort_flag, err, kSiteWgProducer)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(full(stage), Cfg::kStageBytes);
                    tma_load_3d(smem_u32(sA + stage * Cfg::kABytes), &mapP, full(stage), 0,
                                mi * kWgRows, kb);
                    tma_load_3d(smem_u32(sB + stage * Cfg::kBBytes), &mapQ, full(stage), 0, ni * BN, kb);
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                const int outstanding = static_cast<int>(issued < STAGES ? issued : STAGES);
                int s = stage;
                uint32_t p = phase;
                for (int i = 0; i < outstanding; ++i) {
                    if (--s < 0) {
                        s = STAGES - 1;
                        p ^= 1u;
                    }
                    wg_drain(full(s), p, err);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(kWgRows, BN);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int q = blockIdx.x; q < total && ok; q += gridDim.x) {
                const int e = q / per_e;
                const int kb0 = kblk[e], kb1 = kblk[e + 1];
                if (!mbar_wait_bounded(tempty(acc), acc_phase ^ 1u, abort_flag, err, kSiteWgMma)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait_bounded(full(stage), phase, abort_flag, err, kSiteWgMma)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(sA + stage * Cfg::kABytes);
                    const uint32_t b0 = smem_u32(sB + stage * Cfg::kBBytes);
#pragma unroll
                    for (int kk = 0; kk < Cfg::kBK / 16; ++kk)
                        tc_mma_f16(d_tmem, sdesc_kmajor_sw128(a0 + kk * 32), sdesc_kmajor_sw128(b0 + kk * 32),
                                   idesc, (kb != kb0 || kk != 0) ? 1u : 0u);
                    tc_commit(empty(stage));
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                tc_commit(tfull(acc));  // also when the expert has no rows (nothing to wait for)
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            tc_commit(drain_bar);
            wg_drain(drain_bar, 0, err);
        }
    } else {
        // Epilogue: warp w (2..9) reads lanes 32*(w%4).. (rows of the tile)
        // and one half of its BN columns, 32 at a time with the next 32 in
        // flight.  Each 32 x 32 block goes through the warp's staging tile so
        // that every store instruction writes four whole 128-byte row pieces.
        const int quad = warp & 3;
        const int half = (warp - 2) >> 2;
        constexpr int kHalf = BN / 2;
        constexpr int kChunks = kHalf / 32;
        const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
        float *stg = stage_out + (warp - 2) * 32 * 33;
        const int srow = lane >> 3, scol = (lane & 7) * 4;  // store phase: row within 4, column
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int q = blockIdx.x; q < total; q += gridDim.x) {
            const int e = q / per_e, rem = q - e * per_e;
            const int mi = rem / nt, ni = rem - mi * nt;
            const bool empty_e = kblk[e] == kblk[e + 1];
            if (!mbar_wait_bounded(tfull(acc), acc_phase, abort_flag, err, kSiteWgEpilogue)) break;
            tc_fence_after();
            const int col0 = ni * BN + half * kHalf;
            float *obase = out + (static_cast<int64_t>(e) * M + mi * kWgRows + quad * 32) * N + col0;
            if (empty_e) {
                tc_fence_before();
                mbar_arrive(tempty(acc));
                for (int ch = 0; ch < kChunks; ++ch)
                    for (int it = 0; it < 8; ++it)
                        *reinterpret_cast<float4 *>(obase + static_cast<int64_t>(it * 4 + srow) * N +
                                                    ch * 32 + scol) = make_float4(0.f, 0.f, 0.f, 0.f);
            } else {
                const uint32_t tbase =
                    tmem_base + lane_addr + static_cast<uint32_t>(acc * BN + half * kHalf);
                uint32_t v[2][32];
                tmem_ld_32x32b_x32(tbase, v[0]);
#pragma unroll
                for (int ch = 0; ch < kChunks; ++ch) {
                    tmem_ld_wait();
                    if (ch + 1 < kChunks) tmem_ld_32x32b_x32(tbase + (ch + 1) * 32, v[(ch + 1) & 1]);
                    if (ch + 1 == kChunks) {
                        tc_fence_before();
                        mbar_arrive(tempty(acc));
                    }
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 32; ++j) stg[lane * 33 + j] = __uint_as_float(v[ch & 1][j]);
                    __syncwarp();
#pragma unroll
                    for (int it = 0; it < 8; ++it) {
                        const float *src = stg + (it * 4 + srow) * 33 + scol;
                        *reinterpret_cast<float4 *>(obase + static_cast<int64_t>(it * 4 + srow) * N +
                                                    ch * 32 + scol) =
                            make_float4(src[0], src[1], src[2], src[3]);
                    }
                }
            }
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, Cfg::kTmemCols);
}

// 64 x 64 bf16 tile transpose through shared memory with 16-byte global
// loads and stores: rows [r0, r0 + 64) of `in` (row stride ld_in; rows at or
// past `rows` read as zeros) become columns of `out` (row stride ld_out).
// The tile's rows are 66 elements apart so that the column reads of the store
// phase spread over the banks.
__device__ __forceinline__ void tile_transpose_64(const __nv_bfloat16 *__restrict__ in, int64_t ld_in,
                                                  int rows, __nv_bfloat16 *__restrict__ out,
                                                  int64_t ld_out, __nv_bfloat16 (*t)[66]) {
    for (int id = threadIdx.x; id < 64 * 8; id += 256) {
        const int r = id >> 3, ch = id & 7;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (r < rows) v = *reinterpret_cast<const uint4 *>(in + r * ld_in + ch * 8);
        uint32_t *dst = reinterpret_cast<uint32_t *>(&t[r][ch * 8]);
        dst[0] = v.x;
        dst[1] = v.y;
        dst[2] = v.z;
        dst[3] = v.w;
    }
    __syncthreads();
    for (int id = threadIdx.x; id < 64 * 8; id += 256) {
        const int orow = id >> 3, ch = id & 7;
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat16 lo = t[ch * 8 + 2 * i][orow], hi = t[ch * 8 + 2 * i + 1][orow];
            w[i] = static_cast<uint32_t>(__bfloat16_as_ushort(lo)) |
                   (static_cast<uint32_t>(__bfloat16_as_ushort(hi)) << 16);
        }
        *reinterpret_cast<uint4 *>(out + orow * ld_out + ch * 8) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// out[e][c][r] = in[e][r][c] for a stack of n bf16 matrices [R, C] (multiples of 64).
__global__ void __launch_bounds__(256) bt_transpose_w(const __nv_bfloat16 *__restrict__ in, int R,
                                                      int C, __nv_bfloat16 *__restrict__ out) {
    __shared__ __align__(16) __nv_bfloat16 t[64][66];
    const int64_t base = static_cast<int64_t>(blockIdx.z) * R * C;
    const int r0 = blockIdx.y * 64, c0 = blockIdx.x * 64;
    tile_transpose_64(in + base + static_cast<int64_t>(r0) * C + c0, C, 64,
                      out + base + static_cast<int64_t>(c0) * R + r0, R, t);
}

// dE[r] = bf16(G[s] * dy[s / k]) with s = perm[r], one warp per row, 16-byte chunks.
__global__ void __launch_bounds__(256) bt_rows_scaled(const __nv_bfloat16 *__restrict__ dy,
                                                      const float *__restrict__ G,
                                                      const int32_t *__restrict__ perm, int64_t S,
                                                      int d, int k, __nv_bfloat16 *__restrict__ dE,
                                                      int32_t *err) {
    const int64_t r = static_cast<int64_t>(blockIdx.x) * 8 + threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    if (r >= S) return;
    const int32_t s = perm[r];
    uint4 *dst = reinterpret_cast<uint4 *>(dE + r * d);
    if (s < 0 || s >= S) {
        if (lane == 0) report(err, MOE_ERR_DEVICE, kSiteRowsPerm, static_cast<int32_t>(r));
        for (int c = lane; c < d / 8; c += 32) dst[c] = make_uint4(0, 0, 0, 0);
        return;
    }
    const float g = G[s];
    const uint4 *src = reinterpret_cast<const uint4 *>(dy + static_cast<int64_t>(s / k) * d);
    for (int c = lane; c < d / 8; c += 32) {
        const uint4 v = src[c];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 p = *reinterpret_cast<const __nv_bfloat162 *>(&w[i]);
            o[i] = pack_bf16x2(g * __low2float(p), g * __high2float(p));
        }
        dst[c] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// x[i] = 0 where hid[i] <= 0 (ReLU derivative), 8 bf16 per thread.
__global__ void __launch_bounds__(256) bt_mask(__nv_bfloat16 *__restrict__ x,
                                               const __nv_bfloat16 *__restrict__ hid, int64_t n8) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x;
    if (i >= n8) return;
    uint4 v = reinterpret_cast<uint4 *>(x)[i];
    const uint4 m = reinterpret_cast<const uint4 *>(hid)[i];
    uint32_t *vw = reinterpret_cast<uint32_t *>(&v);
    const uint32_t *mw = reinterpret_cast<const uint32_t *>(&m);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const __nv_bfloat162 mp = *reinterpret_cast<const __nv_bfloat162 *>(&mw[j]);
        uint32_t keep = 0;
        if (__low2float(mp) > 0.0f) keep |= 0x0000FFFFu;
        if (__high2float(mp) > 0.0f) keep |= 0xFFFF0000u;
        vw[j] &= keep;
    }
    reinterpret_cast<uint4 *>(x)[i] = v;
}

// out[c, 64*rt + j] = in[offsets[e] + 64*(rt - kblk[e]) + j, c] for the j < 64
// rows of k-block rt (of expert e) that exist, 0 for the others.
__global__ void __launch_bounds__(256) bt_transpose_pad(const __nv_bfloat16 *__restrict__ in, int M,
                                                        const int32_t *__restrict__ offsets,
                                                        const int32_t *__restrict__ kblk, int n,
                                                        int64_t Kcap, __nv_bfloat16 *__restrict__ out) {
    __shared__ __align__(16) __nv_bfloat16 t[64][66];
    const int rt = blockIdx.x;
    if (rt >= kblk[n]) return;
    int lo = 0, hi = n - 1;  // largest e with kblk[e] <= rt
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (kblk[mid] <= rt)
            lo = mid;
        else
            hi = mid - 1;
    }
    const int e = lo;
    const int j0 = (rt - kblk[e]) * 64;
    const int rows = min(64, offsets[e + 1] - offsets[e] - j0);
    const int c0 = blockIdx.y * 64;
    tile_transpose_64(in + static_cast<int64_t>(offsets[e] + j0) * M + c0, M, rows,
                      out + static_cast<int64_t>(c0) * Kcap + static_cast<int64_t>(rt) * 64, Kcap, t);
}

template <int BN, int STAGES>
cudaError_t launch_wg(const CUtensorMap &mP, const CUtensorMap &mQ, const int32_t *kblk, int n,
                      int M, int N, float *out, int32_t *err, cudaStream_t st) {
    using Cfg = WgCfg<BN, STAGES>;
    // Per-context opt-in above 48 KB, set before every launch (cheap).
    const cudaError_t attr_err = cudaFuncSetAttribute(
        wgrad_gemm_tc<BN, STAGES>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
    if (attr_err != cudaSuccess) return attr_err;
    const int64_t total = static_cast<int64_t>(n) * (M / kWgRows) * (N / BN);
    const int grid = static_cast<int>(total < sm_count() ? total : sm_count());
    wgrad_gemm_tc<BN, STAGES><<<grid, kWgThreads, Cfg::kSmem, st>>>(mP, mQ, kblk, n, M, N, out, err);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_wgrad_tc(const __nv_bfloat16 *PT, int M, const __nv_bfloat16 *QT, int N,
                            int64_t Kcap, const int32_t *kblk, int n, float *out, int32_t *err,
                            cudaStream_t st) {
    if (M % kWgRows != 0 || N % 128 != 0 || Kcap % 64 != 0) return cudaErrorInvalidValue;
    const int BN = N % 256 == 0 ? 256 : 128;
    CUtensorMap mP, mQ;
    if (!make_kmajor_map(&mP, PT, static_cast<uint64_t>(Kcap), static_cast<uint64_t>(M), kWgRows) ||
        !make_kmajor_map(&mQ, QT, static_cast<uint64_t>(Kcap), static_cast<uint64_t>(N),
                         static_cast<uint32_t>(BN)))
        return cudaErrorInvalidValue;
    if (BN == 256) return launch_wg<256, 4>(mP, mQ, kblk, n, M, N, out, err, st);
    return launch_wg<128, 6>(mP, mQ, kblk, n, M, N, out, err, st);
}

cudaError_t launch_transpose_experts(const __nv_bfloat16 *in, int n, int R, int C,
                                     __nv_bfloat16 *out, cudaStream_t st) {
    bt_transpose_w<<<dim3(C / 64, R / 64, n), 256, 0, st>>>(in, R, C, out);
    return cudaGetLastError();
}

cudaError_t launch_rows_scaled(const __nv_bfloat16 *dy, const float *G, const int32_t *perm,
                               int64_t S, int d, int k, __nv_bfloat16 *dE, int32_t *err,
                               cudaStream_t st) {
    bt_rows_scaled<<<static_cast<unsigned>((S + 7) / 8), 256, 0, st>>>(dy, G, perm, S, d, k, dE, err);
    return cudaGetLastError();
}

cudaError_t launch_relu_mask(__nv_bfloat16 *x, const __nv_bfloat16 *hid, int64_t count,
                             cudaStream_t st) {
    const int64_t n8 = count / 8;
    bt_mask<<<static_cast<unsigned>((n8 + 255) / 256), 256, 0, st>>>(x, hid, n8);
    return cudaGetLastError();
}

cudaError_t launch_transpose_pad(const __nv_bfloat16 *in, int M, const int32_t *offsets,
                                 const int32_t *kblk, int n, int64_t S, int64_t Kcap,
                                 __nv_bfloat16 *out, cudaStream_t st) {
    const unsigned max_rt = static_cast<unsigned>((S + 63) / 64 + n);
    bt_transpose_pad<<<dim3(max_rt, M / 64), 256, 0, st>>>(in, M, offsets, kblk, n, Kcap, out);
    return cudaGetLastError();
}

}  // namespace moe

// gate_tc.cu -- noisy top-k gating on the tensor cores ("MoE:稀疏门控混合专家",
// sections 三 and 四), for bf16 x.
//
// The scores x.W_g and x.W_noise must be fp32-faithful, but W is fp32.  x is
// exact in bf16, so W is split once per call into two bf16 terms,
// W = W_hi + W_lo (W_hi = bf16(W), W_lo = bf16(W - W_hi); the residual is
// below 2^-16 |W|), and the scores are x.W_hi + x.W_lo accumulated in fp32 by
// tcgen05.mma: every product is exact and the sum carries fp32 rounding only,
// like an fp32 dot product.
//
//   gate_pack       W_g, W_noise [d, C] fp32 -> Bhi, Blo [chunks*128, d] bf16,
//                   K-major: chunk c holds 64 clean-score columns (rows 0..63)
//                   and the same 64 noise-score columns (rows 64..127).
//                   Hierarchical: the G group columns come first (padded to a
//                   chunk boundary), then the n inner columns.
//   gate_tc         persistent over 128-token tiles.  Warp 0 issues TMA loads,
//                   warp 1 issues tcgen05.mma (M=128 tokens, N=128 = 64 clean +
//                   64 noise columns, hi then lo pass into one fp32 accumulator,
//                   double-buffered in tensor memory), warps 2..5 are the
//                   epilogue: thread r owns token r of the tile (tensor-memory
//                   lane r), adds b_g, eps * softplus(noise score), keeps its
//                   running top-k in registers (KeepTopK, ties to the lower
//                   index) and finishes with the softmax over the k survivors.
//                   Hierarchical gating picks the groups from the first chunks
//                   and only then looks at (and reads eps for) the inner
//                   columns of its chosen groups.
// x stays resident in shared memory for the whole tile when d <= 512;
// otherwise each stage carries its x block with the W blocks.
#include "moe_device.cuh"
#include "moe_launch.h"

#include <float.h>
#include <limits.h>

#include <mutex>

namespace moe {

namespace {

constexpr int kGateChunk = 64;       // score columns (clean and noise each) per chunk
constexpr int kGateRows = 128;       // tokens per tile
constexpr int kGateBK = 64;          // d per k-block
constexpr int kKBytes = 128 * 64 * 2;  // one 128 x 64 bf16 block: 16 KB

// ---------------------------------------------------------------------------
// Packing
// ---------------------------------------------------------------------------
// Logical chunk column lc -> source column of W (or -1 for padding).
__host__ __device__ __forceinline__ int gate_source_col(int lc, int C, int groups, int prim_pad) {
    if (groups == 0) return lc < C ? lc : -1;
    if (lc < prim_pad) return lc < groups ? lc : -1;
    const int ic = lc - prim_pad;
    return ic < C - groups ? groups + ic : -1;
}

// Block: 64 d-rows x 64 logical columns of one matrix (clean or noise).
__global__ void __launch_bounds__(256) gate_pack(const float *__restrict__ Wg,
                                                 const float *__restrict__ Wn, int d, int C,
                                                 int groups, int prim_pad, int noisy,
                                                 __nv_bfloat16 *__restrict__ Bhi,
                                                 __nv_bfloat16 *__restrict__ Blo) {
    __shared__ float tile[64][65];
    const int chunk = blockIdx.x;
    const int which = blockIdx.y;  // 0 clean, 1 noise
    const int d0 = blockIdx.z * 64;
    const float *W = which ? Wn : Wg;
    const int tx = threadIdx.x % 64, ty = threadIdx.x / 64;
    const int src = gate_source_col(chunk * kGateChunk + tx, C, groups, prim_pad);
    for (int r = ty; r < 64; r += 4) {
        float v = 0.0f;
        if (src >= 0 && (which == 0 || noisy)) v = W[static_cast<int64_t>(d0 + r) * C + src];
        tile[r][tx] = v;  // tile[d][col]
    }
    __syncthreads();
    // Write rows (one per column) of 64 d-values: thread (col = ty.., dd = tx).
    for (int cc = ty; cc < 64; cc += 4) {
        const float v = tile[tx][cc];
        const __nv_bfloat16 hi = __float2bfloat16_rn(v);
        const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
        const int64_t row = static_cast<int64_t>(chunk) * 128 + which * 64 + cc;
        Bhi[row * d + d0 + tx] = hi;
        Blo[row * d + d0 + tx] = lo;
    }
}

// ---------------------------------------------------------------------------
// Per-token running top-k (registers only; all indices compile-time)
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool better(float a, int ia, float b, int ib) {
    return a > b || (a == b && ia < ib);
}

template <int KM>
struct TopK {
    float v[KM];
    int i[KM];
    __device__ __forceinline__ void reset() {
#pragma unroll
        for (int q = 0; q < KM; ++q) {
            v[q] = -INFINITY;
            i[q] = INT_MAX;
        }
    }
    // Entry kk-1 (kk <= KM) is the current k-th best.
    __device__ __forceinline__ float kth(int kk) const {
        float r = v[0];
#pragma unroll
        for (int q = 0; q < KM; ++q)
            if (q == kk - 1) r = v[q];
        return r;
    }
    __device__ __forceinline__ void insert(float cv, int ci) {
#pragma unroll
        for (int p = 0; p < KM; ++p) {
            if (better(cv, ci, v[p], i[p])) {
                const float tv = v[p];
                const int ti = i[p];
                v[p] = cv;
                i[p] = ci;
                cv = tv;
                ci = ti;
            }
        }
    }
};

// Softmax over the first kk entries (descending): w[q] = e^(v[q]-v[0]) / sum.
template <int KM>
__device__ __forceinline__ void softmax_top(const TopK<KM> &t, int kk, float (&w)[KM]) {
    float s = 0.0f;
#pragma unroll
    for (int q = 0; q < KM; ++q) {
        w[q] = 0.0f;
        if (q < kk) {
            w[q] = expf(t.v[q] - t.v[0]);
            s += w[q];
        }
    }
    const float inv = 1.0f / s;
#pragma unroll
    for (int q = 0; q < KM; ++q) w[q] *= inv;
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
template <bool kResident>
struct GateCfg {
    static constexpr int kStages = kResident ? 5 : 4;
    static constexpr int kStageBytes = kResident ? kKBytes : 3 * kKBytes;
    static constexpr int kXBytes = kResident ? 8 * kKBytes : 0;  // d <= 512
    static constexpr int kBarBytes = 8 * (2 * kStages + 7) + 16;
    static constexpr int kSmem = kXBytes + kStages * kStageBytes + 1024 + kBarBytes;
    static constexpr uint32_t kTmemCols = 256;  // 2 accumulators x 128 columns
};

struct GateArgs {
    const __nv_bfloat16 *x;
    const float *bg;
    const float *eps;
    int32_t *idx;
    float *G;
    int64_t T;
    int d, C, n, k;
    int groups, k_groups, m, prim_pad;
    int chunks, prim_chunks;
    int noisy;
    int32_t *err;
};

// KM: list size for flat (>= k) or for each hierarchical level (>= k_groups, k_inner).
template <bool kResident, bool kHier, int KM>
__global__ void __launch_bounds__(192, 1)
    gate_tc(const __grid_constant__ CUtensorMap mapX, const __grid_constant__ CUtensorMap mapHi,
            const __grid_constant__ CUtensorMap mapLo, const GateArgs a) {
    using Cfg = GateCfg<kResident>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint8_t *sX = smem;                        // resident x tile (kResident)
    uint8_t *sS = smem + Cfg::kXBytes;         // stage ring
    uint64_t *bars = reinterpret_cast<uint64_t *>(sS + Cfg::kStages * Cfg::kStageBytes);
    // full[S], empty[S], tfull[2], tempty[2], xfull, xempty, drain
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * Cfg::kStages + 7);
    volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(tmem_slot + 1);
    constexpr int S = Cfg::kStages;
    auto full = [&](int s) { return smem_u32(bars + s); };
    auto empty = [&](int s) { return smem_u32(bars + S + s); };
    auto tfull = [&](int b) { return smem_u32(bars + 2 * S + b); };
    auto tempty = [&](int b) { return smem_u32(bars + 2 * S + 2 + b); };
    const uint32_t xfull = smem_u32(bars + 2 * S + 4);
    const uint32_t xempty = smem_u32(bars + 2 * S + 5);
    const uint32_t drain_bar = smem_u32(bars + 2 * S + 6);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull(b), 1);
            mbar_init(tempty(b), 128);
        }
        mbar_init(xfull, 1);
        mbar_init(xempty, 1);
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&mapX);
        tma_prefetch_map(&mapHi);
        tma_prefetch_map(&mapLo);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int tiles = static_cast<int>((a.T + kGateRows - 1) / kGateRows);
    const int kblocks = a.d / kGateBK;

    if (warp == 0) {
        // ------------------------------ producer ------------------------------
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, xphase = 0;
            bool ok = true;
            int64_t issued = 0;
            for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
                const int row0 = tile * kGateRows;
                if (kResident) {
                    if (!mbar_wait_bounded(xempty, xphase ^ 1u, abort_flag, a.err, kSiteTcProducer)) {
                        ok = false;
                        break;
                    }
                    xphase ^= 1u;
                    mbar_arrive_expect_tx(xfull, static_cast<uint32_t>(kblocks * kKBytes));
                    for (int kb = 0; kb < kblocks; ++kb)
                        tma_load_2d(smem_u32(sX + kb * kKBytes), &mapX, xfull, kb * kGateBK, row0);
                }
                for (int c = 0; c < a.chunks && ok; ++c) {
                    for (int kb = 0; kb < kblocks && ok; ++kb) {
                        for (int split = 0; split < (kResident ? 2 : 1); ++split) {
                            if (!mbar_wait_bounded(empty(stage), phase ^ 1u, abort_flag, a.err,
                                                   kSiteTcProducer)) {
                                ok = false;
                                break;
                            }
                            uint8_t *st = sS + stage * Cfg::kStageBytes;
                            if (kResident) {
                                mbar_arrive_expect_tx(full(stage), kKBytes);
                                tma_load_2d(smem_u32(st), split ? &mapLo : &mapHi, full(stage),
                                            kb * kGateBK, c * 128);
                            } else {
                                mbar_arrive_expect_tx(full(stage), 3 * kKBytes);
                                tma_load_2d(smem_u32(st), &mapX, full(stage), kb * kGateBK, row0);
                                tma_load_2d(smem_u32(st + kKBytes), &mapHi, full(stage),
                                            kb * kGateBK, c * 128);
                                tma_load_2d(smem_u32(st + 2 * kKBytes), &mapLo, full(stage),
                                            kb * kGateBK, c * 128);
                            }
                            ++issued;
                            if (++stage == S) {
                                stage = 0;
                                phase ^= 1u;
                            }
                        }
                    }
                }
            }
            if (!ok) {  // let issued copies land before the CTA exits
                const int outstanding = static_cast<int>(issued < S ? issued : S);
                int s = stage;
                uint32_t p = phase;
                for (int i = 0; i < outstanding; ++i) {
                    if (--s < 0) {
                        s = S - 1;
                        p ^= 1u;
                    }
                    const uint64_t t0 = global_ns();
                    while (!mbar_try_wait(full(s), p) && global_ns() - t0 < kWaitLimitNs) {
                    }
                }
                if (kResident) {
                    const uint64_t t0 = global_ns();
                    while (!mbar_try_wait(xfull, xphase ^ 1u) && global_ns() - t0 < kWaitLimitNs) {
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------ MMA issuer ----------------------------
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(128, 128);
            int stage = 0;
            uint32_t phase = 0, xphase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
                if (kResident) {
                    if (!mbar_wait_bounded(xfull, xphase, abort_flag, a.err, kSiteTcMma)) break;
                    xphase ^= 1u;
                }
                for (int c = 0; c < a.chunks && ok; ++c) {
                    if (!mbar_wait_bounded(tempty(acc), acc_phase ^ 1u, abort_flag, a.err,
                                           kSiteTcMma)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * 128);
                    for (int kb = 0; kb < kblocks && ok; ++kb) {
                        for (int split = 0; split < (kResident ? 2 : 1); ++split) {
                            if (!mbar_wait_bounded(full(stage), phase, abort_flag, a.err,
                                                   kSiteTcMma)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            const uint32_t st = smem_u32(sS + stage * Cfg::kStageBytes);
                            const uint32_t xa = kResident ? smem_u32(sX + kb * kKBytes) : st;
#pragma unroll
                            for (int kk = 0; kk < kGateBK / 16; ++kk) {
                                const uint64_t ad = sdesc_kmajor_sw128(xa + kk * 32);
                                if (kResident) {
                                    tc_mma_f16(d_tmem, ad, sdesc_kmajor_sw128(st + kk * 32), idesc,
                                               (kb | split | kk) != 0 ? 1u : 0u);
                                } else {
                                    tc_mma_f16(d_tmem, ad,
                                               sdesc_kmajor_sw128(st + kKBytes + kk * 32), idesc,
                                               (kb | kk) != 0 ? 1u : 0u);
                                    tc_mma_f16(d_tmem, ad,
                                               sdesc_kmajor_sw128(st + 2 * kKBytes + kk * 32),
                                               idesc, 1u);
                                }
                            }
                            tc_commit(empty(stage));
                            if (++stage == S) {
                                stage = 0;
                                phase ^= 1u;
                            }
                        }
                    }
                    if (!ok) break;
                    tc_commit(tfull(acc));
                    if (++acc == 2) {
                        acc = 0;
                        acc_phase ^= 1u;
                    }
                }
                if (kResident && ok) tc_commit(xempty);
            }
            // Wait for every MMA issued by this thread before teardown.
            tc_commit(drain_bar);
            const uint64_t t0 = global_ns();
            while (!mbar_try_wait(drain_bar, 0) && global_ns() - t0 < kWaitLimitNs) {
            }
        }
    } else {
        // ------------------------------ epilogue ------------------------------
        const int quad = warp & 3;
        const int r = quad * 32 + lane;
        const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
        const int k_inner = kHier ? a.k / a.k_groups : a.k;
        int acc = 0;
        uint32_t acc_phase = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
            const int64_t t = static_cast<int64_t>(tile) * kGateRows + r;
            const bool valid = t < a.T;
            const float *eps_row = (valid && a.noisy) ? a.eps + t * a.C : nullptr;
            TopK<KM> prim;      // flat: the only list; hierarchical: the groups
            TopK<KM> inner[kHier ? KM : 1];
            prim.reset();
#pragma unroll
            for (int q = 0; q < (kHier ? KM : 1); ++q) inner[q].reset();
            float gw[KM];
            int kk_prim = kHier ? a.k_groups : a.k;
            for (int c = 0; c < a.chunks; ++c) {
                if (!mbar_wait_bounded(tfull(acc), acc_phase, abort_flag, a.err, kSiteTcEpilogue)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (kHier && c == a.prim_chunks) softmax_top<KM>(prim, kk_prim, gw);
#pragma unroll 1
                for (int half = 0; half < 2; ++half) {
                    uint32_t cv[32], nv[32];
                    const uint32_t col = static_cast<uint32_t>(acc * 128 + half * 32);
                    tmem_ld_32x32b_x32(tmem_base + lane_addr + col, cv);
                    tmem_ld_32x32b_x32(tmem_base + lane_addr + col + 64, nv);
                    tmem_ld_wait();
                    if (half == 1) {
                        tc_fence_before();
                        mbar_arrive(tempty(acc));  // accumulator fully read
                    }
                    if (!valid) continue;
                    const int lc0 = c * kGateChunk + half * 32;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int lc = lc0 + j;
                        int col_src;
                        int rank = 0;
                        if (!kHier) {
                            if (lc >= a.C) break;
                            col_src = lc;
                        } else if (c < a.prim_chunks) {
                            if (lc >= a.groups) break;
                            col_src = lc;
                        } else {
                            const int ic = lc - a.prim_pad;
                            if (ic >= a.n) break;
                            const int g = ic / a.m;
                            rank = -1;
#pragma unroll
                            for (int q = 0; q < KM; ++q)
                                if (q < a.k_groups && prim.i[q] == g) rank = q;
                            if (rank < 0) continue;
                            col_src = a.groups + ic;
                        }
                        float hv = __uint_as_float(cv[j]);
                        if (a.bg) hv += a.bg[col_src];
                        if (eps_row) hv += eps_row[col_src] * softplus_f(__uint_as_float(nv[j]));
                        const int id = kHier && c >= a.prim_chunks ? (lc - a.prim_pad) % a.m : col_src;
                        if (!kHier || c < a.prim_chunks) {
                            prim.insert(hv, id);
                        } else {
#pragma unroll
                            for (int q = 0; q < (kHier ? KM : 1); ++q)
                                if (q == rank) inner[q].insert(hv, id);
                        }
                    }
                }
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            if (!ok || !valid) continue;
            if (!kHier) {
                float w[KM];
                softmax_top<KM>(prim, a.k, w);
#pragma unroll
                for (int q = 0; q < KM; ++q)
                    if (q < a.k) {
                        a.idx[t * a.k + q] = prim.i[q];
                        a.G[t * a.k + q] = w[q];
                    }
            } else {
                if (a.prim_chunks == a.chunks) softmax_top<KM>(prim, kk_prim, gw);
#pragma unroll
                for (int q = 0; q < KM; ++q) {
                    if (q >= a.k_groups) break;
                    float wi[KM];
                    softmax_top<KM>(inner[q], k_inner, wi);
                    const int g = prim.i[q];
#pragma unroll
                    for (int e = 0; e < KM; ++e)
                        if (e < k_inner) {
                            a.idx[t * a.k + q * k_inner + e] = g * a.m + inner[q].i[e];
                            a.G[t * a.k + q * k_inner + e] = gw[q] * wi[e];
                        }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, Cfg::kTmemCols);
}

// --- host side --------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn gate_encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

bool gate_map(CUtensorMap *m, const void *base, uint64_t inner, uint64_t rows) {
    EncodeTiledFn enc = gate_encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {inner * 2};
    cuuint32_t box[2] = {64, 128};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool kResident, bool kHier, int KM>
cudaError_t launch_gate_tc_t(const CUtensorMap &mx, const CUtensorMap &mh, const CUtensorMap &ml,
                             const GateArgs &ga, int grid, cudaStream_t st) {
    using Cfg = GateCfg<kResident>;
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [] {
        attr = cudaFuncSetAttribute(gate_tc<kResident, kHier, KM>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
    });
    if (attr != cudaSuccess) return attr;
    gate_tc<kResident, kHier, KM><<<grid, 192, Cfg::kSmem, st>>>(mx, mh, ml, ga);
    return cudaGetLastError();
}

template <bool kResident, bool kHier>
cudaError_t launch_gate_tc_km(int km, const CUtensorMap &mx, const CUtensorMap &mh,
                              const CUtensorMap &ml, const GateArgs &ga, int grid,
                              cudaStream_t st) {
    if (km <= 2) return launch_gate_tc_t<kResident, kHier, 2>(mx, mh, ml, ga, grid, st);
    if (km <= 4) return launch_gate_tc_t<kResident, kHier, 4>(mx, mh, ml, ga, grid, st);
    if constexpr (kHier) {
        return cudaErrorInvalidValue;  // hierarchical lists are limited to 4
    } else {
        if (km <= 8) return launch_gate_tc_t<kResident, kHier, 8>(mx, mh, ml, ga, grid, st);
        return launch_gate_tc_t<kResident, kHier, 16>(mx, mh, ml, ga, grid, st);
    }
}

}  // namespace

size_t gate_tc_pack_bytes(const moe_shape &s) {
    const int C = gate_cols(s);
    int chunks;
    if (s.groups == 0) {
        chunks = (C + kGateChunk - 1) / kGateChunk;
    } else {
        chunks = (s.groups + kGateChunk - 1) / kGateChunk + (s.n + kGateChunk - 1) / kGateChunk;
    }
    return static_cast<size_t>(chunks) * 128 * s.d * 2 * 2;  // hi + lo
}

bool gate_tc_supported(const moe_shape &s) {
    if (s.dtype != MOE_BF16) return false;
    if (s.groups == 0) return s.k <= 16;
    return s.k_groups <= 4 && s.k / s.k_groups <= 4;
}

cudaError_t launch_gate_tc(const moe_shape &s, const void *x, const float *Wg, const float *Wn,
                           const float *bg, const float *eps, int32_t *idx, float *G, void *pack,
                           int32_t *err, cudaStream_t st) {
    const int C = gate_cols(s);
    const int noisy = (s.noisy && eps != nullptr && Wn != nullptr) ? 1 : 0;
    GateArgs ga;
    ga.x = static_cast<const __nv_bfloat16 *>(x);
    ga.bg = bg;
    ga.eps = eps;
    ga.idx = idx;
    ga.G = G;
    ga.T = s.T;
    ga.d = s.d;
    ga.C = C;
    ga.n = s.n;
    ga.k = s.k;
    ga.groups = s.groups;
    ga.k_groups = s.k_groups;
    ga.m = s.groups ? s.n / s.groups : s.n;
    ga.noisy = noisy;
    ga.err = err;
    if (s.groups == 0) {
        ga.prim_pad = 0;
        ga.prim_chunks = 0;
        ga.chunks = (C + kGateChunk - 1) / kGateChunk;
    } else {
        ga.prim_chunks = (s.groups + kGateChunk - 1) / kGateChunk;
        ga.prim_pad = ga.prim_chunks * kGateChunk;
        ga.chunks = ga.prim_chunks + (s.n + kGateChunk - 1) / kGateChunk;
    }
    __nv_bfloat16 *Bhi = static_cast<__nv_bfloat16 *>(pack);
    __nv_bfloat16 *Blo = Bhi + static_cast<size_t>(ga.chunks) * 128 * s.d;
    gate_pack<<<dim3(ga.chunks, 2, s.d / 64), 256, 0, st>>>(Wg, noisy ? Wn : Wg, s.d, C, s.groups,
                                                          ga.prim_pad, noisy, Bhi, Blo);
    CUtensorMap mx, mh, ml;
    if (!gate_map(&mx, x, s.d, static_cast<uint64_t>(s.T)) ||
        !gate_map(&mh, Bhi, s.d, static_cast<uint64_t>(ga.chunks) * 128) ||
        !gate_map(&ml, Blo, s.d, static_cast<uint64_t>(ga.chunks) * 128))
        return cudaErrorInvalidValue;
    const int tiles = static_cast<int>((s.T + kGateRows - 1) / kGateRows);
    const int grid = tiles < sm_count() ? tiles : sm_count();
    const bool resident = s.d <= 512;
    const int km = s.groups ? (s.k_groups > s.k / s.k_groups ? s.k_groups : s.k / s.k_groups) : s.k;
    if (resident)
        return s.groups ? launch_gate_tc_km<true, true>(km, mx, mh, ml, ga, grid, st)
                        : launch_gate_tc_km<true, false>(km, mx, mh, ml, ga, grid, st);
    return s.groups ? launch_gate_tc_km<false, true>(km, mx, mh, ml, ga, grid, st)
                    : launch_gate_tc_km<false, false>(km, mx, mh, ml, ga, grid, st);
}

}  // namespace moe

// ffn_tc.cu -- grouped per-expert GEMM on the 5th-generation tensor cores.
//
// One launch computes, for every expert e and every 128-row block of that
// expert's rows (rows in expert order, offsets[e] .. offsets[e+1]) and every
// BN-column block of the output:
//     out[r, c] = act( sum_k A[r, k] * B[e*N + c, k] + bias[e, c] )
// with A the activations [S, K] (bf16, K contiguous), B the experts' weights
// [n*N, K] (bf16, K contiguous: each expert is an out x in matrix), fp32
// accumulation in tensor memory, act = ReLU or identity, and one RNE rounding
// of the result to bf16.  Used twice per forward pass: the first layer
// (A = x rows in expert order, B = W1, N = h, ReLU) and the second layer
// (A = hidden, B = W2, N = d).  The experts are one-hidden-layer ReLU
// networks ("MoE:稀疏门控混合专家", section 二).
//
// Structure (one CTA per SM, persistent over a static tile sequence):
//   warp 0       TMA producer: per stage one copy each of A (128 rows) and B
//                (BN rows) of one 64-wide k-block, 128-byte swizzle, into a
//                STAGES-deep shared-memory ring (192 KB in all: the weights
//                come from HBM and the ring must cover that latency)
//   warp 1       allocates tensor memory; one lane issues tcgen05.mma
//                (M = 128, N = BN, K = 16) and commits each stage back to the
//                producer and each finished accumulator to the epilogue
//   warps 2..9   epilogue: tcgen05.ld of the accumulator (two warps per
//                32-lane quarter, each one half of the columns, the next 32
//                columns in flight while the current ones are converted),
//                bias, activation, bf16 rounding, 16-byte stores
// The accumulator is double-buffered in tensor memory (2 x BN columns) so
// the epilogue of one tile overlaps the main loop of the next.  Every wait is
// bounded; on a timeout the kernel records MOE_ERR_TIMEOUT, drains its own
// copies and MMAs, frees tensor memory and returns.
#include "moe_device.cuh"
#include "moe_launch.h"

#include <mutex>

namespace moe {

namespace {

template <int BN, int STAGES>
struct TcCfg {
    static constexpr int kBM = kTcRows;
    static constexpr int kBK = 64;       // K per swizzle atom row (128 bytes)
    static constexpr int kKB = 1;        // k-blocks per stage (one 3-D TMA box each)
    static constexpr int kABytes = kBM * kBK * 2 * kKB;
    static constexpr int kBBytes = BN * kBK * 2 * kKB;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kBarBytes = 8 * (2 * STAGES + 5) + 16;
    static constexpr int kSmem = STAGES * kStageBytes + 1024 + kBarBytes;
    static constexpr uint32_t kTmemCols = 2 * BN;
    static_assert(kTmemCols >= 32 && kTmemCols <= 512 && (kTmemCols & (kTmemCols - 1)) == 0, "");
};

struct TileInfo {
    int e, row0, rows, cb;
};

__device__ __forceinline__ TileInfo decode_tile(int q, int ncb, const int32_t *__restrict__ tiles,
                                                int n, const int32_t *__restrict__ offsets) {
    TileInfo ti;
    const int rt = q / ncb;
    ti.cb = q - rt * ncb;
    int lo = 0, hi = n - 1;  // largest e with tiles[e] <= rt
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tiles[mid] <= rt)
            lo = mid;
        else
            hi = mid - 1;
    }
    ti.e = lo;
    ti.row0 = offsets[lo] + (rt - tiles[lo]) * kTcRows;
    ti.rows = min(kTcRows, offsets[lo + 1] - ti.row0);
    return ti;
}

// Bounded wait that ignores the abort flag (used to drain in-flight work).
__device__ __forceinline__ bool mbar_drain(uint32_t bar, uint32_t parity, int32_t *err) {
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_ns() - t0 > kWaitLimitNs) {
            report(err, MOE_ERR_TIMEOUT, kSiteTcDrain);
            return false;
        }
    }
    return true;
}

constexpr int kFfnEpiWarps = 8;  // two per tensor-memory lane quarter
constexpr int kFfnThreads = 32 * (2 + kFfnEpiWarps);

template <int BN, int STAGES>
__global__ void __launch_bounds__(kFfnThreads, 1)
    ffn_gemm_tc(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                const int32_t *__restrict__ offsets, const int32_t *__restrict__ tiles, int n,
                int K, int N, const float *__restrict__ bias, int relu,
                __nv_bfloat16 *__restrict__ out, int out_v8, int32_t *err) {
    using Cfg = TcCfg<BN, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint8_t *sA = smem;
    uint8_t *sB = smem + STAGES * Cfg::kABytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sB + STAGES * Cfg::kBBytes);
    // bars: full[STAGES], empty[STAGES], tfull[2], tempty[2], drain[1]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * STAGES + 5);
    volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(tmem_slot + 1);
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
            mbar_init(tempty(b), 32 * kFfnEpiWarps);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&mapA);
        tma_prefetch_map(&mapB);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int ncb = N / BN;
    const int total = tiles[n] * ncb;
    const int kblocks = K / Cfg::kBK;
    const int kstages = (kblocks + Cfg::kKB - 1) / Cfg::kKB;  // a missing last k-block reads as zeros

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int64_t issued = 0;
            bool ok = true;
            for (int q = blockIdx.x; q < total && ok; q += gridDim.x) {
                const TileInfo ti = decode_tile(q, ncb, tiles, n, offsets);
                const int brow = ti.e * N + ti.cb * BN;
                for (int ks = 0; ks < kstages; ++ks) {
                    if (!mbar_wait_bounded(empty(stage), phase ^ 1u, abort_flag, err,
                                           kSiteTcProducer)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(full(stage), Cfg::kStageBytes);
                    tma_load_3d(smem_u32(sA + stage * Cfg::kABytes), &mapA, full(stage), 0, ti.row0,
                                ks * Cfg::kKB);
                    tma_load_3d(smem_u32(sB + stage * Cfg::kBBytes), &mapB, full(stage), 0, brow,
                                ks * Cfg::kKB);
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                // Let the copies already issued land before the CTA goes away.
                const int outstanding = static_cast<int>(issued < STAGES ? issued : STAGES);
                int s = stage;
                uint32_t p = phase;
                for (int i = 0; i < outstanding; ++i) {
                    if (--s < 0) {
                        s = STAGES - 1;
                        p ^= 1u;
                    }
                    mbar_drain(full(s), p, err);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(kTcRows, BN);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int q = blockIdx.x; q < total && ok; q += gridDim.x) {
                if (!mbar_wait_bounded(tempty(acc), acc_phase ^ 1u, abort_flag, err, kSiteTcMma))
                    break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int ks = 0; ks < kstages; ++ks) {
                    if (!mbar_wait_bounded(full(stage), phase, abort_flag, err, kSiteTcMma)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(sA + stage * Cfg::kABytes);
                    const uint32_t b0 = smem_u32(sB + stage * Cfg::kBBytes);
                    const int nkb = min(Cfg::kKB, kblocks - ks * Cfg::kKB);
                    for (int kb = 0; kb < nkb; ++kb) {
                        const uint32_t ak = a0 + kb * (Cfg::kBM * 128);
                        const uint32_t bk = b0 + kb * (BN * 128);
#pragma unroll
                        for (int kk = 0; kk < Cfg::kBK / 16; ++kk)
                            tc_mma_f16(d_tmem, sdesc_kmajor_sw128(ak + kk * 32),
                                       sdesc_kmajor_sw128(bk + kk * 32), idesc,
                                       (ks | kb | kk) != 0 ? 1u : 0u);
                    }
                    tc_commit(empty(stage));
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                tc_commit(tfull(acc));
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            // Every MMA this thread issued has finished once this arrives.
            tc_commit(drain_bar);
            mbar_drain(drain_bar, 0, err);
        }
    } else {
        // Epilogue: warp w (2..9) reads tensor-memory lanes 32*(w%4).. (rows
        // of the tile) and one half of the tile's columns, 32 at a time; the
        // next 32 columns are already being read while these are converted.
        const int quad = warp & 3;
        const int half = (warp - 2) >> 2;
        constexpr int kHalf = BN / 2;
        constexpr int kChunks = kHalf / 32;
        const int r = quad * 32 + lane;
        const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int q = blockIdx.x; q < total; q += gridDim.x) {
            const TileInfo ti = decode_tile(q, ncb, tiles, n, offsets);
            if (!mbar_wait_bounded(tfull(acc), acc_phase, abort_flag, err, kSiteTcEpilogue)) break;
            tc_fence_after();
            const bool valid = r < ti.rows;
            const int col0 = ti.cb * BN + half * kHalf;
            const float *bp = bias ? bias + static_cast<int64_t>(ti.e) * N + col0 : nullptr;
            __nv_bfloat16 *orow = out + (static_cast<int64_t>(ti.row0) + r) * N + col0;
            const uint32_t tbase = tmem_base + lane_addr + static_cast<uint32_t>(acc * BN + half * kHalf);
            uint32_t v[2][32];
            tmem_ld_32x32b_x32(tbase, v[0]);
#pragma unroll
            for (int ch = 0; ch < kChunks; ++ch) {
                tmem_ld_wait();
                if (ch + 1 < kChunks) tmem_ld_32x32b_x32(tbase + (ch + 1) * 32, v[(ch + 1) & 1]);
                if (ch + 1 == kChunks) {
                    tc_fence_before();
                    mbar_arrive(tempty(acc));  // this half of the accumulator is read
                }
                if (valid) {
                    float b[32];
                    if (bp) {
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const float4 t = __ldg(reinterpret_cast<const float4 *>(bp + ch * 32) + j);
                            b[4 * j] = t.x;
                            b[4 * j + 1] = t.y;
                            b[4 * j + 2] = t.z;
                            b[4 * j + 3] = t.w;
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) b[j] = 0.0f;
                    }
                    uint32_t pk[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        float f0 = __uint_as_float(v[ch & 1][2 * j]) + b[2 * j];
                        float f1 = __uint_as_float(v[ch & 1][2 * j + 1]) + b[2 * j + 1];
                        if (relu) {
                            f0 = fmaxf(f0, 0.0f);
                            f1 = fmaxf(f1, 0.0f);
                        }
                        pk[j] = pack_bf16x2(f0, f1);
                    }
                    if (out_v8) {
                        st_global_v8(orow + ch * 32, pk);
                        st_global_v8(orow + ch * 32 + 16, pk + 8);
                    } else {
                        uint4 *dst = reinterpret_cast<uint4 *>(orow + ch * 32);
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            dst[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
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

template <int BN, int STAGES>
cudaError_t launch_bn(const CUtensorMap &mA, const CUtensorMap &mB, const int32_t *offsets,
                      const int32_t *tiles, int n, int K, int N, const float *bias, int relu,
                      __nv_bfloat16 *out, int32_t *err, int grid, cudaStream_t st) {
    const int out_v8 = (reinterpret_cast<uintptr_t>(out) & 31u) == 0 ? 1 : 0;
    using Cfg = TcCfg<BN, STAGES>;
    // The opt-in above 48 KB of dynamic shared memory belongs to the current
    // device's context, so it is set before every launch (a cheap host call).
    cudaError_t attr_err = cudaFuncSetAttribute(
        ffn_gemm_tc<BN, STAGES>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
    if (attr_err != cudaSuccess) return attr_err;
    ffn_gemm_tc<BN, STAGES><<<grid, kFfnThreads, Cfg::kSmem, st>>>(mA, mB, offsets, tiles, n, K, N, bias,
                                                           relu, out, out_v8, err);
    return cudaGetLastError();
}

}  // namespace

// --- host side: tensor maps -------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
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

// bf16 matrix [rows, K] (K contiguous) seen as a 3-D tensor {64, rows, K/64}
// (strides K*2 and 128 bytes), box {64, box_rows, box_kblocks}: one copy
// brings box_kblocks 64-wide k-blocks of box_rows rows, each landing as a
// 128-byte-swizzled K-major tile; a k-block past K/64 reads as zeros.
bool make_kmajor_map(CUtensorMap *m, const void *base, uint64_t K, uint64_t rows, uint32_t box_rows,
                     uint32_t box_kblocks) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {64, rows, K / 64};
    cuuint64_t strides[2] = {K * 2, 128};
    cuuint32_t box[3] = {64, box_rows, box_kblocks};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_mnmajor_map(CUtensorMap *m, const void *base, uint64_t M, uint64_t rows,
                      uint32_t box_rows, uint32_t box_mblocks) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {64, rows, M / 64};
    cuuint64_t strides[2] = {M * 2, 128};
    cuuint32_t box[3] = {64, box_rows, box_mblocks};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int tc_block_n(int N) {
    if (N % 256 == 0) return 256;
    if (N % 128 == 0) return 128;
    return 64;
}

cudaError_t launch_grouped_gemm_tc(const moe_shape &s, const __nv_bfloat16 *A, int K,
                                   const __nv_bfloat16 *B, int N, const float *bias, int relu,
                                   const int32_t *offsets, const int32_t *tiles,
                                   __nv_bfloat16 *out, int32_t *err, cudaStream_t st) {
    const int64_t S = slots(s);
    CUtensorMap mA, mB;
    const int BN = tc_block_n(N);
    if (!make_kmajor_map(&mA, A, static_cast<uint64_t>(K), static_cast<uint64_t>(S), kTcRows) ||
        !make_kmajor_map(&mB, B, static_cast<uint64_t>(K), static_cast<uint64_t>(s.n) * N,
                  static_cast<uint32_t>(BN)))
        return cudaErrorInvalidValue;
    const int64_t max_tiles = ((S + kTcRows - 1) / kTcRows + s.n) * (N / BN);
    const int grid = static_cast<int>(max_tiles < sm_count() ? max_tiles : sm_count());
    if (BN == 256)
        return launch_bn<256, 4>(mA, mB, offsets, tiles, s.n, K, N, bias, relu, out, err, grid, st);
    if (BN == 128)
        return launch_bn<128, 6>(mA, mB, offsets, tiles, s.n, K, N, bias, relu, out, err, grid, st);
    return launch_bn<64, 8>(mA, mB, offsets, tiles, s.n, K, N, bias, relu, out, err, grid, st);
}

}  // namespace moe

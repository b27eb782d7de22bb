// ffn_pair.cu -- grouped per-expert GEMM on a pair of SMs (tcgen05 cta_group::2),
// with the experts' weight rows on the MMA's M side and the tokens on its N side.
//
// One launch computes, for every expert e, every token tile of e's rows
// (rows in expert order, offsets[e] .. offsets[e+1]) and every 256-row block
// of the expert's output features:
//     out[r, c] = act( sum_k X[r, k] * W[e*Nout + c, k] + bias[e*Nout + c] )
// with X the activations [S, K] (bf16, K contiguous), W the experts' weights
// [n*Nout, K] (bf16, out x in, K contiguous), fp32 accumulation in tensor
// memory, act = ReLU or identity and one RNE rounding to bf16.  Used for both
// layers of the experts' one-hidden-layer ReLU networks ("MoE:稀疏门控混合专家",
// section 二) when the layer's output width is a multiple of 256.
//
// Why this shape.  Each expert sees only about k*b/n rows of a batch
// ("Outrageously Large Neural Networks - 中文验证版", section 瓶颈): a few
// hundred at the widths this library targets.  Putting the tokens on N lets a
// tile take exactly the rows an expert has (N is any multiple of 16 up to
// 256), so no MMA work is spent on padding rows, and an expert of up to 256
// rows reads its weights once.  The pair MMA (M = 256: 128 weight rows from
// each SM, N tokens: N/2 rows from each SM) halves the operand bytes each SM
// takes in per output compared with a single-SM 128 x 256 tile, which is what
// limits the single-SM kernel on these shapes.
//
// Token tiles: an expert with R rows gets ceil(R / 256) tiles of Tn rows,
// Tn = ceil(R / tiles) rounded up to 16 (at most 256); the tile count is then
// ceil(R / Tn), so no tile is empty.  A tile's MMA N is its row count rounded
// up to 32 (so each SM's half is a multiple of 16 rows).  A unit of work is (token tile, block of
// 256 output features); units are numbered tile-major, so the feature blocks
// of one tile run side by side on different pairs and share its rows in L2.
//
// Structure (clusters of two CTAs, one CTA per SM, persistent):
//   warp 0     TMA producer in each CTA: per stage one copy of this CTA's 128
//              weight rows and one of its N/2 token rows (a box of exactly that
//              many rows, so no neighbouring rows are read), each of two 64-wide
//              k-blocks (128-byte swizzle, up to 64 KB); both CTAs' copies
//              complete on the even CTA's barrier.  A copy costs a fixed ~0.3 us of issue
//              time per SM up to 64 KB, so copies are made as large as the
//              three-stage ring allows
//   warp 1     tensor memory (512 columns, allocated by both CTAs together);
//              in the even CTA one lane issues the pair MMAs (M = 256,
//              N = tile rows rounded to 32, K = 16) and commits each stage and
//              each finished accumulator to the barriers of both CTAs
//   warps 2-17 epilogue in each CTA: tcgen05.ld of its 128 accumulator rows
//              (output features) x 32 token columns, bias, activation, bf16,
//              a 32 x 32 transpose through shared memory, and 64-byte row
//              stores of 32 consecutive features of one token
// The accumulator is double-buffered (2 x 256 columns).  Every wait is
// bounded; on a timeout the kernel records MOE_ERR_TIMEOUT and winds down.
#include "moe_device.cuh"
#include "moe_launch.h"

namespace moe {

namespace {

constexpr int kPairTok = 256;      // tokens per tile at most (MMA N)
constexpr int kPairM = 256;        // weight rows per unit (MMA M; 128 per CTA)
constexpr int kPairEpiPerQuad = 4;                      // epilogue warps per lane quarter
constexpr int kPairEpiWarps = 4 * kPairEpiPerQuad;
constexpr int kPairChunks = (kPairTok / 32) / kPairEpiPerQuad;   // 32-column chunks per warp
constexpr int kPairThreads = 32 * (2 + kPairEpiWarps);
constexpr int kPairKB = 2;          // 64-wide k-blocks per copy (one 3-D box)
constexpr int kPairStages = 3;

struct PairCfg {
    static constexpr int kKBlockBytes = 128 * 64 * 2;           // 128 rows x one 64-wide k-block
    static constexpr int kABytes = kPairKB * kKBlockBytes;      // this CTA's 128 weight rows
    static constexpr int kBBytes = kPairKB * kKBlockBytes;      // up to 128 token rows of this CTA
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kStagingBytes = kPairEpiWarps * 32 * 64;   // 32 x 32 bf16 per warp
    static constexpr int kBarBytes = 8 * (2 * kPairStages + 5) + 16;
    static constexpr int kSmem = 1024 + kPairStages * kStageBytes + kStagingBytes + kBarBytes;
    static constexpr uint32_t kTmemCols = 2 * kPairTok;
};
static_assert(PairCfg::kSmem <= 227 * 1024, "shared memory budget");

struct PairUnit {
    int e, row0, rows, N, mt;
};

// Token-row maps of one activation matrix, box i holding 16*(i+1) rows and
// two k-blocks: a unit of N tokens copies exactly its N/2 rows per CTA.
struct XMaps {
    CUtensorMap m[8];
};

// Unit q -> expert, token tile and block of output features, from the
// token-tile table (one 16-byte entry per tile: expert, first row, rows, N).
__device__ __forceinline__ PairUnit unit_of(int4 t, int mt) {
    PairUnit u;
    u.e = t.x;
    u.row0 = t.y;
    u.rows = t.z;
    u.N = t.w;
    u.mt = mt;
    return u;
}

// One block of 1024 threads: tiles[e] = token tiles (at most cap rows each)
// of the experts before e (tiles[n] = all of them), and the table entry of
// every tile.
__global__ void __launch_bounds__(1024) ffn_pair_tiles(const int32_t *__restrict__ offsets, int n,
                                                       int32_t *__restrict__ tiles,
                                                       int4 *__restrict__ tlist, int cap) {
    __shared__ int32_t part[1024];
    const int per = (n + 1023) / 1024;
    const int i0 = threadIdx.x * per, i1 = min(n, i0 + per);
    int32_t sum = 0;
    for (int i = i0; i < i1; ++i) {
        int tn, nt;
        token_tiling(offsets[i + 1] - offsets[i], tn, nt, cap);
        sum += nt;
    }
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
        const int R = offsets[i + 1] - offsets[i];
        int tn, nt;
        token_tiling(R, tn, nt, cap);
        for (int j = 0; j < nt; ++j) {
            const int rows = min(tn, R - j * tn);
            tlist[run + j] = make_int4(i, offsets[i] + j * tn, rows, (rows + 31) & ~31);
        }
        run += nt;
    }
    if (threadIdx.x == 1023) tiles[n] = part[1023];
}

// Bounded wait that ignores the abort flag (used to drain in-flight MMAs).
__device__ __forceinline__ bool pair_drain(uint32_t bar, uint32_t parity, int32_t *err) {
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_ns() - t0 > kWaitLimitNs) {
            report(err, MOE_ERR_TIMEOUT, kSiteTcDrain);
            return false;
        }
    }
    return true;
}

// kAMn: the weights are read in their stored layout [n*K, Nout] (rows k of
// expert e at e*K + k) as an MN-major operand, instead of [n*Nout, K].
template <bool kAMn>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPairThreads, 1)
    ffn_pair_gemm(const __grid_constant__ CUtensorMap mapW, const __grid_constant__ XMaps mapX,
                  const int32_t *__restrict__ tiles, const int4 *__restrict__ tlist, int n,
                  int K, int Nout, const __nv_bfloat16 *__restrict__ Wg,
                  const __nv_bfloat16 *__restrict__ Xg, const float *__restrict__ bias, int relu,
                  __nv_bfloat16 *__restrict__ out, int out_v8, int32_t *err) {
    using Cfg = PairCfg;
    constexpr int STAGES = kPairStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint8_t *sA = smem;                                  // STAGES x 16 KB weight rows
    uint8_t *sB = smem + STAGES * Cfg::kABytes;          // STAGES x 16 KB token rows
    uint8_t *stg = sB + STAGES * Cfg::kBBytes;           // epilogue transposes
    uint64_t *bars = reinterpret_cast<uint64_t *>(stg + Cfg::kStagingBytes);
    // bars: full[STAGES], empty[STAGES], tfull[2], tempty[2], drain
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * STAGES + 5);
    volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(tmem_slot + 1);
    auto full = [&](int s) { return smem_u32(bars + s); };
    auto empty = [&](int s) { return smem_u32(bars + STAGES + s); };
    auto tfull = [&](int b) { return smem_u32(bars + 2 * STAGES + b); };
    auto tempty = [&](int b) { return smem_u32(bars + 2 * STAGES + 2 + b); };
    const uint32_t drain_bar = smem_u32(bars + 2 * STAGES + 4);

    const uint32_t rank = cluster_ctarank();   // 0: the CTA that issues the pair MMAs
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull(b), 1);
            mbar_init(tempty(b), 2 * kPairEpiWarps);   // one arrival per epilogue warp of each CTA
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&mapW);
        for (int i = 0; i < 8; ++i) tma_prefetch_map(&mapX.m[i]);
    }
    // A pair allocation is issued by one warp of each CTA once both CTAs are
    // known to be running; the second cluster barrier publishes the barriers
    // and the allocation to both CTAs before any copy, MMA or remote arrival.
    cluster_sync();
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), Cfg::kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // everything above is local; from here on the previous kernel's results are used
    pdl_wait();
    pdl_launch_dependents();

    const int nmt = Nout / kPairM;
    const int total = tiles[n] * nmt;
    const int kblocks = K / 64;
    const int cl = static_cast<int>(blockIdx.x >> 1), ncl = static_cast<int>(gridDim.x >> 1);

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int4 tcur = cl < total ? __ldg(tlist + cl / nmt) : make_int4(0, 0, 0, 0);
            for (int q = cl; q < total && ok; q += ncl) {
                const PairUnit u = unit_of(tcur, q % nmt);
                if (q + ncl < total) tcur = __ldg(tlist + (q + ncl) / nmt);   // next unit's entry
                const int wrow = u.e * Nout + u.mt * kPairM + static_cast<int>(rank) * 128;
                const int xrow = u.row0 + static_cast<int>(rank) * (u.N >> 1);
                for (int kb = 0; kb < kblocks; kb += kPairKB) {
                    if (!mbar_wait_bounded(empty(stage), phase ^ 1u, abort_flag, err,
                                           kSiteTcProducer)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = mapa_shared(full(stage), 0);
                    // this CTA's N/2 token rows (a multiple of 16) in one box
                    const int hrows = u.N >> 1;
                    if (rank == 0)
                        mbar_arrive_expect_tx(full(stage), 2 * (Cfg::kABytes + hrows * 128 * kPairKB));
                    if constexpr (kAMn) {
                        // K rows kb*64 .. +128 of expert e, this CTA's two 64-wide
                        // blocks of output features
                        tma_load_3d_pair(smem_u32(sA + stage * Cfg::kABytes), &mapW, fb, 0,
                                         u.e * K + kb * 64,
                                         (u.mt * kPairM + static_cast<int>(rank) * 128) / 64);
                    } else {
                        tma_load_3d_pair(smem_u32(sA + stage * Cfg::kABytes), &mapW, fb, 0, wrow, kb);
                    }
                    tma_load_3d_pair(smem_u32(sB + stage * Cfg::kBBytes), &mapX.m[(hrows >> 4) - 1], fb,
                                     0, xrow, kb);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                // Copies already issued complete within microseconds; give them
                // time to land before the CTA can leave.
                const uint64_t t0 = global_ns();
                while (global_ns() - t0 < 200000ull) {
                }
            }
        }
    } else if (warp == 1) {
        if (rank == 0 && lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            int4 tcur = cl < total ? __ldg(tlist + cl / nmt) : make_int4(0, 0, 0, 0);
            for (int q = cl; q < total && ok; q += ncl) {
                const PairUnit u = unit_of(tcur, q % nmt);
                if (q + ncl < total) tcur = __ldg(tlist + (q + ncl) / nmt);
                const uint32_t idesc =
                    kAMn ? idesc_bf16_f32_amn(kPairM, u.N) : idesc_bf16_f32(kPairM, u.N);
                if (!mbar_wait_bounded(tempty(acc), acc_phase ^ 1u, abort_flag, err, kSiteTcMma))
                    break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kPairTok);
                for (int kb = 0; kb < kblocks; kb += kPairKB) {
                    if (!mbar_wait_bounded(full(stage), phase, abort_flag, err, kSiteTcMma)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(sA + stage * Cfg::kABytes);
                    const uint32_t b0 = smem_u32(sB + stage * Cfg::kBBytes);
                    const uint32_t bkb = static_cast<uint32_t>(u.N >> 1) * 128;  // B k-block stride
                    // a k-block past K (the box's zero-filled tail) is skipped
                    const int nkb = min(kPairKB, kblocks - kb);
                    for (int j = 0; j < nkb; ++j) {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            tc_mma_f16_pair(d_tmem,
                                            kAMn ? sdesc_mnmajor_sw128(a0 + j * 64 * 128 + kk * 16 * 128,
                                                                       128 * 128)
                                                 : sdesc_kmajor_sw128(a0 + j * Cfg::kKBlockBytes + kk * 32),
                                            sdesc_kmajor_sw128(b0 + j * bkb + kk * 32),
                                            idesc, (kb | j | kk) != 0 ? 1u : 0u);
                    }
                    tc_commit_pair_both(empty(stage));
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                tc_commit_pair_both(tfull(acc));
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            // Every MMA this thread issued has finished once this arrives.
            tc_commit_pair_both(drain_bar);
            pair_drain(drain_bar, 0, err);
        }
    } else {
        // Epilogue: warp w (2..17) may read tensor-memory lanes 32*(w%4) ..
        // +32 (its output features); the four warps of a lane quarter take
        // every fourth 32-column chunk (tokens) of the tile.
        const int ew = warp - 2;
        const int quad = warp & 3;
        const int sub = ew >> 2;
        uint8_t *my = stg + ew * (32 * 64);
        const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
        int acc = 0;
        uint32_t acc_phase = 0;
        // the unit's table entry and bias value are loaded one unit ahead
        const int fq = static_cast<int>(rank) * 128 + quad * 32 + lane;   // feature in the block
        auto bias_of = [&](int4 t, int q) {
            return bias ? __ldg(bias + static_cast<int64_t>(t.x) * Nout + (q % nmt) * kPairM + fq)
                        : 0.0f;
        };
        int4 tcur = cl < total ? __ldg(tlist + cl / nmt) : make_int4(0, 0, 0, 0);
        float bnext = cl < total ? bias_of(tcur, cl) : 0.0f;
        for (int q = cl; q < total; q += ncl) {
            const PairUnit u = unit_of(tcur, q % nmt);
            const float bv = bnext;
            if (q + ncl < total) {
                tcur = __ldg(tlist + (q + ncl) / nmt);
                bnext = bias_of(tcur, q + ncl);
            }
            const int col0 = u.mt * kPairM + static_cast<int>(rank) * 128 + quad * 32;
            if (!mbar_wait_bounded(tfull(acc), acc_phase, abort_flag, err, kSiteTcEpilogue)) break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + lane_addr + static_cast<uint32_t>(acc * kPairTok);
            // Phase 1: this warp's chunks (32 token columns each) out of tensor
            // memory, biased, activated and packed to bf16 pairs of
            // neighbouring tokens; the accumulator is then released at once,
            // before any global store, so the next unit's MMAs need not wait
            // for the stores.
            uint32_t pk[kPairChunks][16];
#pragma unroll
            for (int i = 0; i < kPairChunks; ++i) {
                const int c = sub + kPairEpiPerQuad * i;
                uint32_t v[32];
                if (c * 32 < u.N) tmem_ld_32x32b_x32(tbase + c * 32, v);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    float f0 = __uint_as_float(v[2 * j]) + bv;
                    float f1 = __uint_as_float(v[2 * j + 1]) + bv;
                    if (relu) {
                        f0 = fmaxf(f0, 0.0f);
                        f1 = fmaxf(f1, 0.0f);
                    }
                    pk[i][j] = pack_bf16x2(f0, f1);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(mapa_shared(tempty(acc), 0));
            // Phase 2: per chunk, a 32 x 32 transpose through shared memory
            // (element (t, lane) of rows of 64 bytes whose four 16-byte pieces
            // are permuted by (t >> 1) & 3), then 64-byte row stores.
#pragma unroll
            for (int i = 0; i < kPairChunks; ++i) {
                const int c = sub + kPairEpiPerQuad * i;
                if (c * 32 >= u.N) continue;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int t0 = 2 * j, t1 = 2 * j + 1;
                    const uint32_t w = pk[i][j];
                    *reinterpret_cast<uint16_t *>(my + t0 * 64 + (((lane >> 3) ^ ((t0 >> 1) & 3)) * 16) +
                                                  (lane & 7) * 2) = static_cast<uint16_t>(w & 0xFFFFu);
                    *reinterpret_cast<uint16_t *>(my + t1 * 64 + (((lane >> 3) ^ ((t1 >> 1) & 3)) * 16) +
                                                  (lane & 7) * 2) = static_cast<uint16_t>(w >> 16);
                }
                __syncwarp();
                const int tok = c * 32 + lane;   // now this thread's token row
                uint4 w4[4];
#pragma unroll
                for (int p = 0; p < 4; ++p)
                    w4[p] = *reinterpret_cast<const uint4 *>(my + lane * 64 +
                                                             ((p ^ ((lane >> 1) & 3)) * 16));
                __syncwarp();
                if (tok < u.rows) {
                    __nv_bfloat16 *dst = out + (static_cast<int64_t>(u.row0) + tok) * Nout + col0;
                    if (out_v8) {
                        st_global_v8(dst, reinterpret_cast<const uint32_t *>(&w4[0]));
                        st_global_v8(dst + 16, reinterpret_cast<const uint32_t *>(&w4[2]));
                    } else {
                        uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
                        for (int p = 0; p < 4; ++p) d4[p] = w4[p];
                    }
                }
            }
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
    }
    __syncwarp();
    tc_fence_before();
    cluster_sync();   // no pair MMA, remote arrival or tensor-memory read is left
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem_base, Cfg::kTmemCols);
}

}  // namespace

// Largest number of CTA pairs of ffn_pair_gemm that fit on the device at once.
static int pair_clusters() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return sm_count() / 2;
    static int cached[64] = {0};
    if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (sm_count() / 2), 1, 1);
    cfg.blockDim = dim3(kPairThreads, 1, 1);
    cfg.dynamicSmemBytes = PairCfg::kSmem;
    int num = 0;
    if (cudaOccupancyMaxActiveClusters(&num, ffn_pair_gemm<false>, &cfg) != cudaSuccess || num <= 0) {
        cudaGetLastError();
        num = sm_count() / 2;
    }
    if (dev >= 0 && dev < 64) cached[dev] = num;
    return num;
}

bool pair_gemm_supported(int Nout) { return Nout % kPairM == 0; }

cudaError_t launch_pair_tiles(const int32_t *offsets, int n, int32_t *tiles, int4 *tlist,
                              cudaStream_t st, int cap) {
    ffn_pair_tiles<<<1, 1024, 0, st>>>(offsets, n, tiles, tlist, cap);
    return cudaGetLastError();
}

template <bool kAMn>
static cudaError_t launch_pair(const moe_shape &s, const CUtensorMap &mW, const XMaps &mX,
                               const int32_t *tiles, const int4 *tlist, int K, int Nout,
                               const __nv_bfloat16 *W, const __nv_bfloat16 *X, const float *bias,
                               int relu, __nv_bfloat16 *out, int32_t *err, cudaStream_t st) {
    const int64_t S = slots(s);
    // The opt-in above 48 KB belongs to the current device's context: set it
    // before every launch (a cheap host call).
    cudaError_t e = cudaFuncSetAttribute(ffn_pair_gemm<kAMn>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, PairCfg::kSmem);
    if (e != cudaSuccess) return e;
    // Upper bound of the unit count: every expert may add one partial tile.
    const int64_t max_units = ((S + kPairTok - 1) / kPairTok + s.n) * (Nout / kPairM);
    int64_t pairs = pair_clusters();
    if (pairs > max_units) pairs = max_units;
    if (pairs < 1) pairs = 1;
    const int out_v8 = (reinterpret_cast<uintptr_t>(out) & 31u) == 0 ? 1 : 0;
    return launch_pdl(ffn_pair_gemm<kAMn>, dim3(static_cast<unsigned>(2 * pairs)), dim3(kPairThreads),
                      PairCfg::kSmem, st, mW, mX, tiles, tlist, s.n, K, Nout, W, X, bias, relu, out,
                      out_v8, err);
}

static bool make_token_maps(XMaps &mX, const moe_shape &s, const __nv_bfloat16 *X, int K) {
    const int64_t S = slots(s);
    for (int i = 0; i < 8; ++i)
        if (!make_kmajor_map(&mX.m[i], X, static_cast<uint64_t>(K), static_cast<uint64_t>(S),
                             static_cast<uint32_t>(16 * (i + 1)), kPairKB))
            return false;
    return true;
}

cudaError_t launch_grouped_gemm_pair(const moe_shape &s, const __nv_bfloat16 *X, int K,
                                     const __nv_bfloat16 *W, int Nout, const float *bias, int relu,
                                     const int32_t *tiles, const int4 *tlist,
                                     __nv_bfloat16 *out, int32_t *err, cudaStream_t st) {
    CUtensorMap mW;
    XMaps mX;
    if (!make_kmajor_map(&mW, W, static_cast<uint64_t>(K), static_cast<uint64_t>(s.n) * Nout, 128,
                         kPairKB) ||
        !make_token_maps(mX, s, X, K))
        return cudaErrorInvalidValue;
    return launch_pair<false>(s, mW, mX, tiles, tlist, K, Nout, W, X, bias, relu, out, err, st);
}

cudaError_t launch_grouped_gemm_pair_wmn(const moe_shape &s, const __nv_bfloat16 *X, int K,
                                         const __nv_bfloat16 *W, int Nout, const int32_t *tiles,
                                         const int4 *tlist, __nv_bfloat16 *out, int32_t *err,
                                         cudaStream_t st) {
    if (!pair_gemm_supported(Nout) || K % 64 != 0) return cudaErrorInvalidValue;
    CUtensorMap mW;
    XMaps mX;
    // box: 128 K rows (two k-blocks) x this CTA's 128 output features (two
    // 64-wide blocks)
    if (!make_mnmajor_map(&mW, W, static_cast<uint64_t>(Nout), static_cast<uint64_t>(s.n) * K,
                          64 * kPairKB, 2) ||
        !make_token_maps(mX, s, X, K))
        return cudaErrorInvalidValue;
    return launch_pair<true>(s, mW, mX, tiles, tlist, K, Nout, W, X, nullptr, 0, out, err, st);
}

}  // namespace moe

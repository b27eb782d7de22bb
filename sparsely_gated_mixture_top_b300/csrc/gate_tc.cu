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
//   gate_pack       W_g, W_noise [d, C] fp32 -> hi/lo bf16 units, one 32 KB
//                   unit per (chunk, 64-wide k-block), stored pre-swizzled so
//                   that one bulk copy fills a pipeline stage: chunk c holds 64
//                   clean-score columns (rows 0..63) and the same 64
//                   noise-score columns (rows 64..127).  Hierarchical: the G
//                   group columns come first (padded to a chunk boundary),
//                   then the n inner columns.
//   gate_tc         persistent over 128-token tiles.  Warp 0 issues TMA loads,
//                   warp 1 issues tcgen05.mma (M=128 tokens, N=128 = 64 clean +
//                   64 noise columns, hi then lo pass into one fp32 accumulator,
//                   four accumulators in tensor memory), warps 2..9 are the
//                   epilogue: two warps per tensor-memory lane quarter, each
//                   owning one half of every chunk's columns for its 32 tokens
//                   (thread r = token r = tensor-memory lane r).  A first,
//                   branch-free pass over 16 columns at a time computes
//                   H = clean (+ b_g) + eps * softplus(noise) (softplus from
//                   the hardware exp/log) and flags the columns that beat the
//                   k-th entry of the running top-k; a second pass inserts the
//                   flagged ones (KeepTopK, ties to the lower index).  The
//                   halves merge their lists through shared memory and the
//                   softmax runs over the k survivors.
//                   Hierarchical gating picks the groups from the first chunks
//                   (both halves merge them) and only then looks at (and reads
//                   eps for) the inner columns of its chosen groups.
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

// Block: 64 d-rows (k-block kb) x 64 logical columns of one matrix (clean or
// noise).  Output: for every (chunk, k-block) a 32 KB unit [hi | lo], each a
// 128-row x 64-element bf16 tile already in the 128-byte-swizzled K-major
// order a TMA copy would produce (16-byte group g of row r stored at group
// g ^ (r % 8)), so that one bulk copy moves it into shared memory.
__global__ void __launch_bounds__(256) gate_pack(const float *__restrict__ Wg,
                                                 const float *__restrict__ Wn, int d, int C,
                                                 int groups, int prim_pad, int noisy,
                                                 uint8_t *__restrict__ pack) {
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
        const int rr = which * 64 + cc;
        const int64_t unit = (static_cast<int64_t>(chunk) * (d / 64) + blockIdx.z) * 2 * kKBytes;
        const int off = rr * 128 + (((tx >> 3) ^ (rr & 7)) << 4) + (tx & 7) * 2;
        *reinterpret_cast<__nv_bfloat16 *>(pack + unit + off) = hi;
        *reinterpret_cast<__nv_bfloat16 *>(pack + unit + kKBytes + off) = lo;
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
    // Entry kk-1 (kk <= KM) is the current k-th best.  The empty asm keeps each
    // entry an opaque register value, so that the compiler does not turn this
    // select into an indexed load (which would move the list to local memory).
    __device__ __forceinline__ float kth(int kk) const {
        float r = v[0];
#pragma unroll
        for (int q = 0; q < KM; ++q) {
            float c = v[q];
            asm("" : "+f"(c));
            if (q == kk - 1) r = c;
        }
        return r;
    }
    // Branch-free: every position takes the better of (its entry, the
    // carried candidate) and passes the other one down.
    __device__ __forceinline__ void insert(float cv, int ci) {
#pragma unroll
        for (int p = 0; p < KM; ++p) {
            const bool b = (cv > v[p]) | ((cv == v[p]) & (ci < i[p]));
            const float tv = v[p];
            const int ti = i[p];
            v[p] = b ? cv : tv;
            i[p] = b ? ci : ti;
            cv = b ? tv : cv;
            ci = b ? ti : ci;
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
constexpr int kGateEpiWarps = 8;                 // two per tensor-memory lane quarter
constexpr int kGateThreads = 32 * (2 + kGateEpiWarps);

template <bool kResident, bool kHier, int KM>
struct GateCfg {
    // Stage: the hi and lo W tiles of one (chunk, k-block) unit (plus, when x
    // is not resident, that k-block of x).
    static constexpr int kStages = kResident ? 2 : 3;
    static constexpr int kStageBytes = kResident ? 2 * kKBytes : 3 * kKBytes;
    static constexpr int kXBytes = kResident ? 8 * kKBytes : 0;  // d <= 512
    // Exchange between the two column halves: the group lists of both halves
    // (hierarchical only) and the final lists of half 1, [slot][token] order.
    static constexpr int kPrimSlots = kHier ? 2 * KM : 0;
    static constexpr int kFinalSlots = kHier ? KM * KM : KM;
    static constexpr int kXchBytes = (kPrimSlots + kFinalSlots) * kGateRows * 8;
    static constexpr int kBarBytes = 8 * (2 * kStages + 11) + 16;
    static constexpr int kSmem = kXBytes + kStages * kStageBytes + kXchBytes + 1024 + kBarBytes;
    static constexpr int kAcc = 4;               // accumulators (128 columns each)
    static constexpr uint32_t kTmemCols = 128 * kAcc;
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

// Named barrier of the eight epilogue warps.
__device__ __forceinline__ void epi_bar() {
    asm volatile("bar.sync 1, %0;" ::"n"(32 * kGateEpiWarps) : "memory");
}

// eps[row][col0 + j] for the 32 columns j of one chunk half whose bit is set
// in `live` (0 elsewhere).  Vector loads when the row stride and col0 allow
// 16-byte alignment (then every live group of 4 is all live).
__device__ __forceinline__ void load_eps32(const float *__restrict__ row, int col0, int C,
                                           bool vec, uint32_t live, float (&ev)[32]) {
    if (vec) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (col0 + 4 * q < C && ((live >> (4 * q)) & 1u))
                v = __ldg(reinterpret_cast<const float4 *>(row + col0 + 4 * q));
            ev[4 * q] = v.x;
            ev[4 * q + 1] = v.y;
            ev[4 * q + 2] = v.z;
            ev[4 * q + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
            ev[j] = (col0 + j < C && ((live >> j) & 1u)) ? __ldg(row + col0 + j) : 0.0f;
    }
}

// KM: list size for flat (>= k) or for each hierarchical level (>= k_groups, k_inner).
template <bool kResident, bool kHier, int KM>
__global__ void __launch_bounds__(kGateThreads, 1)
    gate_tc(const __grid_constant__ CUtensorMap mapX, const uint8_t *__restrict__ wpack,
            const GateArgs a) {
    using Cfg = GateCfg<kResident, kHier, KM>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint8_t *sX = smem;                        // resident x tile (kResident)
    uint8_t *sS = smem + Cfg::kXBytes;         // stage ring
    uint8_t *sXch = sS + Cfg::kStages * Cfg::kStageBytes;
    float *xch_v = reinterpret_cast<float *>(sXch);
    int *xch_i = reinterpret_cast<int *>(sXch + (Cfg::kPrimSlots + Cfg::kFinalSlots) * kGateRows * 4);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sXch + Cfg::kXchBytes);
    // full[S], empty[S], tfull[4], tempty[4], xfull, xempty, drain
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * Cfg::kStages + 11);
    volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(tmem_slot + 1);
    constexpr int S = Cfg::kStages;
    auto full = [&](int s) { return smem_u32(bars + s); };
    auto empty = [&](int s) { return smem_u32(bars + S + s); };
    constexpr int NA = Cfg::kAcc;
    auto tfull = [&](int b) { return smem_u32(bars + 2 * S + b); };
    auto tempty = [&](int b) { return smem_u32(bars + 2 * S + NA + b); };
    const uint32_t xfull = smem_u32(bars + 2 * S + 2 * NA);
    const uint32_t xempty = smem_u32(bars + 2 * S + 2 * NA + 1);
    const uint32_t drain_bar = smem_u32(bars + 2 * S + 2 * NA + 2);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        for (int b = 0; b < NA; ++b) {
            mbar_init(tfull(b), 1);
            mbar_init(tempty(b), 32 * kGateEpiWarps);
        }
        mbar_init(xfull, 1);
        mbar_init(xempty, 1);
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&mapX);
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
                    // the whole x tile (all k-blocks) in one 3-D copy
                    mbar_arrive_expect_tx(xfull, static_cast<uint32_t>(kblocks * kKBytes));
                    tma_load_3d(smem_u32(sX), &mapX, xfull, 0, row0, 0);
                }
                for (int c = 0; c < a.chunks && ok; ++c) {
                    for (int kb = 0; kb < kblocks && ok; ++kb) {
                        if (!mbar_wait_bounded(empty(stage), phase ^ 1u, abort_flag, a.err,
                                               kSiteTcProducer)) {
                            ok = false;
                            break;
                        }
                        uint8_t *st = sS + stage * Cfg::kStageBytes;
                        const uint8_t *unit =
                            wpack + (static_cast<int64_t>(c) * kblocks + kb) * (2 * kKBytes);
                        if (kResident) {
                            mbar_arrive_expect_tx(full(stage), 2 * kKBytes);
                            bulk_load(smem_u32(st), unit, 2 * kKBytes, full(stage));
                        } else {
                            mbar_arrive_expect_tx(full(stage), 3 * kKBytes);
                            tma_load_3d(smem_u32(st), &mapX, full(stage), 0, row0, kb);
                            bulk_load(smem_u32(st + kKBytes), unit, 2 * kKBytes, full(stage));
                        }
                        ++issued;
                        if (++stage == S) {
                            stage = 0;
                            phase ^= 1u;
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
                        if (!mbar_wait_bounded(full(stage), phase, abort_flag, a.err, kSiteTcMma)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t st = smem_u32(sS + stage * Cfg::kStageBytes);
                        const uint32_t xa = kResident ? smem_u32(sX + kb * kKBytes) : st;
                        const uint32_t wb = kResident ? st : st + kKBytes;
#pragma unroll
                        for (int kk = 0; kk < kGateBK / 16; ++kk)  // x . W_hi
                            tc_mma_f16(d_tmem, sdesc_kmajor_sw128(xa + kk * 32),
                                       sdesc_kmajor_sw128(wb + kk * 32), idesc,
                                       (kb | kk) != 0 ? 1u : 0u);
#pragma unroll
                        for (int kk = 0; kk < kGateBK / 16; ++kk)  // + x . W_lo
                            tc_mma_f16(d_tmem, sdesc_kmajor_sw128(xa + kk * 32),
                                       sdesc_kmajor_sw128(wb + kKBytes + kk * 32), idesc, 1u);
                        tc_commit(empty(stage));
                        if (++stage == S) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (!ok) break;
                    tc_commit(tfull(acc));
                    if (++acc == NA) {
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
        // Warp w (2..9) reads tensor-memory lanes 32*(w%4).. (token r of the
        // tile) and column half `half` of every chunk: clean columns
        // half*32 .. +32 and the matching noise columns 64 + half*32 .. +32.
        // Each thread keeps the running top-k of its half; the halves merge
        // through shared memory at the end of the tile (hierarchical: also
        // after the group columns, since both halves need the chosen groups).
        const int half = (warp - 2) >> 2;
        const int quad = warp & 3;
        const int r = quad * 32 + lane;
        const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
        const int k_inner = kHier ? a.k / a.k_groups : a.k;
        const int kk_prim = kHier ? a.k_groups : a.k;
        const bool vec_eps = (a.C & 3) == 0;
        constexpr int kFinalOff = Cfg::kPrimSlots * kGateRows;
        int acc = 0;
        uint32_t acc_phase = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
            const int64_t t = static_cast<int64_t>(tile) * kGateRows + r;
            const bool valid = t < a.T;
            const bool noisy = valid && a.noisy;
            const float *eps_row = noisy ? a.eps + t * a.C : nullptr;
            TopK<KM> prim;  // flat: the only list; hierarchical: the groups
            TopK<KM> inner[kHier ? KM : 1];
            prim.reset();
#pragma unroll
            for (int q = 0; q < (kHier ? KM : 1); ++q) inner[q].reset();
            float gw[KM];
            int glo[KM];  // hierarchical: first inner column of each chosen group
#pragma unroll
            for (int q = 0; q < KM; ++q) {
                gw[q] = 0.0f;
                glo[q] = -0x40000000;
            }
            for (int c = 0; c < a.chunks; ++c) {
                const bool inner_chunk = kHier && c >= a.prim_chunks;
                if (kHier && c == a.prim_chunks) {
                    // both halves publish their group lists and merge the other's
#pragma unroll
                    for (int q = 0; q < KM; ++q) {
                        xch_v[(half * KM + q) * kGateRows + r] = prim.v[q];
                        xch_i[(half * KM + q) * kGateRows + r] = prim.i[q];
                    }
                    epi_bar();
#pragma unroll
                    for (int q = 0; q < KM; ++q)
                        prim.insert(xch_v[((1 - half) * KM + q) * kGateRows + r],
                                    xch_i[((1 - half) * KM + q) * kGateRows + r]);
                    softmax_top<KM>(prim, kk_prim, gw);
#pragma unroll
                    for (int q = 0; q < KM; ++q)
                        if (q < a.k_groups) glo[q] = prim.i[q] * a.m;
                }
                // columns of this chunk half (score index space of the list)
                const int col0 = inner_chunk ? (c - a.prim_chunks) * kGateChunk + half * 32
                                             : c * kGateChunk + half * 32;
                const int ncols = inner_chunk ? a.n : (kHier ? a.groups : a.C);
                const int ecol0 = inner_chunk ? a.groups + col0 : col0;  // eps / bg column
                if (eps_row && !kHier && c + 2 < a.chunks && (c + 2) * kGateChunk + half * 32 < a.C)
                    prefetch_l2(eps_row + (c + 2) * kGateChunk + half * 32);
                float ev[32];
                if (eps_row && col0 < ncols) {
                    uint32_t live = 0xffffffffu;
                    bool vec = vec_eps;
                    if (inner_chunk) {
                        live = 0;
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            #pragma unroll
                            for (int qq = 0; qq < KM; ++qq)
                                if (qq < a.k_groups && static_cast<unsigned>(col0 + j - glo[qq]) <
                                                           static_cast<unsigned>(a.m))
                                    live |= 1u << j;
                        vec = vec && (ecol0 & 3) == 0 && (a.m & 3) == 0;
                    }
                    load_eps32(eps_row, ecol0, a.C, vec, live, ev);
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) ev[j] = 0.0f;
                }
                if (ok && !mbar_wait_bounded(tfull(acc), acc_phase, abort_flag, a.err,
                                             kSiteTcEpilogue))
                    ok = false;
                ok = __all_sync(0xffffffffu, ok);  // warp-uniform: the votes below need every lane
                if (ok) {
                    tc_fence_after();
                    // Pass 1 thresholds: the k-th entry of each list, fixed for the span.
                    const float thr_p = prim.kth(kk_prim);
                    float thr_i[kHier ? KM : 1];
#pragma unroll
                    for (int qq = 0; qq < (kHier ? KM : 1); ++qq) thr_i[qq] = inner[qq].kth(k_inner);
#pragma unroll
                    for (int piece = 0; piece < 2; ++piece) {
                        uint32_t cv[16], nv[16];
                        const uint32_t col = static_cast<uint32_t>(acc * 128 + half * 32 + piece * 16);
                        tmem_ld_32x32b_x16(tmem_base + lane_addr + col, cv);
                        tmem_ld_32x32b_x16(tmem_base + lane_addr + col + 64, nv);
                        tmem_ld_wait();
                        if (piece == 1) {
                            tc_fence_before();
                            mbar_arrive(tempty(acc));  // this half of the accumulator is read
                        }
                        // Pass 1 (branch-free): the noisy score of every column and
                        // which ones beat the k-th entry of their list.  Within a
                        // thread's list the columns arrive in increasing index order,
                        // so an equal score never displaces an entry: '>' is exact.
                        // Tokens past T flag nothing but still take part in the votes.
                        uint32_t pass = 0;
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const int sc = col0 + piece * 16 + j;
                            float h = __uint_as_float(cv[j]);
                            if (a.bg && sc < ncols) h += __ldg(a.bg + ecol0 + piece * 16 + j);
                            if (noisy) h += ev[piece * 16 + j] * softplus_fast(__uint_as_float(nv[j]));
                            cv[j] = __float_as_uint(h);
                            float thr = thr_p;
                            if (inner_chunk) {
                                thr = INFINITY;  // outside the chosen groups
#pragma unroll
                                for (int qq = 0; qq < (kHier ? KM : 1); ++qq)
                                    if (qq < a.k_groups &&
                                        static_cast<unsigned>(sc - glo[qq]) < static_cast<unsigned>(a.m))
                                        thr = thr_i[qq];
                            }
                            if (valid && sc < ncols && h > thr) pass |= 1u << j;
                        }
                        // Pass 2 (rare): insert the flagged columns.  The warp vote
                        // keeps each column's insertion a real branch.
                        if (__any_sync(0xffffffffu, pass != 0)) {
#pragma unroll
                            for (int j = 0; j < 16; ++j) {
                                if (!__any_sync(0xffffffffu, (pass >> j) & 1u)) continue;
                                if (!((pass >> j) & 1u)) continue;
                                const int sc = col0 + piece * 16 + j;
                                const float h = __uint_as_float(cv[j]);
                                if (!inner_chunk) {
                                    prim.insert(h, sc);
                                } else {
#pragma unroll
                                    for (int qq = 0; qq < (kHier ? KM : 1); ++qq)
                                        if (qq < a.k_groups && static_cast<unsigned>(sc - glo[qq]) <
                                                                   static_cast<unsigned>(a.m))
                                            inner[qq].insert(h, sc - glo[qq]);
                                }
                            }
                        }
                    }
                }
                if (++acc == NA) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            // half 1 hands its lists to half 0, which merges and writes the token
            epi_bar();  // half 0 is done with the previous tile's exchange
            if (half == 1) {
                if (!kHier) {
#pragma unroll
                    for (int q = 0; q < KM; ++q) {
                        xch_v[kFinalOff + q * kGateRows + r] = prim.v[q];
                        xch_i[kFinalOff + q * kGateRows + r] = prim.i[q];
                    }
                } else {
#pragma unroll
                    for (int g = 0; g < (kHier ? KM : 1); ++g)
#pragma unroll
                        for (int q = 0; q < KM; ++q) {
                            xch_v[kFinalOff + (g * KM + q) * kGateRows + r] = inner[g].v[q];
                            xch_i[kFinalOff + (g * KM + q) * kGateRows + r] = inner[g].i[q];
                        }
                }
            }
            epi_bar();
            if (half == 0 && ok && valid) {
                if (!kHier) {
#pragma unroll
                    for (int q = 0; q < KM; ++q)
                        prim.insert(xch_v[kFinalOff + q * kGateRows + r],
                                    xch_i[kFinalOff + q * kGateRows + r]);
                    float w[KM];
                    softmax_top<KM>(prim, a.k, w);
#pragma unroll
                    for (int q = 0; q < KM; ++q)
                        if (q < a.k) {
                            a.idx[t * a.k + q] = prim.i[q];
                            a.G[t * a.k + q] = w[q];
                        }
                } else {
#pragma unroll
                    for (int g = 0; g < (kHier ? KM : 1); ++g) {
                        if (g >= a.k_groups) break;
#pragma unroll
                        for (int q = 0; q < KM; ++q)
                            inner[g].insert(xch_v[kFinalOff + (g * KM + q) * kGateRows + r],
                                            xch_i[kFinalOff + (g * KM + q) * kGateRows + r]);
                        float wi[KM];
                        softmax_top<KM>(inner[g], k_inner, wi);
                        const int grp = prim.i[g];
#pragma unroll
                        for (int e = 0; e < KM; ++e)
                            if (e < k_inner) {
                                a.idx[t * a.k + g * k_inner + e] = grp * a.m + inner[g].i[e];
                                a.G[t * a.k + g * k_inner + e] = gw[g] * wi[e];
                            }
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

// x [T, d] bf16 seen as {64, T, d/64} (strides d*2 and 128 bytes); a box of
// 128 tokens x kb_box k-blocks lands as kb_box 128-byte-swizzled K-major tiles.
bool gate_map(CUtensorMap *m, const void *base, uint64_t d, uint64_t rows, uint32_t kb_box) {
    EncodeTiledFn enc = gate_encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {64, rows, d / 64};
    cuuint64_t strides[2] = {d * 2, 128};
    cuuint32_t box[3] = {64, 128, kb_box};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool kResident, bool kHier, int KM>
cudaError_t launch_gate_tc_t(const CUtensorMap &mx, const uint8_t *wpack, const GateArgs &ga,
                             int grid, cudaStream_t st) {
    using Cfg = GateCfg<kResident, kHier, KM>;
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [] {
        attr = cudaFuncSetAttribute(gate_tc<kResident, kHier, KM>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
    });
    if (attr != cudaSuccess) return attr;
    gate_tc<kResident, kHier, KM><<<grid, kGateThreads, Cfg::kSmem, st>>>(mx, wpack, ga);
    return cudaGetLastError();
}

template <bool kResident, bool kHier>
cudaError_t launch_gate_tc_km(int km, const CUtensorMap &mx, const uint8_t *wpack,
                              const GateArgs &ga, int grid, cudaStream_t st) {
    if (km <= 2) return launch_gate_tc_t<kResident, kHier, 2>(mx, wpack, ga, grid, st);
    if (km <= 4) return launch_gate_tc_t<kResident, kHier, 4>(mx, wpack, ga, grid, st);
    if constexpr (kHier) {
        return cudaErrorInvalidValue;  // hierarchical lists are limited to 4
    } else {
        if (km <= 8) return launch_gate_tc_t<kResident, kHier, 8>(mx, wpack, ga, grid, st);
        return launch_gate_tc_t<kResident, kHier, 16>(mx, wpack, ga, grid, st);
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
    uint8_t *wpack = static_cast<uint8_t *>(pack);
    gate_pack<<<dim3(ga.chunks, 2, s.d / 64), 256, 0, st>>>(Wg, noisy ? Wn : Wg, s.d, C, s.groups,
                                                          ga.prim_pad, noisy, wpack);
    const bool resident = s.d <= 512;
    CUtensorMap mx;
    if (!gate_map(&mx, x, s.d, static_cast<uint64_t>(s.T), resident ? s.d / 64 : 1))
        return cudaErrorInvalidValue;
    const int tiles = static_cast<int>((s.T + kGateRows - 1) / kGateRows);
    const int grid = tiles < sm_count() ? tiles : sm_count();
    const int km = s.groups ? (s.k_groups > s.k / s.k_groups ? s.k_groups : s.k / s.k_groups) : s.k;
    if (resident)
        return s.groups ? launch_gate_tc_km<true, true>(km, mx, wpack, ga, grid, st)
                        : launch_gate_tc_km<true, false>(km, mx, wpack, ga, grid, st);
    return s.groups ? launch_gate_tc_km<false, true>(km, mx, wpack, ga, grid, st)
                    : launch_gate_tc_km<false, false>(km, mx, wpack, ga, grid, st);
}

}  // namespace moe

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
//   gate_pack       W_g, W_noise [d, ldw] fp32 -> hi/lo bf16 units, one 32 KB
//                   unit per (chunk, 64-wide k-block), stored pre-swizzled so
//                   that one bulk copy fills a pipeline stage: chunk c holds 64
//                   clean-score columns (rows 0..63) and the same 64
//                   noise-score columns (rows 64..127).  In grouped packing
//                   every group's m columns start on a chunk boundary.
//   gate_tc         persistent over 128-row tiles.  Warp 0 issues the copies,
//                   warp 1 issues tcgen05.mma (M=128 rows, N=128 = 64 clean +
//                   64 noise columns, hi then lo pass into one fp32 accumulator,
//                   four accumulators in tensor memory), warps 2..9 are the
//                   epilogue: two warps per tensor-memory lane quarter, each
//                   owning one half of every chunk's columns for its 32 rows
//                   (thread r = row r = tensor-memory lane r).  A first,
//                   branch-free pass over 16 columns at a time computes
//                   H = clean (+ b_g) + eps * softplus(noise) (softplus from
//                   the hardware exp/log) and flags the columns that beat the
//                   k-th entry of the running top-k; a second pass inserts the
//                   flagged ones (KeepTopK, ties to the lower index).  The
//                   halves merge their lists through shared memory and the
//                   softmax runs over the k survivors.
//
// Flat gating runs gate_tc once over the tokens and all n columns.
// Hierarchical gating (MoE-N-h, section 三: pick the groups, then the experts
// inside each chosen group) runs it twice:
//   1. flat over the G group columns -> the k_g chosen groups of every token
//      and their softmax weights Gp;
//   2. the (token, rank) pairs are routed by group with the dispatch kernels,
//      their x rows gathered into group order, and gate_tc in grouped mode
//      scores each 128-row tile of one group against that group's m columns
//      only; a row's k_i survivors get the weights Gp * softmax.
// So the inner scores cost T * k_g * m columns instead of T * n.
// x (or the gathered rows) stays resident in shared memory for the whole
// tile when d <= 512; otherwise each stage carries its x block with the W
// blocks.
#include "moe_device.cuh"
#include "moe_launch.h"

#include <float.h>
#include <limits.h>

#include <mutex>

namespace moe {

namespace {

constexpr int kGateChunk = 64;         // score columns (clean and noise each) per chunk
constexpr int kGateRows = 128;         // rows per tile
constexpr int kGateBK = 64;            // d per k-block
constexpr int kKBytes = 128 * 64 * 2;  // one 128 x 64 bf16 block: 16 KB

// ---------------------------------------------------------------------------
// Packing
// ---------------------------------------------------------------------------
// Block: 16 d-rows (quarter blockIdx.z % 4 of k-block kb = blockIdx.z / 4)
// x 64 chunk columns of one matrix (clean or noise).  Chunk column lc of
// chunk `chunk` takes W column
//   group_m == 0: col_base + chunk*64 + lc            (if < ncols columns)
//   group_m  > 0: col_base + g*group_m + cl, with g = chunk / mchunks and
//                 cl = (chunk % mchunks)*64 + lc      (if cl < group_m)
// and zero elsewhere.  Output: for every (chunk, k-block) a 32 KB unit
// [hi | lo], each a 128-row x 64-element bf16 tile already in the
// 128-byte-swizzled K-major order a TMA copy would produce (16-byte group g
// of row r stored at group g ^ (r % 8)), so that one bulk copy moves it; this
// block writes the groups 2*quarter and 2*quarter + 1 of its 64 rows.
__global__ void __launch_bounds__(128) gate_pack(const float *__restrict__ Wg,
                                                 const float *__restrict__ Wn, int d, int ldw,
                                                 int col_base, int ncols, int group_m,
                                                 int mchunks, int noisy, int pair,
                                                 uint8_t *__restrict__ pack) {
    __shared__ float tile[16][65];
    // The weights are inputs of the call, not results of the previous kernel
    // (which only ever reads this buffer two launches back, in the previous
    // gate): pack first, and let the gate start its prologue meanwhile.  The
    // wait at the end keeps the stream order for everything after this.
    pdl_launch_dependents();
    const int chunk = blockIdx.x;
    const int which = blockIdx.y;  // 0 clean, 1 noise
    const int kb = blockIdx.z >> 2, quarter = blockIdx.z & 3;
    const int d0 = kb * 64 + quarter * 16;
    const float *W = which ? Wn : Wg;
    const int tx = threadIdx.x % 64, ty = threadIdx.x / 64;
    int src;
    if (group_m == 0) {
        const int col = chunk * kGateChunk + tx;
        src = col < ncols ? col_base + col : -1;
    } else {
        const int g = chunk / mchunks;
        const int cl = (chunk - g * mchunks) * kGateChunk + tx;
        src = cl < group_m ? col_base + g * group_m + cl : -1;
    }
    for (int r = ty; r < 16; r += 2) {
        float v = 0.0f;
        if (src >= 0 && (which == 0 || noisy)) v = W[static_cast<int64_t>(d0 + r) * ldw + src];
        tile[r][tx] = v;  // tile[d][col]
    }
    __syncthreads();
    // Output: this thread's row (one per column) and one 16-byte group of 8
    // d-values, written for hi and for lo.
    const int64_t unit = (static_cast<int64_t>(chunk) * (d / 64) + kb) * 2 * kKBytes;
    const int cc = threadIdx.x >> 1, gl = threadIdx.x & 1;
    const int g = 2 * quarter + gl;
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float v0 = tile[gl * 8 + 2 * e][cc], v1 = tile[gl * 8 + 2 * e + 1][cc];
        const __nv_bfloat16 h0 = __float2bfloat16_rn(v0), h1 = __float2bfloat16_rn(v1);
        const __nv_bfloat16 l0 = __float2bfloat16_rn(v0 - __bfloat162float(h0));
        const __nv_bfloat16 l1 = __float2bfloat16_rn(v1 - __bfloat162float(h1));
        hi[e] = static_cast<uint32_t>(__bfloat16_as_ushort(h0)) |
                (static_cast<uint32_t>(__bfloat16_as_ushort(h1)) << 16);
        lo[e] = static_cast<uint32_t>(__bfloat16_as_ushort(l0)) |
                (static_cast<uint32_t>(__bfloat16_as_ushort(l1)) << 16);
    }
    const int rr = which * 64 + cc;
    if (!pair) {
        const int off = rr * 128 + ((g ^ (rr & 7)) << 4);
        *reinterpret_cast<uint4 *>(pack + unit + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4 *>(pack + unit + kKBytes + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    } else {
        // CTA-pair layout: per (chunk, half) the k-blocks in order, each
        // [hi 64 rows | lo 64 rows] (16 KB), so that one SM of a pair copies
        // its half (clean or noise columns) of two k-blocks in one 32 KB box.
        const int64_t hunit =
            ((static_cast<int64_t>(chunk) * 2 + which) * (d / 64) + kb) * kKBytes;
        const int off = cc * 128 + ((g ^ (cc & 7)) << 4);
        *reinterpret_cast<uint4 *>(pack + hunit + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4 *>(pack + hunit + kKBytes / 2 + off) =
            make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
    pdl_wait();
}

// ---------------------------------------------------------------------------
// Per-row running top-k (registers only; all indices compile-time)
// ---------------------------------------------------------------------------
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
    // carried candidate) and passes the other one down.  Better = larger
    // value, equal values by lower index.
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

// Compare-exchange of two (score, column) entries: a takes the better one
// (larger score, equal scores by lower column).
__device__ __forceinline__ void cas_entry(float &va, int &ia, float &vb, int &ib) {
    const bool sw = (vb > va) | ((vb == va) & (ib < ia));
    const float tv = sw ? vb : va;
    const int ti = sw ? ib : ia;
    vb = sw ? va : vb;
    ib = sw ? ia : ib;
    va = tv;
    ia = ti;
}

// The best four of sixteen entries, in order, by a fixed network: four
// sorted groups of four (5 exchanges each), then three merges of two sorted
// fours into the best four (the better of a[i] and b[3-i] forms a bitonic
// sequence, sorted by 4 exchanges).  Branch-free: the same for every lane.
__device__ __forceinline__ void top4_of16(float (&v)[16], int (&ix)[16], float (&ov)[4],
                                          int (&oi)[4]) {
#pragma unroll
    for (int g = 0; g < 16; g += 4) {
        cas_entry(v[g], ix[g], v[g + 1], ix[g + 1]);
        cas_entry(v[g + 2], ix[g + 2], v[g + 3], ix[g + 3]);
        cas_entry(v[g], ix[g], v[g + 2], ix[g + 2]);
        cas_entry(v[g + 1], ix[g + 1], v[g + 3], ix[g + 3]);
        cas_entry(v[g + 1], ix[g + 1], v[g + 2], ix[g + 2]);
    }
    // merge group b into group a (a, b: first entries of two sorted fours)
    auto merge4 = [&](int a, int b) {
#pragma unroll
        for (int q = 0; q < 4; ++q) cas_entry(v[a + q], ix[a + q], v[b + 3 - q], ix[b + 3 - q]);
        cas_entry(v[a], ix[a], v[a + 2], ix[a + 2]);
        cas_entry(v[a + 1], ix[a + 1], v[a + 3], ix[a + 3]);
        cas_entry(v[a], ix[a], v[a + 1], ix[a + 1]);
        cas_entry(v[a + 2], ix[a + 2], v[a + 3], ix[a + 3]);
    };
    merge4(0, 4);
    merge4(8, 12);
    merge4(0, 8);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        ov[q] = v[q];
        oi[q] = ix[q];
    }
}

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
constexpr int kGateParts = 4;                        // epilogue warps per lane quarter
constexpr int kGateEpiWarps = 4 * kGateParts;
constexpr int kGateThreads = 32 * (2 + kGateEpiWarps);
constexpr int kPartCols = kGateChunk / kGateParts;   // 16 score columns per part and chunk

template <bool kResident, int KM, bool kPair = false>
struct GateCfg {
    // Stage: the hi and lo W tiles of one (chunk, k-block) unit (plus, when x
    // is not resident, that k-block of x).  CTA pair: this SM's half (64
    // columns) of the hi and lo tiles of two k-blocks, 32 KB.
    static constexpr int kStages = kResident ? 2 : 3;
    static constexpr int kStageBytes = kPair ? 2 * kKBytes : (kResident ? 2 * kKBytes : 3 * kKBytes);
    static constexpr int kXBytes = kResident ? 8 * kKBytes : 0;  // d <= 512
    // Exchange of two parts' final lists at a time, [list][slot][row] order.
    static constexpr int kXchBytes = 2 * KM * kGateRows * 8;
    // Each part's k-th score per row after a chunk, two chunks deep (lists
    // of up to 8; the 16-deep lists' exchange leaves no room for it).
    static constexpr bool kShareThr = KM <= 8;
    static constexpr int kThrBytes = kShareThr ? 2 * kGateParts * kGateRows * 4 : 0;
    static constexpr int kAcc = 4;  // accumulators (128 columns each)
    static constexpr int kBarBytes = 8 * (2 * kStages + 2 * kAcc + 3) + 16;
    static constexpr int kSmem =
        kXBytes + kStages * kStageBytes + kXchBytes + kThrBytes + 1024 + kBarBytes;
    static constexpr uint32_t kTmemCols = 128 * kAcc;
    static_assert(kSmem <= 227 * 1024, "shared memory budget");
};

struct GateArgs {
    const float *bg;   // [C] or NULL
    const float *eps;  // rows of ldE floats, or NULL (clean scores)
    int32_t *idx;      // [T, k]
    float *G;          // [T, k]
    int64_t T;         // tokens (flat: rows)
    int d;
    int k;             // outputs per token
    int kk;            // list length used: flat k; grouped k_inner
    int kf;            // list depth kept exact: kk, or kk + 1 in load mode
    int ncols;         // score columns of one row's list (flat: C; grouped: m)
    int chunks;        // chunks per tile
    int ldE;           // eps row stride (floats)
    int noisy;
    int32_t *err;
    // grouped mode (pairs = (token, rank) rows, ordered by group)
    const int32_t *perm_g;     // [T*kg] row -> pair = t*kg + q
    const int32_t *offsets_g;  // [G+1]
    const int32_t *tiles_g;    // [G+1] row-tile starts
    const float *gw;           // [T*kg] group weights
    int groups, kg, m;
    // load mode (flat only): every column's clean score and noise scale, and
    // each token's k-th and (k+1)-th noisy score
    float *c_out;   // [T, ncols] or NULL
    float *s_out;   // [T, ncols]
    float *vk_out;  // [T, 2]
};

// Named barrier of the eight epilogue warps.
__device__ __forceinline__ void epi_bar() {
    asm volatile("bar.sync 1, %0;" ::"n"(32 * kGateEpiWarps) : "memory");
}

// The four warps that read one lane quarter (rows 32*quad ..), one per part.
__device__ __forceinline__ void quad_bar(int quad) {
    asm volatile("bar.sync %0, %1;" ::"r"(2 + quad), "n"(32 * kGateParts) : "memory");
}

// eps[row][col0 + j] for the NC columns j of one chunk part (0 past C).
// Vector loads when the row stride and col0 allow 16-byte alignment.
template <int NC>
__device__ __forceinline__ void load_eps(const float *__restrict__ row, int col0, int C, bool vec,
                                         float (&ev)[NC]) {
    if (vec) {
#pragma unroll
        for (int q = 0; q < NC / 4; ++q) {
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (col0 + 4 * q < C) v = __ldg(reinterpret_cast<const float4 *>(row + col0 + 4 * q));
            ev[4 * q] = v.x;
            ev[4 * q + 1] = v.y;
            ev[4 * q + 2] = v.z;
            ev[4 * q + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < NC; ++j) ev[j] = (col0 + j < C) ? __ldg(row + col0 + j) : 0.0f;
    }
}

struct GateTile {
    int g, row0, rows;
};

template <bool kGrouped, bool kPair = false>
__device__ __forceinline__ GateTile gate_tile(int tile, const GateArgs &a, uint32_t rank = 0) {
    GateTile ti;
    if (!kGrouped) {
        ti.g = 0;
        ti.row0 = tile * (kPair ? 2 : 1) * kGateRows + static_cast<int>(rank) * kGateRows;
        const int64_t left = a.T - ti.row0;
        ti.rows = left < kGateRows ? static_cast<int>(left) : kGateRows;
    } else {
        int lo = 0, hi = a.groups - 1;  // largest g with tiles_g[g] <= tile
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (a.tiles_g[mid] <= tile)
                lo = mid;
            else
                hi = mid - 1;
        }
        ti.g = lo;
        ti.row0 = a.offsets_g[lo] + (tile - a.tiles_g[lo]) * kGateRows;
        ti.rows = min(kGateRows, a.offsets_g[lo + 1] - ti.row0);
    }
    return ti;
}

// KM: list size (>= kk).  kGrouped: rows are (token, rank) pairs of one group
// per tile, scored against that group's columns.
// kPair (flat, resident x only): a cluster of two CTAs scores 256 rows, 128
// per CTA, with one M = 256 MMA whose N = 128 columns are split over the two
// SMs: the even CTA supplies the 64 clean-score columns of each W tile, the
// odd one the 64 noise-score columns.  Each SM so streams half of W, two
// k-blocks per copy (mapW: the packed W viewed as rows of 128 bytes); both
// CTAs' copies complete on the even CTA's barriers, which issues the MMAs and
// commits to the barriers of both.  Each CTA's accumulator holds its 128
// rows x all 128 columns, so the epilogue is the same.
template <bool kResident, bool kGrouped, int KM, bool kPair = false>
__global__ void __launch_bounds__(kGateThreads, 1)
    gate_tc(const __grid_constant__ CUtensorMap mapX, const uint8_t *__restrict__ wpack,
            const GateArgs a, const __grid_constant__ CUtensorMap mapW) {
    static_assert(!kPair || (kResident && !kGrouped), "pair gate: flat, resident x");
    using Cfg = GateCfg<kResident, KM, kPair>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint8_t *sX = smem;                 // resident x tile (kResident)
    uint8_t *sS = smem + Cfg::kXBytes;  // stage ring
    uint8_t *sXch = sS + Cfg::kStages * Cfg::kStageBytes;
    float *xch_v = reinterpret_cast<float *>(sXch);                        // [2][KM][rows]
    int *xch_i = reinterpret_cast<int *>(sXch + 2 * KM * kGateRows * 4);   // [2][KM][rows]
    float *thr_sh = reinterpret_cast<float *>(sXch + Cfg::kXchBytes);   // [2][parts][rows]
    uint64_t *bars = reinterpret_cast<uint64_t *>(sXch + Cfg::kXchBytes + Cfg::kThrBytes);
    constexpr int S = Cfg::kStages;
    constexpr int NA = Cfg::kAcc;
    // full[S], empty[S], tfull[NA], tempty[NA], xfull, xempty, drain
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * S + 2 * NA + 3);
    volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(tmem_slot + 1);
    auto full = [&](int s) { return smem_u32(bars + s); };
    auto empty = [&](int s) { return smem_u32(bars + S + s); };
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
            mbar_init(tempty(b), (kPair ? 2 : 1) * kGateEpiWarps);   // one arrival per epilogue warp
        }
        mbar_init(xfull, 1);
        mbar_init(xempty, 1);
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&mapX);
        if (kPair) tma_prefetch_map(&mapW);
    }
    uint32_t rank = 0;
    if constexpr (kPair) {
        rank = cluster_ctarank();
        // the pair allocation needs both CTAs running (first barrier) and is
        // published to both before any copy, MMA or remote arrival (second)
        cluster_sync();
        if (warp == 1) {
            tmem_alloc_pair(smem_u32(tmem_slot), Cfg::kTmemCols);
            tmem_relinquish_pair();
        }
        tc_fence_before();
        cluster_sync();
        tc_fence_after();
    } else {
        if (warp == 1) {
            tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols);
            tmem_relinquish();
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }
    const uint32_t tmem_base = *tmem_slot;
    const int tile0 = kPair ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
    // Flat gating reads x, an input of the call: the first tile's resident x
    // rows are requested before waiting for the previous kernel (the packed
    // weights).  The grouped pass reads rows the previous kernels gathered.
    const bool x_early = kResident && !kGrouped &&
                         tile0 < static_cast<int>((a.T + (kPair ? 2 : 1) * kGateRows - 1) /
                                                  ((kPair ? 2 : 1) * kGateRows));
    if (x_early && warp == 0 && lane == 0) {
        const GateTile ti = gate_tile<kGrouped, kPair>(tile0, a, rank);
        const int kbl = a.d / kGateBK;
        if constexpr (kPair) {
            if (rank == 0) mbar_arrive_expect_tx(xfull, static_cast<uint32_t>(2 * kbl * kKBytes));
            tma_load_3d_pair(smem_u32(sX), &mapX, mapa_shared(xfull, 0), 0, ti.row0, 0);
        } else {
            mbar_arrive_expect_tx(xfull, static_cast<uint32_t>(kbl * kKBytes));
            tma_load_3d(smem_u32(sX), &mapX, xfull, 0, ti.row0, 0);
        }
    }
    // from here on the previous kernel's results are used
    pdl_wait();
    pdl_launch_dependents();
    // tiles of 128 rows (single CTA) or 256 rows (pair: 128 per CTA)
    const int tiles = kGrouped ? a.tiles_g[a.groups]
                               : static_cast<int>((a.T + (kPair ? 2 : 1) * kGateRows - 1) /
                                                  ((kPair ? 2 : 1) * kGateRows));
    const int tstep = kPair ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
    const int kblocks = a.d / kGateBK;

    if (warp == 0) {
        // ------------------------------ producer ------------------------------
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, xphase = 0;
            bool ok = true;
            int64_t issued = 0;
            for (int tile = tile0; tile < tiles && ok; tile += tstep) {
                const GateTile ti = gate_tile<kGrouped, kPair>(tile, a, rank);
                if (kResident && x_early && tile == tile0) {
                    xphase ^= 1u;  // requested before the wait above
                } else if (kResident) {
                    if (!mbar_wait_bounded(xempty, xphase ^ 1u, abort_flag, a.err, kSiteTcProducer)) {
                        ok = false;
                        break;
                    }
                    xphase ^= 1u;
                    // the whole x tile (all k-blocks) in one 3-D copy
                    if constexpr (kPair) {
                        if (rank == 0)
                            mbar_arrive_expect_tx(xfull, static_cast<uint32_t>(2 * kblocks * kKBytes));
                        tma_load_3d_pair(smem_u32(sX), &mapX, mapa_shared(xfull, 0), 0, ti.row0, 0);
                    } else {
                        mbar_arrive_expect_tx(xfull, static_cast<uint32_t>(kblocks * kKBytes));
                        tma_load_3d(smem_u32(sX), &mapX, xfull, 0, ti.row0, 0);
                    }
                }
                const int64_t unit0 = static_cast<int64_t>(ti.g) * a.chunks;
                if constexpr (kPair) {
                    // this SM's half of two k-blocks of each chunk per stage
                    for (int c = 0; c < a.chunks && ok; ++c) {
                        for (int kb = 0; kb < kblocks && ok; kb += 2) {
                            if (!mbar_wait_bounded(empty(stage), phase ^ 1u, abort_flag, a.err,
                                                   kSiteTcProducer)) {
                                ok = false;
                                break;
                            }
                            if (rank == 0) mbar_arrive_expect_tx(full(stage), 2 * Cfg::kStageBytes);
                            const int wrow = static_cast<int>(
                                (((unit0 + c) * 2 + rank) * kblocks + kb) * (kKBytes / 128));
                            tma_load_2d_pair(smem_u32(sS + stage * Cfg::kStageBytes), &mapW,
                                             mapa_shared(full(stage), 0), 0, wrow);
                            ++issued;
                            if (++stage == S) {
                                stage = 0;
                                phase ^= 1u;
                            }
                        }
                    }
                    continue;
                }
                for (int c = 0; c < a.chunks && ok; ++c) {
                    for (int kb = 0; kb < kblocks && ok; ++kb) {
                        if (!mbar_wait_bounded(empty(stage), phase ^ 1u, abort_flag, a.err,
                                               kSiteTcProducer)) {
                            ok = false;
                            break;
                        }
                        uint8_t *st = sS + stage * Cfg::kStageBytes;
                        const uint8_t *unit = wpack + ((unit0 + c) * kblocks + kb) * (2 * kKBytes);
                        if (kResident) {
                            mbar_arrive_expect_tx(full(stage), 2 * kKBytes);
                            bulk_load(smem_u32(st), unit, 2 * kKBytes, full(stage));
                        } else {
                            mbar_arrive_expect_tx(full(stage), 3 * kKBytes);
                            tma_load_3d(smem_u32(st), &mapX, full(stage), 0, ti.row0, kb);
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
            if (!ok && kPair) {  // copies complete on the even CTA's barriers: give them time
                const uint64_t t0 = global_ns();
                while (global_ns() - t0 < 200000ull) {
                }
            } else if (!ok) {  // let issued copies land before the CTA exits
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
        if (kPair && lane == 0 && rank == 0) {
            // pair MMAs M = 256 (128 rows of each CTA) x N = 128 (64 columns
            // from each CTA), hi then lo, two k-blocks per stage
            constexpr uint32_t idesc = idesc_bf16_f32(256, 128);
            int stage = 0;
            uint32_t phase = 0, xphase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int tile = tile0; tile < tiles && ok; tile += tstep) {
                if (!mbar_wait_bounded(xfull, xphase, abort_flag, a.err, kSiteTcMma)) break;
                xphase ^= 1u;
                for (int c = 0; c < a.chunks && ok; ++c) {
                    if (!mbar_wait_bounded(tempty(acc), acc_phase ^ 1u, abort_flag, a.err,
                                           kSiteTcMma)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * 128);
                    for (int kb = 0; kb < kblocks && ok; kb += 2) {
                        if (!mbar_wait_bounded(full(stage), phase, abort_flag, a.err, kSiteTcMma)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t st = smem_u32(sS + stage * Cfg::kStageBytes);
                        const int nkb = min(2, kblocks - kb);
                        for (int j = 0; j < nkb; ++j) {
                            const uint32_t xa = smem_u32(sX + (kb + j) * kKBytes);
                            const uint32_t wb = st + j * kKBytes;   // [hi 8 KB | lo 8 KB]
#pragma unroll
                            for (int kk = 0; kk < kGateBK / 16; ++kk)  // x . W_hi
                                tc_mma_f16_pair(d_tmem, sdesc_kmajor_sw128(xa + kk * 32),
                                                sdesc_kmajor_sw128(wb + kk * 32), idesc,
                                                (kb | j | kk) != 0 ? 1u : 0u);
#pragma unroll
                            for (int kk = 0; kk < kGateBK / 16; ++kk)  // + x . W_lo
                                tc_mma_f16_pair(d_tmem, sdesc_kmajor_sw128(xa + kk * 32),
                                                sdesc_kmajor_sw128(wb + kKBytes / 2 + kk * 32),
                                                idesc, 1u);
                        }
                        tc_commit_pair_both(empty(stage));
                        if (++stage == S) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (!ok) break;
                    tc_commit_pair_both(tfull(acc));
                    if (++acc == NA) {
                        acc = 0;
                        acc_phase ^= 1u;
                    }
                }
                if (ok) tc_commit_pair_both(xempty);
            }
            tc_commit_pair_both(drain_bar);
            const uint64_t t0 = global_ns();
            while (!mbar_try_wait(drain_bar, 0) && global_ns() - t0 < kWaitLimitNs) {
            }
        } else if (!kPair && lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(128, 128);
            int stage = 0;
            uint32_t phase = 0, xphase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int tile = tile0; tile < tiles && ok; tile += tstep) {
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
        // Warp w (2..17) reads tensor-memory lanes 32*(w%4).. (row r of the
        // tile) and part `part` (0..3) of every chunk: clean columns
        // part*16 .. +16 and the matching noise columns 64 + part*16 .. +16.
        // Each thread keeps the running top-k of its part; the four parts of
        // a row merge through shared memory at the end of the tile.
        const int part = (warp - 2) >> 2;
        const int quad = warp & 3;
        const int r = quad * 32 + lane;
        const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
        int acc = 0;
        uint32_t acc_phase = 0;
        bool ok = true;
        for (int tile = tile0; tile < tiles; tile += tstep) {
            const GateTile ti = gate_tile<kGrouped, kPair>(tile, a, rank);
            const bool valid = r < ti.rows;
            // The row's token, its output slots and the score columns it reads.
            int64_t t = ti.row0 + r;
            int64_t out0 = t * a.k;
            float wrow = 1.0f;
            int col_off = 0;  // eps/bg column of list column 0
            if (kGrouped) {
                t = 0;
                out0 = 0;
                if (valid) {
                    const int pair = a.perm_g[ti.row0 + r];
                    t = pair / a.kg;
                    const int q = pair - static_cast<int>(t) * a.kg;
                    out0 = t * a.k + static_cast<int64_t>(q) * a.kk;
                    wrow = a.gw[pair];
                }
                col_off = a.groups + ti.g * a.m;
            }
            const bool noisy = valid && a.noisy;
            const float *eps_row = noisy ? a.eps + t * a.ldE + col_off : nullptr;
            const float *bg_row = a.bg ? a.bg + col_off : nullptr;
            // 16-byte loads need an aligned row, column base and column count
            const bool vec_eps = ((a.ldE | col_off | a.ncols) & 3) == 0;
            TopK<KM> list;
            list.reset();
            for (int c = 0; c < a.chunks; ++c) {
                const int col0 = c * kGateChunk + part * kPartCols;  // list column of this part
                if (eps_row && c + 2 < a.chunks && col0 + 2 * kGateChunk < a.ncols)
                    prefetch_l2(eps_row + col0 + 2 * kGateChunk);
                float ev[kPartCols];
                if (eps_row && col0 < a.ncols) {
                    load_eps<kPartCols>(eps_row, col0, a.ncols, vec_eps, ev);
                } else {
#pragma unroll
                    for (int j = 0; j < kPartCols; ++j) ev[j] = 0.0f;
                }
                // the gate biases of this part's columns, one per lane (read back by shuffles)
                const float bgl = bg_row && lane < kPartCols && col0 + lane < a.ncols
                                      ? __ldg(bg_row + col0 + lane)
                                      : 0.0f;
                if (ok && !mbar_wait_bounded(tfull(acc), acc_phase, abort_flag, a.err,
                                             kSiteTcEpilogue))
                    ok = false;
                ok = __all_sync(0xffffffffu, ok);  // warp-uniform: the shuffles below need every lane
                // The row's k-th best so far is at least the largest of the
                // four parts' k-th scores after the previous chunk (each part's
                // list holds k of the row's columns): a tighter filter than
                // this part's own list, exact because every column of this
                // chunk has a higher index than every column before it.
                float thr_rows = -INFINITY;
                if (Cfg::kShareThr && c > 0) {
                    quad_bar(quad);
                    const float *tb = thr_sh + ((c - 1) & 1) * kGateParts * kGateRows + r;
                    thr_rows = fmaxf(fmaxf(tb[0], tb[kGateRows]),
                                     fmaxf(tb[2 * kGateRows], tb[3 * kGateRows]));
                }
                if (ok) {
                    tc_fence_after();
                    const float thr = fmaxf(list.kth(a.kf), thr_rows);  // fixed for the span
                    uint32_t cv[16], nv[16];
                    const uint32_t col = static_cast<uint32_t>(acc * 128 + part * kPartCols);
                    tmem_ld_32x32b_x16(tmem_base + lane_addr + col, cv);
                    tmem_ld_32x32b_x16(tmem_base + lane_addr + col + 64, nv);
                    tmem_ld_wait();
                    // this warp's part of the accumulator is read
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        if (kPair)
                            mbar_arrive_remote(mapa_shared(tempty(acc), 0));
                        else
                            mbar_arrive(tempty(acc));
                    }
                    if (a.c_out) {  // load mode: clean score, noise scale
                        // (warp-uniform branch: the bias shuffles need every
                        // lane; only the stores depend on the row)
                        float *crow = a.c_out + t * a.ncols + col0;
                        float *srow = a.s_out + t * a.ncols + col0;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {  // four columns at a time
                            float cc[4], ss[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int j = 4 * q + e;
                                cc[e] = __uint_as_float(cv[j]) + __shfl_sync(0xffffffffu, bgl, j);
                                ss[e] = softplus_fast(__uint_as_float(nv[j]));
                            }
                            if (!valid) continue;
                            if ((a.ncols & 3) == 0) {  // 16-byte rows: float4 stores
                                if (col0 + 4 * q < a.ncols) {
                                    reinterpret_cast<float4 *>(crow)[q] = make_float4(cc[0], cc[1], cc[2], cc[3]);
                                    reinterpret_cast<float4 *>(srow)[q] = make_float4(ss[0], ss[1], ss[2], ss[3]);
                                }
                            } else {
#pragma unroll
                                for (int e = 0; e < 4; ++e)
                                    if (col0 + 4 * q + e < a.ncols) {
                                        crow[4 * q + e] = cc[e];
                                        srow[4 * q + e] = ss[e];
                                    }
                            }
                        }
                    }
                    // Pass 1 (branch-free): the noisy score of every column and
                    // which ones beat the k-th entry of the list.  Within a
                    // thread's list the columns arrive in increasing index order,
                    // so an equal score never displaces an entry: '>' is exact.
                    // Rows past the tile flag nothing.
                    uint32_t pass = 0;
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int sc = col0 + j;
                        float h = __uint_as_float(cv[j]) + __shfl_sync(0xffffffffu, bgl, j);
                        if (noisy) h += ev[j] * softplus_fast(__uint_as_float(nv[j]));
                        cv[j] = __float_as_uint(h);
                        if (valid && sc < a.ncols && h > thr) pass |= 1u << j;
                    }
                    if constexpr (KM == 4) {
                        // First chunk of the tile, empty list: the list is the
                        // best four of these sixteen columns (columns past the
                        // row or the tile rank last), by a fixed network.
                        if (c == 0) {
                            float v16[16];
                            int i16[16];
#pragma unroll
                            for (int j = 0; j < 16; ++j) {
                                const bool use = valid && col0 + j < a.ncols;
                                v16[j] = use ? __uint_as_float(cv[j]) : -INFINITY;
                                i16[j] = use ? col0 + j : INT_MAX;
                            }
                            top4_of16(v16, i16, list.v, list.i);
                            pass = 0u;
                        }
                    }
                    // Pass 2 (rare after the first chunk): each lane inserts its
                    // own flagged columns in increasing index order; the score
                    // leaves the register list through a compile-time select
                    // chain, so the list stays in registers.
                    while (pass != 0u) {
                        const int j = __ffs(pass) - 1;
                        pass &= pass - 1u;
                        float hv = __uint_as_float(cv[0]);
#pragma unroll
                        for (int q = 1; q < 16; ++q)
                            if (q == j) hv = __uint_as_float(cv[q]);
                        list.insert(hv, col0 + j);
                    }
                }
                if (Cfg::kShareThr && c + 1 < a.chunks)
                    thr_sh[(c & 1) * kGateParts * kGateRows + part * kGateRows + r] = list.kth(a.kf);
                if (++acc == NA) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            // The four parts of a row merge in two rounds: parts 2 and 3 hand
            // their lists to parts 0 and 1, then part 1 to part 0, which
            // writes the row.  Every epilogue thread takes part in the barriers.
            epi_bar();  // the previous tile's exchange is read
            if (part >= 2) {
#pragma unroll
                for (int q = 0; q < KM; ++q) {
                    xch_v[((part - 2) * KM + q) * kGateRows + r] = list.v[q];
                    xch_i[((part - 2) * KM + q) * kGateRows + r] = list.i[q];
                }
            }
            epi_bar();
            if (part < 2 && ok && valid) {
#pragma unroll
                for (int q = 0; q < KM; ++q)
                    list.insert(xch_v[(part * KM + q) * kGateRows + r],
                                xch_i[(part * KM + q) * kGateRows + r]);
            }
            epi_bar();
            if (part == 1) {
#pragma unroll
                for (int q = 0; q < KM; ++q) {
                    xch_v[q * kGateRows + r] = list.v[q];
                    xch_i[q * kGateRows + r] = list.i[q];
                }
            }
            epi_bar();
            if (part == 0 && ok && valid) {
#pragma unroll
                for (int q = 0; q < KM; ++q)
                    list.insert(xch_v[q * kGateRows + r], xch_i[q * kGateRows + r]);
                float w[KM];
                softmax_top<KM>(list, a.kk, w);
                if (a.vk_out) {  // the k-th and (k+1)-th noisy score (-inf past the list)
                    a.vk_out[2 * t] = list.kth(a.kk);
                    a.vk_out[2 * t + 1] = a.kk < a.ncols ? list.kth(a.kk + 1) : -INFINITY;
                }
                const int id_off = kGrouped ? ti.g * a.m : 0;
#pragma unroll
                for (int q = 0; q < KM; ++q)
                    if (q < a.kk) {
                        a.idx[out0 + q] = id_off + list.i[q];
                        a.G[out0 + q] = wrow * w[q];
                    }
            }
        }
    }
    if constexpr (kPair) {
        __syncwarp();
        tc_fence_before();
        cluster_sync();   // no pair MMA, remote arrival or tensor-memory read is left
        tc_fence_after();
        if (warp == 1) tmem_dealloc_pair(tmem_base, Cfg::kTmemCols);
    } else {
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (warp == 1) tmem_dealloc(tmem_base, Cfg::kTmemCols);
    }
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

// x [rows, d] bf16 seen as {64, rows, d/64} (strides d*2 and 128 bytes); a box
// of 128 rows x kb_box k-blocks lands as kb_box 128-byte-swizzled K-major tiles.
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

template <bool kResident, bool kGrouped, int KM>
cudaError_t launch_gate_tc_t(const CUtensorMap &mx, const uint8_t *wpack, const GateArgs &ga,
                             int grid, cudaStream_t st) {
    using Cfg = GateCfg<kResident, KM>;
    // Per-context opt-in above 48 KB, set before every launch (cheap).
    const cudaError_t attr = cudaFuncSetAttribute(
        gate_tc<kResident, kGrouped, KM>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
    if (attr != cudaSuccess) return attr;
    return launch_pdl(gate_tc<kResident, kGrouped, KM>, dim3(grid), dim3(kGateThreads), Cfg::kSmem, st,
                      mx, wpack, ga, mx);
}

// Packed W in the pair layout viewed as rows of 128 bytes (64 bf16, no
// swizzle: the bytes are already in the order the MMA reads), boxes of 256
// rows = 32 KB = one SM's half of two k-blocks.
bool gate_pair_wmap(CUtensorMap *m, const void *pack, size_t bytes) {
    EncodeTiledFn enc = gate_encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {64, static_cast<cuuint64_t>(bytes / 128)};
    cuuint64_t strides[1] = {128};
    cuuint32_t box[2] = {64, 256};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(pack), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int KM>
cudaError_t launch_gate_pair_t(const CUtensorMap &mx, const CUtensorMap &mw, const uint8_t *wpack,
                               const GateArgs &ga, int pairs, cudaStream_t st) {
    using Cfg = GateCfg<true, KM, true>;
    auto kern = gate_tc<true, false, KM, true>;
    const cudaError_t attr =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
    if (attr != cudaSuccess) return attr;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * pairs, 1, 1);
    cfg.blockDim = dim3(kGateThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg::kSmem;
    cfg.stream = st;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, mx, wpack, ga, mw);
}

// The CTA-pair gate serves flat gating with x resident (d <= 512).
cudaError_t launch_gate_pair(int km, const CUtensorMap &mx, const uint8_t *wpack, size_t pack_bytes,
                             const GateArgs &ga, cudaStream_t st) {
    CUtensorMap mw;
    if (!gate_pair_wmap(&mw, wpack, pack_bytes)) return cudaErrorInvalidValue;
    const int64_t tiles = (ga.T + 2 * kGateRows - 1) / (2 * kGateRows);
    const int64_t maxp = sm_count() / 2;
    const int pairs = static_cast<int>(tiles < maxp ? tiles : maxp);
    if (km <= 2) return launch_gate_pair_t<2>(mx, mw, wpack, ga, pairs, st);
    if (km <= 4) return launch_gate_pair_t<4>(mx, mw, wpack, ga, pairs, st);
    if (km <= 8) return launch_gate_pair_t<8>(mx, mw, wpack, ga, pairs, st);
    return launch_gate_pair_t<16>(mx, mw, wpack, ga, pairs, st);
}

template <bool kGrouped>
cudaError_t launch_gate_tc_km(bool resident, int km, const CUtensorMap &mx, const uint8_t *wpack,
                              const GateArgs &ga, int grid, cudaStream_t st) {
    if (resident) {
        if (km <= 2) return launch_gate_tc_t<true, kGrouped, 2>(mx, wpack, ga, grid, st);
        if (km <= 4) return launch_gate_tc_t<true, kGrouped, 4>(mx, wpack, ga, grid, st);
        if (km <= 8) return launch_gate_tc_t<true, kGrouped, 8>(mx, wpack, ga, grid, st);
        return launch_gate_tc_t<true, kGrouped, 16>(mx, wpack, ga, grid, st);
    }
    if (km <= 2) return launch_gate_tc_t<false, kGrouped, 2>(mx, wpack, ga, grid, st);
    if (km <= 4) return launch_gate_tc_t<false, kGrouped, 4>(mx, wpack, ga, grid, st);
    if (km <= 8) return launch_gate_tc_t<false, kGrouped, 8>(mx, wpack, ga, grid, st);
    return launch_gate_tc_t<false, kGrouped, 16>(mx, wpack, ga, grid, st);
}

int chunks_of(int cols) { return (cols + kGateChunk - 1) / kGateChunk; }

}  // namespace

size_t gate_tc_pack_bytes(const moe_shape &s) {
    int chunks;
    if (s.groups == 0) {
        chunks = chunks_of(s.n);
    } else {
        chunks = chunks_of(s.groups) + s.groups * chunks_of(s.n / s.groups);
    }
    return static_cast<size_t>(chunks) * 128 * s.d * 2 * 2;  // hi + lo
}

bool gate_tc_supported(const moe_shape &s) { return s.dtype == MOE_BF16; }

cudaError_t launch_gate_tc_load(const moe_shape &s, const void *x, const float *Wg, const float *Wn,
                                const float *bg, const float *eps, int32_t *idx, float *G,
                                float *c_out, float *s_out, float *vk_out, void *ws,
                                const WsLayout &L, cudaStream_t st) {
    // flat, noisy, k + 1 <= 16 (the list keeps the (k+1)-th score too)
    const bool resident = s.d <= 512;
    const int kblocks = s.d / 64;
    uint8_t *pack = ws_ptr<uint8_t>(ws, L.gpack);
    GateArgs ga{};
    ga.bg = bg;
    ga.eps = eps;
    ga.T = s.T;
    ga.d = s.d;
    ga.ldE = s.n;
    ga.noisy = 1;
    ga.err = ws_ptr<int32_t>(ws, 0);
    ga.idx = idx;
    ga.G = G;
    ga.k = ga.kk = s.k;
    ga.kf = s.k + 1;  // the (k+1)-th score must be exact too
    ga.ncols = s.n;
    ga.chunks = chunks_of(s.n);
    ga.c_out = c_out;
    ga.s_out = s_out;
    ga.vk_out = vk_out;
    {
        const cudaError_t pe = launch_pdl(gate_pack, dim3(ga.chunks, 2, 4 * kblocks), dim3(128), 0, st, Wg, Wn, s.d, s.n, 0, s.n, 0, 1, 1, 0, pack);
        if (pe != cudaSuccess) return pe;
    }
    CUtensorMap mx;
    if (!gate_map(&mx, x, s.d, static_cast<uint64_t>(s.T), resident ? kblocks : 1))
        return cudaErrorInvalidValue;
    const int tiles = static_cast<int>((s.T + kGateRows - 1) / kGateRows);
    const int sms = sm_count();
    return launch_gate_tc_km<false>(resident, s.k + 1, mx, pack, ga, tiles < sms ? tiles : sms, st);
}

cudaError_t launch_gate_tc(const moe_shape &s, const void *x, const float *Wg, const float *Wn,
                           const float *bg, const float *eps, int32_t *idx, float *G, void *ws,
                           const WsLayout &L, cudaStream_t st) {
    const int C = gate_cols(s);
    const int noisy = (s.noisy && eps != nullptr && Wn != nullptr) ? 1 : 0;
    const bool resident = s.d <= 512;
    const int kblocks = s.d / 64;
    int32_t *err = ws_ptr<int32_t>(ws, 0);
    uint8_t *pack = ws_ptr<uint8_t>(ws, L.gpack);
    const float *Wnp = noisy ? Wn : Wg;
    GateArgs ga{};
    ga.bg = bg;
    ga.eps = noisy ? eps : nullptr;
    ga.T = s.T;
    ga.d = s.d;
    ga.ldE = C;
    ga.noisy = noisy;
    ga.err = err;
    const int sms = sm_count();
    if (s.groups == 0) {
        // flat: one pass over the tokens and the n columns
        ga.idx = idx;
        ga.G = G;
        ga.k = ga.kk = ga.kf = s.k;
        ga.ncols = s.n;
        ga.chunks = chunks_of(s.n);
        const bool pair = resident;
        {
            const cudaError_t pe = launch_pdl(gate_pack, dim3(ga.chunks, 2, 4 * kblocks), dim3(128), 0, st, Wg, Wnp, s.d, C, 0, s.n, 0, 1,
                                                             noisy, pair ? 1 : 0, pack);
            if (pe != cudaSuccess) return pe;
        }
        CUtensorMap mx;
        if (!gate_map(&mx, x, s.d, static_cast<uint64_t>(s.T), resident ? kblocks : 1))
            return cudaErrorInvalidValue;
        if (pair)
            return launch_gate_pair(s.k, mx, pack,
                                    static_cast<size_t>(ga.chunks) * kblocks * 2 * kKBytes, ga, st);
        const int tiles = static_cast<int>((s.T + kGateRows - 1) / kGateRows);
        return launch_gate_tc_km<false>(resident, s.k, mx, pack, ga, tiles < sms ? tiles : sms, st);
    }

    // hierarchical, pass 1: the groups (flat over the G group columns)
    const int Gn = s.groups, kg = s.k_groups, ki = s.k / s.k_groups, m = s.n / s.groups;
    const int64_t P = s.T * static_cast<int64_t>(kg);  // (token, rank) pairs
    int32_t *gidx = ws_ptr<int32_t>(ws, L.gsel);
    float *gw = reinterpret_cast<float *>(gidx + P);
    const int pchunks = chunks_of(Gn), mchunks = chunks_of(m);
    uint8_t *pack_i = pack + static_cast<size_t>(pchunks) * kblocks * 2 * kKBytes;
    GateArgs gp = ga;
    gp.idx = gidx;
    gp.G = gw;
    gp.k = gp.kk = gp.kf = kg;
    gp.ncols = Gn;
    gp.chunks = pchunks;
    const bool gpair = resident;
    {
        const cudaError_t pe = launch_pdl(gate_pack, dim3(pchunks, 2, 4 * kblocks), dim3(128), 0, st, Wg, Wnp, s.d, C, 0, Gn, 0, 1, noisy,
                                                          gpair ? 1 : 0, pack);
        if (pe != cudaSuccess) return pe;
    }
    CUtensorMap mx;
    if (!gate_map(&mx, x, s.d, static_cast<uint64_t>(s.T), resident ? kblocks : 1))
        return cudaErrorInvalidValue;
    const int ttiles = static_cast<int>((s.T + kGateRows - 1) / kGateRows);
    cudaError_t e =
        gpair ? launch_gate_pair(kg, mx, pack, static_cast<size_t>(pchunks) * kblocks * 2 * kKBytes,
                                 gp, st)
              : launch_gate_tc_km<false>(resident, kg, mx, pack, gp, ttiles < sms ? ttiles : sms, st);
    if (e != cudaSuccess) return e;

    // pass 2: route the pairs by group, gather their x rows, score each group's columns
    moe_shape sg = s;
    sg.n = Gn;
    sg.k = kg;
    sg.groups = 0;
    sg.k_groups = 0;
    int32_t *counts_g = ws_ptr<int32_t>(ws, L.counts);
    int32_t *offsets_g = ws_ptr<int32_t>(ws, L.offsets);
    int32_t *perm_g = ws_ptr<int32_t>(ws, L.perm);
    int32_t *inv_g = ws_ptr<int32_t>(ws, L.inv_perm);
    int32_t *tiles_g = ws_ptr<int32_t>(ws, L.tiles);
    __nv_bfloat16 *xg = ws_ptr<__nv_bfloat16>(ws, L.xperm);
    e = launch_dispatch(sg, gidx, gw, counts_g, offsets_g, perm_g, inv_g,
                        ws_ptr<float>(ws, L.importance), ws_ptr<float>(ws, L.cv2), ws, L, st);
    if (e != cudaSuccess) return e;
    e = launch_row_tiles(offsets_g, Gn, kGateRows, tiles_g, st);
    if (e != cudaSuccess) return e;
    e = launch_gather_rows(static_cast<const __nv_bfloat16 *>(x), perm_g, offsets_g, Gn, P, s.d, kg,
                           xg, err, st);
    if (e != cudaSuccess) return e;
    {
        const cudaError_t pe = launch_pdl(gate_pack, dim3(Gn * mchunks, 2, 4 * kblocks), dim3(128), 0, st, Wg, Wnp, s.d, C, Gn, s.n, m, mchunks,
                                                            noisy, 0, pack_i);
        if (pe != cudaSuccess) return pe;
    }
    CUtensorMap mg;
    if (!gate_map(&mg, xg, s.d, static_cast<uint64_t>(P), resident ? kblocks : 1))
        return cudaErrorInvalidValue;
    GateArgs gi = ga;
    gi.idx = idx;
    gi.G = G;
    gi.k = s.k;
    gi.kk = gi.kf = ki;
    gi.ncols = m;
    gi.chunks = mchunks;
    gi.perm_g = perm_g;
    gi.offsets_g = offsets_g;
    gi.tiles_g = tiles_g;
    gi.gw = gw;
    gi.groups = Gn;
    gi.kg = kg;
    gi.m = m;
    const int64_t max_tiles = (P + kGateRows - 1) / kGateRows + Gn;
    const int grid = static_cast<int>(max_tiles < sms ? max_tiles : sms);
    return launch_gate_tc_km<true>(resident, ki, mg, pack_i, gi, grid, st);
}

}  // namespace moe

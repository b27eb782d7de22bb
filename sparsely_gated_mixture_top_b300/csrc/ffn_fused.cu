// ffn_fused.cu -- both layers of every expert's feed-forward network in one
// persistent kernel on SM pairs (tcgen05 cta_group::2), the hidden activation
// kept on chip.
//
// Each expert is a one-hidden-layer ReLU network ("MoE:稀疏门控混合专家",
// section 二): for the rows r of expert e (expert order, offsets[e] ..
// offsets[e+1])
//     H[r, :] = bf16( ReLU( X[r, :] W1[e]^T + b1[e] ) )       [h]
//     Y[r, :] = bf16( H[r, :] W2[e]^T + b2[e] )               [d]
// with fp32 accumulation and one round-to-nearest-even rounding of each
// layer's output, the same arithmetic as the two separate grouped GEMMs
// (ffn_pair.cu), which write H to memory and read it back.  Here H never
// leaves the pair, a quarter to a third of the expert stage's DRAM traffic
// at the widths this kernel serves (d = 256 or 512, h a multiple of 256).
// Each token tile takes in its expert's weights again, so the library uses
// this kernel only where experts average at most 128 rows
// (fused_ffn_supported).
//
// Unit of work: one token tile of one expert, at most 128 rows (the tile
// table's entries {expert, first row, rows, N = rows rounded up to 32}).
// Tokens sit on the MMA's N side and weight rows on its M side (M = 256,
// 128 per CTA), so a tile takes exactly the rows its expert has.  Per unit,
// the hidden features are taken in chunks of 256:
//     L1(c):  H^T[chunk c] = W1[e, chunk c rows] . X_tile^T      (K = d)
//     epilogue: bias, ReLU, bf16, stored as the K-major B operand of layer 2
//     L2(c):  Y^T += W2[e, :, chunk c columns] . H[chunk c]^T     (K = 256)
// issued in the order L1(0), L1(1), L2(0), L1(2), L2(1), ... so the epilogue
// of chunk c overlaps the first layer of chunk c+1.
//
// Tensor memory (512 columns per CTA): Y^T accumulators at columns 0 and 128
// (one per 256 output features), H^T accumulators at 256 and 384 (double
// buffered).  Shared memory per CTA: three 32 KB weight stages (128 weight
// rows x two 64-wide k-blocks), the tile's N/2 token rows of X (resident for
// all chunks, up to 64 KB) and two 32 KB buffers of H (the CTA's N/2 tokens x
// 256 hidden features, 128-byte swizzled K-major).
//
// The pair split: CTA s holds accumulator rows (features) s*128 .. +128 of
// every M tile, all N token columns, while each CTA must supply its own N/2
// tokens as layer 2's B rows.  So the epilogue of CTA s writes the values of
// tokens in the other CTA's half straight into that CTA's H buffer (32-bit
// stores of two neighbouring features to distributed shared memory), fences
// them for the tensor core and arrives on the issuing CTA's barrier.
//
// Warps (576 threads per CTA, one CTA per SM, clusters of two):
//   warp 0     TMA producer (each CTA): the tile's X rows, then every weight
//              stage in the order the MMAs use them
//   warp 1     tensor memory; in the even CTA one lane issues the pair MMAs
//   warps 2-17 epilogue (each CTA): warp w reads lanes 32*(w%4) .. +32 and
//              the 32-token column chunk (w-2)/4 of each accumulator
// Every wait is bounded; on a timeout the kernel records MOE_ERR_TIMEOUT and
// winds down.
#include "moe_device.cuh"
#include "moe_launch.h"

namespace moe {

namespace {

constexpr int kFTok = 128;            // tokens per tile at most (MMA N)
constexpr int kFM = 256;              // weight rows per MMA (M; 128 per CTA)
constexpr int kFChunk = 256;          // hidden features per chunk
constexpr int kFMaxD = 512;           // model width at most (Y^T accumulators, X tile)
constexpr int kFEpiWarps = 16;
constexpr int kFThreads = 32 * (2 + kFEpiWarps);
constexpr int kFKB = 2;               // 64-wide k-blocks per weight stage
constexpr int kFStages = 3;
constexpr int kFHBufs = 2;            // H buffers in shared memory

struct FusedCfg {
    static constexpr int kKBlockBytes = 128 * 128;                 // 128 rows x 64 bf16
    static constexpr int kStageBytes = kFKB * kKBlockBytes;        // 32 KB
    static constexpr int kXBytes = (kFTok / 2) * 2 * kFMaxD;       // 64 token rows x d
    static constexpr int kHKBlockBytes = (kFTok / 2) * 128;        // 64 token rows x 64 bf16
    static constexpr int kHBytes = (kFChunk / 64) * kHKBlockBytes; // one H buffer
    // full[3], empty[3], xfull, xempty, hacc_full[2], hacc_empty[2],
    // hready[2], hfree[2], yfull, yempty, drain
    static constexpr int kBars = 2 * kFStages + 2 + 8 + 2 + 1;
    static constexpr int kSmem =
        1024 + kFStages * kStageBytes + kXBytes + kFHBufs * kHBytes + 8 * kBars + 16;
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kYCol = 0;      // + m * kFTok
    static constexpr uint32_t kHCol = 256;    // + buffer * kFTok
};
static_assert(FusedCfg::kSmem <= 227 * 1024, "shared memory budget");

// Token-row maps of X: box i holds 16*(i+1) rows and d/64 k-blocks, so a
// tile of N tokens copies exactly its N/2 rows per CTA in one copy.
struct FusedXMaps {
    CUtensorMap m[4];
};

__device__ __forceinline__ bool fused_drain(uint32_t bar, uint32_t parity, int32_t *err) {
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_ns() - t0 > kWaitLimitNs) {
            report(err, MOE_ERR_TIMEOUT, kSiteTcDrain);
            return false;
        }
    }
    return true;
}

// Byte offset of element (token row r, column j) of an H buffer: four
// k-blocks of 64 columns, each 64 rows of 128 bytes whose 16-byte pieces are
// permuted by r & 7 (the layout a 128-byte-swizzled TMA copy writes).
__device__ __forceinline__ uint32_t h_offset(int r, int j) {
    const int kb = j >> 6, cc = j & 63;
    return static_cast<uint32_t>(kb * FusedCfg::kHKBlockBytes + r * 128 +
                                 (((cc >> 3) ^ (r & 7)) << 4) + (cc & 7) * 2);
}

// 18 warps: five of them share one of the SM's four 16K-register
// partitions, so a thread may hold at most 96 registers.
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kFThreads, 1)
    ffn_fused_pair(const __grid_constant__ CUtensorMap mapW1,
                   const __grid_constant__ CUtensorMap mapW2,
                   const __grid_constant__ FusedXMaps mapX, const int32_t *__restrict__ tiles,
                   const int4 *__restrict__ tlist, int n, int d, int h,
                   const float *__restrict__ b1, const float *__restrict__ b2,
                   __nv_bfloat16 *__restrict__ out, int32_t *err) {
    using Cfg = FusedCfg;
    constexpr int STAGES = kFStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint8_t *sW = smem;                                  // STAGES x 32 KB weight rows
    uint8_t *sX = sW + STAGES * Cfg::kStageBytes;        // the tile's token rows of X
    uint8_t *sH = sX + Cfg::kXBytes;                     // 2 x 32 KB hidden buffers
    uint64_t *bars = reinterpret_cast<uint64_t *>(sH + kFHBufs * Cfg::kHBytes);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + Cfg::kBars);
    volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(tmem_slot + 1);
    auto full = [&](int s) { return smem_u32(bars + s); };
    auto empty = [&](int s) { return smem_u32(bars + STAGES + s); };
    const uint32_t xfull = smem_u32(bars + 2 * STAGES);
    const uint32_t xempty = smem_u32(bars + 2 * STAGES + 1);
    auto hacc_full = [&](int b) { return smem_u32(bars + 2 * STAGES + 2 + b); };
    auto hacc_empty = [&](int b) { return smem_u32(bars + 2 * STAGES + 4 + b); };
    auto hready = [&](int b) { return smem_u32(bars + 2 * STAGES + 6 + b); };
    auto hfree = [&](int b) { return smem_u32(bars + 2 * STAGES + 8 + b); };
    const uint32_t yfull = smem_u32(bars + 2 * STAGES + 10);
    const uint32_t yempty = smem_u32(bars + 2 * STAGES + 11);
    const uint32_t drain_bar = smem_u32(bars + 2 * STAGES + 12);

    const uint32_t rank = cluster_ctarank();   // 0: the CTA that issues the pair MMAs
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        mbar_init(xfull, 1);
        mbar_init(xempty, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(hacc_full(b), 1);
            mbar_init(hacc_empty(b), 2 * kFEpiWarps);   // one arrival per epilogue warp of each CTA
            mbar_init(hready(b), 2 * kFEpiWarps);
            mbar_init(hfree(b), 1);
        }
        mbar_init(yfull, 1);
        mbar_init(yempty, 2 * kFEpiWarps);
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&mapW1);
        tma_prefetch_map(&mapW2);
        for (int i = 0; i < 4; ++i) tma_prefetch_map(&mapX.m[i]);
    }
    // A pair allocation is issued by one warp of each CTA once both CTAs are
    // known to be running; the second cluster barrier publishes the barriers
    // and the allocation to both CTAs before any copy, MMA or remote access.
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

    const int total = tiles[n];
    const int nh = h / kFChunk;          // hidden chunks per tile
    const int nm = d / kFM;              // M tiles of the second layer (1 or 2)
    const int kbd = d / 64;              // k-blocks of the first layer
    const int cl = static_cast<int>(blockIdx.x >> 1), ncl = static_cast<int>(gridDim.x >> 1);

    // The MMA order of a unit, as 2*nh operations p = 0 .. 2*nh-1:
    //   p = 0: L1(0);  p odd (< 2nh-1): L1((p+1)/2);  p even > 0: L2(p/2 - 1);
    //   p = 2nh-1: L2(nh-1).
    // L1(c) uses d/64 k-blocks of W1 (d/128 stages), L2(c) 256/64 k-blocks of
    // W2 for each of the nm M tiles (2*nm stages).
    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, xphase = 0;
            bool ok = true;
            for (int q = cl; q < total && ok; q += ncl) {
                const int4 t = __ldg(tlist + q);
                const int hn = t.w >> 1;      // this CTA's token rows (a multiple of 16)
                if (!mbar_wait_bounded(xempty, xphase ^ 1u, abort_flag, err, kSiteTcProducer)) {
                    ok = false;
                    break;
                }
                if (rank == 0) mbar_arrive_expect_tx(xfull, 2 * hn * 128 * kbd);
                tma_load_3d_pair(smem_u32(sX), &mapX.m[(hn >> 4) - 1], mapa_shared(xfull, 0), 0,
                                 t.y + static_cast<int>(rank) * hn, 0);
                xphase ^= 1u;
                const int w1row = t.x * h + static_cast<int>(rank) * 128;
                const int w2row = t.x * d + static_cast<int>(rank) * 128;
                for (int p = 0; p < 2 * nh && ok; ++p) {
                    const bool l1 = p == 0 || ((p & 1) && p != 2 * nh - 1);
                    const int c = l1 ? (p + 1) / 2 : (p == 2 * nh - 1 ? nh - 1 : p / 2 - 1);
                    const int nst = l1 ? kbd / kFKB : nm * (kFChunk / 64 / kFKB);
                    for (int i = 0; i < nst; ++i) {
                        if (!mbar_wait_bounded(empty(stage), phase ^ 1u, abort_flag, err,
                                               kSiteTcProducer)) {
                            ok = false;
                            break;
                        }
                        // this CTA's 128 weight rows, two k-blocks; both CTAs'
                        // copies complete on the even CTA's barrier
                        int row, kb;
                        if (l1) {
                            row = w1row + c * kFChunk;
                            kb = i * kFKB;
                        } else {
                            const int per = kFChunk / 64 / kFKB;   // stages per M tile
                            row = w2row + (i / per) * kFM;
                            kb = c * (kFChunk / 64) + (i % per) * kFKB;
                        }
                        if (rank == 0) mbar_arrive_expect_tx(full(stage), 2 * Cfg::kStageBytes);
                        tma_load_3d_pair(smem_u32(sW + stage * Cfg::kStageBytes), l1 ? &mapW1 : &mapW2,
                                         mapa_shared(full(stage), 0), 0, row, kb);
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
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
            uint32_t phase = 0, xphase = 0, yphase = 0;
            int g = 0;          // hidden chunks of the units before this one
            bool ok = true;
            for (int q = cl; q < total && ok; q += ncl) {
                const int4 t = __ldg(tlist + q);
                const int N = t.w, hn = N >> 1;
                const uint32_t idesc = idesc_bf16_f32(kFM, N);
                const uint32_t xkb = static_cast<uint32_t>(hn) * 128;   // X k-block stride
                if (!mbar_wait_bounded(xfull, xphase, abort_flag, err, kSiteTcMma)) break;
                xphase ^= 1u;
                tc_fence_after();
                for (int p = 0; p < 2 * nh && ok; ++p) {
                    const bool l1 = p == 0 || ((p & 1) && p != 2 * nh - 1);
                    const int c = l1 ? (p + 1) / 2 : (p == 2 * nh - 1 ? nh - 1 : p / 2 - 1);
                    const int gc = g + c, b = gc & 1;   // accumulator of chunk c
                    const uint32_t ph = static_cast<uint32_t>(gc >> 1) & 1u;
                    const int hs = gc % kFHBufs;        // its H buffer
                    const uint32_t hph = static_cast<uint32_t>(gc / kFHBufs) & 1u;
                    if (l1) {
                        // H^T of chunk c into accumulator b, once the epilogue has read it out
                        ok = mbar_wait_bounded(hacc_empty(b), ph ^ 1u, abort_flag, err, kSiteTcMma);
                    } else {
                        // H of chunk c stored by both CTAs' epilogues; for the
                        // first chunk also the previous unit's Y^T read out
                        ok = mbar_wait_cluster_bounded(hready(hs), hph, abort_flag, err, kSiteTcMma) &&
                             (c != 0 ||
                              mbar_wait_bounded(yempty, yphase ^ 1u, abort_flag, err, kSiteTcMma));
                    }
                    if (!ok) break;
                    tc_fence_after();
                    const int per = kFChunk / 64 / kFKB;
                    const int nst = l1 ? kbd / kFKB : nm * per;
                    const uint32_t hb = smem_u32(sH + hs * Cfg::kHBytes);
                    for (int i = 0; i < nst; ++i) {
                        if (!mbar_wait_bounded(full(stage), phase, abort_flag, err, kSiteTcMma)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t a0 = smem_u32(sW + stage * Cfg::kStageBytes);
                        uint32_t d_tmem, b0, bstride;
                        bool first;
                        if (l1) {
                            d_tmem = tmem_base + Cfg::kHCol + static_cast<uint32_t>(b * kFTok);
                            b0 = smem_u32(sX) + static_cast<uint32_t>(i * kFKB) * xkb;
                            bstride = xkb;
                            first = i == 0;
                        } else {
                            d_tmem = tmem_base + Cfg::kYCol + static_cast<uint32_t>((i / per) * kFTok);
                            b0 = hb + static_cast<uint32_t>((i % per) * kFKB * Cfg::kHKBlockBytes);
                            bstride = Cfg::kHKBlockBytes;
                            first = c == 0 && i % per == 0;
                        }
                        for (int j = 0; j < kFKB; ++j) {
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                tc_mma_f16_pair(d_tmem,
                                                sdesc_kmajor_sw128(a0 + j * Cfg::kKBlockBytes + kk * 32),
                                                sdesc_kmajor_sw128(b0 + j * bstride + kk * 32), idesc,
                                                (first && j == 0 && kk == 0) ? 0u : 1u);
                        }
                        tc_commit_pair_both(empty(stage));
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (!ok) break;
                    if (l1) {
                        tc_commit_pair_both(hacc_full(b));
                        if (c == nh - 1) tc_commit_pair_both(xempty);   // X no longer read
                    } else {
                        tc_commit_pair_both(hfree(hs));
                    }
                }
                if (!ok) break;
                tc_commit_pair_both(yfull);
                g += nh;
                yphase ^= 1u;
            }
            // Every MMA this thread issued has finished once this arrives.
            tc_commit_pair_both(drain_bar);
            fused_drain(drain_bar, 0, err);
        }
    } else {
        // Epilogue: warp w (2..17) may read tensor-memory lanes 32*(w%4) ..
        // +32 (features) and takes the 32-token column chunk (w-2)/4.  Values
        // leave as bf16 pairs of neighbouring features: lanes 2i and 2i+1
        // swap halves so that the even lane holds both features of the even
        // token and the odd lane both of the odd token (4-byte stores).
        const int ew = warp - 2;
        const int quad = warp & 3;
        const int sub = ew >> 2;
        const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t hcl0 = mapa_shared(smem_u32(sH), 0), hcl1 = mapa_shared(smem_u32(sH), 1);
        const int jcol = static_cast<int>(rank) * 128 + quad * 32 + lane;   // feature in a 256-block
        const int odd = lane & 1;
        const int jpair = jcol - odd;                                       // first of this lane's pair
        uint32_t yphase = 0;
        int g = 0;
        for (int q = cl; q < total; q += ncl) {
            const int4 t = __ldg(tlist + q);
            const int e = t.x, row0 = t.y, rows = t.z, N = t.w, hn = N >> 1;
            const bool active = sub * 32 < N;   // warp-uniform
            bool ok = true;
            for (int c = 0; c < nh; ++c) {
                const int gc = g + c, b = gc & 1;
                const uint32_t ph = static_cast<uint32_t>(gc >> 1) & 1u;
                const int hs = gc % kFHBufs;
                const uint32_t hph = static_cast<uint32_t>(gc / kFHBufs) & 1u;
                const float bv =
                    b1 ? __ldg(b1 + static_cast<int64_t>(e) * h + c * kFChunk + jcol) : 0.0f;
                if (!mbar_wait_bounded(hacc_full(b), ph, abort_flag, err, kSiteTcEpilogue)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t v[32];
                if (active)
                    tmem_ld_32x32b_x32(tmem_base + lane_addr + Cfg::kHCol +
                                           static_cast<uint32_t>(b * kFTok + sub * 32),
                                       v);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_remote(mapa_shared(hacc_empty(b), 0));
                // the second-layer MMAs that last read this H buffer are done
                if (!mbar_wait_bounded(hfree(hs), hph ^ 1u, abort_flag, err, kSiteTcEpilogue)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (active) {
                    const uint32_t boff = static_cast<uint32_t>(hs * Cfg::kHBytes);
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        // tokens 2i, 2i+1 of the chunk: this lane's feature, bias, ReLU
                        const uint32_t mine = pack_bf16x2(fmaxf(__uint_as_float(v[2 * i]) + bv, 0.0f),
                                                          fmaxf(__uint_as_float(v[2 * i + 1]) + bv, 0.0f));
                        const uint32_t other = __shfl_xor_sync(0xffffffffu, mine, 1);
                        const uint32_t w = odd ? __byte_perm(other, mine, 0x7632)
                                               : __byte_perm(mine, other, 0x5410);
                        const int tk = sub * 32 + 2 * i + odd;
                        const int own = tk >= hn ? 1 : 0;
                        st_cluster_u32((own ? hcl1 : hcl0) + boff + h_offset(tk - own * hn, jpair), w);
                    }
                }
                fence_proxy_async_cluster();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(mapa_shared(hready(hs), 0));
            }
            if (!ok) break;
            if (!mbar_wait_bounded(yfull, yphase, abort_flag, err, kSiteTcEpilogue)) break;
            tc_fence_after();
            uint32_t py[2][16];
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                if (!active || m >= nm) continue;
                uint32_t v[32];
                tmem_ld_32x32b_x32(tmem_base + lane_addr + Cfg::kYCol +
                                       static_cast<uint32_t>(m * kFTok + sub * 32),
                                   v);
                tmem_ld_wait();
                const float bv = b2 ? __ldg(b2 + static_cast<int64_t>(e) * d + m * kFM + jcol) : 0.0f;
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    py[m][i] = pack_bf16x2(__uint_as_float(v[2 * i]) + bv,
                                           __uint_as_float(v[2 * i + 1]) + bv);
            }
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(mapa_shared(yempty, 0));
            if (active) {
#pragma unroll
                for (int m = 0; m < 2; ++m) {
                    if (m >= nm) continue;
                    uint32_t *dst = reinterpret_cast<uint32_t *>(
                        out + static_cast<int64_t>(row0 + sub * 32 + odd) * d + m * kFM + jpair);
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const uint32_t other = __shfl_xor_sync(0xffffffffu, py[m][i], 1);
                        const uint32_t w = odd ? __byte_perm(other, py[m][i], 0x7632)
                                               : __byte_perm(py[m][i], other, 0x5410);
                        if (sub * 32 + 2 * i + odd < rows) *dst = w;
                        dst += d;   // two token rows on (d / 2 words per row)
                    }
                }
            }
            g += nh;
            yphase ^= 1u;
        }
    }
    __syncwarp();
    tc_fence_before();
    cluster_sync();   // no pair MMA, remote access or tensor-memory read is left
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem_base, Cfg::kTmemCols);
}

}  // namespace

// The fused kernel re-reads an expert's weights for every token tile of at
// most 128 rows, while the two separate GEMMs read them once per 256 rows
// and pay for the hidden activation's round trip instead.  Measured on the
// B300 (FFN stage, CUDA events): fused is ahead at 8 to 64 rows per expert
// on average (2048 experts at T = 4096 and 32768: 0.92 vs 0.92 and 0.83 vs
// 0.80 of the copy bandwidth; 4096 experts at 32 rows: 0.90 vs 0.88) and
// behind at 256 (256 experts: 233 us vs 205 us), where each expert has two
// or three tiles.  So it serves shapes whose experts average at most 128 rows.
bool fused_ffn_supported(const moe_shape &s) {
    return s.dtype == MOE_BF16 && s.d % kFM == 0 && s.d <= kFMaxD && s.h % kFChunk == 0 &&
           slots(s) <= static_cast<int64_t>(kFTok) * s.n;
}

// Largest number of CTA pairs of ffn_fused_pair that fit on the device at once.
static int fused_clusters() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return sm_count() / 2;
    static int cached[64] = {0};
    if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (sm_count() / 2), 1, 1);
    cfg.blockDim = dim3(kFThreads, 1, 1);
    cfg.dynamicSmemBytes = FusedCfg::kSmem;
    int num = 0;
    if (cudaOccupancyMaxActiveClusters(&num, ffn_fused_pair, &cfg) != cudaSuccess || num <= 0) {
        cudaGetLastError();
        num = sm_count() / 2;
    }
    if (dev >= 0 && dev < 64) cached[dev] = num;
    return num;
}

cudaError_t launch_ffn_fused(const moe_shape &s, const __nv_bfloat16 *X, const __nv_bfloat16 *W1,
                             const float *b1, const __nv_bfloat16 *W2, const float *b2,
                             const int32_t *tiles, const int4 *tlist, __nv_bfloat16 *Y,
                             int32_t *err, cudaStream_t st) {
    const int64_t S = slots(s);
    if (!fused_ffn_supported(s)) return cudaErrorInvalidValue;
    CUtensorMap m1, m2;
    FusedXMaps mX;
    if (!make_kmajor_map(&m1, W1, static_cast<uint64_t>(s.d), static_cast<uint64_t>(s.n) * s.h, 128,
                         kFKB) ||
        !make_kmajor_map(&m2, W2, static_cast<uint64_t>(s.h), static_cast<uint64_t>(s.n) * s.d, 128,
                         kFKB))
        return cudaErrorInvalidValue;
    for (int i = 0; i < 4; ++i)
        if (!make_kmajor_map(&mX.m[i], X, static_cast<uint64_t>(s.d), static_cast<uint64_t>(S),
                             static_cast<uint32_t>(16 * (i + 1)), static_cast<uint32_t>(s.d / 64)))
            return cudaErrorInvalidValue;
    // The opt-in above 48 KB belongs to the current device's context: set it
    // before every launch (a cheap host call).
    cudaError_t e = cudaFuncSetAttribute(ffn_fused_pair, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         FusedCfg::kSmem);
    if (e != cudaSuccess) return e;
    // Upper bound of the unit count: every expert may add one partial tile.
    const int64_t max_units = (S + kFTok - 1) / kFTok + s.n;
    int64_t pairs = fused_clusters();
    if (pairs > max_units) pairs = max_units;
    if (pairs < 1) pairs = 1;
    return launch_pdl(ffn_fused_pair, dim3(static_cast<unsigned>(2 * pairs)), dim3(kFThreads),
                      FusedCfg::kSmem, st, m1, m2, mX, tiles, tlist, s.n, s.d, s.h, b1, b2, Y, err);
}

}  // namespace moe

// moe_launch.h -- host-side internals shared by the library's .cu files: the
// workspace layout and the launchers of each stage.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

// Launches `kern` on `st` with programmatic stream serialization (the kernel
// calls pdl_wait() before touching what earlier kernels of the stream
// produce), so that its launch and prologue overlap the previous kernel's
// tail.  Cluster dimensions compiled into the kernel still apply.
template <typename... Params, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Params>(args)...);
}

// MOE_OK for cudaSuccess, else MOE_ERR_CUDA, remembering the CUDA error for
// moe_last_cuda_error (per host thread).
moe_status cuda_to_status(cudaError_t e);

constexpr int kRouteChunk = 1024;  // slots ranked per block by the routing kernels
constexpr int kTcRows = 128;       // rows per tensor-core FFN tile (MMA M)
constexpr int kSimtRows = 64;      // rows per fp32 SIMT FFN tile

inline int gate_cols(const moe_shape &s) { return s.groups == 0 ? s.n : s.groups + s.n; }
inline int64_t slots(const moe_shape &s) { return s.T * static_cast<int64_t>(s.k); }
inline size_t dtype_bytes(const moe_shape &s) { return s.dtype == MOE_BF16 ? 2 : 4; }

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Tensor-core gate (gate_tc.cu): whether it handles a shape, and the bytes of
// its packed split-bf16 gate matrices.
bool gate_tc_supported(const moe_shape &s);
size_t gate_tc_pack_bytes(const moe_shape &s);

// Token tiling of the pair FFN for an expert with R rows and tiles of at most
// cap rows (256, or 128 for the fused two-layer kernel): ceil(R / cap) tiles
// of tn rows, tn = ceil(R / tiles) rounded up to 16 (at most cap); the tile
// count is then ceil(R / tn), so no tile is empty.
__host__ __device__ inline void token_tiling(int R, int &tn, int &ntile, int cap = 256) {
    if (R <= 0) {
        tn = 0;
        ntile = 0;
        return;
    }
    const int n0 = (R + cap - 1) / cap;
    int t = (R + n0 - 1) / n0;
    t = (t + 15) & ~15;
    if (t > cap) t = cap;
    tn = t;
    ntile = (R + t - 1) / t;
}

// Entries of the pair FFN's token-tile table: an expert of R rows has at most
// ceil(R / 128) tiles (tiles of at least 128 rows, or the expert's own rows).
inline size_t pair_tile_capacity(int64_t S, int n) { return static_cast<size_t>(S / 128 + n + 1); }

// Byte offsets of every region of a workspace (all 256-byte aligned).
struct WsLayout {
    size_t header = 0;
    size_t scores = 0;      // gate scores H [T, C] fp32 (SIMT gate only)
    size_t gpack = 0;       // packed bf16 hi/lo gate matrices (tensor-core gate only)
    size_t gsel = 0;        // [T*k_groups] int32 chosen groups, then [T*k_groups] fp32
                            // their weights (hierarchical tensor-core gate only)
    size_t local_rank = 0;  // [S] int32, rank of a slot among same-expert slots of its chunk
    size_t chunk = 0;       // [chunks, n] int32, per-chunk expert counts, then bases
    size_t chunk_imp = 0;   // [chunks, n] float, per-chunk gate-weight sums
    size_t imp_acc = 0;     // [n] float, importance summed over the chunks
    size_t counts = 0;      // [n] int32 (used when the caller does not pass counts)
    size_t offsets = 0;     // [n + 1] int32
    size_t perm = 0;        // [S] int32
    size_t inv_perm = 0;    // [S] int32
    size_t importance = 0;  // [n] fp32
    size_t cv2 = 0;         // [1] fp32
    size_t tiles = 0;       // [n + 1] int32 row-tile starts of the FFN schedule
    size_t ptiles = 0;      // [n + 1] int32 token-tile starts of the pair FFN schedule
    size_t plist = 0;       // [S/256 + n + 1] int4 token tiles of the pair FFN schedule
    size_t xperm = 0;       // [S, d] dtype, x rows in expert order
    size_t hidden = 0;      // [S, h] dtype, hidden activations in expert order
    size_t yslot = 0;       // [S, d] dtype, expert outputs in expert order
    size_t total = 0;
};

inline WsLayout ws_layout(const moe_shape &s) {
    WsLayout L;
    const size_t S = static_cast<size_t>(slots(s));
    const size_t n = static_cast<size_t>(s.n);
    const size_t C = static_cast<size_t>(gate_cols(s));
    const size_t chunks = (S + kRouteChunk - 1) / kRouteChunk;
    const size_t eb = dtype_bytes(s);
    size_t o = 256;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = align_up(o + bytes, 256);
        return at;
    };
    const bool tc_gate = gate_tc_supported(s);
    L.scores = take(tc_gate ? 0 : static_cast<size_t>(s.T) * C * 4);
    L.gpack = take(tc_gate ? gate_tc_pack_bytes(s) : 0);
    L.gsel = take(tc_gate && s.groups > 0 ? static_cast<size_t>(s.T) * s.k_groups * 8 : 0);
    L.local_rank = take(S * 4);
    L.chunk = take(chunks * n * 4);
    L.chunk_imp = take(chunks * n * 4);
    L.imp_acc = take(n * 4);
    L.counts = take(n * 4);
    L.offsets = take((n + 1) * 4);
    L.perm = take(S * 4);
    L.inv_perm = take(S * 4);
    L.importance = take(n * 4);
    L.cv2 = take(4);
    L.tiles = take((n + 1) * 4);
    L.ptiles = take((n + 1) * 4);
    L.plist = take(pair_tile_capacity(static_cast<int64_t>(S), s.n) * 16);
    L.xperm = take(S * static_cast<size_t>(s.d) * eb);
    L.hidden = take(S * static_cast<size_t>(s.h) * eb);
    L.yslot = take(S * static_cast<size_t>(s.d) * eb);
    L.total = o;
    return L;
}

template <typename T>
inline T *ws_ptr(void *ws, size_t off) {
    return reinterpret_cast<T *>(static_cast<char *>(ws) + off);
}

// Stage launchers (each returns the launch error, if any).
cudaError_t launch_gate(const moe_shape &s, const void *x, const float *Wg, const float *Wn,
                        const float *bg, const float *eps, int32_t *idx, float *G, void *ws,
                        const WsLayout &L, cudaStream_t st);
// Tensor-core gate.  Hierarchical shapes also use the workspace's routing,
// row-tile and gathered-row regions (free until the dispatch that follows).
cudaError_t launch_gate_tc(const moe_shape &s, const void *x, const float *Wg, const float *Wn,
                           const float *bg, const float *eps, int32_t *idx, float *G, void *ws,
                           const WsLayout &L, cudaStream_t st);

// Extra outputs the forward pass takes from its dispatch: the x rows in
// expert order (bf16) and the schedules of the expert stage's GEMMs, built in
// the same launches instead of launches of their own.
struct DispatchExtras {
    const __nv_bfloat16 *x = nullptr;   // gather x[perm[r] / k] into xperm[r] when set
    __nv_bfloat16 *xperm = nullptr;
    int32_t *rtiles = nullptr;          // row-tile starts for bm-row tiles (when set)
    int bm = 0;
    int32_t *ptiles = nullptr;          // pair token-tile starts and table (when set)
    int4 *plist = nullptr;
    int pcap = 256;                     // rows per pair token tile at most (256 or 128)
};

cudaError_t launch_dispatch(const moe_shape &s, const int32_t *idx, const float *G,
                            int32_t *counts, int32_t *offsets, int32_t *perm, int32_t *inv_perm,
                            float *importance, float *cv2, void *ws, const WsLayout &L,
                            cudaStream_t st, const DispatchExtras *ex = nullptr);

// prepared: the dispatch already built the stage's schedules and (bf16) the x
// rows in expert order (dispatch_extras_for_ffn), so they are not rebuilt.
// keep_hidden: the hidden activations must be left in the workspace's hidden
// region (the backward pass reads them), so the two layers run as separate
// GEMMs even where the fused kernel applies.
cudaError_t launch_expert_ffn(const moe_shape &s, const void *x, const int32_t *perm,
                              const int32_t *offsets, const void *W1, const float *b1,
                              const void *W2, const float *b2, void *Y_slot, void *ws,
                              const WsLayout &L, cudaStream_t st, bool prepared = false,
                              bool keep_hidden = false);

// The DispatchExtras that prepare the expert stage of shape s (ffn.cu).
DispatchExtras dispatch_extras_for_ffn(const moe_shape &s, const void *x, void *ws,
                                       const WsLayout &L);

cudaError_t launch_combine(const moe_shape &s, const void *Y_slot, const int32_t *inv_perm,
                           const float *G, void *y, int32_t *err, cudaStream_t st);

// tiles[e] = sum over e' < e of ceil(rows of e' / bm) for offsets[0..n]; tiles[n] = total.
cudaError_t launch_row_tiles(const int32_t *offsets, int n, int bm, int32_t *tiles,
                             cudaStream_t st);

// out[r] = x[perm[r] / k] (d bf16 values per row) for r < offsets[n].
cudaError_t launch_gather_rows(const __nv_bfloat16 *x, const int32_t *perm, const int32_t *offsets,
                               int n, int64_t S, int d, int k, __nv_bfloat16 *out, int32_t *err,
                               cudaStream_t st);

// Load estimate (load.cu): its own workspace, [T,n] clean scores and noise
// scales, [T,2] k-th / (k+1)-th noisy scores, per-chunk partial sums.
struct LoadLayout {
    size_t c = 0, s = 0, vk = 0, part = 0, load64 = 0, total = 0;
    int chunks = 0;
};
LoadLayout load_layout(const moe_shape &s);

// Tensor-core gate that also writes c, s and the k-th / (k+1)-th scores
// (flat, noisy, bf16, k <= 15).
cudaError_t launch_gate_tc_load(const moe_shape &s, const void *x, const float *Wg, const float *Wn,
                                const float *bg, const float *eps, int32_t *idx, float *G,
                                float *c_out, float *s_out, float *vk_out, void *ws,
                                const WsLayout &L, cudaStream_t st);

cudaError_t launch_load(const moe_shape &s, const int32_t *idx, void *lws, const LoadLayout &L,
                        float *load, float *cv2, cudaStream_t st);

// Number of SMs of the current device (cached per device).
int sm_count();

// Pair (cta_group::2) grouped GEMM with the tokens on the MMA's N side
// (ffn_pair.cu): whether an output width suits it, its token-tile table
// (tiles[e] = token tiles of the experts before e, tiles[n] = total) and the
// GEMM  out[r, c] = act(X[r] . W[e*Nout + c] + bias[e*Nout + c]).
// tlist: one int4 per token tile {expert, first row, rows, rows rounded up to
// 32}, at most pair_tile_capacity(S, n) entries.
bool pair_gemm_supported(int Nout);
cudaError_t launch_pair_tiles(const int32_t *offsets, int n, int32_t *tiles, int4 *tlist,
                              cudaStream_t st, int cap = 256);
cudaError_t launch_grouped_gemm_pair(const moe_shape &s, const __nv_bfloat16 *X, int K,
                                     const __nv_bfloat16 *W, int Nout, const float *bias, int relu,
                                     const int32_t *tiles, const int4 *tlist,
                                     __nv_bfloat16 *out, int32_t *err, cudaStream_t st);

// Both layers of the expert networks in one kernel on SM pairs, the hidden
// activations kept on chip (ffn_fused.cu): bf16, d = 256 or 512, h % 256 == 0,
// at most 128 rows per expert on average (S <= 128 n).  Its token tiles hold
// at most 128 rows (launch_pair_tiles with cap 128).
bool fused_ffn_supported(const moe_shape &s);
cudaError_t launch_ffn_fused(const moe_shape &s, const __nv_bfloat16 *X, const __nv_bfloat16 *W1,
                             const float *b1, const __nv_bfloat16 *W2, const float *b2,
                             const int32_t *tiles, const int4 *tlist, __nv_bfloat16 *Y,
                             int32_t *err, cudaStream_t st);

// Tensor map of a bf16 matrix [rows, K] (K contiguous, K % 64 == 0) seen as a
// 3-D tensor {64, rows, K/64}: a box of box_rows rows and box_kblocks 64-wide
// k-blocks lands as that many 128-byte-swizzled K-major tiles back to back;
// rows or k-blocks past the end read as zeros.
bool make_kmajor_map(CUtensorMap *m, const void *base, uint64_t K, uint64_t rows,
                     uint32_t box_rows, uint32_t box_kblocks = 1);

// Tensor map of a bf16 matrix [rows, M] (M contiguous, M % 64 == 0) read as
// MN-major operand tiles: a 3-D tensor {64, rows, M/64}; a box of box_rows
// rows and box_mblocks 64-wide column blocks lands as that many
// 128-byte-swizzled [box_rows][64] tiles back to back.
bool make_mnmajor_map(CUtensorMap *m, const void *base, uint64_t M, uint64_t rows,
                      uint32_t box_rows, uint32_t box_mblocks);

// The pair GEMM out[r, c] = X[r, :] . W[e*K + k, c] summed over k < K: the
// weights read in their stored layout [n*K, Nout] (MN-major operand) instead
// of transposed, e.g. dA = dE . W2 with W2 [n*d, h].  Nout % 256 == 0.
cudaError_t launch_grouped_gemm_pair_wmn(const moe_shape &s, const __nv_bfloat16 *X, int K,
                                         const __nv_bfloat16 *W, int Nout, const int32_t *tiles,
                                         const int4 *tlist, __nv_bfloat16 *out, int32_t *err,
                                         cudaStream_t st);

}  // namespace moe

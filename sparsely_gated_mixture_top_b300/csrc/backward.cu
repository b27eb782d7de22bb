// backward.cu -- the backward pass of the layer (moe_backward in moe.h), flat
// or hierarchical gating.
//
// The pages train the layer: noise in the gate during training
// ("MoE:稀疏门控混合专家", section 四) and an importance loss beside the task
// loss ("Outrageously Large Neural Networks — MoE 怎样让模型“很大但不每次全算”",
// section 方法怎么做).  With the selection of the forward pass held fixed
// (KeepTopK is piecewise constant), the gradients of
//     L = sum_t <dy_t, y_t> + w_imp * CV^2(importance)
// are the chain rule through the combine, the experts, the softmax over the
// kept scores, the noise scale and the importance sum:
//   z = W1[e] x + b1[e], a = ReLU(z), E = W2[e] a + b2[e]      (per slot, recomputed)
//   dG_j  = <dy_t, E_j> + w_imp dCV^2/dimp_e
//   dH_j  = G_j (dG_j - sum_l G_l dG_l)
//   dc_j  = dH_j,  dr_j = dH_j eps[t,e] sigmoid(x_t . Wn[:,e])
//   dE    = G_j dy_t,  dz = (W2[e]^T dE) * [z > 0]
//   dx_t  = sum_j dc_j Wg[:,e_j] + dr_j Wn[:,e_j] + W1[e_j]^T dz_j
//   dWg[:,e] = sum dc x,  dWn[:,e] = sum dr x,  dbg[e] = sum dc
//   dW2[e] = sum dE a^T,  db2[e] = sum dE,  dW1[e] = sum dz x^T,  db1[e] = sum dz
// For the hierarchical gate ("MoE:稀疏门控混合专家", section 三) the slot weight
// is G = Gp_q Gi_qj and dG passes through both softmax levels to the kept
// group columns and expert columns (bwd_token_hier, below); the expert
// columns sit after the G group columns of Wg, Wn and bg.
//
// bf16 shapes whose widths are multiples of 128 run the contractions on the
// tensor cores (launch_backward_tc below: bf16 operands, fp32 accumulation,
// bf16 intermediates); other shapes run everything in fp32 on the CUDA cores
// (inputs of either dtype are read exactly).  Every sum has a fixed order, so
// results are bit-reproducible either way.  CUDA-core stages, in launch order:
//   dispatch of idx (counts, offsets, perm, inv_perm) and a 64-row tile table
//   bwd_row_gemm  Z = X W1^T + b1 (pre-activation, kept), E = ReLU(Z) W2^T + b2,
//                 dZ = (dE W2) * [Z > 0] with dE rows = G dy rows, dXs = dZ W1
//   bwd_transpose Wg^T, Wn^T;  bwd_gimp  w_imp dCV^2/dimp
//   bwd_token     dG, dH, dc, dr and dx (one warp per token)
//   bwd_gate_part/_fin  dWg, dWn, dbg;  bwd_colsum_part/_fin  db2, db1 (row sums in
//                 256-row chunks, then the chunks of each expert in order)
//   bwd_wgrad     dW2, dW1 (per expert, summed over its rows)
#include "backward_tc.h"
#include "moe_device.cuh"
#include "moe_launch.h"

namespace moe {

// The forward's grouped tensor-core GEMM (ffn_tc.cu): out[r, c] = act(sum_k
// A[r, k] B[e*N + c, k] + bias[e, c]) for the 128-row tiles of each expert, bf16 out.
cudaError_t launch_grouped_gemm_tc(const moe_shape &s, const __nv_bfloat16 *A, int K,
                                   const __nv_bfloat16 *B, int N, const float *bias, int relu,
                                   const int32_t *offsets, const int32_t *tiles,
                                   __nv_bfloat16 *out, int32_t *err, cudaStream_t st);

namespace {

constexpr int32_t kSiteBwdPerm = 20;
constexpr int kBT = 64;  // rows and columns of a SIMT tile
constexpr int kBK = 16;  // k per shared-memory step

// Hierarchical gating: the (token, kept group) pairs routed by group, for
// the gradients of the group columns.
struct PairLayout {
    size_t gidx = 0, gw = 0, counts = 0, offsets = 0, perm = 0, inv = 0, imp = 0, cv2 = 0;
    size_t local_rank = 0, chunk = 0, chunk_imp = 0, imp_acc = 0, dcg = 0, drg = 0, ctiles = 0;
};

template <class Take>
PairLayout take_pairs(const moe_shape &s, Take &&take) {
    PairLayout P;
    if (s.groups == 0) return P;
    const size_t np = static_cast<size_t>(s.T) * s.k_groups, Gn = static_cast<size_t>(s.groups);
    const size_t chunks = (np + kRouteChunk - 1) / kRouteChunk;
    P.gidx = take(np * 4);
    P.gw = take(np * 4);
    P.counts = take(Gn * 4);
    P.offsets = take((Gn + 1) * 4);
    P.perm = take(np * 4);
    P.inv = take(np * 4);
    P.imp = take(Gn * 4);
    P.cv2 = take(4);
    P.local_rank = take(np * 4);
    P.chunk = take(chunks * Gn * 4);
    P.chunk_imp = take(chunks * Gn * 4);
    P.imp_acc = take(Gn * 4);
    P.dcg = take(np * 4);
    P.drg = take(np * 4);
    P.ctiles = take((Gn + 1) * 4);
    return P;
}

struct BwdLayout {
    PairLayout pairs;
    size_t local_rank = 0, chunk = 0, chunk_imp = 0, imp_acc = 0;
    size_t counts = 0, offsets = 0, perm = 0, inv_perm = 0, imp = 0, cv2 = 0, tiles = 0;
    size_t WgT = 0, WnT = 0, gimp = 0, dc = 0, dr = 0;
    size_t Z = 0, dZ = 0, E = 0, dXs = 0;
    size_t ctiles = 0, pg = 0, pn = 0, pb = 0, pc = 0;  // chunked row sums
    size_t total = 0;
};

// Rows are summed in chunks of this many rows of one expert (see row_sums).
constexpr int kRowChunk = 256;
inline size_t row_chunks(const moe_shape &s) {
    return static_cast<size_t>((slots(s) + kRowChunk - 1) / kRowChunk + s.n);
}

BwdLayout bwd_layout(const moe_shape &s) {
    BwdLayout L;
    const size_t S = static_cast<size_t>(slots(s));
    const size_t n = static_cast<size_t>(s.n), d = static_cast<size_t>(s.d),
                 h = static_cast<size_t>(s.h);
    const size_t chunks = (S + kRouteChunk - 1) / kRouteChunk;
    size_t o = kWsHeaderBytes;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = align_up(o + bytes, 256);
        return at;
    };
    L.local_rank = take(S * 4);
    L.chunk = take(chunks * n * 4);
    L.chunk_imp = take(chunks * n * 4);
    L.imp_acc = take(n * 4);
    L.counts = take(n * 4);
    L.offsets = take((n + 1) * 4);
    L.perm = take(S * 4);
    L.inv_perm = take(S * 4);
    L.imp = take(n * 4);
    L.cv2 = take(4);
    L.tiles = take((n + 1) * 4);
    const size_t Cg = static_cast<size_t>(gate_cols(s));
    L.WgT = take(Cg * d * 4);
    L.WnT = take(Cg * d * 4);
    L.gimp = take(n * 4);
    L.dc = take(S * 4);
    L.dr = take(S * 4);
    L.pairs = take_pairs(s, take);
    L.Z = take(S * h * 4);
    L.dZ = take(S * h * 4);
    L.E = take(S * d * 4);
    L.dXs = take(S * d * 4);
    const size_t C = row_chunks(s);
    L.ctiles = take((n + 1) * 4);
    L.pg = take(C * d * 4);
    L.pn = take(C * d * 4);
    L.pb = take(C * 4);
    L.pc = take(C * (d > h ? d : h) * 4);
    L.total = o;
    return L;
}

__device__ __forceinline__ float ldf(const void *p, int64_t i, int bf16) {
    return bf16 ? __bfloat162float(static_cast<const __nv_bfloat16 *>(p)[i])
                : static_cast<const float *>(p)[i];
}

__device__ __forceinline__ int expert_of_tile(const int32_t *__restrict__ tiles, int n, int rt) {
    int lo = 0, hi = n - 1;  // largest e with tiles[e] <= rt
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tiles[mid] <= rt)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

// Row-side operand: value (r, c) = scale * act(P[row(r), c]) where row(r) =
// perm[r] / kdiv when perm is given (else r) and scale = sc[perm[r]] when sc
// is given (else 1); act = ReLU when relu.
struct RowOp {
    const void *p;
    int bf16;
    int64_t ld;
    const int32_t *perm;
    int kdiv;
    const float *sc;
    int relu;
};

// out[r, c] = epi( sum_k A(r, k) B_e(k, c) ) for the rows r of expert e, with
// B_e(k, c) = B[e*bse + k*bsk + c*bsc], epi = + bias[e*N + c], then * [mask[r, c] > 0].
struct RowGemm {
    RowOp a;
    const void *B;
    int b_bf16;
    int64_t bse, bsk, bsc;
    const float *bias;
    const float *mask;
    float *out;
    int K, N;
    const int32_t *offsets, *tiles;
    int n;
    int64_t S;
    int32_t *err;
};

__global__ void __launch_bounds__(256) bwd_row_gemm(const RowGemm g) {
    __shared__ float As[kBK][kBT + 4];
    __shared__ float Bs[kBK][kBT + 4];
    __shared__ int64_t arow[kBT];
    __shared__ float ascale[kBT];
    const int rt = blockIdx.x;
    if (rt >= g.tiles[g.n]) return;
    const int e = expert_of_tile(g.tiles, g.n, rt);
    const int row0 = g.offsets[e] + (rt - g.tiles[e]) * kBT;
    const int rows = min(kBT, g.offsets[e + 1] - row0);
    const int c0 = blockIdx.y * kBT;
    const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
    if (tid < kBT) {
        int64_t ar = -1;
        float sc = 1.0f;
        if (tid < rows) {
            const int64_t r = row0 + tid;
            if (g.a.perm) {
                const int32_t s = g.a.perm[r];
                if (s < 0 || s >= g.S) {
                    report(g.err, MOE_ERR_DEVICE, kSiteBwdPerm, static_cast<int32_t>(r));
                } else {
                    ar = s / g.a.kdiv;
                    if (g.a.sc) sc = g.a.sc[s];
                }
            } else {
                ar = r;
            }
        }
        arow[tid] = ar;
        ascale[tid] = sc;
    }
    __syncthreads();
    const int64_t bbase = static_cast<int64_t>(e) * g.bse;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < g.K; k0 += kBK) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int idx = tid + q * 256;
            {
                const int r = idx / kBK, kk = idx % kBK;
                const int64_t ar = arow[r];
                float v = 0.0f;
                if (ar >= 0) {
                    v = ldf(g.a.p, ar * g.a.ld + k0 + kk, g.a.bf16);
                    if (g.a.relu) v = fmaxf(v, 0.0f);
                    v *= ascale[r];
                }
                As[kk][r] = v;
            }
            {
                // consecutive threads walk the contiguous dimension of B
                int kk, c;
                if (g.bsc == 1) {
                    kk = idx / kBT;
                    c = idx % kBT;
                } else {
                    kk = idx % kBK;
                    c = idx / kBK;
                }
                Bs[kk][c] = ldf(g.B, bbase + (k0 + kk) * g.bsk + (c0 + c) * g.bsc, g.b_bf16);
            }
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < kBK; ++kk) {
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
        const int64_t orow = static_cast<int64_t>(row0 + r) * g.N;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int c = c0 + tx * 4 + j;
            float v = acc[i][j];
            if (g.bias) v += g.bias[static_cast<int64_t>(e) * g.N + c];
            if (g.mask && !(g.mask[orow + c] > 0.0f)) v = 0.0f;
            g.out[orow + c] = v;
        }
    }
}

// out[e][i, j] = sum over the rows r of expert e, in order, of P(r, i) Q(r, j).
__global__ void __launch_bounds__(256) bwd_wgrad(RowOp P, RowOp Q, int M, int N,
                                                 const int32_t *__restrict__ offsets, int64_t S,
                                                 float *__restrict__ out, int32_t *err) {
    __shared__ float Ps[kBK][kBT + 4];
    __shared__ float Qs[kBK][kBT + 4];
    __shared__ int64_t prow[kBK], qrow[kBK];
    __shared__ float psc[kBK], qsc[kBK];
    const int e = blockIdx.z;
    const int i0 = blockIdx.y * kBT, j0 = blockIdx.x * kBT;
    const int r_begin = offsets[e], r_end = offsets[e + 1];
    const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
    float acc[4][4] = {};
    for (int rb = r_begin; rb < r_end; rb += kBK) {
        if (tid < 2 * kBK) {
            const bool isq = tid >= kBK;
            const RowOp op = isq ? Q : P;
            const int rr = tid % kBK;
            const int64_t r = rb + rr;
            int64_t row = -1;
            float sc = 1.0f;
            if (r < r_end) {
                if (op.perm) {
                    const int32_t s = op.perm[r];
                    if (s < 0 || s >= S) {
                        report(err, MOE_ERR_DEVICE, kSiteBwdPerm, static_cast<int32_t>(r));
                    } else {
                        row = s / op.kdiv;
                        if (op.sc) sc = op.sc[s];
                    }
                } else {
                    row = r;
                }
            }
            if (isq) {
                qrow[rr] = row;
                qsc[rr] = sc;
            } else {
                prow[rr] = row;
                psc[rr] = sc;
            }
        }
        __syncthreads();
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int idx = tid + q * 256;
            const int rr = idx / kBT, c = idx % kBT;
            float pv = 0.0f, qv = 0.0f;
            if (prow[rr] >= 0) {
                pv = ldf(P.p, prow[rr] * P.ld + i0 + c, P.bf16);
                if (P.relu) pv = fmaxf(pv, 0.0f);
                pv *= psc[rr];
            }
            if (qrow[rr] >= 0) {
                qv = ldf(Q.p, qrow[rr] * Q.ld + j0 + c, Q.bf16);
                if (Q.relu) qv = fmaxf(qv, 0.0f);
                qv *= qsc[rr];
            }
            Ps[rr][c] = pv;
            Qs[rr][c] = qv;
        }
        __syncthreads();
#pragma unroll
        for (int rr = 0; rr < kBK; ++rr) {
            float pv[4], qv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                pv[i] = Ps[rr][ty * 4 + i];
                qv[i] = Qs[rr][tx * 4 + i];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(pv[i], qv[j], acc[i][j]);
        }
        __syncthreads();
    }
    float *oe = out + static_cast<int64_t>(e) * M * N;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
            oe[static_cast<int64_t>(i0 + ty * 4 + i) * N + j0 + tx * 4 + j] = acc[i][j];
}

// Sums over an expert's rows run in two passes so that an expert holding most
// of the rows does not serialise on one block: chunks of kChunkRows rows of one
// expert (chunk table ctiles, built like a row-tile table) are summed by
// separate blocks, then each expert adds its chunks' partial sums in order.
constexpr int kChunkRows = kRowChunk;

__device__ __forceinline__ bool chunk_rows(const int32_t *__restrict__ ctiles,
                                           const int32_t *__restrict__ offsets, int n, int c,
                                           int *r0, int *r1) {
    if (c >= ctiles[n]) return false;
    const int e = expert_of_tile(ctiles, n, c);
    *r0 = offsets[e] + (c - ctiles[e]) * kChunkRows;
    *r1 = min(*r0 + kChunkRows, offsets[e + 1]);
    return true;
}

// part[c, col] = sum over the rows r of chunk c, in order, of P(r, col).  The
// rows' source rows and scales are staged in shared memory first, so the
// column loop issues only independent loads.
__global__ void __launch_bounds__(256) bwd_colsum_part(RowOp P, int M,
                                                       const int32_t *__restrict__ offsets,
                                                       const int32_t *__restrict__ ctiles, int n,
                                                       int64_t S, float *__restrict__ part,
                                                       int32_t *err) {
    __shared__ int64_t srow[kChunkRows];
    __shared__ float ssc[kChunkRows];
    int r0, r1;
    if (!chunk_rows(ctiles, offsets, n, blockIdx.x, &r0, &r1)) return;
    const int cnt = r1 - r0;
    if (threadIdx.x < cnt) {
        const int r = r0 + threadIdx.x;
        int64_t row = r;
        float sc = 1.0f;
        if (P.perm) {
            const int32_t sl = P.perm[r];
            if (sl < 0 || sl >= S) {
                report(err, MOE_ERR_DEVICE, kSiteBwdPerm, r);
                row = -1;
            } else {
                row = sl / P.kdiv;
                if (P.sc) sc = P.sc[sl];
            }
        }
        srow[threadIdx.x] = row;
        ssc[threadIdx.x] = sc;
    }
    __syncthreads();
    const int col = blockIdx.y * 256 + threadIdx.x;
    if (col >= M) return;
    float acc = 0.0f;
#pragma unroll 8
    for (int i = 0; i < cnt; ++i) {
        const int64_t row = srow[i];
        if (row < 0) continue;
        float v = ldf(P.p, row * P.ld + col, P.bf16);
        if (P.relu) v = fmaxf(v, 0.0f);
        acc = fmaf(v, ssc[i], acc);
    }
    part[static_cast<int64_t>(blockIdx.x) * M + col] = acc;
}

// out[e, col] = sum over e's chunks, in order, of part[c, col] (0 for no rows).
__global__ void __launch_bounds__(256) bwd_colsum_fin(const float *__restrict__ part, int M,
                                                      const int32_t *__restrict__ ctiles,
                                                      float *__restrict__ out) {
    const int e = blockIdx.y;
    const int col = blockIdx.x * 256 + threadIdx.x;
    if (col >= M) return;
    float acc = 0.0f;
    for (int c = ctiles[e]; c < ctiles[e + 1]; ++c) acc += part[static_cast<int64_t>(c) * M + col];
    out[static_cast<int64_t>(e) * M + col] = acc;
}

// WT[i, j] = W[j, i] for W [rows, cols] fp32.
__global__ void bwd_transpose(const float *__restrict__ W, int rows, int cols, float *__restrict__ WT) {
    __shared__ float t[32][33];
    const int c = blockIdx.x * 32 + threadIdx.x;
    for (int i = threadIdx.y; i < 32; i += 8) {
        const int r = blockIdx.y * 32 + i;
        if (r < rows && c < cols) t[i][threadIdx.x] = W[static_cast<int64_t>(r) * cols + c];
    }
    __syncthreads();
    const int r2 = blockIdx.y * 32 + threadIdx.x;
    for (int i = threadIdx.y; i < 32; i += 8) {
        const int c2 = blockIdx.x * 32 + i;
        if (c2 < cols && r2 < rows) WT[static_cast<int64_t>(c2) * rows + r2] = t[threadIdx.x][i];
    }
}

// gimp[e] = w_imp * dCV^2/dimp_e with CV^2 = population variance / mean^2 of
// the n importances (0 where the mean is 0); the sums in fp64, fixed order.
__global__ void __launch_bounds__(256) bwd_gimp(const float *__restrict__ imp, int n, float w_imp,
                                                float *__restrict__ gimp) {
    __shared__ double part[256];
    __shared__ double mu_s, var_s;
    double acc = 0.0;
    for (int e = threadIdx.x; e < n; e += 256) acc += imp ? static_cast<double>(imp[e]) : 0.0;
    part[threadIdx.x] = acc;
    __syncthreads();
    for (int o = 128; o > 0; o >>= 1) {
        if (threadIdx.x < o) part[threadIdx.x] += part[threadIdx.x + o];
        __syncthreads();
    }
    if (threadIdx.x == 0) mu_s = part[0] / n;
    __syncthreads();
    const double mu = mu_s;
    acc = 0.0;
    for (int e = threadIdx.x; e < n; e += 256) {
        const double dv = (imp ? static_cast<double>(imp[e]) : 0.0) - mu;
        acc += dv * dv;
    }
    part[threadIdx.x] = acc;
    __syncthreads();
    for (int o = 128; o > 0; o >>= 1) {
        if (threadIdx.x < o) part[threadIdx.x] += part[threadIdx.x + o];
        __syncthreads();
    }
    if (threadIdx.x == 0) var_s = part[0] / n;
    __syncthreads();
    const double var = var_s;
    for (int e = threadIdx.x; e < n; e += 256) {
        double g = 0.0;
        if (mu != 0.0 && w_imp != 0.0)
            g = w_imp * (2.0 * ((imp ? static_cast<double>(imp[e]) : 0.0) - mu) / (n * mu * mu) -
                         2.0 * var / (n * mu * mu * mu));
        gimp[e] = static_cast<float>(g);
    }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// One warp per token: dG, dH, dc, dr of its k slots and the whole of dx_t.
// One pass over the columns forms <dy_t, E_j> and <x_t, Wn[:, e_j]> for all
// k slots (KM >= k accumulators per lane), then 2k warp reductions.
template <int KM>
__global__ void __launch_bounds__(256) bwd_token(
    int64_t T, int d, int n, int k, const void *__restrict__ x, const void *__restrict__ dy,
    int bf16, const void *__restrict__ E, const void *__restrict__ dXs, int ebf16,
    const int32_t *__restrict__ inv_perm, const int32_t *__restrict__ idx,
    const float *__restrict__ G, const float *__restrict__ gimp, const float *__restrict__ WgT,
    const float *__restrict__ WnT, const float *__restrict__ eps, float *__restrict__ dc,
    float *__restrict__ dr, float *__restrict__ dx, int32_t *err) {
    const int lane = threadIdx.x & 31;
    const int64_t t = static_cast<int64_t>(blockIdx.x) * 8 + threadIdx.x / 32;
    if (t >= T) return;
    const int64_t S = T * k;
    int ex[KM], row[KM];
    float aE[KM], aR[KM];
#pragma unroll
    for (int j = 0; j < KM; ++j) {
        ex[j] = 0;
        row[j] = -1;
        aE[j] = 0.0f;
        aR[j] = 0.0f;
        if (j >= k) continue;
        const int64_t s = t * k + j;
        const int e = idx[s];
        const int r = inv_perm[s];
        if (e < 0 || e >= n || r < 0 || r >= S) {
            if (lane == 0) report(err, MOE_ERR_DEVICE, kSiteBwdPerm, static_cast<int32_t>(s));
            continue;
        }
        ex[j] = e;
        row[j] = r;
    }
#pragma unroll 4
    for (int c = lane; c < d; c += 32) {
        const float dv = ldf(dy, t * d + c, bf16);
        const float xv = eps ? ldf(x, t * d + c, bf16) : 0.0f;
#pragma unroll
        for (int j = 0; j < KM; ++j) {
            if (j >= k) break;
            if (row[j] >= 0) aE[j] = fmaf(dv, ldf(E, static_cast<int64_t>(row[j]) * d + c, ebf16), aE[j]);
            if (eps) aR[j] = fmaf(xv, WnT[static_cast<int64_t>(ex[j]) * d + c], aR[j]);
        }
    }
    float dG[KM], dH[KM], drv[KM];
    float sGdG = 0.0f;
#pragma unroll
    for (int j = 0; j < KM; ++j) {
        if (j >= k) break;
        dG[j] = warp_sum(aE[j]) + gimp[ex[j]];
        sGdG = fmaf(G[t * k + j], dG[j], sGdG);
    }
#pragma unroll
    for (int j = 0; j < KM; ++j) {
        if (j >= k) break;
        const int64_t s = t * k + j;
        dH[j] = G[s] * (dG[j] - sGdG);
        float dv = 0.0f;
        if (eps) {
            const float r = warp_sum(aR[j]);
            dv = dH[j] * eps[t * n + ex[j]] / (1.0f + __expf(-r));
        }
        drv[j] = dv;
        if (lane == 0) {
            dc[s] = dH[j];
            dr[s] = dv;
        }
    }
#pragma unroll 4
    for (int c = lane; c < d; c += 32) {
        float acc = 0.0f;
#pragma unroll
        for (int j = 0; j < KM; ++j) {
            if (j >= k) break;
            const int64_t we = static_cast<int64_t>(ex[j]) * d + c;
            acc = fmaf(dH[j], WgT[we], acc);
            if (eps) acc = fmaf(drv[j], WnT[we], acc);
            if (row[j] >= 0) acc += ldf(dXs, static_cast<int64_t>(row[j]) * d + c, ebf16);
        }
        dx[t * d + c] = acc;
    }
}

// The token kernel for bf16 x, dy, E and dX rows with d a multiple of 256:
// each lane takes 8 consecutive columns per step (16-byte loads of bf16 rows,
// 32-byte loads of the fp32 gate columns, two 16-byte stores of dx).
__device__ __forceinline__ void bf16x8(const __nv_bfloat16 *p, float (&f)[8]) {
    const uint4 v = *reinterpret_cast<const uint4 *>(p);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(&w[i]);
        f[2 * i] = __low2float(b);
        f[2 * i + 1] = __high2float(b);
    }
}

__device__ __forceinline__ void f32x8(const float *p, float (&f)[8]) {
    const float4 a = reinterpret_cast<const float4 *>(p)[0], b = reinterpret_cast<const float4 *>(p)[1];
    f[0] = a.x, f[1] = a.y, f[2] = a.z, f[3] = a.w, f[4] = b.x, f[5] = b.y, f[6] = b.z, f[7] = b.w;
}

template <int KM>
__global__ void __launch_bounds__(256) bwd_token_v8(
    int64_t T, int d, int n, int k, const __nv_bfloat16 *__restrict__ x,
    const __nv_bfloat16 *__restrict__ dy, const __nv_bfloat16 *__restrict__ E,
    const __nv_bfloat16 *__restrict__ dXs, const int32_t *__restrict__ inv_perm,
    const int32_t *__restrict__ idx, const float *__restrict__ G, const float *__restrict__ gimp,
    const float *__restrict__ WgT, const float *__restrict__ WnT, const float *__restrict__ eps,
    float *__restrict__ dc, float *__restrict__ dr, float *__restrict__ dx, int32_t *err) {
    const int lane = threadIdx.x & 31;
    const int64_t t = static_cast<int64_t>(blockIdx.x) * 8 + threadIdx.x / 32;
    if (t >= T) return;
    const int64_t S = T * k;
    int ex[KM], row[KM];
    float aE[KM], aR[KM];
#pragma unroll
    for (int j = 0; j < KM; ++j) {
        ex[j] = 0;
        row[j] = -1;
        aE[j] = 0.0f;
        aR[j] = 0.0f;
        if (j >= k) continue;
        const int64_t s = t * k + j;
        const int e = idx[s];
        const int r = inv_perm[s];
        if (e < 0 || e >= n || r < 0 || r >= S) {
            if (lane == 0) report(err, MOE_ERR_DEVICE, kSiteBwdPerm, static_cast<int32_t>(s));
            continue;
        }
        ex[j] = e;
        row[j] = r;
    }
    for (int c0 = lane * 8; c0 < d; c0 += 256) {
        float dv[8], xv[8];
        bf16x8(dy + t * d + c0, dv);
        if (eps) bf16x8(x + t * d + c0, xv);
#pragma unroll
        for (int j = 0; j < KM; ++j) {
            if (j >= k) break;
            if (row[j] >= 0) {
                float ev[8];
                bf16x8(E + static_cast<int64_t>(row[j]) * d + c0, ev);
#pragma unroll
                for (int i = 0; i < 8; ++i) aE[j] = fmaf(dv[i], ev[i], aE[j]);
            }
            if (eps) {
                float wv[8];
                f32x8(WnT + static_cast<int64_t>(ex[j]) * d + c0, wv);
#pragma unroll
                for (int i = 0; i < 8; ++i) aR[j] = fmaf(xv[i], wv[i], aR[j]);
            }
        }
    }
    float dG[KM], dH[KM], drv[KM];
    float sGdG = 0.0f;
#pragma unroll
    for (int j = 0; j < KM; ++j) {
        if (j >= k) break;
        dG[j] = warp_sum(aE[j]) + gimp[ex[j]];
        sGdG = fmaf(G[t * k + j], dG[j], sGdG);
    }
#pragma unroll
    for (int j = 0; j < KM; ++j) {
        if (j >= k) break;
        const int64_t s = t * k + j;
        dH[j] = G[s] * (dG[j] - sGdG);
        float dv = 0.0f;
        if (eps) {
            const float r = warp_sum(aR[j]);
            dv = dH[j] * eps[t * n + ex[j]] / (1.0f + __expf(-r));
        }
        drv[j] = dv;
        if (lane == 0) {
            dc[s] = dH[j];
            dr[s] = dv;
        }
    }
    for (int c0 = lane * 8; c0 < d; c0 += 256) {
        float acc[8] = {};
#pragma unroll
        for (int j = 0; j < KM; ++j) {
            if (j >= k) break;
            float wg[8];
            f32x8(WgT + static_cast<int64_t>(ex[j]) * d + c0, wg);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = fmaf(dH[j], wg[i], acc[i]);
            if (eps) {
                float wn[8];
                f32x8(WnT + static_cast<int64_t>(ex[j]) * d + c0, wn);
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] = fmaf(drv[j], wn[i], acc[i]);
            }
            if (row[j] >= 0) {
                float xr[8];
                bf16x8(dXs + static_cast<int64_t>(row[j]) * d + c0, xr);
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] += xr[i];
            }
        }
        float4 *o = reinterpret_cast<float4 *>(dx + t * d + c0);
        o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
}

// Launches the token kernel with 4 accumulators per lane when k <= 4.
cudaError_t launch_token(int64_t T, int d, int n, int k, const void *x, const void *dy, int bf16,
                         const void *E, const void *dXs, int ebf16, const int32_t *inv,
                         const int32_t *idx, const float *G, const float *gimp, const float *WgT,
                         const float *WnT, const float *eps, float *dc, float *dr, float *dx,
                         int32_t *err, cudaStream_t st) {
    const unsigned grid = static_cast<unsigned>((T + 7) / 8);
    if (bf16 && ebf16 && d % 256 == 0) {
        using bf = __nv_bfloat16;
        const bf *xb = static_cast<const bf *>(x), *dyb = static_cast<const bf *>(dy);
        const bf *Eb = static_cast<const bf *>(E), *Xb = static_cast<const bf *>(dXs);
        if (k <= 4)
            bwd_token_v8<4><<<grid, 256, 0, st>>>(T, d, n, k, xb, dyb, Eb, Xb, inv, idx, G, gimp, WgT,
                                                  WnT, eps, dc, dr, dx, err);
        else
            bwd_token_v8<MOE_MAX_K><<<grid, 256, 0, st>>>(T, d, n, k, xb, dyb, Eb, Xb, inv, idx, G,
                                                          gimp, WgT, WnT, eps, dc, dr, dx, err);
        return cudaGetLastError();
    }
    if (k <= 4)
        bwd_token<4><<<grid, 256, 0, st>>>(T, d, n, k, x, dy, bf16, E, dXs, ebf16, inv, idx, G, gimp,
                                           WgT, WnT, eps, dc, dr, dx, err);
    else
        bwd_token<MOE_MAX_K><<<grid, 256, 0, st>>>(T, d, n, k, x, dy, bf16, E, dXs, ebf16, inv, idx, G,
                                                   gimp, WgT, WnT, eps, dc, dr, dx, err);
    return cudaGetLastError();
}


// Hierarchical gating, one warp per token.  The k slots hold kg kept
// groups of ki experts each, group-major (slot q*ki + j); G = Gp_q Gi_qj with
// Gp the weights of the kept groups and Gi those of the experts inside group
// q.  Score columns: group g at g, expert e at Gn + e (C in all).  From
// dG_s = <dy, E_s> + gimp[e_s]:
//   dGp_q = sum_j dG_qj Gi_qj,  dGi_qj = dG_qj Gp_q
//   dHi_qj = Gi_qj (dGi_qj - sum_l Gi_ql dGi_ql),  dHp_q = Gp_q (dGp_q - sum_l Gp_l dGp_l)
// and every kept column gives dc = dH, dr = dH eps sigmoid(x . Wn[:, col]) and
// its share of dx.  Slot columns go to dc/dr [S], group columns to dcg/drg
// [T*kg].  The slot loops run over compile-time indices (the per-slot
// arrays stay in registers); slot j belongs to group j / ki.
// The two softmax levels of one token (all lanes hold the warp sums):
// from aE (<dy, E_s> partials), aR / aRg (x . Wn partials of the slot and
// group columns) to dH, dr of the slots and dHg, drg of the kept groups;
// lane 0 writes dc, dr, dcg, drg.
template <int KM>
__device__ __forceinline__ void hier_levels(int lane, int64_t t, int k, int kg, int Gn, int n,
                                            const int (&ex)[KM], const int (&grp)[KM],
                                            const float (&aE)[KM], const float (&aR)[KM],
                                            const float (&aRg)[KM], const float *__restrict__ G,
                                            const float *__restrict__ gimp,
                                            const float *__restrict__ eps, float *__restrict__ dc,
                                            float *__restrict__ dr, float *__restrict__ dcg,
                                            float *__restrict__ drg, float (&dH)[KM],
                                            float (&drv)[KM], float (&dHg)[KM],
                                            float (&drgv)[KM]) {
    const int ki = k / kg, C = Gn + n;
    float dG[KM], Gs[KM];
#pragma unroll
    for (int j = 0; j < KM; ++j) {
        dG[j] = 0.0f;
        Gs[j] = 0.0f;
        if (j >= k) continue;
        dG[j] = warp_sum(aE[j]) + gimp[ex[j]];
        Gs[j] = G[t * k + j];
    }
    float Gp[KM], dGp[KM], sI[KM];
#pragma unroll
    for (int q = 0; q < KM; ++q) {
        Gp[q] = 0.0f;
        dGp[q] = 0.0f;
        sI[q] = 0.0f;
#pragma unroll
        for (int j = 0; j < KM; ++j)
            if (j < k && j / ki == q) Gp[q] += Gs[j];
    }
    float Gi[KM];
#pragma unroll
    for (int j = 0; j < KM; ++j) {
        Gi[j] = 0.0f;
        if (j >= k) continue;
#pragma unroll
        for (int q = 0; q < KM; ++q)
            if (j / ki == q) {
                Gi[j] = Gp[q] != 0.0f ? Gs[j] / Gp[q] : 0.0f;
                dGp[q] = fmaf(dG[j], Gi[j], dGp[q]);
                sI[q] = fmaf(Gi[j], dG[j] * Gp[q], sI[q]);   // sum_l Gi_ql dGi_ql
            }
    }
    float sP = 0.0f;
#pragma unroll
    for (int q = 0; q < KM; ++q)
        if (q < kg) sP = fmaf(Gp[q], dGp[q], sP);
#pragma unroll
    for (int j = 0; j < KM; ++j) {
        dH[j] = 0.0f;
        drv[j] = 0.0f;
        if (j >= k) continue;
#pragma unroll
        for (int q = 0; q < KM; ++q)
            if (j / ki == q) dH[j] = Gi[j] * (dG[j] * Gp[q] - sI[q]);
        if (eps) {
            const float r = warp_sum(aR[j]);
            drv[j] = dH[j] * eps[t * C + Gn + ex[j]] / (1.0f + __expf(-r));
        }
        if (lane == 0) {
            dc[t * k + j] = dH[j];
            dr[t * k + j] = drv[j];
        }
    }
#pragma unroll
    for (int q = 0; q < KM; ++q) {
        dHg[q] = 0.0f;
        drgv[q] = 0.0f;
        if (q >= kg) continue;
        dHg[q] = Gp[q] * (dGp[q] - sP);
        if (eps) {
            const float r = warp_sum(aRg[q]);
            drgv[q] = dHg[q] * eps[t * C + grp[q]] / (1.0f + __expf(-r));
        }
        if (lane == 0) {
            dcg[t * kg + q] = dHg[q];
            drg[t * kg + q] = drgv[q];
        }
    }
}

// The slots' experts, expert rows and kept groups of token t (group of kept
// group q: that of its first slot).  Bad entries are reported and skipped.
template <int KM>
__device__ __forceinline__ void hier_slots(int lane, int64_t t, int64_t S, int k, int kg, int n,
                                           int Gn, const int32_t *__restrict__ idx,
                                           const int32_t *__restrict__ inv_perm, int32_t *err,
                                           int (&ex)[KM], int (&row)[KM], int (&grp)[KM]) {
    const int ki = k / kg, m = n / Gn;
#pragma unroll
    for (int j = 0; j < KM; ++j) {
        ex[j] = 0;
        row[j] = -1;
        grp[j] = 0;
    }
#pragma unroll
    for (int j = 0; j < KM; ++j) {
        if (j >= k) continue;
        const int64_t s = t * k + j;
        const int e = idx[s];
        const int r = inv_perm[s];
        if (e < 0 || e >= n || r < 0 || r >= S) {
            if (lane == 0) report(err, MOE_ERR_DEVICE, kSiteBwdPerm, static_cast<int32_t>(s));
            continue;
        }
        ex[j] = e;
        row[j] = r;
    }
#pragma unroll
    for (int q = 0; q < KM; ++q) {
        if (q >= kg) break;
#pragma unroll
        for (int j = 0; j < KM; ++j)
            if (j < k && j == q * ki) grp[q] = ex[j] / m;
    }
}

// Hierarchical gating, one warp per token.  The k slots hold kg kept
// groups of ki experts each, group-major (slot q*ki + j); G = Gp_q Gi_qj with
// Gp the weights of the kept groups and Gi those of the experts inside group
// q.  Score columns: group g at g, expert e at Gn + e (C in all).  From
// dG_s = <dy, E_s> + gimp[e_s]:
//   dGp_q = sum_j dG_qj Gi_qj,  dGi_qj = dG_qj Gp_q
//   dHi_qj = Gi_qj (dGi_qj - sum_l Gi_ql dGi_ql),  dHp_q = Gp_q (dGp_q - sum_l Gp_l dGp_l)
// and every kept column gives dc = dH, dr = dH eps sigmoid(x . Wn[:, col]) and
// its share of dx.  Slot columns go to dc/dr [S], group columns to dcg/drg
// [T*kg].  The slot loops run over compile-time indices (the per-slot
// arrays stay in registers); slot j belongs to group j / ki.  V8: bf16 rows
// with d a multiple of 256, 8 consecutive columns per lane and step (16-byte
// loads of the bf16 rows, 32-byte loads of the fp32 gate columns); else one
// column per lane and step, any dtype.
template <int KM, bool V8>
__global__ void __launch_bounds__(256) bwd_token_hier(
    int64_t T, int d, int n, int k, int Gn, int kg, const void *__restrict__ x,
    const void *__restrict__ dy, int bf16, const void *__restrict__ E,
    const void *__restrict__ dXs, int ebf16, const int32_t *__restrict__ inv_perm,
    const int32_t *__restrict__ idx, const float *__restrict__ G, const float *__restrict__ gimp,
    const float *__restrict__ WgT, const float *__restrict__ WnT, const float *__restrict__ eps,
    float *__restrict__ dc, float *__restrict__ dr, float *__restrict__ dcg,
    float *__restrict__ drg, float *__restrict__ dx, int32_t *err) {
    const int lane = threadIdx.x & 31;
    const int64_t t = static_cast<int64_t>(blockIdx.x) * 8 + threadIdx.x / 32;
    if (t >= T) return;
    int ex[KM], row[KM], grp[KM];
    hier_slots<KM>(lane, t, T * k, k, kg, n, Gn, idx, inv_perm, err, ex, row, grp);
    float aE[KM], aR[KM], aRg[KM];
#pragma unroll
    for (int j = 0; j < KM; ++j) aE[j] = aR[j] = aRg[j] = 0.0f;
    if constexpr (V8) {
        const auto *xb = static_cast<const __nv_bfloat16 *>(x);
        const auto *dyb = static_cast<const __nv_bfloat16 *>(dy);
        const auto *Eb = static_cast<const __nv_bfloat16 *>(E);
        for (int c0 = lane * 8; c0 < d; c0 += 256) {
            float dv[8], xv[8];
            bf16x8(dyb + t * d + c0, dv);
            if (eps) bf16x8(xb + t * d + c0, xv);
#pragma unroll
            for (int j = 0; j < KM; ++j) {
                if (j >= k) break;
                if (row[j] >= 0) {
                    float ev[8];
                    bf16x8(Eb + static_cast<int64_t>(row[j]) * d + c0, ev);
#pragma unroll
                    for (int i = 0; i < 8; ++i) aE[j] = fmaf(dv[i], ev[i], aE[j]);
                }
                if (eps) {
                    float wv[8];
                    f32x8(WnT + static_cast<int64_t>(Gn + ex[j]) * d + c0, wv);
#pragma unroll
                    for (int i = 0; i < 8; ++i) aR[j] = fmaf(xv[i], wv[i], aR[j]);
                }
            }
            if (eps) {
#pragma unroll
                for (int q = 0; q < KM; ++q) {
                    if (q >= kg) break;
                    float wv[8];
                    f32x8(WnT + static_cast<int64_t>(grp[q]) * d + c0, wv);
#pragma unroll
                    for (int i = 0; i < 8; ++i) aRg[q] = fmaf(xv[i], wv[i], aRg[q]);
                }
            }
        }
    } else {
#pragma unroll 4
        for (int c = lane; c < d; c += 32) {
            const float dv = ldf(dy, t * d + c, bf16);
            const float xv = eps ? ldf(x, t * d + c, bf16) : 0.0f;
#pragma unroll
            for (int j = 0; j < KM; ++j) {
                if (j >= k) break;
                if (row[j] >= 0) aE[j] = fmaf(dv, ldf(E, static_cast<int64_t>(row[j]) * d + c, ebf16), aE[j]);
                if (eps) aR[j] = fmaf(xv, WnT[static_cast<int64_t>(Gn + ex[j]) * d + c], aR[j]);
            }
            if (eps) {
#pragma unroll
                for (int q = 0; q < KM; ++q) {
                    if (q >= kg) break;
                    aRg[q] = fmaf(xv, WnT[static_cast<int64_t>(grp[q]) * d + c], aRg[q]);
                }
            }
        }
    }
    float dH[KM], drv[KM], dHg[KM], drgv[KM];
    hier_levels<KM>(lane, t, k, kg, Gn, n, ex, grp, aE, aR, aRg, G, gimp, eps, dc, dr, dcg, drg,
                    dH, drv, dHg, drgv);
    if constexpr (V8) {
        const auto *dXb = static_cast<const __nv_bfloat16 *>(dXs);
        for (int c0 = lane * 8; c0 < d; c0 += 256) {
            float acc[8] = {};
#pragma unroll
            for (int j = 0; j < KM; ++j) {
                if (j >= k) break;
                const int64_t we = static_cast<int64_t>(Gn + ex[j]) * d + c0;
                float wg[8];
                f32x8(WgT + we, wg);
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] = fmaf(dH[j], wg[i], acc[i]);
                if (eps) {
                    float wn[8];
                    f32x8(WnT + we, wn);
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[i] = fmaf(drv[j], wn[i], acc[i]);
                }
                if (row[j] >= 0) {
                    float xr[8];
                    bf16x8(dXb + static_cast<int64_t>(row[j]) * d + c0, xr);
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[i] += xr[i];
                }
            }
#pragma unroll
            for (int q = 0; q < KM; ++q) {
                if (q >= kg) break;
                const int64_t wq = static_cast<int64_t>(grp[q]) * d + c0;
                float wg[8];
                f32x8(WgT + wq, wg);
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] = fmaf(dHg[q], wg[i], acc[i]);
                if (eps) {
                    float wn[8];
                    f32x8(WnT + wq, wn);
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[i] = fmaf(drgv[q], wn[i], acc[i]);
                }
            }
            float4 *o = reinterpret_cast<float4 *>(dx + t * d + c0);
            o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
            o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
        }
    } else {
#pragma unroll 4
        for (int c = lane; c < d; c += 32) {
            float acc = 0.0f;
#pragma unroll
            for (int j = 0; j < KM; ++j) {
                if (j >= k) break;
                const int64_t we = static_cast<int64_t>(Gn + ex[j]) * d + c;
                acc = fmaf(dH[j], WgT[we], acc);
                if (eps) acc = fmaf(drv[j], WnT[we], acc);
                if (row[j] >= 0) acc += ldf(dXs, static_cast<int64_t>(row[j]) * d + c, ebf16);
            }
#pragma unroll
            for (int q = 0; q < KM; ++q) {
                if (q >= kg) break;
                const int64_t wg = static_cast<int64_t>(grp[q]) * d + c;
                acc = fmaf(dHg[q], WgT[wg], acc);
                if (eps) acc = fmaf(drgv[q], WnT[wg], acc);
            }
            dx[t * d + c] = acc;
        }
    }
}

// (token, kept group) pairs of the forward's selection: pair t*kg + q takes
// the group of slot t*k + q*ki and the weight Gp_q (sum of the group's slots).
__global__ void bwd_pairs(const int32_t *__restrict__ idx, const float *__restrict__ G, int64_t T,
                          int k, int kg, int m, int32_t *__restrict__ gidx, float *__restrict__ gw) {
    const int64_t p = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (p >= T * kg) return;
    const int ki = k / kg;
    const int64_t s0 = (p / kg) * k + (p % kg) * ki;
    const int e = idx[s0];
    gidx[p] = e >= 0 ? e / m : -1;
    float w = 0.0f;
    for (int j = 0; j < ki; ++j) w += G[s0 + j];
    gw[p] = w;
}

cudaError_t launch_token_hier(const moe_shape &s, const void *x, const void *dy, int bf16,
                              const void *E, const void *dXs, int ebf16, const int32_t *inv,
                              const int32_t *idx, const float *G, const float *gimp,
                              const float *WgT, const float *WnT, const float *eps, float *dc,
                              float *dr, float *dcg, float *drg, float *dx, int32_t *err,
                              cudaStream_t st) {
    const dim3 grid(static_cast<unsigned>((s.T + 7) / 8));
    const bool v8 = bf16 && ebf16 && s.d % 256 == 0;
#define MOE_TOKEN_HIER(KM, V)                                                                   \
    bwd_token_hier<KM, V><<<grid, 256, 0, st>>>(s.T, s.d, s.n, s.k, s.groups, s.k_groups, x, dy, \
                                                bf16, E, dXs, ebf16, inv, idx, G, gimp, WgT, WnT, \
                                                eps, dc, dr, dcg, drg, dx, err)
    if (s.k <= 4) {
        if (v8)
            MOE_TOKEN_HIER(4, true);
        else
            MOE_TOKEN_HIER(4, false);
    } else {
        if (v8)
            MOE_TOKEN_HIER(MOE_MAX_K, true);
        else
            MOE_TOKEN_HIER(MOE_MAX_K, false);
    }
#undef MOE_TOKEN_HIER
    return cudaGetLastError();
}


// Gate weight gradients, in the same two passes: per chunk c of one expert's
// rows, pg[c, q] = sum of x[t, q] dc[s], pn[c, q] = sum of x[t, q] dr[s] and
// pb[c] = sum of dc[s] (rows in order; one thread per input column q) ...
__global__ void __launch_bounds__(256) bwd_gate_part(
    int d, int k, int64_t S, const void *__restrict__ x, int bf16, const int32_t *__restrict__ perm,
    const int32_t *__restrict__ offsets, const int32_t *__restrict__ ctiles, int n,
    const float *__restrict__ dc, const float *__restrict__ dr, float *__restrict__ pg,
    float *__restrict__ pn, float *__restrict__ pb, int32_t *err) {
    __shared__ int64_t trow[kChunkRows];
    __shared__ float gdc[kChunkRows], gdr[kChunkRows];
    int r0, r1;
    if (!chunk_rows(ctiles, offsets, n, blockIdx.x, &r0, &r1)) return;
    const int cnt = r1 - r0;
    if (threadIdx.x < cnt) {
        const int r = r0 + threadIdx.x;
        const int32_t sl = perm[r];
        if (sl < 0 || sl >= S) {
            if (blockIdx.y == 0) report(err, MOE_ERR_DEVICE, kSiteBwdPerm, r);
            trow[threadIdx.x] = -1;
            gdc[threadIdx.x] = 0.0f;
            gdr[threadIdx.x] = 0.0f;
        } else {
            trow[threadIdx.x] = sl / k;
            gdc[threadIdx.x] = dc[sl];
            gdr[threadIdx.x] = dr[sl];
        }
    }
    __syncthreads();
    const int64_t c = blockIdx.x;
    if (blockIdx.y == 0 && threadIdx.x == 0) {
        float ab = 0.0f;
        for (int i = 0; i < cnt; ++i) ab += gdc[i];
        pb[c] = ab;
    }
    const int q = blockIdx.y * 256 + threadIdx.x;
    if (q >= d) return;
    float ag = 0.0f, an = 0.0f;
#pragma unroll 8
    for (int i = 0; i < cnt; ++i) {
        const int64_t t = trow[i];
        if (t < 0) continue;
        const float xv = ldf(x, t * d + q, bf16);
        ag = fmaf(xv, gdc[i], ag);
        an = fmaf(xv, gdr[i], an);
    }
    pg[c * d + q] = ag;
    pn[c * d + q] = an;
}

// ... then dWg[q, col0 + e], dWn[q, col0 + e], dbg[col0 + e] = the sums over
// e's chunks in order (row stride ldc: the gate's C score columns).
__global__ void __launch_bounds__(256) bwd_gate_fin(int d, int n, int ldc, int col0,
                                                    const int32_t *__restrict__ ctiles,
                                                    const float *__restrict__ pg,
                                                    const float *__restrict__ pn,
                                                    const float *__restrict__ pb,
                                                    float *__restrict__ dWg, float *__restrict__ dWn,
                                                    float *__restrict__ dbg) {
    const int e = blockIdx.y;
    const int q = blockIdx.x * 256 + threadIdx.x;
    const int c0 = ctiles[e], c1 = ctiles[e + 1];
    if (dbg && blockIdx.x == 0 && threadIdx.x == 0) {
        float ab = 0.0f;
        for (int c = c0; c < c1; ++c) ab += pb[c];
        dbg[col0 + e] = ab;
    }
    if (q >= d) return;
    float ag = 0.0f, an = 0.0f;
    for (int c = c0; c < c1; ++c) {
        ag += pg[static_cast<int64_t>(c) * d + q];
        an += pn[static_cast<int64_t>(c) * d + q];
    }
    dWg[static_cast<int64_t>(q) * ldc + col0 + e] = ag;
    if (dWn) dWn[static_cast<int64_t>(q) * ldc + col0 + e] = an;
}

// Chunk table, gate gradients and bias sums (both paths): the chunked row
// sums of dc/dr into dWg, dWn, dbg, of dE into db2 and of dz into db1.
// Hierarchical gating: the expert columns start at G (the group columns
// come first), and the group columns get the same sums over the (token,
// kept group) pairs, routed by group (Pairs).
struct RowSums {
    int32_t *ctiles;
    float *pg, *pn, *pb, *pc;
};

struct Pairs {
    const int32_t *offsets, *perm;   // the pairs t*kg + q in group order
    const float *dc, *dr;            // per pair
    int32_t *ctiles;                 // [G + 1] chunk table of the pairs
};

cudaError_t row_sums(const moe_shape &s, const RowSums &R, const int32_t *offsets,
                     const int32_t *perm, const void *x, int bf16, const float *dc, const float *dr,
                     float *dWg, float *dWn, float *dbg, const RowOp &dE_op, float *db2,
                     const RowOp &dz_op, float *db1, int32_t *err, cudaStream_t st,
                     const Pairs *pairs = nullptr) {
    const int64_t S = slots(s);
    const int n = s.n, d = s.d, h = s.h;
    const int C = gate_cols(s), col0 = s.groups;
    const unsigned chunks = static_cast<unsigned>((S + kChunkRows - 1) / kChunkRows + n);
    cudaError_t e = launch_row_tiles(offsets, n, kChunkRows, R.ctiles, st);
    if (e != cudaSuccess) return e;
    bwd_gate_part<<<dim3(chunks, (d + 255) / 256), 256, 0, st>>>(d, s.k, S, x, bf16, perm, offsets,
                                                                 R.ctiles, n, dc, dr, R.pg, R.pn,
                                                                 R.pb, err);
    bwd_gate_fin<<<dim3((d + 255) / 256, n), 256, 0, st>>>(d, n, C, col0, R.ctiles, R.pg, R.pn, R.pb,
                                                           dWg, dWn, dbg);
    if (pairs) {
        // the group columns: the same two passes over the pairs of each group
        // (P = T*kg pairs, fewer rows and columns than the slots: the partial
        // buffers fit)
        const int Gn = s.groups, kg = s.k_groups;
        const int64_t P = s.T * kg;
        const unsigned pchunks = static_cast<unsigned>((P + kChunkRows - 1) / kChunkRows + Gn);
        if ((e = launch_row_tiles(pairs->offsets, Gn, kChunkRows, pairs->ctiles, st)) != cudaSuccess)
            return e;
        bwd_gate_part<<<dim3(pchunks, (d + 255) / 256), 256, 0, st>>>(
            d, kg, P, x, bf16, pairs->perm, pairs->offsets, pairs->ctiles, Gn, pairs->dc, pairs->dr,
            R.pg, R.pn, R.pb, err);
        bwd_gate_fin<<<dim3((d + 255) / 256, Gn), 256, 0, st>>>(d, Gn, C, 0, pairs->ctiles, R.pg,
                                                                R.pn, R.pb, dWg, dWn, dbg);
    }
    if (db2) {
        bwd_colsum_part<<<dim3(chunks, (d + 255) / 256), 256, 0, st>>>(dE_op, d, offsets, R.ctiles, n,
                                                                       S, R.pc, err);
        bwd_colsum_fin<<<dim3((d + 255) / 256, n), 256, 0, st>>>(R.pc, d, R.ctiles, db2);
    }
    if (db1) {
        bwd_colsum_part<<<dim3(chunks, (h + 255) / 256), 256, 0, st>>>(dz_op, h, offsets, R.ctiles, n,
                                                                       S, R.pc, err);
        bwd_colsum_fin<<<dim3((h + 255) / 256, n), 256, 0, st>>>(R.pc, h, R.ctiles, db1);
    }
    return cudaGetLastError();
}

// Routes the (token, kept group) pairs of a hierarchical selection by group
// (the dispatch's own kernels on the pairs), for the group columns' sums.
cudaError_t route_pairs(const moe_shape &s, const int32_t *idx, const float *G, void *ws,
                        const PairLayout &P, cudaStream_t st) {
    const int64_t np = s.T * s.k_groups;
    int32_t *gidx = ws_ptr<int32_t>(ws, P.gidx);
    float *gw = ws_ptr<float>(ws, P.gw);
    bwd_pairs<<<static_cast<unsigned>((np + 255) / 256), 256, 0, st>>>(idx, G, s.T, s.k, s.k_groups,
                                                                       s.n / s.groups, gidx, gw);
    moe_shape sg = s;
    sg.n = s.groups;
    sg.k = s.k_groups;
    sg.groups = 0;
    sg.k_groups = 0;
    WsLayout RL{};
    RL.local_rank = P.local_rank;
    RL.chunk = P.chunk;
    RL.chunk_imp = P.chunk_imp;
    RL.imp_acc = P.imp_acc;
    return launch_dispatch(sg, gidx, gw, ws_ptr<int32_t>(ws, P.counts), ws_ptr<int32_t>(ws, P.offsets),
                           ws_ptr<int32_t>(ws, P.perm), ws_ptr<int32_t>(ws, P.inv),
                           ws_ptr<float>(ws, P.imp), ws_ptr<float>(ws, P.cv2), ws, RL, st);
}

// Gate side of both paths: W_g^T and W_noise^T over the C score columns, the
// importance term, the token kernel (flat or two-level) and, for the
// hierarchical gate, the pairs' routing for the group columns' sums.
cudaError_t gate_side(const moe_shape &s, const void *x, const float *Wg, const float *Wn,
                      const float *eps, const int32_t *idx, const float *G,
                      const float *importance, const void *dy, int bf16, float w_imp,
                      const void *E, const void *dXs, int ebf16, const int32_t *inv, float *WgT,
                      float *WnT, float *gimp, float *dc, float *dr, float *dx, void *ws,
                      const PairLayout &P, int32_t *err, cudaStream_t st) {
    const int d = s.d, n = s.n, C = gate_cols(s);
    bwd_transpose<<<dim3((C + 31) / 32, (d + 31) / 32), dim3(32, 8), 0, st>>>(Wg, d, C, WgT);
    if (eps)
        bwd_transpose<<<dim3((C + 31) / 32, (d + 31) / 32), dim3(32, 8), 0, st>>>(Wn, d, C, WnT);
    bwd_gimp<<<1, 256, 0, st>>>(w_imp != 0.0f ? importance : nullptr, n, w_imp, gimp);
    if (s.groups == 0)
        return launch_token(s.T, d, n, s.k, x, dy, bf16, E, dXs, ebf16, inv, idx, G, gimp, WgT, WnT,
                            eps, dc, dr, dx, err, st);
    cudaError_t e = launch_token_hier(s, x, dy, bf16, E, dXs, ebf16, inv, idx, G, gimp, WgT, WnT,
                                      eps, dc, dr, ws_ptr<float>(ws, P.dcg),
                                      ws_ptr<float>(ws, P.drg), dx, err, st);
    if (e != cudaSuccess) return e;
    return route_pairs(s, idx, G, ws, P, st);
}

Pairs pairs_of(const moe_shape &s, void *ws, const PairLayout &P) {
    return Pairs{ws_ptr<int32_t>(ws, P.offsets), ws_ptr<int32_t>(ws, P.perm),
                 ws_ptr<float>(ws, P.dcg), ws_ptr<float>(ws, P.drg), ws_ptr<int32_t>(ws, P.ctiles)};
}

cudaError_t row_gemm(const RowGemm &g, int64_t S, int n, cudaStream_t st) {
    const unsigned max_rt = static_cast<unsigned>((S + kBT - 1) / kBT + n);
    bwd_row_gemm<<<dim3(max_rt, g.N / kBT), 256, 0, st>>>(g);
    return cudaGetLastError();
}

}  // namespace

// --- tensor-core path (bf16) -------------------------------------------------
// The forward's workspace comes first (routing, x rows in expert order,
// hidden activations a = ReLU(z) and expert outputs E, all bf16, from a
// recompute of the expert stage); then:
//   W1T, W2T  the experts' weights transposed ([n, d, h] and [n, h, d]), for
//             the single-SM GEMM (output widths not multiples of 256)
//   dE        [S, d] rows G dy in expert order;  dA -> dZ [S, h];  dXs [S, d]
//   kblk      64-row blocks per expert (tile table), the k-blocks of the
//             weight-gradient contractions
//   PdE, Pa, PdZ, Px  dE, a, dZ, x rows transposed and padded ([M, Kcap])
//   WgT, WnT, gimp, dc, dr  as in the CUDA-core path
struct BtLayout {
    WsLayout fwd;
    int64_t Kcap = 0;
    size_t W1T = 0, W2T = 0, dE = 0, dA = 0, dXs = 0, kblk = 0, PdE = 0, Pa = 0, PdZ = 0, Px = 0;
    size_t WgT = 0, WnT = 0, gimp = 0, dc = 0, dr = 0;
    size_t ctiles = 0, pg = 0, pn = 0, pb = 0, pc = 0;
    PairLayout pairs;
    size_t total = 0;
};

bool backward_tc_supported(const moe_shape &s) {
    return s.dtype == MOE_BF16 && s.d % 128 == 0 && s.h % 128 == 0;
}

BtLayout bt_layout(const moe_shape &s) {
    BtLayout L;
    L.fwd = ws_layout(s);
    const size_t S = static_cast<size_t>(slots(s));
    const size_t n = static_cast<size_t>(s.n), d = static_cast<size_t>(s.d),
                 h = static_cast<size_t>(s.h);
    L.Kcap = 64 * (static_cast<int64_t>((S + 63) / 64) + s.n);
    const size_t K = static_cast<size_t>(L.Kcap);
    size_t o = L.fwd.total;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = align_up(o + bytes, 256);
        return at;
    };
    L.W1T = take(n * d * h * 2);
    L.W2T = take(n * d * h * 2);
    L.dE = take(S * d * 2);
    L.dA = take(S * h * 2);
    L.dXs = take(S * d * 2);
    L.kblk = take((n + 1) * 4);
    L.PdE = take(d * K * 2);
    L.Pa = take(h * K * 2);
    L.PdZ = take(h * K * 2);
    L.Px = take(d * K * 2);
    const size_t Cg = static_cast<size_t>(gate_cols(s));
    L.WgT = take(Cg * d * 4);
    L.WnT = take(Cg * d * 4);
    L.gimp = take(n * 4);
    L.pairs = take_pairs(s, take);
    L.dc = take(S * 4);
    L.dr = take(S * 4);
    const size_t C = row_chunks(s);
    L.ctiles = take((n + 1) * 4);
    L.pg = take(C * d * 4);
    L.pn = take(C * d * 4);
    L.pb = take(C * 4);
    L.pc = take(C * (d > h ? d : h) * 4);
    L.total = o;
    return L;
}

cudaError_t launch_backward_tc(const moe_shape &s, const void *x, const float *Wg, const float *Wn,
                               const float *eps, const void *W1, const float *b1, const void *W2,
                               const float *b2, const int32_t *idx, const float *G,
                               const float *importance, const void *dy, float w_imp, float *dx,
                               float *dWg, float *dWn, float *dbg, float *dW1, float *db1,
                               float *dW2, float *db2, void *ws, cudaStream_t st) {
    const BtLayout B = bt_layout(s);
    const WsLayout &L = B.fwd;
    const int64_t S = slots(s);
    const int n = s.n, d = s.d, h = s.h, k = s.k;
    int32_t *err = ws_ptr<int32_t>(ws, 0);
    int32_t *offsets = ws_ptr<int32_t>(ws, L.offsets);
    int32_t *perm = ws_ptr<int32_t>(ws, L.perm);
    int32_t *inv = ws_ptr<int32_t>(ws, L.inv_perm);
    int32_t *tiles = ws_ptr<int32_t>(ws, L.tiles);     // 128-row blocks (single-SM GEMM)
    int32_t *ptiles = ws_ptr<int32_t>(ws, L.ptiles);   // token tiles (pair GEMM)
    int4 *plist = ws_ptr<int4>(ws, L.plist);
    auto bf = [&](size_t off) { return ws_ptr<__nv_bfloat16>(ws, off); };
    __nv_bfloat16 *xperm = bf(L.xperm), *hid = bf(L.hidden), *E = bf(L.yslot);
    __nv_bfloat16 *W1T = bf(B.W1T), *W2T = bf(B.W2T), *dE = bf(B.dE), *dZ = bf(B.dA), *dXs = bf(B.dXs);
    int32_t *kblk = ws_ptr<int32_t>(ws, B.kblk);
    float *WgT = ws_ptr<float>(ws, B.WgT), *WnT = ws_ptr<float>(ws, B.WnT);
    float *gimp = ws_ptr<float>(ws, B.gimp), *dc = ws_ptr<float>(ws, B.dc), *dr = ws_ptr<float>(ws, B.dr);
    const float *eps_used = s.noisy ? eps : nullptr;
    float *dWn_used = s.noisy ? dWn : nullptr;
    if (!s.noisy && dWn) cudaMemsetAsync(dWn, 0, sizeof(float) * d * gate_cols(s), st);

    cudaError_t e = launch_dispatch(s, idx, G, ws_ptr<int32_t>(ws, L.counts), offsets, perm, inv,
                                    ws_ptr<float>(ws, L.importance), ws_ptr<float>(ws, L.cv2), ws,
                                    L, st);
    // recompute x rows, a = ReLU(x W1^T + b1) and E = a W2^T + b2 (bf16, expert order)
    if (e == cudaSuccess)
        e = launch_expert_ffn(s, x, perm, offsets, W1, b1, W2, b2, E, ws, L, st, false, true);
    // dA = dE W2 (K = d), then dZ = dA * [a > 0];  dXs = dZ W1 (K = h).
    // An output width that suits the SM-pair GEMM reads the weights in their
    // stored layout (an MN-major operand); otherwise the single-SM GEMM reads
    // a transposed copy (W2^T, W1^T rows).  Output widths h and d are the
    // recompute's, so the tile tables it built from the same offsets serve
    // here unchanged.
    if (e == cudaSuccess && !pair_gemm_supported(h))
        e = launch_transpose_experts(static_cast<const __nv_bfloat16 *>(W2), n, d, h, W2T, st);
    if (e == cudaSuccess && !pair_gemm_supported(d))
        e = launch_transpose_experts(static_cast<const __nv_bfloat16 *>(W1), n, h, d, W1T, st);
    if (e == cudaSuccess)
        e = launch_rows_scaled(static_cast<const __nv_bfloat16 *>(dy), G, perm, S, d, k, dE, err, st);
    auto row_gemm = [&](const __nv_bfloat16 *X, int K, const void *W, const __nv_bfloat16 *Wt,
                        int Nout, __nv_bfloat16 *out) {
        return pair_gemm_supported(Nout)
                   ? launch_grouped_gemm_pair_wmn(s, X, K, static_cast<const __nv_bfloat16 *>(W),
                                                  Nout, ptiles, plist, out, err, st)
                   : launch_grouped_gemm_tc(s, X, K, Wt, Nout, nullptr, 0, offsets, tiles, out,
                                            err, st);
    };
    if (e == cudaSuccess) e = row_gemm(dE, d, W2, W2T, h, dZ);
    if (e == cudaSuccess) e = launch_relu_mask(dZ, hid, S * static_cast<int64_t>(h), st);
    if (e == cudaSuccess) e = row_gemm(dZ, h, W1, W1T, d, dXs);
    // weight gradients: rows as the contraction axis, transposed and padded per expert
    if (e == cudaSuccess) e = launch_row_tiles(offsets, n, 64, kblk, st);
    if (e == cudaSuccess) e = launch_transpose_pad(dE, d, offsets, kblk, n, S, B.Kcap, bf(B.PdE), st);
    if (e == cudaSuccess) e = launch_transpose_pad(hid, h, offsets, kblk, n, S, B.Kcap, bf(B.Pa), st);
    if (e == cudaSuccess) e = launch_transpose_pad(dZ, h, offsets, kblk, n, S, B.Kcap, bf(B.PdZ), st);
    if (e == cudaSuccess) e = launch_transpose_pad(xperm, d, offsets, kblk, n, S, B.Kcap, bf(B.Px), st);
    if (e == cudaSuccess) e = launch_wgrad_tc(bf(B.PdE), d, bf(B.Pa), h, B.Kcap, kblk, n, dW2, err, st);
    if (e == cudaSuccess) e = launch_wgrad_tc(bf(B.PdZ), h, bf(B.Px), d, B.Kcap, kblk, n, dW1, err, st);
    if (e != cudaSuccess) return e;

    // gate side and the sums over rows, on the CUDA cores
    if ((e = gate_side(s, x, Wg, Wn, eps_used, idx, G, importance, dy, 1, w_imp, E, dXs, 1, inv, WgT,
                       WnT, gimp, dc, dr, dx, ws, B.pairs, err, st)) != cudaSuccess)
        return e;
    const RowOp dE_op{dy, 1, d, perm, k, G, 0};
    const RowOp dz_op{dZ, 1, h, nullptr, 1, nullptr, 0};
    const RowSums R{ws_ptr<int32_t>(ws, B.ctiles), ws_ptr<float>(ws, B.pg), ws_ptr<float>(ws, B.pn),
                    ws_ptr<float>(ws, B.pb), ws_ptr<float>(ws, B.pc)};
    const Pairs pr = pairs_of(s, ws, B.pairs);
    return row_sums(s, R, offsets, perm, x, 1, dc, dr, dWg, dWn_used, dbg, dE_op, db2, dz_op, db1, err,
                    st, s.groups ? &pr : nullptr);
}

size_t backward_workspace_bytes(const moe_shape &s) {
    return backward_tc_supported(s) ? bt_layout(s).total : bwd_layout(s).total;
}

namespace {

cudaError_t launch_backward(const moe_shape &s, const void *x, const float *Wg, const float *Wn,
                            const float *eps, const void *W1, const float *b1, const void *W2,
                            const float *b2, const int32_t *idx, const float *G,
                            const float *importance, const void *dy, float w_imp, float *dx,
                            float *dWg, float *dWn, float *dbg, float *dW1, float *db1, float *dW2,
                            float *db2, void *ws, cudaStream_t st) {
    const BwdLayout B = bwd_layout(s);
    const int64_t S = slots(s);
    const int n = s.n, d = s.d, h = s.h, k = s.k;
    const int bf16 = s.dtype == MOE_BF16 ? 1 : 0;
    int32_t *err = ws_ptr<int32_t>(ws, 0);
    int32_t *offsets = ws_ptr<int32_t>(ws, B.offsets);
    int32_t *perm = ws_ptr<int32_t>(ws, B.perm);
    int32_t *inv = ws_ptr<int32_t>(ws, B.inv_perm);
    int32_t *tiles = ws_ptr<int32_t>(ws, B.tiles);
    float *WgT = ws_ptr<float>(ws, B.WgT), *WnT = ws_ptr<float>(ws, B.WnT);
    float *gimp = ws_ptr<float>(ws, B.gimp), *dc = ws_ptr<float>(ws, B.dc), *dr = ws_ptr<float>(ws, B.dr);
    float *Z = ws_ptr<float>(ws, B.Z), *dZ = ws_ptr<float>(ws, B.dZ);
    float *E = ws_ptr<float>(ws, B.E), *dXs = ws_ptr<float>(ws, B.dXs);
    const float *eps_used = s.noisy ? eps : nullptr;
    float *dWn_used = s.noisy ? dWn : nullptr;
    if (!s.noisy && dWn) cudaMemsetAsync(dWn, 0, sizeof(float) * d * gate_cols(s), st);

    // routing of the forward's selection (the dispatch's own chunk regions)
    WsLayout RL{};
    RL.local_rank = B.local_rank;
    RL.chunk = B.chunk;
    RL.chunk_imp = B.chunk_imp;
    RL.imp_acc = B.imp_acc;
    cudaError_t e = launch_dispatch(s, idx, G, ws_ptr<int32_t>(ws, B.counts), offsets, perm, inv,
                                    ws_ptr<float>(ws, B.imp), ws_ptr<float>(ws, B.cv2), ws, RL, st);
    if (e == cudaSuccess) e = launch_row_tiles(offsets, n, kBT, tiles, st);
    if (e != cudaSuccess) return e;

    RowGemm g{};
    g.offsets = offsets;
    g.tiles = tiles;
    g.n = n;
    g.S = S;
    g.err = err;
    // Z = X W1^T + b1   (W1[e] is [h, d]: B_e(k, c) = W1[e][c][k])
    g.a = RowOp{x, bf16, d, perm, k, nullptr, 0};
    g.B = W1;
    g.b_bf16 = bf16;
    g.bse = static_cast<int64_t>(h) * d;
    g.bsk = 1;
    g.bsc = d;
    g.bias = b1;
    g.mask = nullptr;
    g.out = Z;
    g.K = d;
    g.N = h;
    if ((e = row_gemm(g, S, n, st)) != cudaSuccess) return e;
    // E = ReLU(Z) W2^T + b2   (W2[e] is [d, h])
    g.a = RowOp{Z, 0, h, nullptr, 1, nullptr, 1};
    g.B = W2;
    g.bse = static_cast<int64_t>(d) * h;
    g.bsk = 1;
    g.bsc = h;
    g.bias = b2;
    g.out = E;
    g.K = h;
    g.N = d;
    if ((e = row_gemm(g, S, n, st)) != cudaSuccess) return e;
    // dZ = (dE W2) * [Z > 0],  dE rows = G[s] dy[t]   (B_e(k, c) = W2[e][k][c])
    g.a = RowOp{dy, bf16, d, perm, k, G, 0};
    g.bsk = h;
    g.bsc = 1;
    g.bias = nullptr;
    g.mask = Z;
    g.out = dZ;
    g.K = d;
    g.N = h;
    if ((e = row_gemm(g, S, n, st)) != cudaSuccess) return e;
    // dXs = dZ W1   (B_e(k, c) = W1[e][k][c])
    g.a = RowOp{dZ, 0, h, nullptr, 1, nullptr, 0};
    g.B = W1;
    g.bse = static_cast<int64_t>(h) * d;
    g.bsk = d;
    g.bsc = 1;
    g.mask = nullptr;
    g.out = dXs;
    g.K = h;
    g.N = d;
    if ((e = row_gemm(g, S, n, st)) != cudaSuccess) return e;

    if ((e = gate_side(s, x, Wg, Wn, eps_used, idx, G, importance, dy, bf16, w_imp, E, dXs, 0, inv,
                       WgT, WnT, gimp, dc, dr, dx, ws, B.pairs, err, st)) != cudaSuccess)
        return e;

    // dW2[e] = sum dE a^T  (M = d, N = h),  dW1[e] = sum dz x^T  (M = h, N = d)
    const RowOp dE_op{dy, bf16, d, perm, k, G, 0};
    const RowOp a_op{Z, 0, h, nullptr, 1, nullptr, 1};
    const RowOp dz_op{dZ, 0, h, nullptr, 1, nullptr, 0};
    const RowOp x_op{x, bf16, d, perm, k, nullptr, 0};
    bwd_wgrad<<<dim3(h / kBT, d / kBT, n), 256, 0, st>>>(dE_op, a_op, d, h, offsets, S, dW2, err);
    bwd_wgrad<<<dim3(d / kBT, h / kBT, n), 256, 0, st>>>(dz_op, x_op, h, d, offsets, S, dW1, err);
    const RowSums R{ws_ptr<int32_t>(ws, B.ctiles), ws_ptr<float>(ws, B.pg), ws_ptr<float>(ws, B.pn),
                    ws_ptr<float>(ws, B.pb), ws_ptr<float>(ws, B.pc)};
    const Pairs pr = pairs_of(s, ws, B.pairs);
    return row_sums(s, R, offsets, perm, x, bf16, dc, dr, dWg, dWn_used, dbg, dE_op, db2, dz_op, db1,
                    err, st, s.groups ? &pr : nullptr);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_backward_workspace_bytes(const moe_shape *s) {
    if (moe_validate(s) != MOE_OK) return 0;
    return backward_workspace_bytes(*s);
}

moe_status moe_backward(const moe_shape *s, const void *x, const float *Wg, const float *Wnoise,
                        const float *eps, const void *W1, const float *b1, const void *W2,
                        const float *b2, const int32_t *idx, const float *G,
                        const float *importance, const void *dy, float w_importance, float *dx,
                        float *dWg, float *dWnoise, float *dbg, float *dW1, float *db1, float *dW2,
                        float *db2, void *ws, size_t ws_bytes, void *stream) {
    moe_status v = moe_validate(s);
    if (v != MOE_OK) return v;
    auto al = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    auto req = [&](const void *p) { return p != nullptr && al(p); };
    auto opt = [&](const void *p) { return p == nullptr || al(p); };
    if (!req(Wg) || !req(W1) || !req(W2) || !req(dWg) || !req(dW1) || !req(dW2))
        return MOE_ERR_INVALID_ARG;
    if (!opt(b1) || !opt(b2) || !opt(dbg) || !opt(db1) || !opt(db2) || !opt(Wnoise) || !opt(eps) ||
        !opt(dWnoise) || !opt(importance))
        return MOE_ERR_INVALID_ARG;
    if (s->noisy && (!req(Wnoise) || !req(dWnoise))) return MOE_ERR_INVALID_ARG;
    if (w_importance != 0.0f && !req(importance)) return MOE_ERR_INVALID_ARG;
    if (!(w_importance == w_importance)) return MOE_ERR_INVALID_ARG;  // NaN
    if (s->T > 0 && (!req(x) || !req(idx) || !req(G) || !req(dy) || !req(dx)))
        return MOE_ERR_INVALID_ARG;
    if (s->T > 0 && s->noisy && !req(eps)) return MOE_ERR_INVALID_ARG;
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 ||
        ws_bytes < backward_workspace_bytes(*s))
        return MOE_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int64_t n = s->n, d = s->d, h = s->h, C = gate_cols(*s);
    if (s->T == 0) {
        // no slot: every gradient is zero
        cudaMemsetAsync(dWg, 0, sizeof(float) * d * C, st);
        if (dWnoise) cudaMemsetAsync(dWnoise, 0, sizeof(float) * d * C, st);
        if (dbg) cudaMemsetAsync(dbg, 0, sizeof(float) * C, st);
        cudaMemsetAsync(dW1, 0, sizeof(float) * n * h * d, st);
        cudaMemsetAsync(dW2, 0, sizeof(float) * n * d * h, st);
        if (db1) cudaMemsetAsync(db1, 0, sizeof(float) * n * h, st);
        if (db2) cudaMemsetAsync(db2, 0, sizeof(float) * n * d, st);
        return cuda_to_status(cudaGetLastError());
    }
    const auto run = backward_tc_supported(*s) ? launch_backward_tc : launch_backward;
    const cudaError_t e = run(*s, x, Wg, Wnoise, eps, W1, b1, W2, b2, idx, G, importance, dy,
                              w_importance, dx, dWg, dWnoise, dbg, dW1, db1, dW2, db2, ws, st);
    return cuda_to_status(e);
}

}  // extern "C"

// balanced.cu -- the layer with balanced routing (moe_forward_balanced in moe.h).
//
// "Outrageously Large Neural Networks - 中文验证版", section 方法适配: in some
// translation experiments a per-batch mask gives every expert the same batch
// size during training, and per-expert thresholds approximate that at
// inference.  The pages give no formula; the reading taken:
//   H[t, e]    the flat gate's noisy score, c + eps * softplus(r)
//   batchwise  (thr NULL) expert e keeps the m = floor(k*T/n) tokens with the
//              largest H[:, e], equal scores going to the lower token index
//   threshold  (thr given) expert e keeps token t iff H[t, e] > thr[e]
//   weights    softmax of H[t, .] over the experts that kept t
//   y[t]       sum over those experts, in increasing e, of w E_e(x_t); 0 if none
// Stages, in launch order:
//   scores            H [T, n]: noisy bf16 shapes from the tensor-core gate's
//                     load mode (c and softplus(r) per expert, fp32-faithful,
//                     H = c + eps * s formed by bal_transpose); other shapes
//                     bal_scores, fp32 on the CUDA cores (64 x 64 tiles)
//   bal_transpose     HT [n, T], each expert's scores contiguous; the row map
//                     reset to -1
//   bal_count         per expert: the m-th largest score by a 4-pass 8-bit
//                     radix select on order-preserving keys, and how many of
//                     the tied scores to keep (batchwise); or the number of
//                     scores above thr[e] (threshold)
//   bal_scan          offsets = exclusive scan of the counts, clamped to the
//                     row capacity (an overflow is reported)
//   bal_write         per expert, its kept tokens in token order into rows
//                     offsets[e].. (ordered block compaction), and the map
//                     rowmap[t, e] = row
//   bal_weights       one warp per token: the softmax over its kept experts
//   expert FFN        the forward's stage on the rows (x row = the token)
//   bal_combine       one warp per token: y = sum over kept e (increasing) of w Y[row]
#include "moe_device.cuh"
#include "moe_launch.h"

#include <algorithm>

namespace moe {
namespace {

constexpr int32_t kSiteBalRows = 40;
constexpr int kBT = 64, kBK = 16;

struct BalLayout {
    moe_shape ffn;  // the expert stage's shape: one slot per row
    WsLayout fwd;
    size_t H = 0, HT = 0, rowmap = 0, row_token = 0, row_weight = 0, kstar = 0, quota = 0, cnt = 0;
    size_t sN = 0, gidx = 0, gG = 0, vk = 0;  // tensor-core scores: noise scale, its top-k, k-th
    size_t total = 0;
    int64_t rows = 0;  // row capacity
};

// Noisy bf16 shapes take the scores from the tensor-core gate, which in its
// load mode writes the clean score c = x.Wg + bg and the noise scale
// softplus(x.Wnoise) of every (token, expert), fp32-faithful; H = c + eps * s.
bool bal_tc_scores(const moe_shape &s) {
    return s.dtype == MOE_BF16 && s.noisy && s.k < MOE_MAX_K && gate_tc_supported(s);
}

moe_shape ffn_shape(const moe_shape &s, int64_t rows_cap) {
    moe_shape f = s;
    f.T = std::max<int64_t>(rows_cap, s.T);  // gathered token ids stay below T <= f.T
    f.k = 1;
    f.groups = 0;
    f.k_groups = 0;
    return f;
}

BalLayout bal_layout(const moe_shape &s, int64_t rows_cap) {
    BalLayout B;
    B.ffn = ffn_shape(s, rows_cap);
    B.fwd = ws_layout(B.ffn);
    B.rows = rows_cap;
    const size_t Tn = static_cast<size_t>(s.T) * s.n;
    const size_t R = static_cast<size_t>(B.ffn.T);
    size_t o = B.fwd.total;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = align_up(o + bytes, 256);
        return at;
    };
    B.H = take(Tn * 4);
    B.HT = take(Tn * 4);
    B.rowmap = take(Tn * 4);
    B.row_token = take(R * 4);
    B.row_weight = take(R * 4);
    B.kstar = take(static_cast<size_t>(s.n) * 4);
    B.quota = take(static_cast<size_t>(s.n) * 4);
    B.cnt = take(static_cast<size_t>(s.n) * 4);
    if (bal_tc_scores(s)) {
        B.sN = take(Tn * 4);
        B.gidx = take(static_cast<size_t>(s.T) * s.k * 4);
        B.gG = take(static_cast<size_t>(s.T) * s.k * 4);
        B.vk = take(static_cast<size_t>(s.T) * 2 * 4);
    }
    B.total = o;
    return B;
}

// H[t, e] = x_t . Wg[:, e] + bg[e] (+ eps[t, e] softplus(x_t . Wn[:, e])), fp32.
template <typename TX>
__global__ void __launch_bounds__(256) bal_scores(const TX *__restrict__ x, const float *__restrict__ Wg,
                                                  const float *__restrict__ Wn,
                                                  const float *__restrict__ bg,
                                                  const float *__restrict__ eps, int64_t T, int d,
                                                  int n, float *__restrict__ H) {
    __shared__ float Xs[kBK][kBT + 4];
    __shared__ float Gs[kBK][kBT + 4];
    __shared__ float Ns[kBK][kBT + 4];
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kBT;
    const int e0 = blockIdx.y * kBT;
    const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
    float c[4][4] = {}, r[4][4] = {};
    for (int k0 = 0; k0 < d; k0 += kBK) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int idx = tid + q * 256;
            {
                const int row = idx / kBK, kk = idx % kBK;
                const int64_t t = t0 + row;
                Xs[kk][row] = t < T ? to_f(x[t * d + k0 + kk]) : 0.0f;
            }
            {
                const int kk = idx / kBT, col = idx % kBT;
                const int e = e0 + col;
                const int64_t at = static_cast<int64_t>(k0 + kk) * n + e;
                Gs[kk][col] = e < n ? Wg[at] : 0.0f;
                Ns[kk][col] = (e < n && eps) ? Wn[at] : 0.0f;
            }
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < kBK; ++kk) {
            float xv[4], gv[4], nv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                xv[i] = Xs[kk][ty * 4 + i];
                gv[i] = Gs[kk][tx * 4 + i];
                nv[i] = Ns[kk][tx * 4 + i];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    c[i][j] = fmaf(xv[i], gv[j], c[i][j]);
                    r[i][j] = fmaf(xv[i], nv[j], r[i][j]);
                }
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t t = t0 + ty * 4 + i;
        if (t >= T) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int e = e0 + tx * 4 + j;
            if (e >= n) continue;
            float v = c[i][j] + (bg ? bg[e] : 0.0f);
            if (eps) v += eps[t * n + e] * softplus_f(r[i][j]);
            H[t * n + e] = v;
        }
    }
}

// HT[e, t] = H[t, e]: each expert's scores contiguous for the per-expert
// select and compaction (32 x 32 tiles through shared memory).  With sc and
// eps given, H holds the clean scores c on entry and becomes the noisy
// scores c + eps * s first (in place).  The row map [T, n] is reset to -1 on
// the way (the compaction then writes the kept entries).
__global__ void bal_transpose(float *__restrict__ H, const float *__restrict__ sc,
                              const float *__restrict__ eps, int64_t T, int n,
                              float *__restrict__ HT, int32_t *__restrict__ rowmap) {
    __shared__ float tile[32][33];
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * 32;
    const int e0 = blockIdx.y * 32;
    for (int i = threadIdx.y; i < 32; i += 8) {
        const int64_t t = t0 + i;
        const int e = e0 + threadIdx.x;
        float v = 0.0f;
        if (t < T && e < n) {
            const int64_t at = t * n + e;
            v = H[at];
            if (sc) {
                v = fmaf(eps[at], sc[at], v);
                H[at] = v;
            }
            rowmap[at] = -1;
        }
        tile[i][threadIdx.x] = v;
    }
    __syncthreads();
    for (int i = threadIdx.y; i < 32; i += 8) {
        const int e = e0 + i;
        const int64_t t = t0 + threadIdx.x;
        if (e < n && t < T) HT[static_cast<int64_t>(e) * T + t] = tile[threadIdx.x][i];
    }
}

// Scores a thread keeps in registers across the passes of the per-expert
// select (up to 16384 tokens; longer columns are read again from memory).
constexpr int kBalKeys = 16;

// Order-preserving key of a float: larger float, larger key.
__device__ __forceinline__ uint32_t fkey(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// One block of 1024 threads per expert.  Batchwise (thr == nullptr): kstar[e]
// = key of the m-th largest score, quota[e] = how many scores equal to it are
// kept (the lowest token indices), cnt[e] = m.  Threshold: cnt[e] = number of
// scores above thr[e].
__global__ void __launch_bounds__(1024) bal_count(const float *__restrict__ HT, int64_t T, int n,
                                                  int64_t m, const float *__restrict__ thr,
                                                  uint32_t *__restrict__ kstar,
                                                  int32_t *__restrict__ quota,
                                                  int32_t *__restrict__ cnt) {
    __shared__ uint32_t hist[256];
    __shared__ uint32_t sel_digit;
    __shared__ int64_t sel_above;
    __shared__ int32_t part[32];
    const int e = blockIdx.x;
    const int tid = threadIdx.x;
    if (thr) {
        const float th = thr[e];
        int32_t c = 0;
        const float *col = HT + static_cast<int64_t>(e) * T;
        for (int64_t t = tid; t < T; t += 1024) c += col[t] > th ? 1 : 0;
        for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
        if ((tid & 31) == 0) part[tid >> 5] = c;
        __syncthreads();
        if (tid == 0) {
            int32_t s = 0;
            for (int w = 0; w < 32; ++w) s += part[w];
            cnt[e] = s;
            kstar[e] = 0;
            quota[e] = 0;
        }
        return;
    }
    if (m <= 0) {
        if (tid == 0) {
            cnt[e] = 0;
            kstar[e] = 0xFFFFFFFFu;
            quota[e] = 0;
        }
        return;
    }
    // Up to kBalKeys scores per thread stay in registers across the passes.
    const float *col = HT + static_cast<int64_t>(e) * T;
    const bool cached = T <= static_cast<int64_t>(kBalKeys) * 1024;
    uint32_t keys[kBalKeys];
    if (cached) {
#pragma unroll
        for (int i = 0; i < kBalKeys; ++i) {
            const int64_t t = tid + static_cast<int64_t>(i) * 1024;
            keys[i] = t < T ? fkey(__ldg(col + t)) : 0u;
        }
    }
    uint32_t prefix = 0, pmask = 0;
    int64_t remaining = m;
    for (int p = 3; p >= 0; --p) {
        for (int i = tid; i < 256; i += 1024) hist[i] = 0;
        __syncthreads();
        if (cached) {
#pragma unroll
            for (int i = 0; i < kBalKeys; ++i) {
                const int64_t t = tid + static_cast<int64_t>(i) * 1024;
                if (t < T && (keys[i] & pmask) == prefix)
                    atomicAdd(&hist[(keys[i] >> (8 * p)) & 255u], 1u);
            }
        } else {
            for (int64_t t = tid; t < T; t += 1024) {
                const uint32_t key = fkey(col[t]);
                if ((key & pmask) == prefix) atomicAdd(&hist[(key >> (8 * p)) & 255u], 1u);
            }
        }
        __syncthreads();
        if (tid < 32) {
            // The digit: going down from 255, the first whose count brings
            // the candidates at or above it to `remaining` (digit 0 if none
            // before it); sel_above = the candidates above it.  Lane l holds
            // digits 255 - 8l .. 248 - 8l.
            const int lane = tid;
            uint32_t hv[8];
            uint32_t sl = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                hv[j] = hist[255 - 8 * lane - j];
                sl += hv[j];
            }
            uint32_t inc = sl;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t u = __shfl_up_sync(0xffffffffu, inc, o);
                if (lane >= o) inc += u;
            }
            const unsigned cross = __ballot_sync(0xffffffffu, static_cast<int64_t>(inc) >= remaining);
            const int L = cross ? __ffs(cross) - 1 : 31;
            if (lane == L) {
                int64_t cum = static_cast<int64_t>(inc - sl);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int dg = 255 - 8 * lane - j;
                    if (dg == 0 || cum + hv[j] >= remaining) {
                        sel_digit = static_cast<uint32_t>(dg);
                        sel_above = cum;
                        break;
                    }
                    cum += hv[j];
                }
            }
        }
        __syncthreads();
        remaining -= sel_above;
        prefix |= sel_digit << (8 * p);
        pmask |= 0xFFu << (8 * p);
        __syncthreads();
    }
    if (tid == 0) {
        kstar[e] = prefix;
        quota[e] = static_cast<int32_t>(remaining);
        cnt[e] = static_cast<int32_t>(m);
    }
}

// offsets = exclusive scan of cnt (n + 1 entries), each clamped to `cap`; a
// total above the capacity is reported.  One block of 1024 threads.
__global__ void __launch_bounds__(1024) bal_scan(const int32_t *__restrict__ cnt, int n, int64_t cap,
                                                 int32_t *__restrict__ offsets,
                                                 int32_t *__restrict__ counts_out, int32_t *err) {
    __shared__ int64_t part[1024];
    const int per = (n + 1023) / 1024;
    const int i0 = threadIdx.x * per, i1 = min(n, i0 + per);
    int64_t sum = 0;
    for (int i = i0; i < i1; ++i) sum += cnt[i];
    part[threadIdx.x] = sum;
    __syncthreads();
    for (int off = 1; off < 1024; off <<= 1) {
        const int64_t v = threadIdx.x >= off ? part[threadIdx.x - off] : 0;
        __syncthreads();
        part[threadIdx.x] += v;
        __syncthreads();
    }
    int64_t run = threadIdx.x ? part[threadIdx.x - 1] : 0;
    for (int i = i0; i < i1; ++i) {
        offsets[i] = static_cast<int32_t>(run < cap ? run : cap);
        if (counts_out) counts_out[i] = cnt[i];
        run += cnt[i];
    }
    if (threadIdx.x == 1023) {
        offsets[n] = static_cast<int32_t>(part[1023] < cap ? part[1023] : cap);
        if (part[1023] > cap) report(err, MOE_ERR_DEVICE, kSiteBalRows, static_cast<int32_t>(cap));
    }
}

// Exclusive scan of one value per thread over a block of 1024 threads.
__device__ __forceinline__ int32_t block_exscan(int32_t v, int32_t *warp_tot) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int32_t inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t u = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += u;
    }
    if (lane == 31) warp_tot[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        int32_t w = warp_tot[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t u = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += u;
        }
        warp_tot[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const int32_t base = warp ? warp_tot[warp - 1] : 0;
    const int32_t out = base + inc - v;
    __syncthreads();
    return out;
}

// One block of 1024 threads per expert: its kept tokens in token order into
// rows offsets[e] .. offsets[e+1]-1 (thread i owns a contiguous token range).
__global__ void __launch_bounds__(1024) bal_write(const float *__restrict__ HT, int64_t T, int n,
                                                  const float *__restrict__ thr,
                                                  const uint32_t *__restrict__ kstar,
                                                  const int32_t *__restrict__ quota,
                                                  const int32_t *__restrict__ offsets,
                                                  int32_t *__restrict__ row_token,
                                                  int32_t *__restrict__ rowmap) {
    __shared__ int32_t warp_tot[32];
    const int e = blockIdx.x;
    const int64_t per = (T + 1023) / 1024;
    const int64_t t0 = threadIdx.x * per, t1 = min(T, t0 + per);
    const uint32_t ks = kstar[e];
    const int32_t qt = quota[e];
    const float th = thr ? thr[e] : 0.0f;
    const float *col = HT + static_cast<int64_t>(e) * T;
    const int32_t r0 = offsets[e], r1 = offsets[e + 1];
    if (per <= kBalKeys) {
        // the thread's scores (tokens t0 .. t1) in registers for all three passes
        float v[kBalKeys];
#pragma unroll
        for (int i = 0; i < kBalKeys; ++i) v[i] = t0 + i < t1 ? __ldg(col + t0 + i) : 0.0f;
        int32_t eq = 0;   // ties at the m-th score in this thread's range
        if (!thr) {
#pragma unroll
            for (int i = 0; i < kBalKeys; ++i) eq += (t0 + i < t1 && fkey(v[i]) == ks) ? 1 : 0;
        }
        const int32_t eq_base = block_exscan(eq, warp_tot);
        bool keep[kBalKeys];
        int32_t cnt = 0, seen = 0;
#pragma unroll
        for (int i = 0; i < kBalKeys; ++i) {
            bool k = false;
            if (t0 + i < t1) {
                if (thr) {
                    k = v[i] > th;
                } else {
                    const uint32_t key = fkey(v[i]);
                    k = key > ks || (key == ks && eq_base + seen++ < qt);
                }
            }
            keep[i] = k;
            cnt += k ? 1 : 0;
        }
        int32_t row = r0 + block_exscan(cnt, warp_tot);
#pragma unroll
        for (int i = 0; i < kBalKeys; ++i) {
            if (!keep[i]) continue;
            if (row < r1) {  // rows past the capacity were reported by bal_scan
                row_token[row] = static_cast<int32_t>(t0 + i);
                rowmap[(t0 + i) * n + e] = row;
            }
            ++row;
        }
        return;
    }
    // ties at the m-th score before this thread's range
    int32_t eq = 0;
    if (!thr)
        for (int64_t t = t0; t < t1; ++t) eq += fkey(col[t]) == ks ? 1 : 0;
    const int32_t eq_base = block_exscan(eq, warp_tot);
    auto kept = [&](int64_t t, int32_t &seen) {
        if (thr) return col[t] > th;
        const uint32_t key = fkey(col[t]);
        if (key > ks) return true;
        if (key == ks) return eq_base + seen++ < qt;
        return false;
    };
    int32_t cnt = 0, seen = 0;
    for (int64_t t = t0; t < t1; ++t) cnt += kept(t, seen) ? 1 : 0;
    const int32_t pos = block_exscan(cnt, warp_tot);
    int32_t row = r0 + pos;
    seen = 0;
    for (int64_t t = t0; t < t1; ++t) {
        if (!kept(t, seen)) continue;
        if (row < r1) {  // rows past the capacity were reported by bal_scan
            row_token[row] = static_cast<int32_t>(t);
            rowmap[t * n + e] = row;
        }
        ++row;
    }
}

// One warp per token: w = softmax of H[t, .] over its kept experts, written
// per row and (optionally) densely as W[t, e] (0 where not kept).
__global__ void __launch_bounds__(256) bal_weights(const float *__restrict__ H,
                                                   const int32_t *__restrict__ rowmap, int64_t T,
                                                   int n, float *__restrict__ row_weight,
                                                   float *__restrict__ W) {
    const int lane = threadIdx.x & 31;
    const int64_t t = static_cast<int64_t>(blockIdx.x) * 8 + threadIdx.x / 32;
    if (t >= T) return;
    const float *h = H + t * n;
    const int32_t *rm = rowmap + t * n;
    if (n <= 256) {
        // the token's row map and scores read once, eight per lane
        int32_t r[8];
        float hv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = 32 * i + lane;
            r[i] = e < n ? __ldg(rm + e) : -1;
            hv[i] = e < n ? __ldg(h + e) : 0.0f;
        }
        float mx = -INFINITY;
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (r[i] >= 0) mx = fmaxf(mx, hv[i]);
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        float sum = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (r[i] >= 0) sum += __expf(hv[i] - mx);
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = 32 * i + lane;
            if (e >= n) continue;
            const float w = r[i] >= 0 ? __expf(hv[i] - mx) / sum : 0.0f;
            if (r[i] >= 0) row_weight[r[i]] = w;
            if (W) W[t * n + e] = w;
        }
        return;
    }
    float mx = -INFINITY;
    for (int e = lane; e < n; e += 32)
        if (rm[e] >= 0) mx = fmaxf(mx, h[e]);
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float sum = 0.0f;
    for (int e = lane; e < n; e += 32)
        if (rm[e] >= 0) sum += __expf(h[e] - mx);
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    for (int e = lane; e < n; e += 32) {
        const int32_t r = rm[e];
        const float w = r >= 0 ? __expf(h[e] - mx) / sum : 0.0f;
        if (r >= 0) row_weight[r] = w;
        if (W) W[t * n + e] = w;
    }
}

// 16-byte pieces of bf16 or fp32 rows as fp32.
__device__ __forceinline__ void piece_to_f(const uint4 &u, float (&v)[8]) {
    const __nv_bfloat162 *b = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(b[i]);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
}
__device__ __forceinline__ void piece_to_f(const uint4 &u, float (&v)[4]) {
    v[0] = __uint_as_float(u.x);
    v[1] = __uint_as_float(u.y);
    v[2] = __uint_as_float(u.z);
    v[3] = __uint_as_float(u.w);
}
__device__ __forceinline__ uint4 piece_from_f(const float (&v)[8]) {
    return make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                      pack_bf16x2(v[6], v[7]));
}
__device__ __forceinline__ uint4 piece_from_f(const float (&v)[4]) {
    return make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]),
                      __float_as_uint(v[3]));
}

// Sums up to four queued experts' pieces into acc0/acc1 in queue order: all
// rows are requested before any is summed.
template <typename TY, int V>
__device__ __forceinline__ void bal_flush(const TY *__restrict__ Y, int d, int p0, int p1, bool has0,
                                          bool has1, const int32_t (&r)[4], const float (&w)[4],
                                          int cnt, float (&acc0)[V], float (&acc1)[V]) {
    uint4 u[4][2];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        u[q][0] = u[q][1] = make_uint4(0, 0, 0, 0);
        if (q < cnt) {
            const uint4 *src4 = reinterpret_cast<const uint4 *>(Y + static_cast<int64_t>(r[q]) * d);
            if (has0) u[q][0] = __ldg(src4 + p0);
            if (has1) u[q][1] = __ldg(src4 + p1);
        }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        if (q >= cnt) continue;
        float a[V], b[V];
        piece_to_f(u[q][0], a);
        piece_to_f(u[q][1], b);
#pragma unroll
        for (int i = 0; i < V; ++i) {
            acc0[i] = fmaf(w[q], a[i], acc0[i]);
            acc1[i] = fmaf(w[q], b[i], acc1[i]);
        }
    }
}

// One warp per token: y_t = sum over its kept experts, in increasing e, of
// w Y[row]; fp32 accumulation, one rounding to the output type.  Each lane
// owns two 16-byte pieces of every 64-piece span of the row.  The row map
// of 256 experts (and the kept ones' weights) is read at once; the kept
// experts are then found 32 at a time by a ballot and queued (warp-uniform
// registers), and every four queued experts' rows are requested together
// before they are summed in order.
template <typename TY>
__global__ void __launch_bounds__(256) bal_combine(const TY *__restrict__ Y,
                                                   const int32_t *__restrict__ rowmap,
                                                   const float *__restrict__ row_weight, int64_t T,
                                                   int n, int d, TY *__restrict__ y) {
    constexpr int V = 16 / static_cast<int>(sizeof(TY));   // elements per 16-byte piece
    const int lane = threadIdx.x & 31;
    const int64_t t = static_cast<int64_t>(blockIdx.x) * 8 + threadIdx.x / 32;
    if (t >= T) return;
    const int32_t *rm = rowmap + t * n;
    const int pieces = d / V;
    for (int p0 = lane; p0 - lane < pieces; p0 += 64) {
        const int p1 = p0 + 32;
        const bool has0 = p0 < pieces, has1 = p1 < pieces;
        float acc0[V], acc1[V];
#pragma unroll
        for (int i = 0; i < V; ++i) acc0[i] = acc1[i] = 0.0f;
        int32_t qr[4] = {-1, -1, -1, -1};
        float qw[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        int qn = 0;
        for (int eb0 = 0; eb0 < n; eb0 += 256) {
            // 256 experts' row-map entries, then the kept ones' weights, all
            // requested before the first ballot
            int32_t mr[8];
            float mw[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int e = eb0 + 32 * i + lane;
                mr[i] = e < n ? __ldg(rm + e) : -1;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) mw[i] = mr[i] >= 0 ? __ldg(row_weight + mr[i]) : 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                unsigned bits = __ballot_sync(0xffffffffu, mr[i] >= 0);
                while (bits) {   // warp-uniform
                    const int src = __ffs(bits) - 1;
                    bits &= bits - 1;
                    const int32_t rr = __shfl_sync(0xffffffffu, mr[i], src);
                    const float ww = __shfl_sync(0xffffffffu, mw[i], src);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        if (q == qn) {
                            qr[q] = rr;
                            qw[q] = ww;
                        }
                    if (++qn == 4) {
                        bal_flush<TY, V>(Y, d, p0, p1, has0, has1, qr, qw, 4, acc0, acc1);
                        qn = 0;
                    }
                }
            }
        }
        if (qn) bal_flush<TY, V>(Y, d, p0, p1, has0, has1, qr, qw, qn, acc0, acc1);
        uint4 *dst = reinterpret_cast<uint4 *>(y + t * d);
        if (has0) dst[p0] = piece_from_f(acc0);
        if (has1) dst[p1] = piece_from_f(acc1);
    }
}

}  // namespace

size_t balanced_workspace_bytes(const moe_shape &s, int64_t rows_cap) {
    return bal_layout(s, rows_cap).total;
}

cudaError_t launch_forward_balanced(const moe_shape &s, const void *x, const float *Wg,
                                    const float *Wn, const float *bg, const float *eps,
                                    const float *thr, int64_t rows_cap, const void *W1,
                                    const float *b1, const void *W2, const float *b2, void *y,
                                    int32_t *counts, float *W, void *ws, cudaStream_t st) {
    const BalLayout B = bal_layout(s, rows_cap);
    const WsLayout &L = B.fwd;
    const int64_t T = s.T;
    const int n = s.n, d = s.d;
    int32_t *err = ws_ptr<int32_t>(ws, 0);
    float *H = ws_ptr<float>(ws, B.H);
    int32_t *rowmap = ws_ptr<int32_t>(ws, B.rowmap);
    int32_t *row_token = ws_ptr<int32_t>(ws, B.row_token);
    float *row_weight = ws_ptr<float>(ws, B.row_weight);
    int32_t *offsets = ws_ptr<int32_t>(ws, L.offsets);
    const float *eps_used = s.noisy ? eps : nullptr;
    const dim3 sgrid(static_cast<unsigned>((T + kBT - 1) / kBT), static_cast<unsigned>((n + kBT - 1) / kBT));
    const float *noisy_sc = nullptr;
    if (bal_tc_scores(s) && eps_used) {
        float *sN = ws_ptr<float>(ws, B.sN);
        cudaError_t ge = launch_gate_tc_load(s, x, Wg, Wn, bg, eps_used, ws_ptr<int32_t>(ws, B.gidx),
                                             ws_ptr<float>(ws, B.gG), H, sN, ws_ptr<float>(ws, B.vk),
                                             ws, L, st);
        if (ge != cudaSuccess) return ge;
        noisy_sc = sN;   // H = c + eps * s is formed by the transpose
    } else if (s.dtype == MOE_BF16)
        bal_scores<__nv_bfloat16><<<sgrid, 256, 0, st>>>(static_cast<const __nv_bfloat16 *>(x), Wg, Wn,
                                                        bg, eps_used, T, d, n, H);
    else
        bal_scores<float><<<sgrid, 256, 0, st>>>(static_cast<const float *>(x), Wg, Wn, bg, eps_used,
                                                 T, d, n, H);
    float *HT = ws_ptr<float>(ws, B.HT);
    bal_transpose<<<dim3(static_cast<unsigned>((T + 31) / 32), static_cast<unsigned>((n + 31) / 32)),
                    dim3(32, 8), 0, st>>>(H, noisy_sc, noisy_sc ? eps_used : nullptr, T, n, HT,
                                          rowmap);
    const int64_t m = thr ? 0 : static_cast<int64_t>(s.k) * T / n;
    bal_count<<<n, 1024, 0, st>>>(HT, T, n, m, thr, ws_ptr<uint32_t>(ws, B.kstar),
                                  ws_ptr<int32_t>(ws, B.quota), ws_ptr<int32_t>(ws, B.cnt));
    bal_scan<<<1, 1024, 0, st>>>(ws_ptr<int32_t>(ws, B.cnt), n, rows_cap, offsets, counts, err);
    bal_write<<<n, 1024, 0, st>>>(HT, T, n, thr, ws_ptr<uint32_t>(ws, B.kstar),
                                  ws_ptr<int32_t>(ws, B.quota), offsets, row_token, rowmap);
    bal_weights<<<static_cast<unsigned>((T + 7) / 8), 256, 0, st>>>(H, rowmap, T, n, row_weight, W);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    void *Yrows = ws_ptr<void>(ws, L.yslot);
    e = launch_expert_ffn(B.ffn, x, row_token, offsets, W1, b1, W2, b2, Yrows, ws, L, st);
    if (e != cudaSuccess) return e;
    if (s.dtype == MOE_BF16)
        bal_combine<__nv_bfloat16><<<static_cast<unsigned>((T + 7) / 8), 256, 0, st>>>(
            static_cast<const __nv_bfloat16 *>(Yrows), rowmap, row_weight, T, n, d,
            static_cast<__nv_bfloat16 *>(y));
    else
        bal_combine<float><<<static_cast<unsigned>((T + 7) / 8), 256, 0, st>>>(
            static_cast<const float *>(Yrows), rowmap, row_weight, T, n, d, static_cast<float *>(y));
    return cudaGetLastError();
}

}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_balanced_workspace_bytes(const moe_shape *s, int64_t rows_cap) {
    if (moe_validate(s) != MOE_OK || s->groups != 0 || rows_cap < 0) return 0;
    if (static_cast<int64_t>(s->T) * s->n > MOE_MAX_SLOTS || rows_cap > MOE_MAX_SLOTS) return 0;
    return balanced_workspace_bytes(*s, rows_cap);
}

moe_status moe_forward_balanced(const moe_shape *s, const void *x, const float *Wg, const float *Wn,
                                const float *bg, const float *eps, const float *thr,
                                int64_t rows_cap, const void *W1, const float *b1, const void *W2,
                                const float *b2, void *y, int32_t *counts, float *W, void *ws,
                                size_t ws_bytes, void *stream) {
    moe_status v = moe_validate(s);
    if (v != MOE_OK) return v;
    if (s->groups != 0) return MOE_ERR_UNSUPPORTED;
    if (rows_cap < 0 || rows_cap > MOE_MAX_SLOTS || static_cast<int64_t>(s->T) * s->n > MOE_MAX_SLOTS)
        return MOE_ERR_UNSUPPORTED;
    auto al = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    auto req = [&](const void *p) { return p != nullptr && al(p); };
    auto opt = [&](const void *p) { return p == nullptr || al(p); };
    if (!req(Wg) || !req(W1) || !req(W2) || !req(counts) || !opt(bg) || !opt(b1) || !opt(b2) ||
        !opt(Wn) || !opt(eps) || !opt(thr) || !opt(W))
        return MOE_ERR_INVALID_ARG;
    if (s->T > 0 && (!req(x) || !req(y))) return MOE_ERR_INVALID_ARG;
    if (s->T > 0 && s->noisy && (!req(Wn) || !req(eps))) return MOE_ERR_INVALID_ARG;
    // batchwise needs room for m rows of every expert
    if (!thr && rows_cap < static_cast<int64_t>(s->k) * s->T / s->n * s->n) return MOE_ERR_INVALID_ARG;
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 ||
        ws_bytes < balanced_workspace_bytes(*s, rows_cap))
        return MOE_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (s->T == 0) {
        cudaMemsetAsync(counts, 0, sizeof(int32_t) * s->n, st);
        return cuda_to_status(cudaGetLastError());
    }
    const cudaError_t e = launch_forward_balanced(*s, x, Wg, Wn, bg, eps, thr, rows_cap, W1, b1, W2, b2,
                                                  y, counts, W, ws, st);
    return cuda_to_status(e);
}

}  // extern "C"

// backward_tc.h -- launchers of the tensor-core pieces of the bf16 backward
// pass (backward_tc.cu).  Internal to the library, not part of the ABI.
#pragma once

#include "moe_launch.h"

namespace moe {

// out[e][i, j] = sum over the 64-wide column blocks kblk[e] .. kblk[e+1]-1 of
// PT[i, :] . QT[j, :]  (PT [M, Kcap], QT [N, Kcap] bf16, K contiguous; out
// [n, M, N] fp32; zeros for an expert with no blocks).  M % 128 == 0,
// N % 128 == 0, Kcap % 64 == 0.
cudaError_t launch_wgrad_tc(const __nv_bfloat16 *PT, int M, const __nv_bfloat16 *QT, int N,
                            int64_t Kcap, const int32_t *kblk, int n, float *out, int32_t *err,
                            cudaStream_t st);

// out[e] = in[e]^T for n bf16 matrices [R, C] (R, C multiples of 64).
cudaError_t launch_transpose_experts(const __nv_bfloat16 *in, int n, int R, int C,
                                     __nv_bfloat16 *out, cudaStream_t st);

// dE[r] = bf16(G[perm[r]] * dy[perm[r] / k]) for r < S (d a multiple of 8).
cudaError_t launch_rows_scaled(const __nv_bfloat16 *dy, const float *G, const int32_t *perm,
                               int64_t S, int d, int k, __nv_bfloat16 *dE, int32_t *err,
                               cudaStream_t st);

// x = 0 where hid <= 0, elementwise over `count` bf16 values (a multiple of 8).
cudaError_t launch_relu_mask(__nv_bfloat16 *x, const __nv_bfloat16 *hid, int64_t count,
                             cudaStream_t st);

// Transposed, per-expert padded copy of expert-ordered rows in [S, M]: column
// block kblk[e] + b of out [M, Kcap] holds rows 64b .. 64b+63 of expert e
// (zeros past its last row).  kblk = tile table of 64-row blocks.
cudaError_t launch_transpose_pad(const __nv_bfloat16 *in, int M, const int32_t *offsets,
                                 const int32_t *kblk, int n, int64_t S, int64_t Kcap,
                                 __nv_bfloat16 *out, cudaStream_t st);

}  // namespace moe

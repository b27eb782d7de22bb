// selftest.cu -- exercises the library's bounded wait until it runs out.
//
// Every spin in the tensor-core kernels goes through mbar_wait_bounded: after
// kWaitLimitNs (2 s) it records MOE_ERR_TIMEOUT in the workspace's error word,
// raises the CTA's abort flag and returns, so a stalled pipeline ends the
// kernel with a status the host reads instead of hanging the GPU.  This
// kernel waits, through that same helper, on an mbarrier that nothing ever
// arrives at; the wait runs out and the kernel returns.  Nothing faults or
// traps, and the context stays usable.
#include "moe_device.cuh"
#include "moe_launch.h"

namespace moe {
namespace {

constexpr int32_t kSiteSelftest = 50;

__global__ void selftest_wait(int32_t *err) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int32_t abort_flag;
    if (threadIdx.x != 0) return;
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
    // phase 0 never completes: no thread arrives
    mbar_wait_bounded(smem_u32(&bar), 0, &abort_flag, err, kSiteSelftest);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

moe_status moe_selftest_timeout(void *ws, size_t ws_bytes, void *stream) {
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || ws_bytes < kWsHeaderBytes)
        return MOE_ERR_WORKSPACE;
    selftest_wait<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<int32_t *>(ws));
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // extern "C"

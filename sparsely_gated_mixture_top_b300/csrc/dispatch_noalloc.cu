// dispatch_noalloc.cu -- moe_dispatch_noalloc: the dispatch step for callers
// that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at all, or may not hand this library a
// workspace: code that runs inside another framework's memory pool with a
// fixed budget, plug-ins loaded into a host that owns every device
// allocation, or a real-time path where an allocation could block or fail.
// This entry point runs the same routing kernels as moe_dispatch, but their
// scratch (slot ranks, per-chunk counts and importance sums, an error word)
// lives in one array with static storage in this library's device image.
// The array is created when the library's module is loaded on a device and
// stays resident on every device that loads it until the process exits.
#include "moe_device.cuh"
#include "moe_launch.h"

namespace moe {

namespace {

constexpr size_t kNoAllocScratchBytes = static_cast<size_t>(8) << 20;  // 8 MiB

// Shared by every call on a device: contents persist from call to call.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// The scratch regions moe_dispatch would take from a workspace, packed into
// the static array (header with the error word first).
WsLayout noalloc_layout(const moe_shape &s) {
    WsLayout L;
    const size_t S = static_cast<size_t>(slots(s));
    const size_t n = static_cast<size_t>(s.n);
    const size_t chunks = (S + kRouteChunk - 1) / kRouteChunk;
    size_t o = kWsHeaderBytes;
    L.local_rank = o;
    o = align_up(o + S * 4, 256);
    L.chunk = o;
    o = align_up(o + chunks * n * 4, 256);
    L.chunk_imp = o;
    o = align_up(o + chunks * n * 4, 256);
    L.imp_acc = o;
    o = align_up(o + n * 4, 256);
    L.total = o;
    return L;
}

// Device address of the static array on the current device.  Host code only
// sees a host-side stand-in for the symbol, so the address is queried, with
// the device current, on every call: the lookup is a cheap host operation
// once the module is loaded, and a fresh lookup stays right after a device
// reset (which reloads the module, possibly at another address).  The first
// call on a device may load the module there.
cudaError_t scratch_address(void **out) {
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    *out = p;
    return p ? cudaSuccess : cudaErrorInvalidSymbol;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" MOE_API moe_status moe_dispatch_noalloc(const moe_shape *s, const int32_t *idx,
                                                   const float *G, int32_t *counts,
                                                   int32_t *offsets, int32_t *perm,
                                                   int32_t *inv_perm, float *importance,
                                                   float *cv2, void *stream) {
    moe_status v = moe_validate(s);
    if (v != MOE_OK) return v;
    const auto aligned = [](const void *p) {
        return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
    };
    if (!aligned(counts) || !aligned(offsets) || !aligned(importance) || !aligned(cv2))
        return MOE_ERR_INVALID_ARG;
    if (s->T > 0 && (!aligned(idx) || !aligned(G) || !aligned(perm) || !aligned(inv_perm)))
        return MOE_ERR_INVALID_ARG;
    const WsLayout L = noalloc_layout(*s);
    if (L.total > kNoAllocScratchBytes) return MOE_ERR_UNSUPPORTED;
    void *scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // The error word must start at zero; every other region is fully written
    // before it is read within one call.
    if (cudaMemsetAsync(scratch, 0, kWsHeaderBytes, st) != cudaSuccess) return MOE_ERR_CUDA;
    return launch_dispatch(*s, idx, G, counts, offsets, perm, inv_perm, importance, cv2, scratch,
                           L, st) == cudaSuccess
               ? MOE_OK
               : MOE_ERR_CUDA;
}

// api.cu -- the C ABI declared in include/moe.h: validation of shapes and
// pointers, the workspace layout, and the launch sequence of each entry point.
// Every host-detectable error returns before anything is enqueued.
#include "moe_device.cuh"
#include "moe_launch.h"

#include <mutex>

namespace moe {

int sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (cached[dev] == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
            v = 148;
        cached[dev] = v;
    }
    return cached[dev];
}

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// NULL or misaligned required pointer -> MOE_ERR_INVALID_ARG.
bool ok_ptr(const void *p) { return p != nullptr && aligned16(p); }
// Optional pointer: NULL is fine, otherwise it must be aligned.
bool ok_opt(const void *p) { return p == nullptr || aligned16(p); }

moe_status check_ws(const moe_shape *s, const void *ws, size_t ws_bytes) {
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MOE_ERR_WORKSPACE;
    if (ws_bytes < ws_layout(*s).total) return MOE_ERR_WORKSPACE;
    return MOE_OK;
}

moe_status cuda_status(cudaError_t e) { return cuda_to_status(e); }

thread_local int32_t g_last_cuda_error = 0;

}  // namespace

moe_status cuda_to_status(cudaError_t e) {
    if (e == cudaSuccess) return MOE_OK;
    g_last_cuda_error = static_cast<int32_t>(e);
    return MOE_ERR_CUDA;
}

}  // namespace moe

using namespace moe;

extern "C" {

int32_t moe_version(void) { return 100; }

int32_t moe_last_cuda_error(void) { return g_last_cuda_error; }

const char *moe_cuda_error_name(int32_t code) {
    return cudaGetErrorName(static_cast<cudaError_t>(code));
}

const char *moe_status_string(moe_status s) {
    switch (s) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported size";
        case MOE_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case MOE_ERR_CUDA: return "CUDA error";
        case MOE_ERR_TIMEOUT: return "device wait timed out";
        case MOE_ERR_DEVICE: return "invalid data found on the device";
        default: return "unknown status";
    }
}

moe_status moe_validate(const moe_shape *s) {
    if (s == nullptr) return MOE_ERR_INVALID_ARG;
    if (s->T < 0 || s->d <= 0 || s->h <= 0 || s->n <= 0 || s->k <= 0 || s->k > s->n)
        return MOE_ERR_INVALID_ARG;
    if (s->dtype != MOE_F32 && s->dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
    if (s->noisy != 0 && s->noisy != 1) return MOE_ERR_INVALID_ARG;
    if (s->groups < 0) return MOE_ERR_INVALID_ARG;
    if (s->groups == 0) {
        if (s->k_groups != 0) return MOE_ERR_INVALID_ARG;
    } else {
        if (s->n % s->groups != 0 || s->k_groups <= 0 || s->k_groups > s->groups ||
            s->k % s->k_groups != 0 || s->k / s->k_groups > s->n / s->groups)
            return MOE_ERR_INVALID_ARG;
    }
    if (s->d % 64 != 0 || s->h % 64 != 0 || s->d > 8192 || s->h > 16384) return MOE_ERR_UNSUPPORTED;
    if (s->k > MOE_MAX_K) return MOE_ERR_UNSUPPORTED;
    if (gate_cols(*s) > MOE_MAX_COLS) return MOE_ERR_UNSUPPORTED;
    if (s->T > static_cast<int64_t>(MOE_MAX_SLOTS) / s->k) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

size_t moe_workspace_bytes(const moe_shape *s) {
    if (moe_validate(s) != MOE_OK) return 0;
    return ws_layout(*s).total;
}

moe_status moe_workspace_init(void *ws, size_t ws_bytes, void *stream) {
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || ws_bytes < kWsHeaderBytes)
        return MOE_ERR_WORKSPACE;
    return cuda_status(
        cudaMemsetAsync(ws, 0, kWsHeaderBytes, static_cast<cudaStream_t>(stream)));
}

moe_status moe_gate(const moe_shape *s, const void *x, const float *Wg, const float *Wn,
                    const float *bg, const float *eps, int32_t *idx, float *G, void *ws,
                    size_t ws_bytes, void *stream) {
    moe_status v = moe_validate(s);
    if (v != MOE_OK) return v;
    if (s->T > 0 && (!ok_ptr(x) || !ok_ptr(Wg) || !ok_ptr(idx) || !ok_ptr(G)))
        return MOE_ERR_INVALID_ARG;
    if (s->T > 0 && s->noisy && (!ok_ptr(Wn) || !ok_ptr(eps))) return MOE_ERR_INVALID_ARG;
    if (!ok_opt(bg) || !ok_opt(Wn) || !ok_opt(eps)) return MOE_ERR_INVALID_ARG;
    if ((v = check_ws(s, ws, ws_bytes)) != MOE_OK) return v;
    if (s->T == 0) return MOE_OK;
    const WsLayout L = ws_layout(*s);
    return cuda_status(launch_gate(*s, x, Wg, s->noisy ? Wn : nullptr, bg, s->noisy ? eps : nullptr,
                                   idx, G, ws, L, static_cast<cudaStream_t>(stream)));
}

moe_status moe_dispatch(const moe_shape *s, const int32_t *idx, const float *G, int32_t *counts,
                        int32_t *offsets, int32_t *perm, int32_t *inv_perm, float *importance,
                        float *cv2, void *ws, size_t ws_bytes, void *stream) {
    moe_status v = moe_validate(s);
    if (v != MOE_OK) return v;
    if (!ok_ptr(counts) || !ok_ptr(offsets) || !ok_ptr(importance) || !ok_ptr(cv2))
        return MOE_ERR_INVALID_ARG;
    if (s->T > 0 && (!ok_ptr(idx) || !ok_ptr(G) || !ok_ptr(perm) || !ok_ptr(inv_perm)))
        return MOE_ERR_INVALID_ARG;
    if ((v = check_ws(s, ws, ws_bytes)) != MOE_OK) return v;
    const WsLayout L = ws_layout(*s);
    return cuda_status(launch_dispatch(*s, idx, G, counts, offsets, perm, inv_perm, importance, cv2,
                                       ws, L, static_cast<cudaStream_t>(stream)));
}

moe_status moe_expert_ffn(const moe_shape *s, const void *x, const int32_t *perm,
                          const int32_t *offsets, const void *W1, const float *b1, const void *W2,
                          const float *b2, void *Y_slot, void *ws, size_t ws_bytes,
                          void *stream) {
    moe_status v = moe_validate(s);
    if (v != MOE_OK) return v;
    if (!ok_ptr(offsets) || !ok_ptr(W1) || !ok_ptr(W2) || !ok_opt(b1) || !ok_opt(b2))
        return MOE_ERR_INVALID_ARG;
    if (s->T > 0 && (!ok_ptr(x) || !ok_ptr(perm) || !ok_ptr(Y_slot))) return MOE_ERR_INVALID_ARG;
    if ((v = check_ws(s, ws, ws_bytes)) != MOE_OK) return v;
    const WsLayout L = ws_layout(*s);
    return cuda_status(launch_expert_ffn(*s, x, perm, offsets, W1, b1, W2, b2, Y_slot, ws, L,
                                         static_cast<cudaStream_t>(stream)));
}

moe_status moe_combine(const moe_shape *s, const void *Y_slot, const int32_t *inv_perm,
                       const float *G, void *y, void *ws, size_t ws_bytes, void *stream) {
    moe_status v = moe_validate(s);
    if (v != MOE_OK) return v;
    if (s->T > 0 && (!ok_ptr(Y_slot) || !ok_ptr(inv_perm) || !ok_ptr(G) || !ok_ptr(y)))
        return MOE_ERR_INVALID_ARG;
    if ((v = check_ws(s, ws, ws_bytes)) != MOE_OK) return v;
    return cuda_status(launch_combine(*s, Y_slot, inv_perm, G, y, ws_ptr<int32_t>(ws, 0),
                                      static_cast<cudaStream_t>(stream)));
}

moe_status moe_forward(const moe_shape *s, const void *x, const float *Wg, const float *Wn,
                       const float *bg, const float *eps, const void *W1, const float *b1,
                       const void *W2, const float *b2, void *y, float *G, int32_t *idx,
                       float *importance, float *cv2, int32_t *counts, void *ws,
                       size_t ws_bytes, void *stream) {
    moe_status v = moe_validate(s);
    if (v != MOE_OK) return v;
    if (!ok_ptr(Wg) || !ok_ptr(W1) || !ok_ptr(W2) || !ok_opt(b1) || !ok_opt(b2) || !ok_opt(bg))
        return MOE_ERR_INVALID_ARG;
    if (!ok_opt(importance) || !ok_opt(cv2) || !ok_opt(counts) || !ok_opt(Wn) || !ok_opt(eps))
        return MOE_ERR_INVALID_ARG;
    if (s->T > 0 && (!ok_ptr(x) || !ok_ptr(y) || !ok_ptr(G) || !ok_ptr(idx)))
        return MOE_ERR_INVALID_ARG;
    if (s->T > 0 && s->noisy && (!ok_ptr(Wn) || !ok_ptr(eps))) return MOE_ERR_INVALID_ARG;
    if ((v = check_ws(s, ws, ws_bytes)) != MOE_OK) return v;
    const WsLayout L = ws_layout(*s);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t *cnt = counts ? counts : ws_ptr<int32_t>(ws, L.counts);
    float *imp = importance ? importance : ws_ptr<float>(ws, L.importance);
    float *c2 = cv2 ? cv2 : ws_ptr<float>(ws, L.cv2);
    int32_t *off = ws_ptr<int32_t>(ws, L.offsets);
    int32_t *perm = ws_ptr<int32_t>(ws, L.perm);
    int32_t *inv = ws_ptr<int32_t>(ws, L.inv_perm);
    void *yslot = ws_ptr<void>(ws, L.yslot);
    cudaError_t e = cudaSuccess;
    if (s->T > 0)
        e = launch_gate(*s, x, Wg, s->noisy ? Wn : nullptr, bg, s->noisy ? eps : nullptr, idx, G,
                        ws, L, st);
    // The dispatch also gathers the x rows and builds the expert stage's
    // schedules, so the expert stage starts with its GEMMs.
    const DispatchExtras ex = dispatch_extras_for_ffn(*s, x, ws, L);
    if (e == cudaSuccess)
        e = launch_dispatch(*s, idx, G, cnt, off, perm, inv, imp, c2, ws, L, st, &ex);
    if (e == cudaSuccess)
        e = launch_expert_ffn(*s, x, perm, off, W1, b1, W2, b2, yslot, ws, L, st, true);
    if (e == cudaSuccess) e = launch_combine(*s, yslot, inv, G, y, ws_ptr<int32_t>(ws, 0), st);
    return cuda_status(e);
}

static bool load_supported(const moe_shape *s) {
    return s->groups == 0 && s->noisy == 1 && s->dtype == MOE_BF16 && s->k < MOE_MAX_K;
}

size_t moe_load_workspace_bytes(const moe_shape *s) {
    if (moe_validate(s) != MOE_OK || !load_supported(s)) return 0;
    return load_layout(*s).total;
}

moe_status moe_gate_load(const moe_shape *s, const void *x, const float *Wg, const float *Wn,
                         const float *bg, const float *eps, int32_t *idx, float *G, float *load,
                         float *load_cv2, void *ws, size_t ws_bytes, void *lws, size_t lws_bytes,
                         void *stream) {
    moe_status v = moe_validate(s);
    if (v != MOE_OK) return v;
    if (!load_supported(s)) return MOE_ERR_UNSUPPORTED;
    if (!ok_ptr(Wg) || !ok_ptr(Wn) || !ok_opt(bg) || !ok_ptr(load) || !ok_ptr(load_cv2))
        return MOE_ERR_INVALID_ARG;
    if (s->T > 0 && (!ok_ptr(x) || !ok_ptr(eps) || !ok_ptr(idx) || !ok_ptr(G)))
        return MOE_ERR_INVALID_ARG;
    if ((v = check_ws(s, ws, ws_bytes)) != MOE_OK) return v;
    const LoadLayout LL = load_layout(*s);
    if (lws == nullptr || (reinterpret_cast<uintptr_t>(lws) & 255u) != 0 || lws_bytes < LL.total)
        return MOE_ERR_WORKSPACE;
    const WsLayout L = ws_layout(*s);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    if (s->T > 0)
        e = launch_gate_tc_load(*s, x, Wg, Wn, bg, eps, idx, G, ws_ptr<float>(lws, LL.c),
                                ws_ptr<float>(lws, LL.s), ws_ptr<float>(lws, LL.vk), ws, L, st);
    if (e == cudaSuccess) e = launch_load(*s, idx, lws, LL, load, load_cv2, st);
    return cuda_status(e);
}

moe_status moe_check(void *ws, void *stream) {
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MOE_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    WsHeader h{};
    if (cudaMemcpyAsync(&h, ws, sizeof(h), cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
    if (h.err != MOE_OK) {
        if (cudaMemsetAsync(ws, 0, sizeof(h), st) != cudaSuccess) return MOE_ERR_CUDA;
        if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
    }
    return h.err;
}

}  // extern "C"

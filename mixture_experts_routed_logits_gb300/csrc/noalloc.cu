// noalloc.cu -- ts_moe_forward_noalloc: the expert half of the layer for callers that cannot
// allocate device memory.
//
// Some callers of this library cannot call cudaMalloc or use an allocator at the point where
// they run the layer: a host application that owns all device memory and hands out nothing,
// an embedding in a runtime whose allocator is not reachable from the calling thread, or code
// that must not allocate while it runs (latency-critical serving loops).  ts_moe_forward needs
// a caller-provided workspace for its route lists and intermediate activations; this entry
// point instead uses a fixed scratch array that lives in the library's own device memory.
//
// The scratch is a file-scope __device__ array of kScratchBytes (16 MiB).  Every GPU on which
// this code is loaded keeps that array until the process exits.  Host code cannot use the
// array's name as a device address (on the host it is only a stand-in symbol), so its device
// address is looked up once per device with cudaGetSymbolAddress and cached.  That lookup
// happens inside the first call on each device.
#include <cstdio>

#include "../../include/ts_moe.h"
#include "internal.h"

namespace {

ts_status record_error(int status, const char* msg) {
    return static_cast<ts_status>(tsmoe::record_error_code(status, msg));
}

constexpr size_t kScratchBytes = static_cast<size_t>(16) << 20;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

// Device address of g_scratch on the current device (looked up once per device).
cudaError_t scratch_address(void** out) {
    static void* addr[64] = {nullptr};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_scratch);
        if (e != cudaSuccess) return e;
        addr[dev] = p;
    }
    *out = addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" ts_status ts_moe_forward_noalloc(const void* x, int32_t adt, int32_t T,
                                            const ts_moe_experts* ex, const int32_t* idx,
                                            const float* w, int32_t k,
                                            const ts_moe_experts* shared, void* y, float* y_f32,
                                            void* stream) {
    char msg[256];
    if (!ex) return record_error(TS_ERR_INVALID_ARG, "ts_moe_forward_noalloc: experts is NULL");
    const size_t need = ts_moe_workspace_size(T, k, ex, shared);
    if (need == 0 && T > 0)
        return record_error(TS_ERR_INVALID_ARG,
                                   "ts_moe_forward_noalloc: invalid T, k or expert shapes");
    if (need > kScratchBytes) {
        snprintf(msg, sizeof(msg),
                 "ts_moe_forward_noalloc: this call needs %zu bytes of scratch but the library's "
                 "static scratch holds %zu; use ts_moe_forward with a workspace",
                 need, kScratchBytes);
        return record_error(TS_ERR_WORKSPACE, msg);
    }
    if (T == 0)
        return ts_moe_forward(x, adt, T, ex, idx, w, k, shared, y, y_f32, nullptr, 0, stream);
    void* scratch = nullptr;
    cudaError_t e = scratch_address(&scratch);
    // the first word of the scratch is the device status word: start every call from zero
    if (e == cudaSuccess) e = cudaMemsetAsync(scratch, 0, 256, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        snprintf(msg, sizeof(msg), "ts_moe_forward_noalloc: %s (%s)", cudaGetErrorName(e),
                 cudaGetErrorString(e));
        (void)cudaGetLastError();
        return record_error(TS_ERR_CUDA, msg);
    }
    return ts_moe_forward(x, adt, T, ex, idx, w, k, shared, y, y_f32, scratch, kScratchBytes,
                          stream);
}

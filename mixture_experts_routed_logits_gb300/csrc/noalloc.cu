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
// address is looked up with cudaGetSymbolAddress, with the device current, and cached per
// device.  The cache entry remembers the id of the CUDA context it was looked up in: a device
// reset destroys that context (and the module's copy of the array with it), and the next call
// finds a new context id and looks the address up again.  The cache is filled under a mutex,
// so host threads may call concurrently (their GPU work still races, see ts_moe.h).
#include <cuda.h>

#include <cstdio>
#include <mutex>

#include "../../include/ts_moe.h"
#include "internal.h"

namespace {

ts_status record_error(int status, const char* msg) {
    return static_cast<ts_status>(tsmoe::record_error_code(status, msg));
}

constexpr size_t kScratchBytes = static_cast<size_t>(16) << 20;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

// Id of the calling thread's current CUDA context (0 if none is current or the driver cannot
// say), through the driver entry points the runtime hands out.
unsigned long long current_context_id() {
    using GetCurrent = CUresult (*)(CUcontext*);
    using GetId = CUresult (*)(CUcontext, unsigned long long*);
    static GetCurrent get_current = nullptr;
    static GetId get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrent>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetId>(p);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// Device address of g_scratch on the current device, in the current context.
cudaError_t scratch_address(void** out) {
    struct Slot { unsigned long long ctx; void* addr; };
    static Slot slots[64];
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    const unsigned long long ctx = current_context_id();
    if (ctx != 0 && slots[dev].ctx == ctx && slots[dev].addr) {
        *out = slots[dev].addr;
        return cudaSuccess;
    }
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);      // makes the device's context current if needed
    if (e != cudaSuccess) return e;
    slots[dev].ctx = current_context_id();
    slots[dev].addr = p;
    *out = p;
    return cudaSuccess;
}

ts_status cuda_error(const char* what, cudaError_t e) {
    char msg[256];
    snprintf(msg, sizeof(msg), "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
    (void)cudaGetLastError();
    return record_error(TS_ERR_CUDA, msg);
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
    if (e != cudaSuccess) return cuda_error("ts_moe_forward_noalloc", e);
    return ts_moe_forward(x, adt, T, ex, idx, w, k, shared, y, y_f32, scratch, kScratchBytes,
                          stream);
}

// The status word of the scratch (its first int) is where the kernels of the last
// ts_moe_forward_noalloc call on this device reported a device-side failure.
extern "C" ts_status ts_moe_noalloc_device_status(int32_t* code, void* stream) {
    if (!code) return record_error(TS_ERR_INVALID_ARG, "ts_moe_noalloc_device_status: code is NULL");
    void* scratch = nullptr;
    cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess) return cuda_error("ts_moe_noalloc_device_status", e);
    return ts_moe_device_status(scratch, code, stream);
}

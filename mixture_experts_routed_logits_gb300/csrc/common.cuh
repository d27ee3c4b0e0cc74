// common.cuh -- device helpers shared by the ts_moe kernels (sm_103a).
//
// Inline PTX below is written from the public PTX ISA: mbarrier, cp.async.bulk (the
// bulk-copy engine behind TMA), mma.sync m16n8k16, griddepcontrol.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace tsmoe {

// Raises a kernel's dynamic shared-memory limit once per device (to `bytes` or more), so that
// launches made later -- e.g. while a stream is being captured into a graph -- need no
// attribute call.
template <typename K>
inline cudaError_t ensure_smem(K kernel, size_t bytes) {
    // one slot per (kernel, device); the table is tiny and filled on first use
    struct Slot { const void* fn; int dev; int bytes; };
    static Slot table[64];
    static int used = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const void* fn = reinterpret_cast<const void*>(kernel);
    for (int i = 0; i < used; ++i)
        if (table[i].fn == fn && table[i].dev == dev && table[i].bytes >= static_cast<int>(bytes))
            return cudaSuccess;
    // raise the limit once to the most this kernel can use (opt-in maximum minus its static
    // shared memory), so that later, larger requests need no further attribute call
    cudaFuncAttributes fa;
    int optin = 0;
    e = cudaFuncGetAttributes(&fa, kernel);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) { (void)cudaGetLastError(); return e; }
    const int want = optin - static_cast<int>(fa.sharedSizeBytes);
    if (static_cast<int>(bytes) > want) return cudaErrorInvalidValue;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, want);
    if (e != cudaSuccess) { (void)cudaGetLastError(); return e; }
    if (used < 64) table[used++] = Slot{fn, dev, want};
    return e;
}

// ------------------------------------------------------------------------------------------
// device status word: the first int of every workspace.  Kernels that give up waiting or
// detect a bad index write a TS_ERR_* code here (first writer wins) and skip their work.
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ void report_error(int* status, int code) {
    if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------------------------------
// mbarrier (shared::cta) helpers
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait: gives up after ~2^31 SM clocks (about a second) and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (clock64() - t0 > (1ll << 31)) return false;
    }
}

// 1-D bulk copy global -> shared, completion signalled on `bar` (complete_tx bytes).
// dst/src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Named barrier over `nthreads` threads (multiple of 32) with id `id` (1..15).
__device__ __forceinline__ int ld_acquire_gpu_s32(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void named_bar(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Programmatic dependent launch controls (no-ops when the launch did not enable PDL).
__device__ __forceinline__ void pdl_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launch with programmatic dependent launch allowed: the kernel may be scheduled while the
// previous kernel of the stream is still running (hiding the launch gap); it calls pdl_wait()
// before it reads anything an earlier kernel wrote.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// ------------------------------------------------------------------------------------------
// tensor-core fragments (legacy warp-level mma; used by the streaming GEMV path, where the
// tensor pipe only has to keep pace with HBM)
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ void mma_f16_16816(float d[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_bf16_16816(float d[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ------------------------------------------------------------------------------------------
// 16-bit conversions
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ float adt_load(const uint16_t* p, int adt) {
    const uint16_t b = *p;
    return adt == 0 ? __half2float(__ushort_as_half(b)) : __bfloat162float(__ushort_as_bfloat16(b));
}
__device__ __forceinline__ float adt_bits_to_float(uint16_t b, int adt) {
    return adt == 0 ? __half2float(__ushort_as_half(b)) : __bfloat162float(__ushort_as_bfloat16(b));
}
__device__ __forceinline__ uint16_t float_to_adt_bits(float v, int adt) {
    return adt == 0 ? __half_as_ushort(__float2half_rn(v))
                    : __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

// e8m0 block scale 2^(b-127) as f32 (b == 0 is the subnormal 2^-127).
__device__ __forceinline__ float e8m0_to_float(uint32_t b) {
    return b ? __uint_as_float(b << 23) : __uint_as_float(0x00400000u);
}

// Two e2m1 codes (low nibble -> .x, high nibble -> .y) to f16x2, via the CUDA fp4 header.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
    __half2_raw r = __nv_cvt_fp4x2_to_halfraw2(static_cast<__nv_fp4x2_storage_t>(byte & 0xFF),
                                                __NV_E2M1);
    return static_cast<uint32_t>(r.x) | (static_cast<uint32_t>(r.y) << 16);
}

// Four bytes of e2m1 pairs (byte j -> out[j]: low nibble in .x, high nibble in .y) with the
// hardware converter, from one 32-bit register.
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t out[4]) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(out[0]), "=r"(out[1]), "=r"(out[2]), "=r"(out[3])
        : "r"(w));
}

// Unsigned 4-bit codes to f16x2 via the 1024-offset trick: (0x6400 | q) is the f16 1024+q.
// Returns the pair (nibble at bit s, nibble at bit s+16) as f16 values q, exactly.
__device__ __forceinline__ uint32_t u4pair_to_f16x2(uint32_t w, int s) {
    const uint32_t t = ((w >> s) & 0x000F000Fu) | 0x64006400u;
    __half2 h = *reinterpret_cast<const __half2*>(&t);
    const __half2 k1024 = __halves2half2(__ushort_as_half(0x6400), __ushort_as_half(0x6400));
    h = __hsub2(h, k1024);
    return *reinterpret_cast<uint32_t*>(&h);
}

// Gated-FFN activations in f32: SiLU-GLU, gelu-tanh-GLU, and the clamped SwiGLU of gpt-oss
// (biases already added to g and u; the clamp comes before the gate).
__device__ __forceinline__ float act_fn(int act, float g, float u, float limit, float alpha) {
    if (act == ACT_SILU) return g / (1.0f + expf(-g)) * u;
    if (act == ACT_GELU) {
        const float c = 0.7978845608028654f;   // sqrt(2/pi)
        return 0.5f * g * (1.0f + tanhf(c * (g + 0.044715f * g * g * g))) * u;
    }
    g = fminf(g, limit);
    u = fminf(fmaxf(u, -limit), limit);
    return g / (1.0f + expf(-alpha * g)) * (u + 1.0f);
}

__device__ __forceinline__ float warp_sum_xor(float v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Fixed-order f32 dot product of a warp: lane l sums fmaf(a[l+32j], b[l+32j]) over j, then an
// xor butterfly 16, 8, 4, 2, 1.  Every lane returns the same bits.
template <typename LoadB>
__device__ __forceinline__ float warp_dot_fixed(const float* a, LoadB loadb, int H, int lane) {
    float p = 0.0f;
#pragma unroll 8
    for (int j = lane; j < H; j += 32) p = __fmaf_rn(a[j], loadb(j), p);
    return warp_sum_xor(p);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

}  // namespace tsmoe

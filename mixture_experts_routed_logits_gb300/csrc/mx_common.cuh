// mx_common.cuh -- helpers of the block-scaled (MXFP4 x split-bf16) tensor-core kernels:
// tcgen05.mma kind::mxf8f6f4 with e8m0 block scales in TMEM, the scale-atom copy into TMEM, TMEM
// loads, and the exact two-term e4m3 split of bf16 values.  Inline PTX written from the public
// PTX ISA; the descriptor fields and the TMEM scale layout were checked on GB300 against a host
// computation (exact match for N = 16 .. 256).
#pragma once

#include <cuda_fp8.h>

#include "tc_common.cuh"

namespace tsmoe {

__device__ __forceinline__ void umma_mx(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t tsfa, uint32_t tsfb, uint32_t accum) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
        ::"r"(tmem_d), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(tsfa), "r"(tsfb), "r"(accum)
        : "memory");
}

// 32 rows x 16 bytes of shared memory (no swizzle, rows contiguous) into TMEM lanes 0-31,
// columns +0..3, replicated to the four lane quarters
__device__ __forceinline__ void tmem_cp_atom(uint32_t taddr, const void* src) {
    uint64_t d = static_cast<uint64_t>((smem_u32(src) & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(128 >> 4) << 16;      // leading byte offset
    d |= static_cast<uint64_t>(128 >> 4) << 32;      // stride byte offset: 8-row groups
    d |= static_cast<uint64_t>(1) << 46;
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(d) : "memory");
}

// Instruction descriptor, kind::mxf8f6f4: A e2m1, B e4m3, both K-major, e8m0 scales, M = 128.
__device__ __forceinline__ uint32_t idesc_mx(int N, int sf_id) {
    return (static_cast<uint32_t>(sf_id) << 4) | (5u << 7) | (0u << 10) |
           (static_cast<uint32_t>(N >> 3) << 17) | (1u << 23) | ((128u >> 4) << 24) |
           (static_cast<uint32_t>(sf_id) << 29);
}

__device__ __forceinline__ void tmem_ld8x4(uint32_t t0, uint32_t t1, uint32_t t2, uint32_t t3,
                                           float a[8], float b[8], float c[8], float d[8]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%32];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%8,%9,%10,%11,%12,%13,%14,%15}, [%33];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%16,%17,%18,%19,%20,%21,%22,%23}, [%34];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%24,%25,%26,%27,%28,%29,%30,%31}, [%35];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(t0), "r"(t1), "r"(t2), "r"(t3)
        : "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        a[i] = __uint_as_float(r[i]);
        b[i] = __uint_as_float(r[8 + i]);
        c[i] = __uint_as_float(r[16 + i]);
        d[i] = __uint_as_float(r[24 + i]);
    }
}

// Block scale exponent s of a 32-block with max |v| = amax: amax / 2^s in [128, 256), held in
// [-123, 120] so that 2^s and 2^(s-4) are e8m0 values and 2^-s a normal f32.
__device__ __forceinline__ int mx_scale_exp(float amax) {
    if (!(amax > 0.0f)) return 0;
    const int e = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu) - 127;
    return max(-123, min(120, e - 7));
}

// v / 2^s -> (t1, t2) e4m3 codes with v / 2^s = t1 + t2 / 16 (see the file header).
__device__ __forceinline__ void mx_split2(float a, float b, uint32_t& t1, uint32_t& t2) {
    const __nv_fp8x2_storage_t q1 = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
    const __half2_raw h1 = __nv_cvt_fp8x2_to_halfraw2(q1, __NV_E4M3);
    const float ra = __fmul_rn(__fsub_rn(a, __half2float(__ushort_as_half(h1.x))), 16.0f);
    const float rb = __fmul_rn(__fsub_rn(b, __half2float(__ushort_as_half(h1.y))), 16.0f);
    const __nv_fp8x2_storage_t q2 = __nv_cvt_float2_to_fp8x2(make_float2(ra, rb), __NV_SATFINITE, __NV_E4M3);
    t1 = q1;
    t2 = q2;
}

}  // namespace tsmoe

// tail.cu -- the Gemma sandwich tail that follows the routed phase 2.
//
// Source page (docs.rs, turbospark-runtime 0.3.0): Gemma-4 batched routed prefill
// (src/families/gemma4/moe_batch.rs), the per-token tail encoded on the same command buffer after
// the fused phase 2: rms_norm_bf16w of the routed output with post_feedforward_layernorm_2 (in
// place), residual_add into the dense branch h1, rms_norm_bf16w of h1 with
// post_feedforward_layernorm, residual_add into the residual stream x, scalar_mul of x by the
// layer scalar.  Every buffer is 16-bit, so each step rounds to the activation type; the weight
// multiply reads plainly as v * r * w, and the sum of squares takes the fixed order of the
// pre-routing RMSNorm (lane l: fmaf over j, then the xor butterfly), so results are bit-exact
// against the oracle.
#include "common.cuh"

namespace tsmoe {

namespace {

constexpr int kTailThreads = 1024;
constexpr int kTailPer = kTailMaxH / kTailThreads;     // elements per thread at most (8)

// One CTA per token row.  Every thread loads all it needs (its elements of y, h1, x and of the
// two weight rows) before any arithmetic, so a row costs one memory round trip; the row under
// normalisation sits in shared memory as f32 for warp 0's fixed-order sum of squares.
__global__ void __launch_bounds__(kTailThreads) gemma_tail_kernel(TailArgs a) {
    __shared__ float v[kTailMaxH];
    __shared__ float rs;
    pdl_wait();                 // y comes from the previous kernel
    pdl_launch_dependents();
    const int t = blockIdx.x;
    if (t >= a.T) return;
    const int H = a.H, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint16_t* y = a.y + static_cast<size_t>(t) * H;
    uint16_t* h1 = a.h1 + static_cast<size_t>(t) * H;
    uint16_t* x = a.x + static_cast<size_t>(t) * H;
    uint16_t yv[kTailPer], hv[kTailPer], xv[kTailPer], w2v[kTailPer], w1v[kTailPer];
#pragma unroll
    for (int i = 0; i < kTailPer; ++i) {
        const int j = threadIdx.x + i * kTailThreads;
        if (j < H) {
            yv[i] = y[j];
            hv[i] = h1[j];
            xv[i] = x[j];
            w2v[i] = a.w_post2[j];
            w1v[i] = a.w_post[j];
        }
    }
    // r = 1/sqrt(mean(v^2) + eps) of the staged row, by warp 0, for every thread
    auto rscale = [&]() {
        __syncthreads();
        if (warp == 0) {
            const float ss = warp_dot_fixed(v, [&](int j) { return v[j]; }, H, lane);
            const float ms = __fdiv_rn(ss, static_cast<float>(H));
            if (lane == 0) rs = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, a.eps)));
        }
        __syncthreads();
        return rs;
    };
    auto wnorm = [&](float vj, float r, uint16_t w) {      // adt((v * r) * w)
        return float_to_adt_bits(__fmul_rn(__fmul_rn(vj, r), __bfloat162float(__ushort_as_bfloat16(w))), a.adt);
    };

#pragma unroll
    for (int i = 0; i < kTailPer; ++i) {
        const int j = threadIdx.x + i * kTailThreads;
        if (j < H) v[j] = adt_bits_to_float(yv[i], a.adt);
    }
    const float r2 = rscale();
#pragma unroll
    for (int i = 0; i < kTailPer; ++i) {
        const int j = threadIdx.x + i * kTailThreads;
        if (j >= H) continue;
        const uint16_t yb = wnorm(v[j], r2, w2v[i]);
        y[j] = yb;
        const uint16_t hb = float_to_adt_bits(
            __fadd_rn(adt_bits_to_float(hv[i], a.adt), adt_bits_to_float(yb, a.adt)), a.adt);
        h1[j] = hb;
        hv[i] = hb;
    }
#pragma unroll
    for (int i = 0; i < kTailPer; ++i) {
        const int j = threadIdx.x + i * kTailThreads;
        if (j < H) v[j] = adt_bits_to_float(hv[i], a.adt);
    }
    const float r1 = rscale();
#pragma unroll
    for (int i = 0; i < kTailPer; ++i) {
        const int j = threadIdx.x + i * kTailThreads;
        if (j >= H) continue;
        const uint16_t fb = wnorm(v[j], r1, w1v[i]);
        const uint16_t xb = float_to_adt_bits(
            __fadd_rn(adt_bits_to_float(xv[i], a.adt), adt_bits_to_float(fb, a.adt)), a.adt);
        x[j] = float_to_adt_bits(__fmul_rn(adt_bits_to_float(xb, a.adt), a.layer_scalar), a.adt);
    }
}

}  // namespace

cudaError_t launch_gemma_tail(const TailArgs& a, cudaStream_t s) {
    if (a.T <= 0) return cudaSuccess;
    return launch_pdl(gemma_tail_kernel, dim3(a.T), dim3(kTailThreads), 0, s, a);
}

}  // namespace tsmoe

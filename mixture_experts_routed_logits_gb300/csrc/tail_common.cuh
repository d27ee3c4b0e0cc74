// tail_common.cuh -- the Gemma sandwich tail of one token row, shared by the tail launch
// (tail.cu) and the GEMV phase 2 that runs it inside its fused combine (gemv.cu).
//
// Source page (docs.rs, turbospark-runtime 0.3.0): Gemma-4 batched routed prefill
// (src/families/gemma4/moe_batch.rs), the per-token tail after the fused phase 2:
// rms_norm_bf16w of the routed output with post_feedforward_layernorm_2 (in place),
// residual_add into the dense branch h1, rms_norm_bf16w of h1 with post_feedforward_layernorm,
// residual_add into the residual stream x, scalar_mul of x by the layer scalar.  Every buffer is
// 16-bit, so each step rounds to the activation type; the weight multiply reads plainly as
// v * r * w, and the sum of squares takes the fixed order of the pre-routing RMSNorm (lane l:
// fmaf over j, then the xor butterfly), so results are bit-exact against the oracle.
#pragma once
#include "common.cuh"

namespace tsmoe {

// Tail of the nb token rows t0 .. t0 + nb - 1 by nthr threads (this one is tix; nthr >= 32 nb,
// warp w < nb of them takes the sums of squares of row t0 + w).  v: shared f32 [nb][H]; rs: shared
// f32 [nb]; sync(): a barrier over the nthr threads.  Ends with a barrier, so v and rs may be
// reused at once.
template <typename Sync>
__device__ __forceinline__ void gemma_tail_rows(const TailArgs& a, int t0, int nb, float* v, float* rs,
                                                int tix, int nthr, Sync sync) {
    const int H = a.H, lane = tix & 31, w = tix >> 5, n = nb * H;
    const size_t base = static_cast<size_t>(t0) * H;
    // r = 1/sqrt(mean(v^2) + eps) of every staged row
    auto rscale = [&]() {
        sync();
        if (w < nb) {
            const float* vr = v + static_cast<size_t>(w) * H;
            const float ss = warp_dot_fixed(vr, [&](int j) { return vr[j]; }, H, lane);
            const float ms = __fdiv_rn(ss, static_cast<float>(H));
            if (lane == 0) rs[w] = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, a.eps)));
        }
        sync();
    };
    auto wnorm = [&](float vj, float r, uint16_t wt) {      // adt((v * r) * w)
        return float_to_adt_bits(__fmul_rn(__fmul_rn(vj, r), __bfloat162float(__ushort_as_bfloat16(wt))), a.adt);
    };
#pragma unroll 4
    for (int i = tix; i < n; i += nthr) v[i] = adt_bits_to_float(__ldcg(a.y + base + i), a.adt);
    rscale();
#pragma unroll 4
    for (int i = tix; i < n; i += nthr) {
        const int j = i % H;
        const uint16_t yb = wnorm(v[i], rs[i / H], a.w_post2[j]);
        a.y[base + i] = yb;
        const uint16_t hb = float_to_adt_bits(
            __fadd_rn(adt_bits_to_float(a.h1[base + i], a.adt), adt_bits_to_float(yb, a.adt)), a.adt);
        a.h1[base + i] = hb;
        v[i] = adt_bits_to_float(hb, a.adt);
    }
    rscale();
#pragma unroll 4
    for (int i = tix; i < n; i += nthr) {
        const int j = i % H;
        const uint16_t fb = wnorm(v[i], rs[i / H], a.w_post[j]);
        const uint16_t xb = float_to_adt_bits(
            __fadd_rn(adt_bits_to_float(a.x[base + i], a.adt), adt_bits_to_float(fb, a.adt)), a.adt);
        a.x[base + i] = float_to_adt_bits(__fmul_rn(adt_bits_to_float(xb, a.adt), a.layer_scalar), a.adt);
    }
    sync();
}

// As gemma_tail_rows (the same operations on the same values), 8 consecutive elements a thread
// at a time with 16-byte accesses, every load of a row batch issued up front (at most kTailV
// vectors per thread: nb * H / 8 <= kTailV * nthr): h1, x and the two weight rows first, then
// ready() (which returns once y may be read: the caller's wait for y goes there, overlapping
// those loads), then y.  y, h1, x, w_post2 and w_post 16-byte aligned, H a multiple of 8.
// Named barrier `bar` over the nthr threads.  Returns false (nothing written) if ready() did.
constexpr int kTailV = 2;
template <typename Ready>
__device__ __forceinline__ bool gemma_tail_rows_v8(const TailArgs a, int t0, int nb, float* v, float* rs,
                                                   int tix, int nthr, int bar, Ready ready) {
    const int H = a.H, lane = tix & 31, w = tix >> 5, n8 = nb * H / 8;
    const size_t base = static_cast<size_t>(t0) * H;
    const uint4* __restrict__ y4 = reinterpret_cast<const uint4*>(a.y + base);
    const uint4* __restrict__ h4 = reinterpret_cast<const uint4*>(a.h1 + base);
    const uint4* __restrict__ x4 = reinterpret_cast<const uint4*>(a.x + base);
    const uint4* __restrict__ w24 = reinterpret_cast<const uint4*>(a.w_post2);
    const uint4* __restrict__ w14 = reinterpret_cast<const uint4*>(a.w_post);
    uint4* __restrict__ yo4 = reinterpret_cast<uint4*>(a.y + base);
    uint4* __restrict__ ho4 = reinterpret_cast<uint4*>(a.h1 + base);
    uint4* __restrict__ xo4 = reinterpret_cast<uint4*>(a.x + base);
    const int adt = a.adt;
    const float eps = a.eps, scalar = a.layer_scalar;
    const int h8 = H / 8;
    uint4 yv[kTailV], hv[kTailV], xv[kTailV], w2v[kTailV], w1v[kTailV];
#pragma unroll
    for (int m = 0; m < kTailV; ++m) {
        const int q = tix + m * nthr;
        if (q < n8) {
            hv[m] = h4[q];
            xv[m] = x4[q];
            w2v[m] = w24[q % h8];
            w1v[m] = w14[q % h8];
        }
    }
    if (!ready()) return false;
#pragma unroll
    for (int m = 0; m < kTailV; ++m) {
        const int q = tix + m * nthr;
        if (q < n8) yv[m] = __ldcg(y4 + q);
    }
    auto sync = [&]() { asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(nthr) : "memory"); };
    auto rscale = [&]() {
        sync();
        if (w < nb) {
            const float* vr = v + static_cast<size_t>(w) * H;
            const float ss = warp_dot_fixed(vr, [&](int j) { return vr[j]; }, H, lane);
            const float ms = __fdiv_rn(ss, static_cast<float>(H));
            if (lane == 0) rs[w] = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
        }
        sync();
    };
    auto lo = [](uint32_t u) { return static_cast<uint16_t>(u & 0xFFFFu); };
    auto hi = [](uint32_t u) { return static_cast<uint16_t>(u >> 16); };
    auto wn = [&](float vj, float r, uint16_t wt) {      // adt((v * r) * w)
        return float_to_adt_bits(__fmul_rn(__fmul_rn(vj, r), __bfloat162float(__ushort_as_bfloat16(wt))), adt);
    };
#pragma unroll
    for (int m = 0; m < kTailV; ++m) {
        const int q = tix + m * nthr;
        if (q < n8) {
            const uint32_t u[4] = {yv[m].x, yv[m].y, yv[m].z, yv[m].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                v[8 * q + 2 * e] = adt_bits_to_float(lo(u[e]), adt);
                v[8 * q + 2 * e + 1] = adt_bits_to_float(hi(u[e]), adt);
            }
        }
    }
    rscale();
#pragma unroll
    for (int m = 0; m < kTailV; ++m) {
        const int q = tix + m * nthr;
        if (q < n8) {
            const float r = rs[(8 * q) / H];
            const uint32_t wv[4] = {w2v[m].x, w2v[m].y, w2v[m].z, w2v[m].w};
            const uint32_t hu[4] = {hv[m].x, hv[m].y, hv[m].z, hv[m].w};
            uint32_t yo[4], ho[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                uint32_t yy = 0, hh = 0;
#pragma unroll
                for (int b = 0; b < 2; ++b) {
                    const int i = 8 * q + 2 * e + b;
                    const uint16_t yb = wn(v[i], r, b ? hi(wv[e]) : lo(wv[e]));
                    const uint16_t hb = float_to_adt_bits(
                        __fadd_rn(adt_bits_to_float(b ? hi(hu[e]) : lo(hu[e]), adt), adt_bits_to_float(yb, adt)),
                        adt);
                    v[i] = adt_bits_to_float(hb, adt);
                    yy |= static_cast<uint32_t>(yb) << (16 * b);
                    hh |= static_cast<uint32_t>(hb) << (16 * b);
                }
                yo[e] = yy;
                ho[e] = hh;
            }
            yo4[q] = make_uint4(yo[0], yo[1], yo[2], yo[3]);
            ho4[q] = make_uint4(ho[0], ho[1], ho[2], ho[3]);
        }
    }
    rscale();
#pragma unroll
    for (int m = 0; m < kTailV; ++m) {
        const int q = tix + m * nthr;
        if (q < n8) {
            const float r = rs[(8 * q) / H];
            const uint32_t wv[4] = {w1v[m].x, w1v[m].y, w1v[m].z, w1v[m].w};
            const uint32_t xu[4] = {xv[m].x, xv[m].y, xv[m].z, xv[m].w};
            uint32_t xo[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                uint32_t xx = 0;
#pragma unroll
                for (int b = 0; b < 2; ++b) {
                    const int i = 8 * q + 2 * e + b;
                    const uint16_t fb = wn(v[i], r, b ? hi(wv[e]) : lo(wv[e]));
                    const uint16_t xb = float_to_adt_bits(
                        __fadd_rn(adt_bits_to_float(b ? hi(xu[e]) : lo(xu[e]), adt), adt_bits_to_float(fb, adt)),
                        adt);
                    xx |= static_cast<uint32_t>(float_to_adt_bits(__fmul_rn(adt_bits_to_float(xb, adt), scalar),
                                                                  adt)) << (16 * b);
                }
                xo[e] = xx;
            }
            xo4[q] = make_uint4(xo[0], xo[1], xo[2], xo[3]);
        }
    }
    sync();
    return true;
}

}  // namespace tsmoe

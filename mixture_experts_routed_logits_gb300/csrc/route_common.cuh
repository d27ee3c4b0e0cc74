// route_common.cuh -- the per-token selection step of the router (keys, top-k, weights), shared by
// the router kernel and the decode prep kernel that routes its own tokens.
//
// Source pages (docs.rs, turbospark-runtime 0.3.0):
//   gpt-oss routed-expert pass (src/families/gptoss/moe.rs): the bias is added to the logits
//     before the top-k; the top-k runs on the raw biased logits; the weights are the softmax over
//     the selected k without renormalisation.
//   Gemma-4 batched routed prefill (src/families/gemma4/moe_batch.rs): per_expert_scale.
//   Llama/Mixtral decode flow (src/families/llama/mod.rs): MiniMax biased sigmoid scores with
//     unbiased weights.
#pragma once

#include "common.cuh"

namespace tsmoe {

// Order-preserving map of an f32 to u32 (larger float -> larger integer); -0 folds to +0 so
// that equal keys tie and fall back to the expert id, as the f32 comparison does.
__device__ __forceinline__ uint32_t mono_u32(float v) {
    const uint32_t u = __float_as_uint(__fadd_rn(v, 0.0f));
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Key for a max-reduction: value first, then the LOWER expert id wins a tie.
__device__ __forceinline__ uint64_t sel_key(float v, int e) {
    return (static_cast<uint64_t>(mono_u32(v)) << 32) | static_cast<uint32_t>(0xFFFFFFFFu - e);
}

__device__ __forceinline__ uint64_t shfl_xor_u64(uint64_t v, int o) {
    uint32_t lo = static_cast<uint32_t>(v), hi = static_cast<uint32_t>(v >> 32);
    lo = __shfl_xor_sync(0xffffffffu, lo, o);
    hi = __shfl_xor_sync(0xffffffffu, hi, o);
    return (static_cast<uint64_t>(hi) << 32) | lo;
}

// One warp: token t's keys, top-k by repeated warp arg-max, and weights, from its E logits (read
// through lg(e)); bias_r holds lane + 32 i's bias.  scr is 4 E floats of the warp's shared
// memory.  Writes idx/w (and the logits if logits_out); an aborted token gets idx -1.
template <typename LoadLogit>
__device__ __forceinline__ void route_token_warp(LoadLogit lg, const float (&bias_r)[kMaxExperts / 32],
                                                 int E, int k, int mode, bool has_bias,
                                                 const float* scale, float* scr, int t,
                                                 int32_t* idx, float* w, float* logits_out,
                                                 bool aborted, int lane) {
    float* key = scr;
    float* sg = scr + E;
    float* ex = scr + 2 * E;
    int* sel = reinterpret_cast<int*>(scr + 3 * E);
    for (int e = lane; e < E; e += 32) {
        const float l = lg(e);
        if (logits_out) logits_out[static_cast<size_t>(t) * E + e] = l;
        float b = 0.0f;
#pragma unroll
        for (int i = 0; i < kMaxExperts / 32; ++i)
            if (e == lane + 32 * i) b = bias_r[i];
        float kv;
        if (mode == MODE_SIGMOID_BIASED) {
            const float sv = __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-l)));
            sg[e] = sv;
            kv = has_bias ? __fadd_rn(sv, b) : sv;
        } else {
            kv = has_bias ? __fadd_rn(l, b) : l;
        }
        key[e] = kv;
    }
    __syncwarp();
    // top-k by repeated warp arg-max; each lane owns experts lane + 32 i
    uint64_t own[kMaxExperts / 32];
#pragma unroll
    for (int i = 0; i < kMaxExperts / 32; ++i) {
        const int e = lane + 32 * i;
        own[i] = e < E ? sel_key(key[e], e) : 0ull;
    }
    for (int s = 0; s < k; ++s) {
        uint64_t best = 0ull;
#pragma unroll
        for (int i = 0; i < kMaxExperts / 32; ++i) best = own[i] > best ? own[i] : best;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            const uint64_t other = shfl_xor_u64(best, o);
            best = other > best ? other : best;
        }
        const int e = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(best));
        if ((e & 31) == lane) {
#pragma unroll
            for (int i = 0; i < kMaxExperts / 32; ++i)
                if (lane + 32 * i == e) own[i] = 0ull;
        }
        if (lane == 0) sel[s] = e;
    }
    __syncwarp();
    if (mode == MODE_SIGMOID_BIASED) {
        for (int s = lane; s < k; s += 32) ex[s] = sg[sel[s]];
    } else {
        const float m = key[sel[0]];
        for (int s = lane; s < k; s += 32) ex[s] = expf(__fsub_rn(key[sel[s]], m));
    }
    __syncwarp();
    float sum = 0.0f;
    if (lane == 0)
        for (int s = 0; s < k; ++s) sum = __fadd_rn(sum, ex[s]);   // slot order
    sum = __shfl_sync(0xffffffffu, sum, 0);
    for (int s = lane; s < k; s += 32) {
        float wv = __fdiv_rn(ex[s], sum);
        if (mode == MODE_SOFTMAX_K_SCALED) wv = __fmul_rn(wv, scale[sel[s]]);
        idx[static_cast<size_t>(t) * k + s] = aborted ? -1 : sel[s];   // -1: a wait gave up
        w[static_cast<size_t>(t) * k + s] = wv;
    }
}

}  // namespace tsmoe

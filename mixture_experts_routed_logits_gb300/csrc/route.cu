// route.cu -- steps 1-3 of the routed-expert layer on sm_103a:
//   fused (optional RMSNorm) + router GEMV + bias + top-k + weights, one warp per token, and
//   the deterministic route-list builder (counting sort by expert).
//
// Source pages (docs.rs, turbospark-runtime 0.3.0):
//   gpt-oss routed-expert pass (src/families/gptoss/moe.rs): module header (bias added to the
//     logits before the top-k; top-k on the raw biased logits; softmax over the selected k with
//     no renormalisation, router_topk_gemma4's contract) and the "THE BIAS, BEFORE THE TOP-K"
//     step of encode_gpt_oss_layer_moe.
//   Gemma-4 batched routed prefill (src/families/gemma4/moe_batch.rs): router_topk_gemma4 with
//     per_expert_scale; RMS_EPS; encode_routes (route list for the batched kernels).
//   Llama/Mixtral decode flow (src/families/llama/mod.rs): "r = family_topk(m @ router)";
//     MiniMax "biased sigmoid scores with unbiased weights".
// The pages run the top-k on the host after a blocking readback of the logits; here it stays
// on the device, so the whole layer is one asynchronous stream of kernels.
#include "common.cuh"

namespace tsmoe {

namespace {

constexpr int kRouterWarps = 8;   // warps per token (experts are spread over them)


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

// Fixed-order f32 dot product of a warp: lane l sums fmaf(a[l+32j], b[l+32j]) over j, then an
// xor butterfly 16, 8, 4, 2, 1.  Every lane returns the same bits.
template <typename LoadB>
__device__ __forceinline__ float warp_dot_fixed(const float* a, LoadB loadb, int H, int lane) {
    float p = 0.0f;
    for (int j = lane; j < H; j += 32) p = __fmaf_rn(a[j], loadb(j), p);
    return warp_sum_xor(p);
}

// One CTA per token.  The router weights stream through shared memory in stages of `rb` rows
// (one 1-D bulk copy per stage, up to `ns` stages in flight, mbarrier completion); warp w
// computes the logit of row w of each stage.  The summation order of every logit is the fixed
// one (lane l: fmaf over j, then the xor butterfly), so which warp computes it does not matter.
struct RouterPlan {
    int rb, ns;           // rows per stage, stages in flight
    size_t smem;
};

__host__ inline RouterPlan router_plan(int H, int has_x) {
    RouterPlan p{8, 3, 0};
    if (!has_x) return p;
    const size_t budget = 200 * 1024;
    const size_t xs = static_cast<size_t>(H) * 4;
    while (p.rb > 1 || p.ns > 1) {
        const size_t need = xs + static_cast<size_t>(p.ns) * p.rb * H * 2 + 64;
        if (need <= budget) break;
        if (p.ns > 1) --p.ns; else p.rb /= 2;
    }
    p.smem = xs + static_cast<size_t>(p.ns) * p.rb * H * 2 + 64;
    return p;
}

__global__ void __launch_bounds__(kRouterWarps * 32)
router_kernel(RouteArgs a, int rb, int ns) {
    extern __shared__ __align__(128) unsigned char rsm[];
    __shared__ float key[kMaxExperts];
    __shared__ float sg[kMaxExperts];
    __shared__ float ex[kMaxExperts];
    __shared__ int sel[kMaxExperts];
    __shared__ float rnorm;
    __shared__ __align__(8) uint64_t full[3];
    __shared__ __align__(8) uint64_t empty[3];
    __shared__ volatile int abort_flag;
    pdl_wait();                 // x may come from the previous kernel
    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x;
    const int E = a.E, H = a.H, k = a.k;
    if (t >= a.T) return;

    // ---- step 1: optional RMSNorm + raw logits ------------------------------------------
    if (a.x) {
        float* xs = reinterpret_cast<float*>(rsm);
        uint16_t* wst = reinterpret_cast<uint16_t*>(rsm + static_cast<size_t>(H) * 4);
        const size_t stage_elems = static_cast<size_t>(rb) * H;
        const int nst = (E + rb - 1) / rb;
        const uint16_t* W = static_cast<const uint16_t*>(a.Wr);
        if (threadIdx.x == 0) {
            abort_flag = 0;
            for (int q = 0; q < ns; ++q) {
                mbar_init(&full[q], 1);
                mbar_init(&empty[q], kRouterWarps);
            }
            fence_mbar_init();
        }
        __syncthreads();
        auto issue = [&](int st) {
            const int e0 = st * rb;
            const int rows = min(rb, E - e0);
            const uint32_t bytes = static_cast<uint32_t>(rows) * H * 2;
            const int slot = st % ns;
            mbar_arrive_expect_tx(&full[slot], bytes);
            bulk_g2s(wst + slot * stage_elems, W + static_cast<size_t>(e0) * H, bytes, &full[slot]);
        };
        if (threadIdx.x == 0)
            for (int st = 0; st < min(ns, nst); ++st) issue(st);
        const uint16_t* xr = static_cast<const uint16_t*>(a.x) + static_cast<size_t>(t) * H;
        for (int j = threadIdx.x; j < H; j += blockDim.x) xs[j] = adt_bits_to_float(xr[j], a.adt);
        __syncthreads();
        if (a.rmsnorm) {
            if (warp == 0) {
                const float ss = warp_dot_fixed(xs, [&](int j) { return xs[j]; }, H, lane);
                const float ms = __fdiv_rn(ss, static_cast<float>(H));
                if (lane == 0) rnorm = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, a.eps)));
            }
            __syncthreads();
            const float r = rnorm;
            uint16_t* xo = static_cast<uint16_t*>(a.xn_out) + static_cast<size_t>(t) * H;
            for (int j = threadIdx.x; j < H; j += blockDim.x) {
                const uint16_t b = float_to_adt_bits(__fmul_rn(xs[j], r), a.adt);
                xo[j] = b;
                xs[j] = adt_bits_to_float(b, a.adt);
            }
            __syncthreads();
        }
        for (int st = 0; st < nst; ++st) {
            const int slot = st % ns;
            const bool ok = !abort_flag && mbar_wait_bounded(&full[slot], (st / ns) & 1);
            if (!ok) {
                if (lane == 0) abort_flag = 1;
            } else if (warp < rb && st * rb + warp < E) {
                const uint16_t* wr = wst + slot * stage_elems + static_cast<size_t>(warp) * H;
                const float l = warp_dot_fixed(xs, [&](int j) { return adt_bits_to_float(wr[j], a.adt); },
                                               H, lane);
                if (lane == 0) key[st * rb + warp] = l;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
            if (threadIdx.x == 0 && st + ns < nst && !abort_flag) {
                // the slot is refilled once every warp has read it
                if (mbar_wait_bounded(&empty[slot], (st / ns) & 1)) issue(st + ns);
                else abort_flag = 1;
            }
        }
        // no copy may still be in flight when the CTA exits
        if (threadIdx.x == 0)
            for (int st = max(0, nst - ns); st < nst; ++st)
                mbar_wait_bounded(&full[st % ns], (st / ns) & 1);
    } else {
        const float* lr = a.logits_in + static_cast<size_t>(t) * E;
        for (int e = threadIdx.x; e < E; e += blockDim.x) key[e] = lr[e];
    }
    __syncthreads();
    if (warp != 0) return;

    // ---- step 2: keys per mode --------------------------------------------------------------
    for (int e = lane; e < E; e += 32) {
        const float l = key[e];
        if (a.logits_out) a.logits_out[static_cast<size_t>(t) * E + e] = l;
        const float b = a.bias ? a.bias[e] : 0.0f;
        float kv;
        if (a.mode == MODE_SIGMOID_BIASED) {
            const float s = __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-l)));
            sg[e] = s;
            kv = a.bias ? __fadd_rn(s, b) : s;
        } else {
            kv = a.bias ? __fadd_rn(l, b) : l;
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

    // ---- weights ------------------------------------------------------------------------------
    if (a.mode == MODE_SIGMOID_BIASED) {
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
    const bool aborted = a.x && abort_flag;
    for (int s = lane; s < k; s += 32) {
        float wv = __fdiv_rn(ex[s], sum);
        if (a.mode == MODE_SOFTMAX_K_SCALED) wv = __fmul_rn(wv, a.scale[sel[s]]);
        a.idx[static_cast<size_t>(t) * k + s] = aborted ? -1 : sel[s];   // -1: the wait gave up
        a.w[static_cast<size_t>(t) * k + s] = wv;
    }
}

// ------------------------------------------------------------------------------------------
// Route list: off[E+1], perm (route ids grouped by expert, ascending id inside an expert),
// inv.  One CTA, deterministic: counts, exclusive scan, then a stable scatter in chunks of
// 1024 routes (rank inside a chunk from warp match masks plus earlier warps' counts).
// ------------------------------------------------------------------------------------------
constexpr int kBuildThreads = 1024;

__global__ void __launch_bounds__(kBuildThreads)
build_routes_kernel(const int32_t* __restrict__ idx, int n, int E, int32_t* __restrict__ off,
                    int32_t* __restrict__ perm, int32_t* __restrict__ inv, int* status) {
    __shared__ int cnt[kMaxExperts];
    __shared__ int cursor[kMaxExperts];
    __shared__ int wcnt[kBuildThreads / 32][kMaxExperts];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pdl_wait();                 // idx comes from the previous kernel
    pdl_launch_dependents();
    for (int e = tid; e < E; e += kBuildThreads) cnt[e] = 0;
    __syncthreads();
    for (int r = tid; r < n; r += kBuildThreads) {
        const int e = idx[r];
        if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);
        else report_error(status, DEV_ERR_INVALID);
    }
    __syncthreads();
    if (tid == 0) {
        int acc = 0;
        for (int e = 0; e < E; ++e) {
            off[e] = acc;
            cursor[e] = acc;
            acc += cnt[e];
        }
        off[E] = acc;
    }
    __syncthreads();
    for (int base = 0; base < n; base += kBuildThreads) {
        for (int i = tid; i < (kBuildThreads / 32) * E; i += kBuildThreads)
            wcnt[i / E][i % E] = 0;
        __syncthreads();
        const int r = base + tid;
        int e = -1;
        if (r < n) {
            e = idx[r];
            if (e < 0 || e >= E) e = -1;
        }
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        const int rank = __popc(peers & ((1u << lane) - 1u));
        if (e >= 0 && rank == 0) wcnt[warp][e] = __popc(peers);
        __syncthreads();
        if (e >= 0) {
            int pos = cursor[e] + rank;
            for (int w2 = 0; w2 < warp; ++w2) pos += wcnt[w2][e];
            perm[pos] = r;
            inv[r] = pos;
        }
        __syncthreads();
        for (int e2 = tid; e2 < E; e2 += kBuildThreads) {
            int add = 0;
            for (int w2 = 0; w2 < kBuildThreads / 32; ++w2) add += wcnt[w2][e2];
            cursor[e2] += add;
        }
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_router(const RouteArgs& a, cudaStream_t s) {
    if (a.T <= 0) return cudaSuccess;
    const RouterPlan p = router_plan(a.H, a.x != nullptr);
    if (p.smem > 40 * 1024) {
        cudaError_t e = ensure_smem(router_kernel, p.smem);
        if (e != cudaSuccess) return e;
    }
    return launch_pdl(router_kernel, dim3(a.T), dim3(kRouterWarps * 32), p.smem, s, a, p.rb, p.ns);
}

cudaError_t launch_build_routes(const int32_t* idx, int T, int E, int k, int32_t* off,
                                int32_t* perm, int32_t* inv, int* status, cudaStream_t s) {
    return launch_pdl(build_routes_kernel, dim3(1), dim3(kBuildThreads), 0, s, idx, T * k, E, off,
                      perm, inv, status);
}

}  // namespace tsmoe

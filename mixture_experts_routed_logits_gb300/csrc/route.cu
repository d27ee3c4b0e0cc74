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
#include <algorithm>

#include "common.cuh"

namespace tsmoe {

namespace {

constexpr int kRouterWarps = 8;   // warps per CTA


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

// Router layout.  A CTA takes a tile of `tt` tokens and a group of `ec` experts; the `cl` expert
// groups of a token tile form one thread-block cluster, so a decode batch of a few tokens still
// spreads over many SMs.  The CTA's router rows stream through shared memory in stages of `rb`
// rows (1-D bulk copies, `ns` stages in flight, mbarrier completion); each warp computes whole
// logits (one row against every token of the tile, the tokens giving independent fma chains).
// The summation order of every logit is the fixed one (lane l: fmaf over j, then the xor
// butterfly), whichever warp or CTA computes it.  Rank 0 of the cluster then gathers each
// token's E logits from the cluster's shared memory (distributed shared memory) and runs the
// top-k, one warp per token.
constexpr int kRouterTT = 8;      // tokens per CTA at most (one top-k warp each)

struct RouterPlan {
    int tt, cl, ec;       // tokens per CTA, CTAs per cluster, experts per CTA
    int rb, ns;           // router rows per stage, stages in flight
    int ntiles;           // token tiles
    size_t xs_off, ring_off, lg_off, scr_off, smem;
};

__host__ inline RouterPlan router_plan_tt(int T, int H, int E, int has_x, int tt) {
    RouterPlan p{};
    const size_t budget = 210 * 1024;
    p.tt = tt;
    p.ntiles = (T + p.tt - 1) / p.tt;
    if (has_x) {
        p.cl = 1;
        while (p.cl < 8 && p.cl * 2 <= E && static_cast<long long>(p.ntiles) * p.cl < 128) p.cl *= 2;
        p.ec = (E + p.cl - 1) / p.cl;
    } else {
        p.cl = 1;
        p.ec = E;
    }
    p.xs_off = 0;
    const size_t xs = has_x ? static_cast<size_t>(p.tt) * H * 4 : 0;
    const size_t lg = static_cast<size_t>(p.tt) * p.ec * 4;
    const size_t scr = static_cast<size_t>(kRouterWarps) * (2 * E + 2 * E) * 4;   // key, sg, ex, sel
    const size_t fixed = ((xs + 127) & ~size_t(127)) + ((lg + 127) & ~size_t(127)) + scr + 256;
    p.rb = std::min(p.ec, 32);
    p.ns = 3;
    while (has_x && p.rb > 1 && fixed + static_cast<size_t>(p.ns) * p.rb * H * 2 > budget) {
        if (p.ns > 2) --p.ns; else p.rb = (p.rb + 1) / 2;
    }
    if (has_x && fixed + static_cast<size_t>(p.ns) * p.rb * H * 2 > budget) p.ns = 1;
    p.ring_off = (xs + 127) & ~size_t(127);
    const size_t ring = has_x ? static_cast<size_t>(p.ns) * p.rb * H * 2 : 0;
    p.lg_off = p.ring_off + ((ring + 127) & ~size_t(127));
    p.scr_off = p.lg_off + ((lg + 127) & ~size_t(127));
    p.smem = p.scr_off + scr + 128;
    return p;
}

// Tokens per CTA: 1 for decode batches; for prefill as many as fit (f32 rows within 96 KB) while a
// stage still holds a router row for every warp.
__host__ inline RouterPlan router_plan(int T, int H, int E, int has_x) {
    if (!has_x) return router_plan_tt(T, H, E, 0, kRouterTT);
    int tt = T <= 64 ? 1 : static_cast<int>(std::min<size_t>(kRouterTT, (96 * 1024) / (static_cast<size_t>(H) * 4)));
    if (tt < 1) tt = 1;
    RouterPlan p = router_plan_tt(T, H, E, 1, tt);
    while (p.tt > 1 && p.rb < std::min(p.ec, kRouterWarps)) p = router_plan_tt(T, H, E, 1, p.tt - 1);
    return p;
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ float ld_cluster_f32(const float* local, uint32_t rank) {
    uint32_t addr;
    float v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(addr) : "r"(smem_u32(local)), "r"(rank));
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

__global__ void __launch_bounds__(kRouterWarps * 32)
router_kernel(RouteArgs a, RouterPlan p) {
    extern __shared__ __align__(128) unsigned char rsm[];
    __shared__ __align__(8) uint64_t full[3];
    __shared__ __align__(8) uint64_t empty[3];
    __shared__ float rnorm[kRouterTT];
    __shared__ volatile int abort_flag;
    pdl_wait();                 // x may come from the previous kernel
    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = a.E, H = a.H, k = a.k;
    const uint32_t rank = p.cl > 1 ? cluster_rank() : 0u;
    const int tile = blockIdx.x / p.cl;
    const int t0 = tile * p.tt;
    const int ntok = max(0, min(p.tt, a.T - t0));
    const int e0 = static_cast<int>(rank) * p.ec;
    const int ne = max(0, min(p.ec, E - e0));
    float* xs = reinterpret_cast<float*>(rsm + p.xs_off);          // [tt][H] f32
    uint16_t* wst = reinterpret_cast<uint16_t*>(rsm + p.ring_off); // stages of rb rows
    float* lg = reinterpret_cast<float*>(rsm + p.lg_off);          // [tt][ec] logits
    if (threadIdx.x == 0) abort_flag = 0;
    // the top-k warps fetch their router biases now, off the critical path
    float bias_r[kMaxExperts / 32];
#pragma unroll
    for (int i = 0; i < kMaxExperts / 32; ++i) {
        const int e = lane + 32 * i;
        bias_r[i] = (a.bias && rank == 0 && warp < ntok && e < E) ? a.bias[e] : 0.0f;
    }

    // ---- step 1: optional RMSNorm + raw logits of this CTA's experts -----------------------
    if (a.x) {
        const size_t stage_elems = static_cast<size_t>(p.rb) * H;
        const int nst = (ne + p.rb - 1) / p.rb;
        const uint16_t* W = static_cast<const uint16_t*>(a.Wr) + static_cast<size_t>(e0) * H;
        if (threadIdx.x == 0) {
            for (int q = 0; q < p.ns; ++q) {
                mbar_init(&full[q], 1);
                mbar_init(&empty[q], kRouterWarps);
            }
            fence_mbar_init();
        }
        __syncthreads();
        auto issue = [&](int st) {
            const int r0 = st * p.rb;
            const int rows = min(p.rb, ne - r0);
            const uint32_t bytes = static_cast<uint32_t>(rows) * H * 2;
            const int slot = st % p.ns;
            mbar_arrive_expect_tx(&full[slot], bytes);
            bulk_g2s(wst + slot * stage_elems, W + static_cast<size_t>(r0) * H, bytes, &full[slot]);
        };
        if (threadIdx.x == 0)
            for (int st = 0; st < min(p.ns, nst); ++st) issue(st);
        // token rows -> f32 in shared memory (16-byte loads, all issued before use: for a
        // multi-token tile every token's at once, rows of up to 2 x 8 x blockDim elements;
        // otherwise token by token)
        const bool vec_ok = (H & 7) == 0 && (reinterpret_cast<uintptr_t>(a.x) & 15) == 0;
        if (ntok > 1 && vec_ok && H / 8 <= 2 * static_cast<int>(blockDim.x)) {
            const int nv = H / 8;
            uint4 v[kRouterTT][2];
#pragma unroll
            for (int q = 0; q < kRouterTT; ++q)
#pragma unroll
                for (int m = 0; m < 2; ++m) {
                    const int i = threadIdx.x + m * blockDim.x;
                    if (q < ntok && i < nv)
                        v[q][m] = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.x) +
                                                                        static_cast<size_t>(t0 + q) * H) + i);
                }
#pragma unroll
            for (int q = 0; q < kRouterTT; ++q)
#pragma unroll
                for (int m = 0; m < 2; ++m) {
                    const int i = threadIdx.x + m * blockDim.x;
                    if (q < ntok && i < nv) {
                        float* xq = xs + static_cast<size_t>(q) * H + 8 * i;
                        const uint32_t w4[4] = {v[q][m].x, v[q][m].y, v[q][m].z, v[q][m].w};
#pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            xq[2 * h] = adt_bits_to_float(static_cast<uint16_t>(w4[h] & 0xFFFF), a.adt);
                            xq[2 * h + 1] = adt_bits_to_float(static_cast<uint16_t>(w4[h] >> 16), a.adt);
                        }
                    }
                }
        } else {
            for (int q = 0; q < ntok; ++q) {
                const uint16_t* xr = static_cast<const uint16_t*>(a.x) + static_cast<size_t>(t0 + q) * H;
                float* xq = xs + static_cast<size_t>(q) * H;
                if ((H & 7) == 0 && (reinterpret_cast<uintptr_t>(xr) & 15) == 0) {
                    constexpr int kMaxV = 8;
                    const int nv = H / 8;
                    uint4 v[kMaxV];
    #pragma unroll
                    for (int i8 = 0; i8 < kMaxV; ++i8) {
                        const int i = threadIdx.x + i8 * blockDim.x;
                        if (i < nv) v[i8] = __ldg(reinterpret_cast<const uint4*>(xr) + i);
                    }
    #pragma unroll
                    for (int i8 = 0; i8 < kMaxV; ++i8) {
                        const int i = threadIdx.x + i8 * blockDim.x;
                        if (i < nv) {
                            const uint32_t w4[4] = {v[i8].x, v[i8].y, v[i8].z, v[i8].w};
    #pragma unroll
                            for (int h = 0; h < 4; ++h) {
                                xq[8 * i + 2 * h] = adt_bits_to_float(static_cast<uint16_t>(w4[h] & 0xFFFF), a.adt);
                                xq[8 * i + 2 * h + 1] = adt_bits_to_float(static_cast<uint16_t>(w4[h] >> 16), a.adt);
                            }
                        }
                    }
                    for (int j = kMaxV * blockDim.x * 8 + threadIdx.x; j < H; j += blockDim.x)
                        xq[j] = adt_bits_to_float(xr[j], a.adt);
                } else {
                    for (int j = threadIdx.x; j < H; j += blockDim.x) xq[j] = adt_bits_to_float(xr[j], a.adt);
                }
            }
        }
        __syncthreads();
        if (a.rmsnorm) {
            if (warp < ntok) {
                const float* xq = xs + static_cast<size_t>(warp) * H;
                const float ss = warp_dot_fixed(xq, [&](int j) { return xq[j]; }, H, lane);
                const float ms = __fdiv_rn(ss, static_cast<float>(H));
                if (lane == 0) rnorm[warp] = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, a.eps)));
            }
            __syncthreads();
            for (int q = 0; q < ntok; ++q) {
                const float r = rnorm[q];
                float* xq = xs + static_cast<size_t>(q) * H;
                uint16_t* xo = static_cast<uint16_t*>(a.xn_out) + static_cast<size_t>(t0 + q) * H;
                for (int j = threadIdx.x; j < H; j += blockDim.x) {
                    const uint16_t b = float_to_adt_bits(__fmul_rn(xq[j], r), a.adt);
                    if (rank == 0) xo[j] = b;
                    xq[j] = adt_bits_to_float(b, a.adt);
                }
            }
            __syncthreads();
        }
        for (int st = 0; st < nst; ++st) {
            const int slot = st % p.ns;
            const int rows = min(p.rb, ne - st * p.rb);
            const bool ok = !abort_flag && mbar_wait_bounded(&full[slot], (st / p.ns) & 1);
            if (!ok) {
                if (lane == 0) abort_flag = 1;
            } else {
                for (int rr = warp; rr < rows; rr += kRouterWarps) {
                    const uint16_t* wr = wst + slot * stage_elems + static_cast<size_t>(rr) * H;
                    float acc[kRouterTT];
#pragma unroll
                    for (int q = 0; q < kRouterTT; ++q) acc[q] = 0.0f;
#pragma unroll 4
                    for (int j = lane; j < H; j += 32) {
                        const float wv = adt_bits_to_float(wr[j], a.adt);
#pragma unroll
                        for (int q = 0; q < kRouterTT; ++q)
                            if (q < ntok) acc[q] = __fmaf_rn(xs[static_cast<size_t>(q) * H + j], wv, acc[q]);
                    }
#pragma unroll
                    for (int q = 0; q < kRouterTT; ++q) {
                        if (q >= ntok) break;
                        const float l = warp_sum_xor(acc[q]);
                        if (lane == 0) lg[q * p.ec + st * p.rb + rr] = l;
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
            if (threadIdx.x == 0 && st + p.ns < nst && !abort_flag) {
                // the slot is refilled once every warp has read it
                if (mbar_wait_bounded(&empty[slot], (st / p.ns) & 1)) issue(st + p.ns);
                else abort_flag = 1;
            }
        }
        // no copy may still be in flight when the CTA exits
        if (threadIdx.x == 0)
            for (int st = max(0, nst - p.ns); st < nst; ++st)
                mbar_wait_bounded(&full[st % p.ns], (st / p.ns) & 1);
    } else {
        for (int i = threadIdx.x; i < ntok * E; i += blockDim.x)
            lg[i] = a.logits_in[static_cast<size_t>(t0) * E + i];
    }
    __syncthreads();
    if (p.cl > 1) cluster_sync_all();        // every CTA's logits are in its shared memory

    // ---- step 2: per token (one warp each, cluster rank 0): keys, top-k, weights --------------
    if (rank == 0 && warp < ntok) {
        const int t = t0 + warp;
        float* key = reinterpret_cast<float*>(rsm + p.scr_off) + static_cast<size_t>(warp) * 4 * E;
        float* sg = key + E;
        float* ex = key + 2 * E;
        int* sel = reinterpret_cast<int*>(key + 3 * E);
        for (int e = lane; e < E; e += 32) {
            const uint32_t owner = static_cast<uint32_t>(e / p.ec);
            const float* src = lg + warp * p.ec + (e - static_cast<int>(owner) * p.ec);
            const float l = p.cl > 1 ? ld_cluster_f32(src, owner) : *src;
            if (a.logits_out) a.logits_out[static_cast<size_t>(t) * E + e] = l;
            float b = 0.0f;
#pragma unroll
            for (int i = 0; i < kMaxExperts / 32; ++i)
                if (e == lane + 32 * i) b = bias_r[i];
            float kv;
            if (a.mode == MODE_SIGMOID_BIASED) {
                const float sv = __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-l)));
                sg[e] = sv;
                kv = a.bias ? __fadd_rn(sv, b) : sv;
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
            a.idx[static_cast<size_t>(t) * k + s] = aborted ? -1 : sel[s];   // -1: a wait gave up
            a.w[static_cast<size_t>(t) * k + s] = wv;
        }
    }
    // the other CTAs of the cluster keep their shared memory until rank 0 has read it
    if (p.cl > 1) cluster_sync_all();
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
    // Every position starts as a valid route id and every route as unplaced, so that the list
    // stays inside 0..n-1 even if idx holds ids outside 0..E-1 or changes between the two
    // passes below (the placement never leaves an expert's counted range).
    for (int r = tid; r < n; r += kBuildThreads) {
        perm[r] = 0;
        inv[r] = -1;
    }
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
            cnt[e] = acc;               // end of expert e's range
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
            if (pos < cnt[e]) {
                perm[pos] = r;
                inv[r] = pos;
            } else {
                report_error(status, DEV_ERR_INVALID);   // idx changed since it was counted
            }
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
    const RouterPlan p = router_plan(a.T, a.H, a.E, a.x != nullptr);
    cudaError_t e = ensure_smem(router_kernel, p.smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.ntiles * p.cl);
    cfg.blockDim = dim3(kRouterWarps * 32);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = s;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    at[1].id = cudaLaunchAttributeClusterDimension;
    at[1].val.clusterDim.x = static_cast<unsigned>(p.cl);
    at[1].val.clusterDim.y = 1;
    at[1].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, router_kernel, a, p);
}

cudaError_t launch_build_routes(const int32_t* idx, int T, int E, int k, int32_t* off,
                                int32_t* perm, int32_t* inv, int* status, cudaStream_t s) {
    return launch_pdl(build_routes_kernel, dim3(1), dim3(kBuildThreads), 0, s, idx, T * k, E, off,
                      perm, inv, status);
}

}  // namespace tsmoe

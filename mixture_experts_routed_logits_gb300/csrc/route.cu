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

#include "mx_common.cuh"
#include "route_common.cuh"

namespace tsmoe {

namespace {

constexpr int kRouterWarps = 8;   // warps per CTA

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

// PREP: the launch also does the block-scaled decode kernels' prep (a.mxd_xs set; that code
// exists only in this instantiation)
template <bool PREP>
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
        if (PREP) {
            // ---- the block-scaled decode kernels' prep (their x image and counters), folded in
            // while the router rows are in flight: each token row is split into two e4m3 terms
            // under one scale, 2^s with s = floor(log2 max|x_t|) - 7; the CTAs of the cluster
            // take its 16-column chunks in turn (the image holds the K stages [KG][16 rows][128
            // B] as the decode kernel's shared memory holds them, 128-byte swizzle, then the
            // scale atom of the 16 rows) ----
            const int KG = (H + 127) / 128;
            unsigned char* atom = a.mxd_xs + static_cast<size_t>(KG) * kMxdBStage;
            for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < a.mxd_ncnt; i += gridDim.x * blockDim.x)
                a.mxd_cnt[i] = 0;
            __shared__ float red[kRouterWarps];
            for (int q = 0; q < ntok; ++q) {
                const int t = t0 + q;
                const float* xq = xs + static_cast<size_t>(q) * H;
                float mx = 0.0f;
                for (int j = threadIdx.x; j < H; j += blockDim.x) mx = fmaxf(mx, fabsf(xq[j]));
                mx = warp_max(mx);
                if (lane == 0) red[warp] = mx;
                __syncthreads();
                mx = red[0];
#pragma unroll
                for (int i = 1; i < kRouterWarps; ++i) mx = fmaxf(mx, red[i]);
                __syncthreads();
                const int se = mx_scale_exp(mx);
                const float inv = __uint_as_float(static_cast<uint32_t>(127 - se) << 23);
                for (int c = static_cast<int>(rank) + p.cl * threadIdx.x; c < KG * 8; c += p.cl * blockDim.x) {
                    uint32_t q1[4] = {0u, 0u, 0u, 0u}, q2[4] = {0u, 0u, 0u, 0u};
#pragma unroll
                    for (int h = 0; h < 8; ++h) {
                        const int col = c * 16 + 2 * h;
                        const float f0 = col < H ? xq[col] : 0.0f, f1 = col + 1 < H ? xq[col + 1] : 0.0f;
                        uint32_t t1, t2;
                        mx_split2(__fmul_rn(f0, inv), __fmul_rn(f1, inv), t1, t2);
                        q1[h >> 1] |= (t1 & 0xFFFFu) << (16 * (h & 1));
                        q2[h >> 1] |= (t2 & 0xFFFFu) << (16 * (h & 1));
                    }
                    unsigned char* sx = a.mxd_xs + static_cast<size_t>(c >> 3) * kMxdBStage;
                    const int cc = c & 7;
                    *reinterpret_cast<uint4*>(sx + t * 128 + ((cc ^ t) << 4)) = make_uint4(q1[0], q1[1], q1[2], q1[3]);
                    *reinterpret_cast<uint4*>(sx + (8 + t) * 128 + ((cc ^ t) << 4)) = make_uint4(q2[0], q2[1], q2[2], q2[3]);
                }
                if (rank == 0 && threadIdx.x == 0) {
                    // rows t (2^s) and 8 + t (2^(s-4)) of the atom; rows 16..31 zero
                    const uint32_t w0 = static_cast<uint32_t>(se + 127) * 0x01010101u;
                    *reinterpret_cast<uint4*>(atom + 16 * t) = make_uint4(w0, 0u, 0u, 0u);
                    *reinterpret_cast<uint4*>(atom + 16 * (8 + t)) = make_uint4(w0 - 0x04040404u, 0u, 0u, 0u);
                    *reinterpret_cast<uint4*>(atom + 16 * (16 + t)) = make_uint4(0u, 0u, 0u, 0u);
                    *reinterpret_cast<uint4*>(atom + 16 * (24 + t)) = make_uint4(0u, 0u, 0u, 0u);
                }
            }
            if (blockIdx.x == 0) {
                // the token slots past T: zero rows, and the scale atoms a zero row gets (s = 0)
                const int nz = (kMxdTokens - a.T) * KG * 16;
                for (int u = threadIdx.x; u < nz; u += blockDim.x) {
                    const int t = a.T + u / (KG * 16), r = u % (KG * 16);
                    const int kg = r >> 4, row = ((r >> 3) & 1) * 8 + t, chunk = r & 7;
                    *reinterpret_cast<uint4*>(a.mxd_xs + static_cast<size_t>(kg) * kMxdBStage + row * 128 + chunk * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                const int t = a.T + static_cast<int>(threadIdx.x);
                if (t < kMxdTokens) {
                    *reinterpret_cast<uint4*>(atom + 16 * t) = make_uint4(0x7F7F7F7Fu, 0u, 0u, 0u);
                    *reinterpret_cast<uint4*>(atom + 16 * (8 + t)) = make_uint4(0x7B7B7B7Bu, 0u, 0u, 0u);
                    *reinterpret_cast<uint4*>(atom + 16 * (16 + t)) = make_uint4(0u, 0u, 0u, 0u);
                    *reinterpret_cast<uint4*>(atom + 16 * (24 + t)) = make_uint4(0u, 0u, 0u, 0u);
                }
            }
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
        float* scr = reinterpret_cast<float*>(rsm + p.scr_off) + static_cast<size_t>(warp) * 4 * E;
        auto logit = [&](int e) {
            const uint32_t owner = static_cast<uint32_t>(e / p.ec);
            const float* src = lg + warp * p.ec + (e - static_cast<int>(owner) * p.ec);
            return p.cl > 1 ? ld_cluster_f32(src, owner) : *src;
        };
        route_token_warp(logit, bias_r, E, k, a.mode, a.bias != nullptr, a.scale, scr, t, a.idx, a.w,
                         a.logits_out, a.x && abort_flag, lane);
    }
    // the other CTAs of the cluster keep their shared memory until rank 0 has read it
    if (p.cl > 1) cluster_sync_all();
}

// Router for prefill-sized calls (no RMSNorm, at most 32 experts, router rows that fit in shared
// memory): every CTA holds all E router rows (one bulk copy, split in pieces) and takes rounds of
// `tpc` tokens.  A token's row is copied into a shared-memory buffer (16-byte loads, all issued
// at once) by the EG warps that share it; warp g of them keeps the partial sums of experts
// 8 g .. 8 g + 7 over x[t][l + 32 m] (lane l), so every logit has the fixed order of the cluster
// path above (lane l: fmaf over m ascending, then the xor butterfly) and the two paths give the
// same bits; then one warp per token runs the top-k.  No cluster barriers, and the router rows
// are loaded once per SM instead of once per tile of a few tokens.  Measured (one GB300, router
// launch against the cluster path): Mixtral T=2048 (E=8) 43.8 -> 24.4 us, gpt-oss T=512 (E=32,
// four warps per token) 26.1 -> 21.8 us.
constexpr int kWideMaxWarps = 16;
constexpr size_t kWideSmem = 227 * 1024;      // shared memory of one CTA
constexpr int kWideMaxV = 16;                 // 16-byte pieces of a token row per lane (H <= 4096)
constexpr uint32_t kWidePiece = 32 * 1024;    // bytes per bulk copy of the router rows

template <int EG>   // warps per token: experts in groups of 8, E <= 8 EG
__global__ void __launch_bounds__(kWideMaxWarps * 32, 1) router_wide_kernel(RouteArgs a) {
    extern __shared__ __align__(128) unsigned char rsm[];
    __shared__ __align__(8) uint64_t wfull;
    pdl_wait();                 // x may come from the previous kernel
    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tpc = (blockDim.x >> 5) / EG;                     // token slots per round
    const int ts = warp / EG, g = warp - ts * EG;               // this warp's slot and expert group
    const int E = a.E, H = a.H;
    const uint32_t wbytes = static_cast<uint32_t>(E) * H * 2;
    const size_t wal = (wbytes + 127) & ~127u;
    const uint16_t* ws = reinterpret_cast<const uint16_t*>(rsm);                       // [E][H]
    uint16_t* xb = reinterpret_cast<uint16_t*>(rsm + wal) + static_cast<size_t>(ts) * H;    // [tpc][H]
    float* lg = reinterpret_cast<float*>(rsm + wal + static_cast<size_t>(tpc) * H * 2) +
                static_cast<size_t>(ts) * E;                                            // [tpc][E]
    float* scr = reinterpret_cast<float*>(rsm + wal + static_cast<size_t>(tpc) * H * 2) +
                 static_cast<size_t>(tpc) * E + static_cast<size_t>(ts) * 4 * E;      // [tpc][4E]
    if (threadIdx.x == 0) {
        mbar_init(&wfull, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(&wfull, wbytes);
        for (uint32_t o = 0; o < wbytes; o += kWidePiece)
            bulk_g2s(rsm + o, static_cast<const unsigned char*>(a.Wr) + o, min(kWidePiece, wbytes - o), &wfull);
    }
    float bias_r[kMaxExperts / 32];
#pragma unroll
    for (int i = 0; i < kMaxExperts / 32; ++i) bias_r[i] = (i == 0 && a.bias && lane < E) ? a.bias[lane] : 0.0f;
    __syncthreads();            // the barrier is initialised before anyone waits on it
    const bool ok = mbar_wait_bounded(&wfull, 0);
    const uint16_t* xg = static_cast<const uint16_t*>(a.x);
    const int nv = H / 8;
    for (int base = blockIdx.x * tpc; base < a.T; base += gridDim.x * tpc) {
        const int t = base + ts;
        const bool have = t < a.T;
        if (have) {
            // the token row into its buffer: the slot's EG warps take its 16-byte pieces in turn
            const uint4* src = reinterpret_cast<const uint4*>(xg + static_cast<size_t>(t) * H);
#pragma unroll
            for (int h = 0; h < kWideMaxV / EG; h += 8) {
                uint4 v[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int pc = lane + 32 * (g + EG * (h + q));
                    if (pc < nv) v[q] = __ldg(src + pc);
                }
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int pc = lane + 32 * (g + EG * (h + q));
                    if (pc < nv) reinterpret_cast<uint4*>(xb)[pc] = v[q];
                }
            }
        }
        // rows in (and the last round's top-k done with lg and scr); one warp per token needs
        // no more than its own barrier
        if (EG > 1) __syncthreads(); else __syncwarp();
        if (have) {
            float acc[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
            const int e0 = 8 * g;
            if (ok) {
#pragma unroll 4
                for (int j = lane; j < H; j += 32) {
                    const float xv = adt_bits_to_float(xb[j], a.adt);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        if (e0 + i < E)
                            acc[i] = __fmaf_rn(xv, adt_bits_to_float(ws[static_cast<size_t>(e0 + i) * H + j], a.adt), acc[i]);
                }
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (e0 + i < E) {
                    const float l = warp_sum_xor(acc[i]);
                    if (lane == i) lg[e0 + i] = l;
                }
            }
        }
        if (EG > 1) __syncthreads(); else __syncwarp();    // the token's logits in
        if (have && g == 0)
            route_token_warp([&](int e) { return lg[e]; }, bias_r, E, a.k, a.mode, a.bias != nullptr, a.scale, scr,
                             t, a.idx, a.w, a.logits_out, !ok, lane);
    }
    // no copy may still be in flight when the CTA exits
    if (!ok && threadIdx.x == 0) mbar_wait_bounded(&wfull, 0);
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
    // prefill sizes: the router rows held in shared memory, rounds of whole tokens per CTA
    const int EG = (a.E + 7) / 8;
    const size_t wal = (static_cast<size_t>(a.E) * a.H * 2 + 127) & ~size_t(127);
    const size_t per_slot = static_cast<size_t>(a.H) * 2 + static_cast<size_t>(5) * a.E * 4;
    const int tpc = wal + per_slot <= kWideSmem
                        ? static_cast<int>(std::min<size_t>(kWideMaxWarps / EG, (kWideSmem - wal) / per_slot)) : 0;
    if (a.x && !a.rmsnorm && !a.mxd_xs && a.T > 64 && a.E <= 32 && a.H % 8 == 0 && a.H <= 8 * 32 * kWideMaxV &&
        tpc >= 2 && (reinterpret_cast<uintptr_t>(a.Wr) & 15) == 0 && (reinterpret_cast<uintptr_t>(a.x) & 15) == 0) {
        int dev = 0, sms = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        const size_t smem = wal + static_cast<size_t>(tpc) * per_slot;
        const int grid = std::min(sms, (a.T + tpc - 1) / tpc);
        auto kern = EG == 1 ? router_wide_kernel<1> : EG == 2 ? router_wide_kernel<2>
                  : EG == 3 ? router_wide_kernel<3> : router_wide_kernel<4>;
        e = ensure_smem(kern, smem);
        if (e != cudaSuccess) return e;
        return launch_pdl(kern, dim3(grid), dim3(tpc * EG * 32), smem, s, a);
    }
    const RouterPlan p = router_plan(a.T, a.H, a.E, a.x != nullptr);
    auto kern = a.mxd_xs ? router_kernel<true> : router_kernel<false>;
    cudaError_t e = ensure_smem(kern, p.smem);
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
    return cudaLaunchKernelEx(&cfg, kern, a, p);
}

cudaError_t launch_build_routes(const int32_t* idx, int T, int E, int k, int32_t* off,
                                int32_t* perm, int32_t* inv, int* status, cudaStream_t s) {
    return launch_pdl(build_routes_kernel, dim3(1), dim3(kBuildThreads), 0, s, idx, T * k, E, off,
                      perm, inv, status);
}

}  // namespace tsmoe

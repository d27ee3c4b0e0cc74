// gemv.cu -- steps 4-5 of the routed-expert layer for small token counts (decode): the
// per-expert gated FFN as a weight-streaming GEMV on sm_103a.
//
// Source pages (docs.rs, turbospark-runtime 0.3.0):
//   gpt-oss routed-expert pass (src/families/gptoss/moe.rs): phase 1 (gate/up + activation
//     into the 16-bit acts buffer) and phase 2 (down projection), encode_moe_phase{1,2}_any;
//     module header: the clamped SwiGLU and the per-expert biases ride inside the MXFP4 pair,
//     has_bias follows from a non-zero bias offset.
//   Gemma-4 batched routed prefill (src/families/gemma4/moe_batch.rs): the INT4-affine blobs
//     and the shared expert (a dense gated FFN on every token).
//   Llama/Mixtral decode flow (src/families/llama/mod.rs): use_silu, else gelu-tanh.
//
// Design (GB300):
//   * A unit is (touched expert, 16-row tile, group of <= 8 tokens routed to that expert).
//     Every touched expert's weights are streamed from HBM once per call, whatever the number
//     of tokens routed to it (<= 8 per group).
//   * One producer warp streams the units' weight tiles into a ring of shared-memory stages
//     with cp.async.bulk (the bulk-copy engine), completion on mbarriers.  Quantised weights
//     are pre-packed (ts_moe_pack) so a 16-row tile chunk is ONE contiguous copy.
//   * Eight consumer warps split each tile's 32-column blocks.  They dequantise in registers
//     (e2m1 pairs through the hardware converter, INT4 through the 1024-offset f16 trick) and
//     feed mma.sync m16n8k16 (16 weight rows x 8 tokens): the tensor pipe takes the
//     multiply-adds so the ALUs only pay for the dequantisation and keep pace with HBM.
//     MXFP4 blocks are multiplied unscaled and the e8m0 scale is applied to the block's f32
//     partial product, so no scale range restriction arises.
//   * Activations enter the f16 mma with a per-token power-of-two prescale (max |x| in
//     [2^14, 2^15)), exact for bf16 inputs in f16's range, undone in f32 after the sum.
//   * Partial sums of the eight warps are reduced through shared memory in fixed warp order:
//     results are deterministic run to run.
#include "common.cuh"

namespace tsmoe {

namespace {

constexpr int kNCW = 16;                      // consumer warps
constexpr int kThreads = (kNCW + 2) * 32;     // + one producer warp + one reducer warp
constexpr int kMaxLocalRoutes = 512;          // route lists built inside the kernel up to this
constexpr int kStageBytes = 24576;
constexpr int kMaxStages = 6;
constexpr int kSmemBudget = 225 * 1024;

struct Plan {                                 // host-computed launch shape
    int nstages, tg, nb;                      // ring stages, tokens per group, blocks per stage
    int row_stride;                           // 16-bit formats: smem bytes per row in a stage
    int xstride;                              // smem bytes per staged activation row
    size_t smem;
};

__host__ __device__ inline int round_up(int v, int m) { return (v + m - 1) / m * m; }

__host__ inline Plan make_plan(int fmt, int K, int tg_cap) {
    Plan p{};
    const int nblk = K / kBlockK;
    if (fmt == FMT_MXFP4 || fmt == FMT_INT4) {
        p.nb = kStageBytes / packed_block_bytes(fmt);
        p.row_stride = 0;
    } else {
        // 16 rows x (nb*64 + 64) bytes, nb even so the row stride is 64 mod 128 (no bank
        // conflicts on the 16-byte fragment loads)
        p.nb = ((kStageBytes / kRowTile - 64) / 64) & ~1;
        p.row_stride = p.nb * 64 + 64;
    }
    if (p.nb > nblk) {
        p.nb = nblk;
        if (p.row_stride) p.row_stride = round_up(p.nb, 2) * 64 + 64;
    }
    p.xstride = round_up(2 * K, 128) + 64;
    const size_t fixed = static_cast<size_t>(2) * kNCW * 2 * kRowTile * 8 * 4   // reduction x2
                         + static_cast<size_t>(nblk) * 8 * 4                  // INT4 x sums
                         + 8 * 4                                             // inverse prescale
                         + 2 * kMaxStages * 8                                // mbarriers
                         + (3 * kMaxExperts + 1 + 8) * 4                     // unit tables
                         + 2 * 8 * 4 + 4 * 8                                 // reducer hand-off
                         + (kMaxExperts + 1 + kMaxLocalRoutes) * 4            // in-kernel routes
                         + 16 * 16;                                           // region padding
    for (int ns = kMaxStages; ns >= 2; --ns) {
        const size_t ring = static_cast<size_t>(ns) * kStageBytes;
        if (ring + fixed >= static_cast<size_t>(kSmemBudget)) continue;
        int tg = static_cast<int>((kSmemBudget - ring - fixed) / p.xstride);
        if (tg > 8) tg = 8;
        if (tg >= tg_cap || ns == 2) {
            p.nstages = ns;
            p.tg = tg < tg_cap ? tg : tg_cap;
            break;
        }
    }
    if (p.tg < 1) { p.tg = 0; return p; }
    p.smem = static_cast<size_t>(p.nstages) * kStageBytes + static_cast<size_t>(p.tg) * p.xstride +
             fixed + 128;
    return p;
}

struct KParams {
    GemvArgs a;
    Plan p;
};

// smem carve-up (all offsets 16-byte aligned)
struct Carve {
    unsigned char* ring;
    unsigned char* xs;
    float* xsum;      // [nblk][8]
    float* xinv;      // [8]
    float* red;       // [2 buffers][kNCW][2][16][8]
    uint64_t* full;   // [nstages]
    uint64_t* empty;  // [nstages]
    int* touched;     // [256]
    int* cnt;         // [256]
    int* goff;        // [257]
    int* misc;        // [8]: 0 = ntouched, 1 = abort flag
    float* rinv;      // [2][8]: prescale inverses travelling with the partials
    uint64_t* rfull;  // [2]: partials of a unit written (16 compute warps arrive)
    uint64_t* rempty; // [2]: partial buffer read by the reducer
    int* off_s;       // [257]: route offsets built in the kernel
    int* perm_s;      // [512]: route list built in the kernel
};

__device__ inline Carve carve(unsigned char* base, const Plan& p, int K) {
    Carve c;
    unsigned char* q = base;
    // every region starts on a 16-byte boundary (the mbarriers need 8)
    auto take = [&](size_t bytes) {
        unsigned char* r = q;
        q += (bytes + 15) & ~static_cast<size_t>(15);
        return r;
    };
    c.ring = take(static_cast<size_t>(p.nstages) * kStageBytes);
    c.xs = take(static_cast<size_t>(p.tg) * p.xstride);
    c.xsum = reinterpret_cast<float*>(take(static_cast<size_t>(K / kBlockK) * 8 * 4));
    c.xinv = reinterpret_cast<float*>(take(8 * 4));
    c.red = reinterpret_cast<float*>(take(2 * kNCW * 2 * kRowTile * 8 * 4));
    c.full = reinterpret_cast<uint64_t*>(take(kMaxStages * 8));
    c.empty = reinterpret_cast<uint64_t*>(take(kMaxStages * 8));
    c.rfull = reinterpret_cast<uint64_t*>(take(2 * 8));
    c.rempty = reinterpret_cast<uint64_t*>(take(2 * 8));
    c.touched = reinterpret_cast<int*>(take(kMaxExperts * 4));
    c.cnt = reinterpret_cast<int*>(take(kMaxExperts * 4));
    c.goff = reinterpret_cast<int*>(take((kMaxExperts + 1) * 4));
    c.misc = reinterpret_cast<int*>(take(8 * 4));
    c.rinv = reinterpret_cast<float*>(take(2 * 8 * 4));
    c.off_s = reinterpret_cast<int*>(take((kMaxExperts + 1) * 4));
    c.perm_s = reinterpret_cast<int*>(take(kMaxLocalRoutes * 4));
    return c;
}

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

// Unit u -> (touched index j, row tile, group).  `j` is a running hint (units are visited in
// increasing order).
__device__ __forceinline__ void decode_unit(int u, int RT, const int* goff, int nt, int& j,
                                            int& rt, int& g, const int* cnt, int tg) {
    while (j + 1 < nt && u >= RT * goff[j + 1]) ++j;
    const int ng = (cnt[j] + tg - 1) / tg;
    const int local = u - RT * goff[j];
    rt = local / ng;
    g = local % ng;
}

// Stages one activation row into shared memory in the mma operand type: f16 with a
// power-of-two prescale (max |x| * 2^ks in [2^14, 2^15)) when bf16 activations feed the f16
// mma, else the bits as they are; element order inside each 8-group is natural, or
// (0,4,1,5,2,6,3,7) for INT4.  For K <= 3072 the row is read once, with every load issued
// before any is used; returns the inverse prescale.
template <int FMT>
__device__ __forceinline__ float stage_row(const uint16_t* __restrict__ src, unsigned char* xrow,
                                           float* xsum, int col, int K, int nblk, bool prescale,
                                           bool copy_bits, int lane) {
    auto store_block = [&](int blk, const uint32_t (&wv)[16], float scl) {
        uint16_t o[32];
        float bsum = 0.0f;
#pragma unroll
        for (int q = 0; q < 32; ++q) {
            const uint16_t bits = static_cast<uint16_t>((q & 1) ? (wv[q >> 1] >> 16) : (wv[q >> 1] & 0xFFFF));
            uint16_t ob;
            if (copy_bits) {
                ob = bits;
            } else {
                const float v = __fmul_rn(__bfloat162float(__ushort_as_bfloat16(bits)), scl);
                ob = __half_as_ushort(__float2half_rn(v));
            }
            if (FMT == FMT_INT4) bsum += __half2float(__ushort_as_half(ob));
            o[q] = ob;
        }
        uint32_t pk[16];
#pragma unroll
        for (int q8 = 0; q8 < 4; ++q8) {
#pragma unroll
            for (int pr = 0; pr < 4; ++pr) {
                uint16_t lo, hi;
                if (FMT == FMT_INT4) { lo = o[q8 * 8 + pr]; hi = o[q8 * 8 + pr + 4]; }
                else { lo = o[q8 * 8 + 2 * pr]; hi = o[q8 * 8 + 2 * pr + 1]; }
                pk[q8 * 4 + pr] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
            }
        }
        uint4* d4 = reinterpret_cast<uint4*>(xrow + static_cast<size_t>(blk) * 64);
#pragma unroll
        for (int h = 0; h < 4; ++h) d4[h] = make_uint4(pk[4 * h], pk[4 * h + 1], pk[4 * h + 2], pk[4 * h + 3]);
        if (FMT == FMT_INT4) xsum[blk * 8 + col] = bsum;
    };
    auto absmax16 = [&](const uint32_t (&wv)[16]) {
        float mx = 0.0f;
#pragma unroll
        for (int h = 0; h < 16; ++h) {
            mx = fmaxf(mx, fabsf(__bfloat162float(__ushort_as_bfloat16(wv[h] & 0xFFFF))));
            mx = fmaxf(mx, fabsf(__bfloat162float(__ushort_as_bfloat16(wv[h] >> 16))));
        }
        return mx;
    };
    auto prescale_of = [&](float mx, float& scl, float& inv) {
        scl = inv = 1.0f;
        if (mx > 0.0f && mx < 3.0e38f) {
            int ex;
            frexpf(mx, &ex);            // mx = f * 2^ex, f in [0.5, 1)
            const int ks = max(-120, min(120, 15 - ex));
            scl = __uint_as_float(static_cast<uint32_t>(ks + 127) << 23);
            inv = __uint_as_float(static_cast<uint32_t>(127 - ks) << 23);
        }
    };
    float scl = 1.0f, inv = 1.0f;
    if (nblk <= 96) {
        uint32_t wv[3][16];
#pragma unroll
        for (int q = 0; q < 3; ++q) {
            const int blk = lane + 32 * q;
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                uint4 v = make_uint4(0, 0, 0, 0);
                if (blk < nblk) v = __ldg(reinterpret_cast<const uint4*>(src + blk * kBlockK) + h);
                wv[q][4 * h] = v.x; wv[q][4 * h + 1] = v.y; wv[q][4 * h + 2] = v.z; wv[q][4 * h + 3] = v.w;
            }
        }
        if (prescale) {
            float mx = fmaxf(fmaxf(absmax16(wv[0]), absmax16(wv[1])), absmax16(wv[2]));
            prescale_of(warp_max(mx), scl, inv);
        }
#pragma unroll
        for (int q = 0; q < 3; ++q)
            if (lane + 32 * q < nblk) store_block(lane + 32 * q, wv[q], scl);
        return inv;
    }
    if (prescale) {
        float mx = 0.0f;
        for (int blk = lane; blk < nblk; blk += 32) {
            uint32_t wv[16];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const uint4 v = __ldg(reinterpret_cast<const uint4*>(src + blk * kBlockK) + h);
                wv[4 * h] = v.x; wv[4 * h + 1] = v.y; wv[4 * h + 2] = v.z; wv[4 * h + 3] = v.w;
            }
            mx = fmaxf(mx, absmax16(wv));
        }
        prescale_of(warp_max(mx), scl, inv);
    }
    for (int blk = lane; blk < nblk; blk += 32) {
        uint32_t wv[16];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(src + blk * kBlockK) + h);
            wv[4 * h] = v.x; wv[4 * h + 1] = v.y; wv[4 * h + 2] = v.z; wv[4 * h + 3] = v.w;
        }
        store_block(blk, wv, scl);
    }
    return inv;
}

template <int FMT>
__global__ void __launch_bounds__(kThreads, 1) gemv_kernel(const __grid_constant__ KParams P) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const GemvArgs& a = P.a;
    const Plan& p = P.p;
    const int K = a.K, R = a.R;
    const int nblk = K / kBlockK;
    const int RT = R / kRowTile;
    const int nmat = a.phase == 0 ? 2 : 1;
    const int nchunk = (nblk + p.nb - 1) / p.nb;
    const int tg = p.tg;
    constexpr bool kPacked = (FMT == FMT_MXFP4 || FMT == FMT_INT4);
    constexpr int BB = kPacked ? packed_block_bytes(FMT) : 0;
    constexpr bool kMmaBf16 = (FMT == FMT_BF16);
    const bool prescale = !kMmaBf16 && a.adt == 1;

    Carve c = carve(smem_raw, p, K);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // ---- route list (built here for decode sizes), unit tables --------------------------------
    const int* OFF = a.off;
    const int* PERM = a.perm;
    if (a.idx) {
        OFF = c.off_s;
        PERM = c.perm_s;
    }
    if (threadIdx.x == 0) {
        if (a.idx) {
            // counting sort of the route ids by expert, ascending id inside an expert
            const int n = a.T * a.k;
            for (int e = 0; e <= a.E; ++e) c.off_s[e] = 0;
            for (int r = 0; r < n; ++r) {
                const int e = a.idx[r];
                if (e >= 0 && e < a.E) c.off_s[e + 1] += 1;
                else report_error(a.status, DEV_ERR_INVALID);
            }
            for (int e = 0; e < a.E; ++e) c.off_s[e + 1] += c.off_s[e];
            for (int e = 0; e < a.E; ++e) c.cnt[e] = c.off_s[e];     // cursors (cnt reused)
            for (int r = 0; r < n; ++r) {
                const int e = a.idx[r];
                if (e >= 0 && e < a.E) c.perm_s[c.cnt[e]++] = r;
            }
        }
        int nt = 0, acc = 0;
        if (a.dense) {
            c.touched[0] = 0;
            c.cnt[0] = a.T;
            c.goff[0] = 0;
            acc = (a.T + tg - 1) / tg;
            nt = 1;
        } else {
            for (int e = 0; e < a.E; ++e) {
                const int n = OFF[e + 1] - OFF[e];
                if (n > 0) {
                    c.touched[nt] = e;
                    c.cnt[nt] = n;
                    c.goff[nt] = acc;
                    acc += (n + tg - 1) / tg;
                    ++nt;
                }
            }
        }
        c.goff[nt] = acc;
        c.misc[0] = nt;
        c.misc[1] = 0;
        for (int s = 0; s < p.nstages; ++s) {
            mbar_init(&c.full[s], 1);
            mbar_init(&c.empty[s], kNCW);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&c.rfull[b], kNCW);
            mbar_init(&c.rempty[b], 1);
        }
        fence_mbar_init();
    }
    // the phase-1 launch clears the combine counters the phase-2 launch will count with
    if (a.cmb_mode == 1 && blockIdx.x == 0)
        for (int i = threadIdx.x; i < a.cmb_n; i += blockDim.x) a.cmb_cnt[i] = 0;
    __syncthreads();
    const int nt = c.misc[0];
    const int U = RT * c.goff[nt];
    const int u0 = static_cast<int>((static_cast<long long>(U) * blockIdx.x) / gridDim.x);
    const int u1 = static_cast<int>((static_cast<long long>(U) * (blockIdx.x + 1)) / gridDim.x);
    if (u0 >= u1) return;

    if (warp == kNCW + 1) {
        // ================================ reducer warp ======================================
        // Sums the 16 compute warps' partials of each unit in fixed warp order, applies the
        // prescale inverse, bias and activation, stores the unit's outputs; in phase 2 of a
        // routed decode call the last unit of each 16-row tile also runs the slot-ordered
        // combine for that tile.
        int j = 0;
        for (int u = u0; u < u1; ++u) {
            int rt, g;
            decode_unit(u, RT, c.goff, nt, j, rt, g, c.cnt, tg);
            const int e = c.touched[j];
            const int cnt_g = min(tg, c.cnt[j] - g * tg);
            const int rbase = a.dense ? g * tg : OFF[e] + g * tg;
            const int nl = u - u0, b = nl & 1;
            const bool ok = c.misc[1] == 0 && mbar_wait_bounded(&c.rfull[b], (nl >> 1) & 1);
            if (!ok) {
                if (lane == 0 && c.misc[1] == 0) {
                    c.misc[1] = 1;
                    report_error(a.status, DEV_ERR_TIMEOUT);
                }
            } else {
                const float* redb = c.red + static_cast<size_t>(b) * kNCW * 2 * kRowTile * 8;
                for (int o = lane; o < kRowTile * 8; o += 32) {
                    const int n = o / kRowTile, row = o % kRowTile;
                    if (n >= cnt_g) continue;
                    const int rid = a.dense ? rbase + n : PERM[rbase + n];
                    const int orow = rt * kRowTile + row;
                    float s0 = 0.0f, s1 = 0.0f;
                    for (int w = 0; w < kNCW; ++w) {
                        s0 += redb[(w * 2 + 0) * kRowTile * 8 + row * 8 + n];
                        if (nmat == 2) s1 += redb[(w * 2 + 1) * kRowTile * 8 + row * 8 + n];
                    }
                    const float inv = c.rinv[b * 8 + n];
                    s0 *= inv;
                    s1 *= inv;
                    const size_t bidx = static_cast<size_t>(e) * R + orow;
                    if (a.b0) s0 += __bfloat162float(__ushort_as_bfloat16(a.b0[bidx]));
                    if (a.phase == 0) {
                        if (a.b1) s1 += __bfloat162float(__ushort_as_bfloat16(a.b1[bidx]));
                        const float h = act_fn(a.act, s0, s1, a.limit, a.alpha);
                        static_cast<uint16_t*>(a.out)[static_cast<size_t>(rid) * R + orow] = float_to_adt_bits(h, a.adt);
                    } else {
                        static_cast<float*>(a.out)[static_cast<size_t>(rid) * R + orow] = s0;
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&c.rempty[b]);
        }
        if (a.cmb_mode == 2 && c.misc[1] == 0) {
            // Fused combine: every unit of a 16-row tile (over all CTAs) bumps that tile's
            // counter once this CTA's outputs are globally visible (one fence for all of them);
            // the CTA that completes a tile's count runs the slot-ordered combine for it.
            __threadfence();
            __syncwarp();
            j = 0;
            for (int u = u0; u < u1; ++u) {
                int rt, g;
                decode_unit(u, RT, c.goff, nt, j, rt, g, c.cnt, tg);
                int last = 0;
                if (lane == 0) last = (atomicAdd(a.cmb_cnt + rt, 1) + 1 == c.goff[nt]);
                last = __shfl_sync(0xffffffffu, last, 0);
                if (!last) continue;
                __threadfence();
                const float* ev = static_cast<const float*>(a.out);
                for (int o = lane; o < a.T * kRowTile; o += 32) {
                    const int t = o / kRowTile, orow = rt * kRowTile + o % kRowTile;
                    const size_t yo = static_cast<size_t>(t) * R + orow;
                    float accv = a.seed ? __ldcg(a.seed + yo) : 0.0f;
                    for (int q = 0; q < a.k; ++q) {
                        const size_t r = static_cast<size_t>(t) * a.k + q;
                        accv = __fadd_rn(accv, __fmul_rn(a.w[r], __ldcg(ev + r * R + orow)));
                    }
                    if (a.y_f32) a.y_f32[yo] = accv;
                    static_cast<uint16_t*>(a.y)[yo] = float_to_adt_bits(accv, a.adt);
                }
                if (lane == 0) a.cmb_cnt[rt] = 0;
            }
        }
        return;
    }

    if (warp == kNCW) {
        // ================================ producer warp =====================================
        int it = 0, j = 0;
        for (int u = u0; u < u1; ++u) {
            int rt, g;
            decode_unit(u, RT, c.goff, nt, j, rt, g, c.cnt, tg);
            const int e = c.touched[j];
            for (int m = 0; m < nmat; ++m) {
                const uint8_t* wbase = (m == 0 ? a.w0 : a.w1) + static_cast<size_t>(e) * a.mat_bytes;
                for (int ch = 0; ch < nchunk; ++ch, ++it) {
                    const int s = it % p.nstages;
                    const uint32_t par = ((it / p.nstages) & 1) ^ 1;
                    const int b0 = ch * p.nb;
                    const int nbc = min(p.nb, nblk - b0);
                    bool ok = true;
                    if (lane == 0) ok = c.misc[1] || mbar_wait_bounded(&c.empty[s], par);
                    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0);
                    if (!ok) {
                        if (lane == 0) { c.misc[1] = 1; report_error(a.status, DEV_ERR_TIMEOUT); }
                    }
                    __syncwarp();
                    if (c.misc[1]) continue;
                    unsigned char* dst = c.ring + static_cast<size_t>(s) * kStageBytes;
                    if (kPacked) {
                        if (lane == 0) {
                            const uint32_t bytes = static_cast<uint32_t>(nbc) * BB;
                            const uint8_t* src = wbase + (static_cast<size_t>(rt) * nblk + b0) * BB;
                            mbar_arrive_expect_tx(&c.full[s], bytes);
                            bulk_g2s(dst, src, bytes, &c.full[s]);
                        }
                    } else {
                        if (lane == 0)
                            mbar_arrive_expect_tx(&c.full[s], static_cast<uint32_t>(nbc) * 64 * kRowTile);
                        __syncwarp();
                        if (lane < kRowTile) {
                            const size_t row = static_cast<size_t>(rt) * kRowTile + lane;
                            const uint8_t* src = wbase + (row * K + static_cast<size_t>(b0) * kBlockK) * 2;
                            bulk_g2s(dst + lane * p.row_stride, src, static_cast<uint32_t>(nbc) * 64,
                                     &c.full[s]);
                        }
                    }
                    __syncwarp();
                }
            }
        }
        // if the consumers gave up, wait (bounded) for the copies still in flight
        if (c.misc[1] && lane == 0) {
            for (int q = (it > p.nstages ? it - p.nstages : 0); q < it; ++q)
                mbar_wait_bounded(&c.full[q % p.nstages], (q / p.nstages) & 1);
        }
        return;
    }

    // ================================== consumer warps =========================================
    const int gid = lane >> 2, tid = lane & 3;
    int it = 0, j = 0;
    int staged_j = -1, staged_g = -1;
    const uint16_t* in = a.in;
    const bool copy_bits = kMmaBf16 || a.adt == 0;
    // Phase 1 with at most tg tokens: every token's row is staged once here (x is per token and
    // shared by every expert), and the units index it by token; otherwise rows are staged per
    // group of routes when the group changes.
    const bool tokmode = a.phase == 0 && a.T <= tg;
    if (tokmode) {
        if (warp < 8) {
            const int t = warp;
            float inv = 0.0f;
            if (t < a.T) {
                inv = stage_row<FMT>(in + static_cast<size_t>(t) * K, c.xs + static_cast<size_t>(t) * p.xstride,
                                     c.xsum, t, K, nblk, prescale, copy_bits, lane);
            } else if (FMT == FMT_INT4) {
                for (int blk = lane; blk < nblk; blk += 32) c.xsum[blk * 8 + t] = 0.0f;
            }
            if (lane == 0) c.xinv[t] = inv;
        }
        named_bar(1, kNCW * 32);
    }

    for (int u = u0; u < u1; ++u) {
        int rt, g;
        decode_unit(u, RT, c.goff, nt, j, rt, g, c.cnt, tg);
        const int e = c.touched[j];
        const int cnt_g = min(tg, c.cnt[j] - g * tg);
        const int rbase = a.dense ? g * tg : OFF[e] + g * tg;
        // staged row of each of the unit's columns (routes): the token in token mode
        auto row_of = [&](int n) {
            if (!tokmode) return n < tg ? n : 0;
            if (n >= cnt_g) return 0;
            return a.dense ? rbase + n : PERM[rbase + n] / a.k;
        };
        const int brow = row_of(gid);                 // activation row this lane feeds the mma
        const int xc0 = row_of(2 * tid), xc1 = row_of(2 * tid + 1);   // INT4 x-sum columns

        // ---- stage this group's activations (f16 with prescale, or as-is) -----------------
        if (!tokmode && (j != staged_j || g != staged_g)) {
            // every compute warp must be done with the previous group's activations
            if (staged_j >= 0) named_bar(1, kNCW * 32);
            staged_j = j;
            staged_g = g;
            if (warp < 8) {
                const int n = warp;
                float inv = 0.0f;
                if (n < cnt_g) {
                    const int rid = a.dense ? rbase + n : PERM[rbase + n];
                    size_t row;
                    if (a.phase == 0) row = a.dense ? static_cast<size_t>(rid) : static_cast<size_t>(rid / a.k);
                    else row = static_cast<size_t>(rid);
                    inv = stage_row<FMT>(in + row * K, c.xs + static_cast<size_t>(n) * p.xstride, c.xsum, n,
                                         K, nblk, prescale, copy_bits, lane);
                } else {
                    if (n < tg) {
                        unsigned char* xrow = c.xs + static_cast<size_t>(n) * p.xstride;
                        for (int q = lane; q < K / 8; q += 32)
                            reinterpret_cast<uint4*>(xrow)[q] = make_uint4(0, 0, 0, 0);
                    }
                    if (FMT == FMT_INT4)
                        for (int blk = lane; blk < nblk; blk += 32) c.xsum[blk * 8 + n] = 0.0f;
                }
                if (lane == 0) c.xinv[n] = inv;
            }
            named_bar(1, kNCW * 32);
        }

        // ---- stream the unit's weight chunks ---------------------------------------------------
        float acc[2][4];
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[m][q] = 0.0f;

        for (int m = 0; m < nmat; ++m) {
            for (int ch = 0; ch < nchunk; ++ch, ++it) {
                const int s = it % p.nstages;
                const uint32_t par = (it / p.nstages) & 1;
                const int b0 = ch * p.nb;
                const int nbc = min(p.nb, nblk - b0);
                bool ok = c.misc[1] == 0 && mbar_wait_bounded(&c.full[s], par);
                if (!ok) {
                    if (lane == 0 && c.misc[1] == 0) {
                        c.misc[1] = 1;
                        report_error(a.status, DEV_ERR_TIMEOUT);
                    }
                } else {
                    const unsigned char* st = c.ring + static_cast<size_t>(s) * kStageBytes;
                    const unsigned char* xrow = c.xs + static_cast<size_t>(brow) * p.xstride + tid * 16;
                    float* ac = acc[m];
                    auto block = [&](int i) {
                        const uint4 bx = *reinterpret_cast<const uint4*>(xrow + static_cast<size_t>(b0 + i) * 64);
                        if (FMT == FMT_MXFP4) {
                            const unsigned char* blk = st + static_cast<size_t>(i) * BB;
                            const uint2 cw = *reinterpret_cast<const uint2*>(blk + lane * 8);
                            const uint32_t sc = *reinterpret_cast<const uint16_t*>(blk + 256 + gid * 2);
                            uint32_t pa[4], pb[4];
                            e2m1x8_to_f16x2x4(cw.x, pa);
                            e2m1x8_to_f16x2x4(cw.y, pb);
                            float d[4] = {0.f, 0.f, 0.f, 0.f};
                            mma_f16_16816(d, pa[0], pb[0], pa[1], pb[1], bx.x, bx.y);
                            mma_f16_16816(d, pa[2], pb[2], pa[3], pb[3], bx.z, bx.w);
                            const float s0 = e8m0_to_float(sc & 0xFF), s1 = e8m0_to_float(sc >> 8);
                            ac[0] = fmaf(d[0], s0, ac[0]);
                            ac[1] = fmaf(d[1], s0, ac[1]);
                            ac[2] = fmaf(d[2], s1, ac[2]);
                            ac[3] = fmaf(d[3], s1, ac[3]);
                        } else if (FMT == FMT_INT4) {
                            const unsigned char* blk = st + static_cast<size_t>(i) * BB;
                            const uint2 cw = *reinterpret_cast<const uint2*>(blk + lane * 8);
                            const uint2 smv = *reinterpret_cast<const uint2*>(blk + 256 + gid * 8);
                            const float2 xsm = make_float2(c.xsum[(b0 + i) * 8 + xc0], c.xsum[(b0 + i) * 8 + xc1]);
                            float d[4] = {0.f, 0.f, 0.f, 0.f};
                            mma_f16_16816(d, u4pair_to_f16x2(cw.x, 0), u4pair_to_f16x2(cw.y, 0),
                                          u4pair_to_f16x2(cw.x, 4), u4pair_to_f16x2(cw.y, 4), bx.x, bx.y);
                            mma_f16_16816(d, u4pair_to_f16x2(cw.x, 8), u4pair_to_f16x2(cw.y, 8),
                                          u4pair_to_f16x2(cw.x, 12), u4pair_to_f16x2(cw.y, 12), bx.z, bx.w);
                            const float sg = __half2float(__ushort_as_half(smv.x & 0xFFFF));
                            const float mg = __half2float(__ushort_as_half(smv.x >> 16));
                            const float sg8 = __half2float(__ushort_as_half(smv.y & 0xFFFF));
                            const float mg8 = __half2float(__ushort_as_half(smv.y >> 16));
                            ac[0] = fmaf(sg, d[0], fmaf(mg, xsm.x, ac[0]));
                            ac[1] = fmaf(sg, d[1], fmaf(mg, xsm.y, ac[1]));
                            ac[2] = fmaf(sg8, d[2], fmaf(mg8, xsm.x, ac[2]));
                            ac[3] = fmaf(sg8, d[3], fmaf(mg8, xsm.y, ac[3]));
                        } else {
                            const unsigned char* ra = st + static_cast<size_t>(gid) * p.row_stride + i * 64 + tid * 16;
                            const uint4 wa = *reinterpret_cast<const uint4*>(ra);
                            const uint4 wb = *reinterpret_cast<const uint4*>(ra + 8 * p.row_stride);
                            float d[4] = {0.f, 0.f, 0.f, 0.f};
                            if (kMmaBf16) {
                                mma_bf16_16816(d, wa.x, wb.x, wa.y, wb.y, bx.x, bx.y);
                                mma_bf16_16816(d, wa.z, wb.z, wa.w, wb.w, bx.z, bx.w);
                            } else {
                                mma_f16_16816(d, wa.x, wb.x, wa.y, wb.y, bx.x, bx.y);
                                mma_f16_16816(d, wa.z, wb.z, wa.w, wb.w, bx.z, bx.w);
                            }
                            ac[0] += d[0];
                            ac[1] += d[1];
                            ac[2] += d[2];
                            ac[3] += d[3];
                        }
                    };
                    // two blocks in flight per warp: independent fragments, interleavable
                    int i = warp;
                    for (; i + kNCW < nbc; i += 2 * kNCW) {
                        block(i);
                        block(i + kNCW);
                    }
                    if (i < nbc) block(i);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&c.empty[s]);
            }
        }

        // ---- hand the partials to the reducer warp (double-buffered, no CTA barrier) ---------
        {
            const int nl = u - u0, b = nl & 1;
            const bool ok = c.misc[1] == 0 && mbar_wait_bounded(&c.rempty[b], ((nl >> 1) & 1) ^ 1);
            if (!ok) {
                if (lane == 0 && c.misc[1] == 0) {
                    c.misc[1] = 1;
                    report_error(a.status, DEV_ERR_TIMEOUT);
                }
            }
            float* rw = c.red + (static_cast<size_t>(b) * kNCW + warp) * 2 * kRowTile * 8;
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                if (m >= nmat) break;
                float* rm = rw + m * kRowTile * 8;
                rm[gid * 8 + 2 * tid] = acc[m][0];
                rm[gid * 8 + 2 * tid + 1] = acc[m][1];
                rm[(gid + 8) * 8 + 2 * tid] = acc[m][2];
                rm[(gid + 8) * 8 + 2 * tid + 1] = acc[m][3];
            }
            if (warp == 0 && lane < 8) c.rinv[b * 8 + lane] = c.xinv[row_of(lane)];
            __syncwarp();
            if (lane == 0) mbar_arrive(&c.rfull[b]);
        }
    }
}

}  // namespace

int gemv_pick_tg(int K) { return make_plan(FMT_F16, K, 8).tg; }

size_t gemv_smem_bytes(int fmt, int K, int tg) { return make_plan(fmt, K, tg).smem; }

cudaError_t launch_gemv(const GemvArgs& a, int num_sms, cudaStream_t s) {
    KParams P;
    P.a = a;
    const int tmax = a.dense ? a.T : a.T;   // tokens per expert never exceed T
    P.p = make_plan(a.fmt, a.K, tmax < 8 ? (tmax > 0 ? tmax : 1) : 8);
    if (P.p.tg < 1) return cudaErrorInvalidValue;
    P.a.tg = P.p.tg;
    void (*kern)(const KParams);
    switch (a.fmt) {
        case FMT_F16: kern = gemv_kernel<FMT_F16>; break;
        case FMT_BF16: kern = gemv_kernel<FMT_BF16>; break;
        case FMT_MXFP4: kern = gemv_kernel<FMT_MXFP4>; break;
        default: kern = gemv_kernel<FMT_INT4>; break;
    }
    cudaError_t e;
    switch (a.fmt) {
        case FMT_F16: e = ensure_smem(gemv_kernel<FMT_F16>, P.p.smem); break;
        case FMT_BF16: e = ensure_smem(gemv_kernel<FMT_BF16>, P.p.smem); break;
        case FMT_MXFP4: e = ensure_smem(gemv_kernel<FMT_MXFP4>, P.p.smem); break;
        default: e = ensure_smem(gemv_kernel<FMT_INT4>, P.p.smem); break;
    }
    if (e != cudaSuccess) return e;
    kern<<<num_sms, kThreads, P.p.smem, s>>>(P);
    return cudaGetLastError();
}

}  // namespace tsmoe

// gemv_sk.cu -- steps 4-5 of the routed-expert layer for few tokens (decode) with packed INT4
// weights (the block code also covers MXFP4): a weight-streaming GEMV in which every warp works
// on its own.
//
// Source pages (docs.rs, turbospark-runtime 0.3.0):
//   gpt-oss routed-expert pass (src/families/gptoss/moe.rs): phase 1 (gate/up + activation into
//     the 16-bit acts buffer) and phase 2 (down projection), encode_moe_phase{1,2}_any; the
//     clamped SwiGLU and the per-expert biases ride inside the MXFP4 pair.
//   Gemma-4 batched routed prefill (src/families/gemma4/moe_batch.rs): the INT4-affine blobs.
//
// Design (GB300):
//   * A unit is (touched expert, 16-row tile, group of <= 8 routes of that expert); each unit's
//     weights are streamed once per call whatever its number of routes.  The units of a CTA
//     are cut into chunks (a run of up to `cb` 32-column blocks of one matrix, one contiguous
//     piece of the packed layout), and the CTA's chunk sequence is split evenly over its 16
//     warps: each warp owns a contiguous range of chunks.
//   * Every warp streams its own chunks through its own three-slot ring (one cp.async.bulk per
//     chunk issued by the warp itself, mbarrier completion): no producer warp, no stage shared
//     between warps, no per-unit hand-off.
//   * Per block: e2m1 pairs (or INT4 codes) to f16 in registers, two mma.sync m16n8k16 (16
//     weight rows x 8 routes) against the staged activations, the e8m0 scale applied to the
//     block's f32 partial (so any scale is exact).
//   * A unit that lies entirely in one warp's range is finished by that warp: prescale inverse,
//     bias, activation, store.  A unit split between consecutive warps is finished by the last
//     of them to arrive: each writes its partial sums to shared memory, and the last sums the
//     parts in warp order (= K order), so the result does not depend on timing.
//   * Activations: f16 with a per-row power-of-two prescale (max |x| in [2^14, 2^15)).  In phase
//     1 with at most 8 tokens every token's row is staged once and the units index it by
//     token; otherwise the rows of a route group are restaged when the group changes (all
//     warps step through the groups together).
#include "gemv_common.cuh"

namespace tsmoe {

namespace {

constexpr int kW = 16;                       // warps per CTA, all compute
constexpr int kThr = kW * 32;
constexpr int kSlots = 3;                    // ring slots per warp
constexpr int kSkBudget = 225 * 1024;
constexpr int kChunkMx = 9;                  // blocks per chunk, MXFP4 (2448 bytes)
constexpr int kChunkI4 = 8;                  // blocks per chunk, INT4 (2560 bytes)
constexpr int kPrefetch = 0;                 // chunks pulled into L2 beyond the ring (0: none)

// Bulk prefetch of global memory into L2 (no destination, no completion); src 16-byte
// aligned, bytes a multiple of 16.
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

struct SkPlan {
    int cb;                                  // 32-column blocks per chunk
    int slot_bytes;                          // bytes per ring slot (multiple of 128)
    int nchk;                                // chunks per matrix
    int tg;                                  // routes per group (mma columns), <= 8
    int xstride;                             // bytes per staged activation row
    size_t smem;
};

struct SkCarve {
    unsigned char* ring;                     // [kW][kSlots][slot_bytes]
    unsigned char* xs;                       // [tg][xstride]
    float* xsum;                             // [nblk][8] (INT4)
    float* xinv;                             // [8]
    float* piece;                            // [kW][2][32][8] partial sums of split units
    int* pcnt;                               // [kW] arrivals per split unit (by first warp)
    uint64_t* full;                          // [kW][kSlots]
    int* touched;
    int* cnt;
    int* goff;
    int* misc;                               // 0 ntouched, 1 abort, 2 combine on, 3 tiles
    int* off_s;
    int* perm_s;
    int* tok_s;
    int* ctile;                              // [32]
};

__host__ __device__ inline size_t sk_align(size_t v) { return (v + 127) & ~static_cast<size_t>(127); }

// Byte offsets of the shared-memory regions (16 entries, the last one the total).
__host__ __device__ inline size_t sk_layout(int fmt, int K, const SkPlan& p, size_t (&off)[16]) {
    const int nblk = K / kBlockK;
    const size_t bytes[15] = {
        static_cast<size_t>(kW) * kSlots * p.slot_bytes,            // 0 ring
        static_cast<size_t>(p.tg) * p.xstride,                      // 1 staged activations
        fmt == FMT_INT4 ? static_cast<size_t>(nblk) * 8 * 4 : 0,    // 2 INT4 x sums
        8 * 4,                                                      // 3 inverse prescales
        static_cast<size_t>(kW) * 2 * 32 * 8 * 4,                   // 4 split-unit partials
        kW * 4,                                                     // 5 split-unit arrivals
        static_cast<size_t>(kW) * kSlots * 8,                       // 6 ring mbarriers
        kMaxExperts * 4,                                            // 7 touched
        kMaxExperts * 4,                                            // 8 cnt
        (kMaxExperts + 1) * 4,                                      // 9 goff
        8 * 4,                                                      // 10 misc
        (kMaxExperts + 1) * 4,                                      // 11 off_s
        kMaxLocalRoutes * 4,                                        // 12 perm_s
        kMaxLocalRoutes * 4,                                        // 13 tok_s
        32 * 4};                                                    // 14 ctile
    size_t o = 0;
    for (int i = 0; i < 15; ++i) {
        off[i] = o;
        o += sk_align(bytes[i]);
    }
    off[15] = o;
    return o;
}

__device__ inline SkCarve sk_carve(unsigned char* base, int fmt, int K, const SkPlan& p) {
    size_t o[16];
    sk_layout(fmt, K, p, o);
    SkCarve c;
    c.ring = base + o[0];
    c.xs = base + o[1];
    c.xsum = reinterpret_cast<float*>(base + o[2]);
    c.xinv = reinterpret_cast<float*>(base + o[3]);
    c.piece = reinterpret_cast<float*>(base + o[4]);
    c.pcnt = reinterpret_cast<int*>(base + o[5]);
    c.full = reinterpret_cast<uint64_t*>(base + o[6]);
    c.touched = reinterpret_cast<int*>(base + o[7]);
    c.cnt = reinterpret_cast<int*>(base + o[8]);
    c.goff = reinterpret_cast<int*>(base + o[9]);
    c.misc = reinterpret_cast<int*>(base + o[10]);
    c.off_s = reinterpret_cast<int*>(base + o[11]);
    c.perm_s = reinterpret_cast<int*>(base + o[12]);
    c.tok_s = reinterpret_cast<int*>(base + o[13]);
    c.ctile = reinterpret_cast<int*>(base + o[14]);
    return c;
}

__host__ inline SkPlan sk_plan(int fmt, int K, int tg_cap) {
    SkPlan p{};
    const int nblk = K / kBlockK;
    const int BB = packed_block_bytes(fmt);
    p.xstride = static_cast<int>(((2 * static_cast<size_t>(K) + 127) / 128) * 128 + 64);
    // largest route group first, then the largest chunk that fits
    for (int tg = tg_cap; tg >= 1; --tg) {
        p.tg = tg;
        for (int cb = (fmt == FMT_MXFP4 ? kChunkMx : kChunkI4); cb >= 2; --cb) {
            p.cb = cb < nblk ? cb : nblk;
            p.slot_bytes = static_cast<int>(sk_align(static_cast<size_t>(p.cb) * BB));
            p.nchk = (nblk + p.cb - 1) / p.cb;
            size_t o[16];
            p.smem = sk_layout(fmt, K, p, o) + 128;
            if (p.smem <= static_cast<size_t>(kSkBudget)) return p;
        }
    }
    p.tg = 0;
    return p;
}

struct SkParams {
    GemvArgs a;
    SkPlan p;
};

// Unit walk in group-major order inside an expert: unit u = RT * goff[j] + g * RT + rt, so the
// units of one route group are contiguous.
struct SkCursor {
    int j, g, rt, ng;
    __device__ __forceinline__ void seek(int u, int RT, const int* goff, int nt) {
        j = 0;
        while (j + 1 < nt && u >= RT * goff[j + 1]) ++j;
        ng = goff[j + 1] - goff[j];
        const int local = u - RT * goff[j];
        g = local / RT;
        rt = local - g * RT;
    }
    // call only while a next unit exists
    __device__ __forceinline__ void next(int RT, const int* goff) {
        if (++rt == RT) {
            rt = 0;
            if (++g == ng) {
                g = 0;
                ++j;
                ng = goff[j + 1] - goff[j];
            }
        }
    }
};

// Chunk walk over a warp's range: chunk q of a segment -> (unit cursor, matrix m, chunk ch).
struct ChunkWalk {
    SkCursor cu;
    int m, ch;
    __device__ __forceinline__ void next(int RT, const int* goff, int nchk, int nmat, bool more) {
        if (++ch == nchk) {
            ch = 0;
            if (++m == nmat) {
                m = 0;
                if (more) cu.next(RT, goff);
            }
        }
    }
};

template <int FMT>
__global__ void __launch_bounds__(kThr, 1) gemv_sk_kernel(const __grid_constant__ SkParams P) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const GemvArgs& a = P.a;
    const SkPlan& p = P.p;
    constexpr int BB = packed_block_bytes(FMT);
    const int K = a.K, R = a.R;
    const int nblk = K / kBlockK;
    const int RT = R / kRowTile;
    const int nmat = a.phase == 0 ? 2 : 1;
    const int C = nmat * p.nchk;                   // chunks per unit
    const int tg = p.tg;
    const bool prescale = a.adt == 1;
    const bool copy_bits = a.adt == 0;

    SkCarve c = sk_carve(smem_raw, FMT, K, p);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, tid = lane & 3;
    pdl_wait();                 // inputs of this launch may come from the previous kernel
    pdl_launch_dependents();
    const int* OFF = a.idx ? c.off_s : a.off;
    const int* PERM = a.idx ? c.perm_s : a.perm;
    const bool tokmode = a.phase == 0 && a.T <= tg;
    uint64_t* myfull = c.full + warp * kSlots;

    // ---- setup: ring barriers, route tables (last warp), token rows (warps 0-7) ------------
    if (lane == 0) {
        for (int s = 0; s < kSlots; ++s) mbar_init(&myfull[s], 1);
        fence_mbar_init();
    }
    if (warp == kW - 1) {
        build_route_tables(a, tg, lane, c.off_s, c.perm_s, c.tok_s, c.touched, c.cnt, c.goff, c.misc);
    } else if (tokmode && warp < 8) {
        const int t = warp;
        float inv = 0.0f;
        if (t < a.T) {
            inv = stage_row<FMT>(a.in + static_cast<size_t>(t) * K, c.xs + static_cast<size_t>(t) * p.xstride,
                                 c.xsum, t, K, nblk, prescale, copy_bits, lane);
        } else if (FMT == FMT_INT4) {
            for (int blk = lane; blk < nblk; blk += 32) c.xsum[blk * 8 + t] = 0.0f;
        }
        if (lane == 0) c.xinv[t] = inv;
    }
    if (threadIdx.x < kW) c.pcnt[threadIdx.x] = 0;
    // the phase-1 launch clears the combine counters the phase-2 launch will count with
    if (a.cmb_mode == 1 && blockIdx.x == 0)
        for (int i = threadIdx.x; i < a.cmb_n; i += blockDim.x) a.cmb_cnt[i] = 0;
    __syncthreads();
    const int nt = c.misc[0];
    const int U = RT * c.goff[nt];
    const int u0 = static_cast<int>((static_cast<long long>(U) * blockIdx.x) / gridDim.x);
    const int u1 = static_cast<int>((static_cast<long long>(U) * (blockIdx.x + 1)) / gridDim.x);
    if (u0 >= u1) return;

    auto aborted = [&]() { return *reinterpret_cast<volatile int*>(&c.misc[1]) != 0; };
    auto fail_timeout = [&]() {
        if (lane == 0 && c.misc[1] == 0) {
            c.misc[1] = 1;
            report_error(a.status, DEV_ERR_TIMEOUT);
        }
    };

    // ring slot state of this warp (persists across segments)
    int slot_c = 0, slot_i = 0;                    // next slot to consume / to fill
    uint32_t ph_c = 0;                             // phase parity of slot_c
    int inflight = 0;                              // copies issued and not yet consumed
    uint32_t pend = 0;                             // slots whose copy has not been seen complete
    uint32_t lastpar = 0;                          // parity of the last completion issued per slot

    SkCursor seg;
    seg.seek(u0, RT, c.goff, nt);
    int sa = u0;
    bool first_seg = true;
    while (sa < u1) {
        // ---- one segment: units [sa, sb) sharing the staged activation rows ----------------
        const int sb = tokmode ? u1 : min(u1, sa + (RT - seg.rt));
        const int gj = seg.j, gg = seg.g;
        if (!tokmode) {
            if (!first_seg) named_bar(1, kThr);    // every warp is done with the previous rows
            if (warp < 8) {
                const int e = c.touched[gj];
                const int cnt_g = min(tg, c.cnt[gj] - gg * tg);
                const int rbase = a.dense ? gg * tg : OFF[e] + gg * tg;
                const int n = warp;
                float inv = 0.0f;
                if (n < cnt_g) {
                    const int rid = a.dense ? rbase + n : PERM[rbase + n];
                    size_t row;
                    if (a.phase == 0) row = a.dense ? static_cast<size_t>(rid) : static_cast<size_t>(rid / a.k);
                    else row = static_cast<size_t>(rid);
                    inv = stage_row<FMT>(a.in + row * K, c.xs + static_cast<size_t>(n) * p.xstride, c.xsum, n,
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
            named_bar(1, kThr);
        }

        const long long N = static_cast<long long>(sb - sa) * C;
        const int c0 = static_cast<int>((warp * N) / kW);
        const int c1 = static_cast<int>(((warp + 1) * N) / kW);
        auto owner = [&](long long q) {            // the warp whose range holds chunk q
            return static_cast<int>((kW * (q + 1) - 1) / N);
        };
        auto start_of = [&](int w) { return static_cast<int>((w * N) / kW); };

        if (c0 < c1) {
            // walkers: `cw` over the chunks being consumed, `iw` over the chunks being issued
            ChunkWalk cw, iw;
            {
                const int du = c0 / C, win = c0 - du * C;
                cw.cu = seg;
                for (int q = 0; q < du; ++q) cw.cu.next(RT, c.goff);
                cw.m = win / p.nchk;
                cw.ch = win - cw.m * p.nchk;
                iw = cw;
            }
            ChunkWalk pw = cw;                     // prefetch walk, kPrefetch chunks past the ring
            int pq = c0;
            auto prefetch_one = [&]() {
                if (pq >= c1) return;
                if (lane == 0) {
                    const int e = c.touched[pw.cu.j];
                    const uint8_t* wb = (pw.m == 0 ? a.w0 : a.w1) + static_cast<size_t>(e) * a.mat_bytes;
                    const int b0 = pw.ch * p.cb;
                    const int nb = min(p.cb, nblk - b0);
                    prefetch_l2(wb + (static_cast<size_t>(pw.cu.rt) * nblk + b0) * BB, static_cast<uint32_t>(nb) * BB);
                }
                ++pq;
                pw.next(RT, c.goff, p.nchk, nmat, pq < c1);
            };
            if (kPrefetch > 0) {
                // skip the chunks the ring loads straight away, then run kPrefetch ahead
                for (int q = 0; q < kSlots && pq < c1; ++q) {
                    ++pq;
                    pw.next(RT, c.goff, p.nchk, nmat, pq < c1);
                }
                for (int q = 0; q < kPrefetch; ++q) prefetch_one();
            }
            int iq = c0;                           // next chunk to issue
            int du = c0 / C;                       // unit offset (in the segment) of chunk q
            auto issue_one = [&]() {
                const int e = c.touched[iw.cu.j];
                const uint8_t* wb = (iw.m == 0 ? a.w0 : a.w1) + static_cast<size_t>(e) * a.mat_bytes;
                const int b0 = iw.ch * p.cb;
                const int nb = min(p.cb, nblk - b0);
                const uint32_t bytes = static_cast<uint32_t>(nb) * BB;
                unsigned char* dst = c.ring + (static_cast<size_t>(warp) * kSlots + slot_i) * p.slot_bytes;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&myfull[slot_i], bytes);
                    bulk_g2s(dst, wb + (static_cast<size_t>(iw.cu.rt) * nblk + b0) * BB, bytes, &myfull[slot_i]);
                }
                pend |= 1u << slot_i;
                lastpar ^= 1u << slot_i;                   // bit = parity of this issue's completion ^ 1
                if (++slot_i == kSlots) slot_i = 0;
                ++inflight;
                ++iq;
                iw.next(RT, c.goff, p.nchk, nmat, iq < c1);
                if (kPrefetch > 0 && iq > c0 + kSlots) prefetch_one();
            };
            // generic-proxy reads of a slot must be ordered before the async copy that refills it
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            while (iq < c1 && inflight < kSlots) issue_one();

            float acc[2][4];                       // [matrix][fragment], indexed statically only
#pragma unroll
            for (int m = 0; m < 2; ++m)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[m][q] = 0.0f;
            // per-unit state, set when the walk enters a unit
            int brow = 0, xc0 = 0, xc1 = 0, cnt_g = 0, rbase = 0, e_cur = 0;
            float bias_r[2][2] = {{0.f, 0.f}, {0.f, 0.f}};     // [matrix][row gid / gid + 8]
            auto enter_unit = [&]() {
                const int j = cw.cu.j, g = cw.cu.g;
                e_cur = c.touched[j];
                cnt_g = min(tg, c.cnt[j] - g * tg);
                rbase = a.dense ? g * tg : OFF[e_cur] + g * tg;
                auto row_of = [&](int n) {
                    if (!tokmode) return n < tg ? n : 0;
                    if (n >= cnt_g) return 0;
                    if (a.dense) return rbase + n;
                    return a.idx ? c.tok_s[rbase + n] : PERM[rbase + n] / a.k;
                };
                brow = row_of(gid);
                xc0 = row_of(2 * tid);
                xc1 = row_of(2 * tid + 1);
                // biases of rows gid and gid + 8 of both matrices, for whichever warp finishes
                const size_t bi = static_cast<size_t>(e_cur) * R + cw.cu.rt * kRowTile + gid;
                bias_r[0][0] = a.b0 ? __bfloat162float(__ushort_as_bfloat16(a.b0[bi])) : 0.0f;
                bias_r[0][1] = a.b0 ? __bfloat162float(__ushort_as_bfloat16(a.b0[bi + 8])) : 0.0f;
                bias_r[1][0] = (a.phase == 0 && a.b1) ? __bfloat162float(__ushort_as_bfloat16(a.b1[bi])) : 0.0f;
                bias_r[1][1] = (a.phase == 0 && a.b1) ? __bfloat162float(__ushort_as_bfloat16(a.b1[bi + 8])) : 0.0f;
            };
            enter_unit();
            // finish a unit from its summed partials (this lane's 4 outputs per matrix)
            auto finish = [&](const float (&s)[2][4], int rt) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int row = gid + 8 * (q >> 1), col = 2 * tid + (q & 1);
                    if (col >= cnt_g) continue;
                    const int rid = a.dense ? rbase + col : PERM[rbase + col];
                    const float inv = c.xinv[tokmode ? (a.dense ? rbase + col : (a.idx ? c.tok_s[rbase + col] : PERM[rbase + col] / a.k)) : col];
                    const size_t o = static_cast<size_t>(rid) * R + rt * kRowTile + row;
                    const float v0 = s[0][q] * inv + bias_r[0][q >> 1];
                    if (a.phase == 0) {
                        const float v1 = s[1][q] * inv + bias_r[1][q >> 1];
                        static_cast<uint16_t*>(a.out)[o] = float_to_adt_bits(act_fn(a.act, v0, v1, a.limit, a.alpha), a.adt);
                    } else {
                        static_cast<float*>(a.out)[o] = v0;
                    }
                }
            };

            const unsigned char* xbase = c.xs + tid * 16;
            for (int q = c0; q < c1; ++q) {
                const int s = slot_c;
                const uint32_t par = ph_c;
                if (++slot_c == kSlots) {
                    slot_c = 0;
                    ph_c ^= 1;
                }
                const bool ok = !aborted() && mbar_wait_bounded(&myfull[s], par);
                --inflight;
                if (ok) pend &= ~(1u << s);
                else fail_timeout();
                const int b0 = cw.ch * p.cb;
                const int nb = min(p.cb, nblk - b0);
                if (ok) {
                    const unsigned char* st = c.ring + (static_cast<size_t>(warp) * kSlots + s) * p.slot_bytes;
                    const unsigned char* xrow = xbase + static_cast<size_t>(brow) * p.xstride + static_cast<size_t>(b0) * 64;
                    float ac[4] = {0.f, 0.f, 0.f, 0.f};   // this chunk's sum, added to acc[m] below
                    auto block = [&](int i) {
                        const uint4 bx = *reinterpret_cast<const uint4*>(xrow + i * 64);
                        const unsigned char* blk = st + i * BB;
                        const uint2 cwd = *reinterpret_cast<const uint2*>(blk + lane * 8);
                        float d[4] = {0.f, 0.f, 0.f, 0.f};
                        if (FMT == FMT_MXFP4) {
                            const uint32_t sc = *reinterpret_cast<const uint16_t*>(blk + 256 + gid * 2);
                            uint32_t pa[4], pb[4];
                            e2m1x8_to_f16x2x4(cwd.x, pa);
                            e2m1x8_to_f16x2x4(cwd.y, pb);
                            mma_f16_16816(d, pa[0], pb[0], pa[1], pb[1], bx.x, bx.y);
                            mma_f16_16816(d, pa[2], pb[2], pa[3], pb[3], bx.z, bx.w);
                            // 2^(e-127) as f32 bits e << 23; e = 0 gives the subnormal 2^-127 (0x00400000)
                            const float s0 = __uint_as_float(max((sc << 23) & 0x7F800000u, 0x00400000u));
                            const float s1 = __uint_as_float(max((sc << 15) & 0x7F800000u, 0x00400000u));
                            ac[0] = fmaf(d[0], s0, ac[0]);
                            ac[1] = fmaf(d[1], s0, ac[1]);
                            ac[2] = fmaf(d[2], s1, ac[2]);
                            ac[3] = fmaf(d[3], s1, ac[3]);
                        } else {
                            const uint2 smv = *reinterpret_cast<const uint2*>(blk + 256 + gid * 8);
                            const int bi = b0 + i;
                            const float xs0 = c.xsum[bi * 8 + xc0], xs1 = c.xsum[bi * 8 + xc1];
                            mma_f16_16816(d, u4pair_to_f16x2(cwd.x, 0), u4pair_to_f16x2(cwd.y, 0),
                                          u4pair_to_f16x2(cwd.x, 4), u4pair_to_f16x2(cwd.y, 4), bx.x, bx.y);
                            mma_f16_16816(d, u4pair_to_f16x2(cwd.x, 8), u4pair_to_f16x2(cwd.y, 8),
                                          u4pair_to_f16x2(cwd.x, 12), u4pair_to_f16x2(cwd.y, 12), bx.z, bx.w);
                            const float sg = __half2float(__ushort_as_half(smv.x & 0xFFFF));
                            const float mg = __half2float(__ushort_as_half(smv.x >> 16));
                            const float sg8 = __half2float(__ushort_as_half(smv.y & 0xFFFF));
                            const float mg8 = __half2float(__ushort_as_half(smv.y >> 16));
                            ac[0] = fmaf(sg, d[0], fmaf(mg, xs0, ac[0]));
                            ac[1] = fmaf(sg, d[1], fmaf(mg, xs1, ac[1]));
                            ac[2] = fmaf(sg8, d[2], fmaf(mg8, xs0, ac[2]));
                            ac[3] = fmaf(sg8, d[3], fmaf(mg8, xs1, ac[3]));
                        }
                    };
                    constexpr int kCB = FMT == FMT_MXFP4 ? kChunkMx : kChunkI4;
                    if (nb == kCB) {
                        // the common full chunk: straight-line code, every load issued early
#pragma unroll
                        for (int i = 0; i < kCB; ++i) block(i);
                    } else {
                        for (int i = 0; i < nb; ++i) block(i);
                    }
                    if (cw.m == 0) {
#pragma unroll
                        for (int r = 0; r < 4; ++r) acc[0][r] += ac[r];
                    } else {
#pragma unroll
                        for (int r = 0; r < 4; ++r) acc[1][r] += ac[r];
                    }
                }
                // refill the slot just read with the chunk kSlots further on
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (iq < c1 && !aborted()) issue_one();

                const bool unit_end = (cw.m == nmat - 1 && cw.ch == p.nchk - 1) || q == c1 - 1;
                if (unit_end) {
                    const int ufirst = du * C;                      // first chunk of the unit
                    const bool whole = c0 <= ufirst && c1 >= ufirst + C;
                    if (whole) {
                        finish(acc, cw.cu.rt);
                    } else {
                        // split unit: park the partials; the last warp to arrive sums them
                        const int which = c0 >= ufirst ? 0 : 1;
                        float4* pc = reinterpret_cast<float4*>(c.piece + ((warp * 2 + which) * 32 + lane) * 8);
                        pc[0] = make_float4(acc[0][0], acc[0][1], acc[0][2], acc[0][3]);
                        pc[1] = make_float4(acc[1][0], acc[1][1], acc[1][2], acc[1][3]);
                        const int wf = owner(ufirst), wl = owner(static_cast<long long>(ufirst) + C - 1);
                        // warps between wf and wl whose range is empty hold no part
                        int nparts = 0;
                        for (int w = wf; w <= wl; ++w) nparts += start_of(w) < start_of(w + 1);
                        __threadfence_block();
                        __syncwarp();
                        int last = 0;
                        if (lane == 0) last = atomicAdd(&c.pcnt[wf], 1) == nparts - 1;
                        last = __shfl_sync(0xffffffffu, last, 0);
                        if (last) {
                            __threadfence_block();
                            float sum[2][4];
#pragma unroll
                            for (int m = 0; m < 2; ++m)
#pragma unroll
                                for (int r = 0; r < 4; ++r) sum[m][r] = 0.0f;
                            for (int w = wf; w <= wl; ++w) {        // K order
                                if (start_of(w) >= start_of(w + 1)) continue;   // empty range
                                const int wh = start_of(w) >= ufirst ? 0 : 1;
                                const float4* pw = reinterpret_cast<const float4*>(c.piece + ((w * 2 + wh) * 32 + lane) * 8);
                                const float4 p0 = pw[0], p1 = pw[1];
                                sum[0][0] += p0.x; sum[0][1] += p0.y; sum[0][2] += p0.z; sum[0][3] += p0.w;
                                sum[1][0] += p1.x; sum[1][1] += p1.y; sum[1][2] += p1.z; sum[1][3] += p1.w;
                            }
                            finish(sum, cw.cu.rt);
                            if (lane == 0) c.pcnt[wf] = 0;
                        }
                    }
#pragma unroll
                    for (int m = 0; m < 2; ++m)
#pragma unroll
                        for (int r = 0; r < 4; ++r) acc[m][r] = 0.0f;
                }
                const bool more = q + 1 < c1;
                const bool crossing = cw.m == nmat - 1 && cw.ch == p.nchk - 1;
                cw.next(RT, c.goff, p.nchk, nmat, more);
                if (crossing) ++du;
                if (crossing && more) enter_unit();
            }
            // copies not seen complete (only after a failed wait) must land before the CTA exits
            if (pend && lane == 0)
                for (int t = 0; t < kSlots; ++t)
                    if (pend & (1u << t)) mbar_wait_bounded(&myfull[t], ((lastpar >> t) & 1u) ^ 1u);
            pend = 0;
            __syncwarp();
        }
        // next segment
        for (int q = sa; q < sb; ++q)
            if (q + 1 < u1) seg.next(RT, c.goff);
        sa = sb;
        first_seg = false;
    }

    // ---- fused combine (phase 2 of a routed decode call) -------------------------------------
    if (a.cmb_mode == 2) {
        // every output of this CTA is stored before the barrier; the counting atomics release them
        if (warp == 0 && lane == 0) c.misc[2] = c.misc[1] == 0;
        named_bar(2, kThr);
        if (c.misc[2]) {
            SkCursor cc;
            cc.seek(u0, RT, c.goff, nt);
            for (int ub = u0; ub < u1; ub += 32) {
                if (warp == 0) {
                    // lane l bumps the counter of unit ub + l (walk the cursor to it)
                    int rt = 0, last = 0;
                    SkCursor lc = cc;
                    for (int q = 0; q < lane && ub + q + 1 < u1; ++q) lc.next(RT, c.goff);
                    if (ub + lane < u1) {
                        rt = lc.rt;
                        last = count_tile_unit(a.cmb_cnt, rt, c.goff[nt]);
                    }
                    const unsigned lm = __ballot_sync(0xffffffffu, last);
                    if (last) {
                        c.ctile[__popc(lm & ((1u << lane) - 1u))] = rt;
                        a.cmb_cnt[rt] = 0;              // complete: ready for the next call
                    }
                    if (lane == 0) c.misc[3] = __popc(lm);
                }
                for (int q = 0; q < 32 && ub + q + 1 < u1; ++q) cc.next(RT, c.goff);
                named_bar(2, kThr);              // tile list ready
                const int ntile = c.misc[3];
                combine_tiles(a, c.ctile, ntile, kRowTile, threadIdx.x, kThr);
                named_bar(2, kThr);              // tile list consumed
            }
        }
    }
}

}  // namespace

bool gemv_sk_fits(int fmt, int K, int T) {
    return sk_plan(fmt, K, T < 8 ? (T > 0 ? T : 1) : 8).tg >= 1;
}

cudaError_t launch_gemv_sk(const GemvArgs& a, int num_sms, cudaStream_t s) {
    SkParams P;
    P.a = a;
    P.p = sk_plan(a.fmt, a.K, a.T < 8 ? (a.T > 0 ? a.T : 1) : 8);
    if (P.p.tg < 1) return cudaErrorInvalidValue;
    P.a.tg = P.p.tg;
    // only INT4 is routed here (MXFP4 measured faster on the producer/reducer kernel of gemv.cu);
    // the MXFP4 block code above is kept for that comparison but not instantiated
    if (a.fmt != FMT_INT4) return cudaErrorInvalidValue;
    cudaError_t e = ensure_smem(gemv_sk_kernel<FMT_INT4>, P.p.smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(gemv_sk_kernel<FMT_INT4>, dim3(num_sms), dim3(kThr), P.p.smem, s, P);
}

}  // namespace tsmoe

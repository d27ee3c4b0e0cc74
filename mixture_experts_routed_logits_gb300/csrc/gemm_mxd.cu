// gemm_mxd.cu -- steps 3-5 of the routed-expert layer for decode batches (T <= 8 tokens) with
// MXFP4 experts and bf16 activations, on the block-scaled tensor cores, in three launches:
//   prep:    the T token rows split into two e4m3 terms (one e8m0 scale per row), written once
//            as the shared-memory image of B that phase 1 copies; the counters zeroed;
//   phase 1: the route tables from idx, gate and up of every touched expert streamed once, bias
//            + activation, h split into two e4m3 terms (one e8m0 scale per 32 values) and
//            written as the B image of phase 2's K stage;
//   phase 2: down of every touched expert streamed once, bias, e per route, and the slot-ordered
//            combine into y by the CTA that finishes a row block last.
//
// Source pages (docs.rs, turbospark-runtime 0.3.0):
//   gpt-oss routed-expert pass (src/families/gptoss/moe.rs): the decode pair of encoders (phase 1
//     gate/up + clamped SwiGLU + biases into the 16-bit acts, phase 2 down), the slot order of the
//     reduction (router rank, slot-index order), the zero residual seed.
//   Gemma-4 batched routed prefill (src/families/gemma4/moe_batch.rs): the route list.
//
// Design (GB300, one CTA per SM, persistent):
//   * Every CTA builds the route tables itself from idx (T*k <= 64 entries): the touched experts in
//     ascending order and, per (touched expert, token), the route id or none.  No route-list
//     launch.
//   * B = the T token rows, computed for every touched expert (N = 16 whatever the routing: the
//     MMA costs the same up to N = 128).  An activation v under scale 2^s, s = floor(log2 max) -
//     7 (max over the values sharing the scale), splits into e4m3 terms t1 + t2 / 16 exactly
//     for |v| >= max 2^-14, with an error below max 2^-23 for smaller values.  x has one scale
//     per row, so its scale atom reaches TMEM once per launch; h has one scale per 32 values,
//     which lets the CTA that finishes a 128-row tile of phase 1 split it on the spot: the tile
//     is exactly one 128-column K stage of phase 2.  Each stage's 2 KB of B rows is copied into
//     the ring slot beside the weights (from L2).
//   * The weights stream from HBM through a ring of 6 slots; a 4-bit code takes a byte in
//     shared memory in the block-scaled MMA's operand layout, so shared memory caps the bytes in
//     flight (about 96 KB of HBM data per SM).  An L2 prefetch ahead of the ring was measured
//     slower (its copies compete with the ring's at the start and cost the producer an
//     instruction per stage), so there is none.
//   * Stream-K: the work units (touched expert, block of weight rows, K stage) are cut into
//     equal contiguous ranges, one per CTA; a tile split between CTAs parks its partial sums and
//     the CTA that brings the last part finishes it, summing the parts in K (= CTA) order, so
//     results are deterministic.
//   * Warps: 0 weight producer (one 16 KB tensor copy per stage), 7 scale and activation producer
//     (bulk copies), 6 scale copies into TMEM, 1 MMA issuer, 2-5 epilogue.
//     Every mbarrier wait is bounded.
#include "mx_common.cuh"

namespace tsmoe {

namespace {

constexpr int kDThreads = 256;
constexpr int kDMaxSlots = 8;
constexpr int kDAtom = 512;
constexpr int kDAbox = 16384;          // shared bytes of 128 rows x 128 padded codes
constexpr int kDBstage = kMxdBStage;  // one K stage of B: 16 rows x 128 bytes
constexpr uint32_t kDColSfb = 64;      // TMEM: accumulators [0, 64), x scales [64, 68),
constexpr uint32_t kDColSf = 80;       // scales of slot s at 80 + 16 s (A: 8 columns, phase 2 B: 4)

struct MxdLayout {
    int nslot, slot_bytes, sfa_off, b_off;   // ring slot: A codes 32 KB, scale atoms 1 KB, B stage
                                             // 2 KB (phase 2: + its scale atom 512 B)
    int sfb_off;                             // phase 1: x scale atom (512 B)
    int tail_off;
};

struct MxdParams {
    CUtensorMap tmA;
    MxdArgs a;
    MxdLayout ly;
};

struct MxdTail {
    uint64_t full[kDMaxSlots];      // weight codes, scale atoms and the B stage landed
    uint64_t sfull[kDMaxSlots];     // the slot's scales copied into TMEM
    uint64_t empty[kDMaxSlots];     // the slot's MMAs done
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t bready;                // phase 1: the x scale atom landed
    uint32_t tmem_base;
    volatile int abort_flag;
    int nt;
    int touched[kMxdMaxTouched];
    int rid[kMxdMaxTouched][kMxdTokens];
    float wr[kMxdTokens * kMxdMaxK];  // phase 2: routing weights [t][s]
};

template <int PHASE>
__global__ void __launch_bounds__(kDThreads, 1) mxd_kernel(const __grid_constant__ MxdParams P) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const MxdArgs& a = P.a;
    const MxdLayout& Ly = P.ly;
    unsigned char* base = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    unsigned char* ring = base;
    unsigned char* sfb = base + Ly.sfb_off;
    MxdTail* tl = reinterpret_cast<MxdTail*>(base + Ly.tail_off);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int G = PHASE == 0 ? 2 : 1;
    constexpr int RPI = PHASE == 0 ? 128 : 256;       // weight rows per tile
    const int R = a.R, K = a.K, T = a.T, k = a.k;
    const int MB = mx_units(G, R);
    const int KG = mx_kg(K);
    const int NS = Ly.nslot;
    const uint8_t* sfa_base = a.w + mx_sf_offset(G, a.E, R, K);
    // Phase 1 reads idx and the x image; phase 2 reads idx early (the router finished before
    // phase 1 passed its own wait, and phase 2 starts only after that) and waits before touching
    // what phase 1 writes.
    if (PHASE == 0) pdl_wait();
    pdl_launch_dependents();

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&tl->full[s], 1);
            mbar_init(&tl->sfull[s], 1);
            mbar_init(&tl->empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tl->tfull[b], 1);
            mbar_init(&tl->tempty[b], 4);
        }
        mbar_init(&tl->bready, 1);
        tl->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 256;" ::"r"(
                         smem_u32(&tl->tmem_base))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (warp == 2) {
        // ---- route tables: touched experts ascending, route id per (touched expert, token) ----
        const int n = T * k;
        const int e0 = lane < n ? __ldcg(a.idx + lane) : -1;
        const int e1 = lane + 32 < n ? __ldcg(a.idx + lane + 32) : -1;
        const bool v0 = e0 >= 0 && e0 < a.E, v1 = e1 >= 0 && e1 < a.E;
        if ((lane < n && !v0) || (lane + 32 < n && !v1)) report_error(a.status, DEV_ERR_INVALID);
        // touched experts as a bit mask (E <= 256), reduced over the warp; an expert's rank is
        // the number of touched experts below it
        uint32_t msk[kMaxExperts / 32];
        int nt = 0;
#pragma unroll
        for (int w = 0; w < kMaxExperts / 32; ++w) {
            const uint32_t bits = ((v0 && (e0 >> 5) == w) ? 1u << (e0 & 31) : 0u) |
                                  ((v1 && (e1 >> 5) == w) ? 1u << (e1 & 31) : 0u);
            msk[w] = __reduce_or_sync(0xffffffffu, bits);
            nt += __popc(msk[w]);
        }
        auto rank_of = [&](int e) {
            int r = __popc(msk[e >> 5] & ((1u << (e & 31)) - 1u));
#pragma unroll
            for (int w = 0; w < kMaxExperts / 32; ++w) r += (w < (e >> 5)) ? __popc(msk[w]) : 0;
            return r;
        };
        const int rank0 = v0 ? rank_of(e0) : 0, rank1 = v1 ? rank_of(e1) : 0;
        for (int i = lane; i < kMxdMaxTouched * kMxdTokens; i += 32) (&tl->rid[0][0])[i] = -1;
        __syncwarp();
        if (v0) { tl->touched[rank0] = e0; tl->rid[rank0][lane / k] = lane; }
        if (v1) { tl->touched[rank1] = e1; tl->rid[rank1][(lane + 32) / k] = lane + 32; }
        if (lane == 0) tl->nt = nt;
        if (PHASE == 1) {
            if (lane < n) tl->wr[lane] = __ldcg(a.wr + lane);
            if (lane + 32 < n) tl->wr[lane + 32] = __ldcg(a.wr + lane + 32);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tl->tmem_base;
    const int nt = tl->nt;
    const int tiles = nt * MB;
    const long long U = static_cast<long long>(tiles) * KG;
    // at most U CTAs take part, so that every range holds at least one unit (the part counts
    // below assume it); the others have empty ranges
    const int Gc = static_cast<int>(U < gridDim.x ? (U > 0 ? U : 1) : gridDim.x);
    const bool in_grid = static_cast<int>(blockIdx.x) < Gc;
    const int u0 = in_grid ? static_cast<int>(U * blockIdx.x / Gc) : 0;
    const int u1 = in_grid ? static_cast<int>(U * (blockIdx.x + 1) / Gc) : 0;
    // the CTA whose range holds unit u
    auto cta_of = [&](long long u) { return static_cast<int>(((u + 1) * Gc + U - 1) / U - 1); };

    // Segments: the maximal runs of one tile inside this CTA's range.  They are processed first,
    // last, then the middle ones: the first and last segments are the ones that may share their
    // tile with a neighbour, so their parts meet early and the CTA ends on a whole tile, whose
    // finish needs no other CTA.
    struct Seg { int tile, j, mb, kg0, kg1; };
    const int tile0 = u0 / KG;
    const int nseg_all = u1 > u0 ? (u1 - 1) / KG - tile0 + 1 : 0;
    auto seg_of = [&](int i, Seg& s) {
        const int r = (i == 0 || nseg_all < 3) ? i : (i == 1 ? nseg_all - 1 : i - 1);
        s.tile = tile0 + r;
        s.kg0 = r == 0 ? u0 - tile0 * KG : 0;
        s.kg1 = r == nseg_all - 1 ? u1 - s.tile * KG : KG;
        s.j = s.tile / MB;
        s.mb = s.tile - s.j * MB;
    };
    // stage cursor over the segments
    struct Stage { int i, kg; Seg sg; };
    auto first_stage = [&](Stage& c) { c.i = -1; c.kg = 0; c.sg.kg1 = 0; };
    auto next_stage = [&](Stage& c) -> bool {
        if (c.i >= 0 && c.kg + 1 < c.sg.kg1) { ++c.kg; return true; }
        if (++c.i >= nseg_all) return false;
        seg_of(c.i, c.sg);
        c.kg = c.sg.kg0;
        return true;
    };
    auto a_load = [&](int e, int mb, int kg, void* dst, uint64_t* bar) {
        if (PHASE == 0) tma_load_5d(dst, &P.tmA, 0, mb * RPI, 0, kg, e, bar);
        else tma_load_4d(dst, &P.tmA, 0, mb * RPI, kg, e, bar);
    };
    auto sfa_src = [&](int e, int mb, int kg) {
        return sfa_base + ((static_cast<size_t>(e) * MB + mb) * KG + kg) * (2 * kDAtom);
    };

    if (warp == 0 || warp == 7) {
        if (lane == 0) {
            // ================= producers: weight codes (warp 0), scale atoms (warp 7) ===========
            const bool wts = warp == 0;
            // warp 7 also copies each stage's B rows: the x image (phase 1; its scale atom once,
            // first) or the split h stage with its atom (phase 2, after phase 1 has finished)
            if (PHASE == 1 && !wts) pdl_wait();
            if (PHASE == 0 && !wts) {
                mbar_arrive_expect_tx(&tl->bready, kDAtom);
                bulk_g2s(sfb, a.xs + static_cast<size_t>(KG) * kDBstage, kDAtom, &tl->bready);
            }
            int it = 0;
            int issued[kDMaxSlots];
            for (int q = 0; q < kDMaxSlots; ++q) issued[q] = -1;
            Stage c;
            first_stage(c);
            while (next_stage(c)) {
                const int s = it % NS;
                if (tl->abort_flag || !mbar_wait_bounded(&tl->empty[s], ((it / NS) & 1) ^ 1)) {
                    tl->abort_flag = 1;
                    report_error(a.status, DEV_ERR_TIMEOUT);
                    break;
                }
                // test setting: the first stage's copies are withheld, so the consumers' bounded
                // waits on it run out (reported as TS_ERR_TIMEOUT)
                if (PHASE == 0 && a.stall && it == 0) {
                    ++it;
                    continue;
                }
                unsigned char* st = ring + static_cast<size_t>(s) * Ly.slot_bytes;
                const int e = tl->touched[c.sg.j];
                if (wts) {
                    mbar_arrive_expect_tx(&tl->full[s], 2 * 8192 + 2 * kDAtom + (PHASE == 1 ? kMxdHImage : kDBstage));
                    a_load(e, c.sg.mb, c.kg, st, &tl->full[s]);
                } else {
                    bulk_g2s(st + Ly.sfa_off, sfa_src(e, c.sg.mb, c.kg), 2 * kDAtom, &tl->full[s]);
                    if (PHASE == 1)
                        bulk_g2s(st + Ly.b_off, a.hs + (static_cast<size_t>(c.sg.j) * KG + c.kg) * kMxdHImage,
                                 kMxdHImage, &tl->full[s]);
                    else
                        bulk_g2s(st + Ly.b_off, a.xs + static_cast<size_t>(c.kg) * kDBstage, kDBstage, &tl->full[s]);
                }
                issued[s] = it;
                ++it;
            }
            for (int q = 0; q < NS; ++q)
                if (issued[q] >= 0) mbar_wait_bounded(&tl->full[q], (issued[q] / NS) & 1);
        }
    } else if (warp == 6) {
        // ===================== scale atoms into TMEM, one commit per stage =====================
        int it = 0;
        bool stop = false;
        if (PHASE == 0) {
            // the resident x scales, once
            int ok = 1;
            if (lane == 0) {
                ok = mbar_wait_bounded(&tl->bready, 0);
                if (ok) {
                    tc_fence_after();
                    tmem_cp_atom(tmem + kDColSfb, sfb);
                }
            }
            if (!__shfl_sync(0xffffffffu, ok, 0)) {
                if (lane == 0) { tl->abort_flag = 1; report_error(a.status, DEV_ERR_TIMEOUT); }
                stop = true;
            }
        }
        if (lane == 0 && !stop) {
            for (int i = 0; i < nseg_all && !stop; ++i) {
                Seg sg;
                seg_of(i, sg);
                for (int kg = sg.kg0; kg < sg.kg1; ++kg, ++it) {
                    const int s = it % NS;
                    if (tl->abort_flag || !mbar_wait_bounded(&tl->full[s], (it / NS) & 1)) {
                        tl->abort_flag = 1;
                        report_error(a.status, DEV_ERR_TIMEOUT);
                        stop = true;
                        break;
                    }
                    tc_fence_after();
                    const unsigned char* st = ring + static_cast<size_t>(s) * Ly.slot_bytes;
                    const uint32_t tsf = tmem + kDColSf + 16u * s;
                    tmem_cp_atom(tsf, st + Ly.sfa_off);
                    tmem_cp_atom(tsf + 4, st + Ly.sfa_off + kDAtom);
                    if (PHASE == 1) tmem_cp_atom(tsf + 8, st + Ly.b_off + kDBstage);
                    umma_commit(&tl->sfull[s]);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ================================= MMA issuer ====================================
            bool ok = PHASE == 1 || mbar_wait_bounded(&tl->bready, 0);
            if (!ok) { tl->abort_flag = 1; report_error(a.status, DEV_ERR_TIMEOUT); }
            int it = 0;
            for (int nseg = 0; nseg < nseg_all && ok && !tl->abort_flag; ++nseg) {
                Seg sg;
                seg_of(nseg, sg);
                const bool has1 = PHASE == 0 || sg.mb * RPI + 128 < R;
                const int tb = nseg & 1;
                const uint32_t acc0 = tmem + static_cast<uint32_t>(tb * 32);
                const uint32_t acc1 = acc0 + 16;

                if (!mbar_wait_bounded(&tl->tempty[tb], ((nseg >> 1) & 1) ^ 1)) {
                    tl->abort_flag = 1;
                    report_error(a.status, DEV_ERR_TIMEOUT);
                    break;
                }
                tc_fence_after();
                for (int kg = sg.kg0; kg < sg.kg1; ++kg, ++it) {
                    const int s = it % NS;
                    if (!mbar_wait_bounded(&tl->full[s], (it / NS) & 1) ||
                        !mbar_wait_bounded(&tl->sfull[s], (it / NS) & 1)) {
                        tl->abort_flag = 1;
                        report_error(a.status, DEV_ERR_TIMEOUT);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const unsigned char* st = ring + static_cast<size_t>(s) * Ly.slot_bytes;
                    const uint32_t tsf = tmem + kDColSf + 16u * s;
                    const uint32_t tsfb = PHASE == 0 ? tmem + kDColSfb : tsf + 8;
                    const uint64_t dA0 = sdesc_sw128(smem_u32(st));
                    const uint64_t dA1 = sdesc_sw128(smem_u32(st + kDAbox));
                    const uint64_t dB = sdesc_sw128(smem_u32(st + Ly.b_off));
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        const uint32_t acc = (kg > sg.kg0 || ks > 0) ? 1u : 0u;
                        const uint32_t idesc = idesc_mx(2 * kMxdTokens, ks);
                        umma_mx(acc0, dA0 + 2 * ks, dB + 2 * ks, idesc, tsf, tsfb, acc);
                        if (has1) umma_mx(acc1, dA1 + 2 * ks, dB + 2 * ks, idesc, tsf + 4, tsfb, acc);
                    }
                    umma_commit(&tl->empty[s]);
                }
                if (!ok) break;
                umma_commit(&tl->tfull[tb]);
            }
        }
    } else {
        // =================================== epilogue ==========================================
        const int q = warp & 3;                     // TMEM lane quarter: rows 32q .. 32q + 31
        if (PHASE == 1) pdl_wait();                // parts, counters and e of phase 1's launch
        const uint32_t tq = tmem + (static_cast<uint32_t>(32 * q) << 16);
        for (int nseg = 0; nseg < nseg_all; ++nseg) {
            Seg sg;
            seg_of(nseg, sg);
            const int tb = nseg & 1;
            const bool go = __shfl_sync(0xffffffffu, tl->abort_flag, 0) == 0;
            if (!__all_sync(0xffffffffu, go && mbar_wait_bounded(&tl->tfull[tb], (nseg >> 1) & 1))) {
                if (lane == 0) { tl->abort_flag = 1; report_error(a.status, DEV_ERR_TIMEOUT); }
                break;
            }
            tc_fence_after();
            float d0[8], d0b[8], d1[8], d1b[8];
            const uint32_t t0 = tq + static_cast<uint32_t>(tb * 32);
            tmem_ld8x4(t0, t0 + 8, t0 + 16, t0 + 24, d0, d0b, d1, d1b);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tl->tempty[tb]);
            float x0[8], x1[8];
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                x0[t] = d0[t] + d0b[t];
                x1[t] = d1[t] + d1b[t];
            }
            const int e = tl->touched[sg.j];
            const int ra = sg.mb * RPI + 32 * q + lane;      // row of acc0 (acc1: + 128, phase 2)
            if (!(sg.kg0 == 0 && sg.kg1 == KG)) {
                // a tile split between CTAs: park this part; the last part's CTA finishes
                const int slot = (u0 >= sg.tile * KG) ? 0 : 1;   // this CTA's first or last segment
                float* pp = a.part + ((static_cast<size_t>(blockIdx.x) * 2 + slot) * 2) * 128 * 8;
                float4* p0 = reinterpret_cast<float4*>(pp + (32 * q + lane) * 8);
                float4* p1 = reinterpret_cast<float4*>(pp + (128 + 32 * q + lane) * 8);
                p0[0] = make_float4(x0[0], x0[1], x0[2], x0[3]);
                p0[1] = make_float4(x0[4], x0[5], x0[6], x0[7]);
                p1[0] = make_float4(x1[0], x1[1], x1[2], x1[3]);
                p1[1] = make_float4(x1[4], x1[5], x1[6], x1[7]);
                // the warp barrier orders the lanes' stores before lane 0's release
                __syncwarp();
                const long long tu0 = static_cast<long long>(sg.tile) * KG;
                const int b0 = cta_of(tu0), b1 = cta_of(tu0 + KG - 1);
                int last = 0;
                if (lane == 0) {
                    int old;
                    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old)
                                 : "l"(a.tcnt + sg.tile * 4 + q) : "memory");
                    last = old + 1 == b1 - b0 + 1;
                    if (last) a.tcnt[sg.tile * 4 + q] = 0;
                }
                if (!__shfl_sync(0xffffffffu, last, 0)) continue;
                __syncwarp();                       // lane 0's acquire, then every lane's loads
                // sum the parts in K order (CTAs b0 .. b1)
#pragma unroll
                for (int t = 0; t < 8; ++t) { x0[t] = 0.0f; x1[t] = 0.0f; }
                for (int b = b0; b <= b1; b += 4) {
                    // up to four parts' loads in flight, added in CTA order
                    float4 pv[4][4];
#pragma unroll
                    for (int bb = 0; bb < 4; ++bb) {
                        if (b + bb > b1) {
#pragma unroll
                            for (int i = 0; i < 4; ++i) pv[bb][i] = make_float4(0.f, 0.f, 0.f, 0.f);
                            continue;
                        }
                        const int bslot = (static_cast<long long>(U * (b + bb) / Gc) >= tu0) ? 0 : 1;
                        const float* qp = a.part + ((static_cast<size_t>(b + bb) * 2 + bslot) * 2) * 128 * 8;
                        const float4* q0 = reinterpret_cast<const float4*>(qp + (32 * q + lane) * 8);
                        const float4* q1 = reinterpret_cast<const float4*>(qp + (128 + 32 * q + lane) * 8);
                        pv[bb][0] = __ldcg(q0);
                        pv[bb][1] = __ldcg(q0 + 1);
                        pv[bb][2] = __ldcg(q1);
                        pv[bb][3] = __ldcg(q1 + 1);
                    }
#pragma unroll
                    for (int bb = 0; bb < 4; ++bb) {
                        if (b + bb > b1) continue;
                        x0[0] += pv[bb][0].x; x0[1] += pv[bb][0].y; x0[2] += pv[bb][0].z; x0[3] += pv[bb][0].w;
                        x0[4] += pv[bb][1].x; x0[5] += pv[bb][1].y; x0[6] += pv[bb][1].z; x0[7] += pv[bb][1].w;
                        x1[0] += pv[bb][2].x; x1[1] += pv[bb][2].y; x1[2] += pv[bb][2].z; x1[3] += pv[bb][2].w;
                        x1[4] += pv[bb][3].x; x1[5] += pv[bb][3].y; x1[6] += pv[bb][3].z; x1[7] += pv[bb][3].w;
                    }
                }
            }
            if (PHASE == 0) {
                // ---- finish: bias, activation, h rounded to bf16, then split for phase 2: this
                // 128-row tile is K stage mb of phase 2 (B rows plane * 8 + t, 128-byte swizzle),
                // warp q's 32 rows its scale block q ----
                unsigned char* img = a.hs + (static_cast<size_t>(sg.j) * MB + sg.mb) * kMxdHImage;
                const bool live = sg.mb * RPI + 32 * q < R;          // rows past I stay zero
                float hv[8];
                if (live) {
                    const size_t bi = static_cast<size_t>(e) * R + ra;
                    const float bg = a.b0 ? __bfloat162float(__ushort_as_bfloat16(a.b0[bi])) : 0.0f;
                    const float bu = a.b1 ? __bfloat162float(__ushort_as_bfloat16(a.b1[bi])) : 0.0f;
#pragma unroll
                    for (int t = 0; t < 8; ++t)
                        hv[t] = __bfloat162float(__float2bfloat16_rn(act_fn(a.act, x0[t] + bg, x1[t] + bu, a.limit, a.alpha)));
                } else {
#pragma unroll
                    for (int t = 0; t < 8; ++t) hv[t] = 0.0f;
                }
                const int chunk = 2 * q + (lane >> 4);               // 16-byte chunk of the row
                int se_mine = 0;                                    // lane t: token t's exponent
#pragma unroll
                for (int t = 0; t < 8; t += 2) {
                    const int s0 = mx_scale_exp(warp_max(fabsf(hv[t])));
                    const int s1 = mx_scale_exp(warp_max(fabsf(hv[t + 1])));
                    se_mine = lane == t ? s0 : (lane == t + 1 ? s1 : se_mine);
                    uint32_t t1, t2;
                    mx_split2(__fmul_rn(hv[t], __uint_as_float(static_cast<uint32_t>(127 - s0) << 23)),
                              __fmul_rn(hv[t + 1], __uint_as_float(static_cast<uint32_t>(127 - s1) << 23)), t1, t2);
#pragma unroll
                    for (int tt = 0; tt < 2; ++tt) {
                        const int r = t + tt;
                        const int off = ((chunk ^ r) << 4) + (lane & 15);
                        img[r * 128 + off] = static_cast<unsigned char>(t1 >> (8 * tt));
                        img[(8 + r) * 128 + off] = static_cast<unsigned char>(t2 >> (8 * tt));
                    }
                }
                // the scale atom: byte 16 n + q of row n = plane * 8 + t holds 2^s (plane 0) or
                // 2^(s-4) (plane 1)
                if (lane < 8) {
                    img[kDBstage + 16 * lane + q] = static_cast<unsigned char>(se_mine + 127);
                    img[kDBstage + 16 * (8 + lane) + q] = static_cast<unsigned char>(se_mine + 123);
                }
            } else {
                // ---- finish: bias, e per route; the last tile of a row block runs its combine ----
                const int rb = ra + 128;
                const bool va = sg.mb * RPI + 32 * q < R, vb = sg.mb * RPI + 128 + 32 * q < R;
                const float bga = (a.b0 && va) ? __bfloat162float(__ushort_as_bfloat16(a.b0[static_cast<size_t>(e) * R + ra])) : 0.0f;
                const float bgb = (a.b0 && vb) ? __bfloat162float(__ushort_as_bfloat16(a.b0[static_cast<size_t>(e) * R + rb])) : 0.0f;
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    const int r = tl->rid[sg.j][t];
                    if (r < 0) continue;
                    if (va) a.e_out[static_cast<size_t>(r) * R + ra] = x0[t] + bga;
                    if (vb) a.e_out[static_cast<size_t>(r) * R + rb] = x1[t] + bgb;
                }
                __syncwarp();                       // the lanes' stores, then lane 0's release
                int last = 0;
                if (lane == 0) {
                    int old;
                    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old)
                                 : "l"(a.rbcnt + sg.mb * 4 + q) : "memory");
                    last = old + 1 == nt;
                    if (last) a.rbcnt[sg.mb * 4 + q] = 0;
                }
                if (__shfl_sync(0xffffffffu, last, 0)) {
                    __syncwarp();                   // lane 0's acquire, then every lane's loads
                    // slot-ordered combine of this slice's rows (ra, rb) for every token: the
                    // loads of four slots of all tokens are issued before their sums
                    uint16_t* y = static_cast<uint16_t*>(a.y);
                    float acc[kMxdTokens][2];
#pragma unroll
                    for (int t = 0; t < kMxdTokens; ++t)
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            const bool v = t < T && (hh ? vb : va);
                            acc[t][hh] = (v && a.seed) ? __ldcg(a.seed + static_cast<size_t>(t) * R + (hh ? rb : ra)) : 0.0f;
                        }
                    for (int s0 = 0; s0 < k; s0 += 4) {
                        float ev[kMxdTokens][2][4];
#pragma unroll
                        for (int t = 0; t < kMxdTokens; ++t)
#pragma unroll
                            for (int s = 0; s < 4; ++s) {
                                const bool vt = t < T && s0 + s < k;
                                const float* src = a.e_out + static_cast<size_t>(vt ? t * k + s0 + s : 0) * R;
                                ev[t][0][s] = (vt && va) ? __ldcg(src + ra) : 0.0f;
                                ev[t][1][s] = (vt && vb) ? __ldcg(src + rb) : 0.0f;
                            }
#pragma unroll
                        for (int t = 0; t < kMxdTokens; ++t)
#pragma unroll
                            for (int s = 0; s < 4; ++s) {
                                const bool vt = t < T && s0 + s < k;
                                const float wv = tl->wr[vt ? t * k + s0 + s : 0];
                                const float n0 = __fadd_rn(acc[t][0], __fmul_rn(wv, ev[t][0][s]));
                                const float n1 = __fadd_rn(acc[t][1], __fmul_rn(wv, ev[t][1][s]));
                                acc[t][0] = vt ? n0 : acc[t][0];
                                acc[t][1] = vt ? n1 : acc[t][1];
                            }
                    }
#pragma unroll
                    for (int t = 0; t < kMxdTokens; ++t)
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            if (t >= T || !(hh ? vb : va)) continue;
                            const size_t yo = static_cast<size_t>(t) * R + (hh ? rb : ra);
                            if (a.y_f32) a.y_f32[yo] = acc[t][hh];
                            y[yo] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[t][hh]));
                        }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 256;" ::"r"(tmem) : "memory");
}

inline bool make_map_mxd_codes(CUtensorMap* m, const void* blob, int G, int K, int R, int E) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t kg = static_cast<cuuint64_t>(mx_kg(K)), r = static_cast<cuuint64_t>(R);
    const cuuint32_t es[5] = {1, 1, 1, 1, 1};
    if (G == 2) {
        const cuuint64_t dims[5] = {128, r, 2, kg, static_cast<cuuint64_t>(E)};
        const cuuint64_t strides[4] = {64, r * 64, 2 * r * 64, kg * 2 * r * 64};
        const cuuint32_t box[5] = {128, 128, 2, 1, 1};
        return fn(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 5, const_cast<void*>(blob), dims, strides, box,
                  es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    }
    const cuuint64_t dims[4] = {128, r, kg, static_cast<cuuint64_t>(E)};
    const cuuint64_t strides[3] = {64, r * 64, kg * r * 64};
    const cuuint32_t box[4] = {128, 256, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 4, const_cast<void*>(blob), dims, strides, box,
              es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The x image: CTA t splits token row t (zeros for t >= T) under one scale, 2^s with s =
// floor(log2 max|x_t|) - 7; thread c takes the 16-column chunk c of every K stage (K <= 4096);
// the image holds the K stages [KG][16 rows][128 B] as phase 1's shared memory holds them
// (128-byte swizzle), then the scale atom of the 16 rows.  The CTAs also zero the counters.
__global__ void __launch_bounds__(256) mxd_prep_kernel(const MxdArgs a) {
    pdl_wait();
    pdl_launch_dependents();
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < a.ncnt; i += gridDim.x * blockDim.x) a.tcnt[i] = 0;
    __shared__ float red[8];
    const int t = blockIdx.x, c = threadIdx.x, K = a.K, KG = mx_kg(K);
    uint4 v0 = make_uint4(0u, 0u, 0u, 0u), v1 = v0;
    if (t < a.T && c * 16 < K) {
        const uint4* src = reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(t) * K + c * 16);
        v0 = __ldg(src);
        v1 = __ldg(src + 1);
    }
    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    float mx = 0.0f;
#pragma unroll
    for (int h = 0; h < 8; ++h)
        mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(w[h] << 16)), fabsf(__uint_as_float(w[h] & 0xFFFF0000u))));
    mx = warp_max(mx);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
    __syncthreads();
    mx = red[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) mx = fmaxf(mx, red[i]);
    const int se = mx_scale_exp(mx);
    const float inv = __uint_as_float(static_cast<uint32_t>(127 - se) << 23);
    if (c < KG * 8) {
        uint32_t q1[4] = {0u, 0u, 0u, 0u}, q2[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int h = 0; h < 8; ++h) {
            uint32_t t1, t2;
            mx_split2(__fmul_rn(__uint_as_float(w[h] << 16), inv),
                      __fmul_rn(__uint_as_float(w[h] & 0xFFFF0000u), inv), t1, t2);
            q1[h >> 1] |= (t1 & 0xFFFFu) << (16 * (h & 1));
            q2[h >> 1] |= (t2 & 0xFFFFu) << (16 * (h & 1));
        }
        unsigned char* st = a.xs + static_cast<size_t>(c >> 3) * kDBstage;
        const int cc = c & 7;
        *reinterpret_cast<uint4*>(st + t * 128 + ((cc ^ t) << 4)) = make_uint4(q1[0], q1[1], q1[2], q1[3]);
        *reinterpret_cast<uint4*>(st + (8 + t) * 128 + ((cc ^ t) << 4)) = make_uint4(q2[0], q2[1], q2[2], q2[3]);
    }
    if (threadIdx.x == 0) {
        // rows t (2^s) and 8 + t (2^(s-4)) of the atom; rows 16..31 zero
        unsigned char* atom = a.xs + static_cast<size_t>(KG) * kDBstage;
        const uint32_t w0 = static_cast<uint32_t>(se + 127) * 0x01010101u;
        *reinterpret_cast<uint4*>(atom + 16 * t) = make_uint4(w0, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(atom + 16 * (8 + t)) = make_uint4(w0 - 0x04040404u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(atom + 16 * (16 + t)) = make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(atom + 16 * (24 + t)) = make_uint4(0u, 0u, 0u, 0u);
    }
}

}  // namespace

cudaError_t launch_mxd_prep(const MxdArgs& a, cudaStream_t s) {
    if (a.K > kMxdMaxH || a.T > kMxdTokens) return cudaErrorInvalidValue;
    return launch_pdl(mxd_prep_kernel, dim3(kMxdTokens), dim3(256), 0, s, a);
}

cudaError_t launch_mxd(const MxdArgs& a, int num_sms, cudaStream_t s) {
    MxdParams P;
    memset(&P, 0, sizeof(P));
    P.a = a;
    MxdLayout& L = P.ly;
    const int KG = mx_kg(a.K);
    L.sfa_off = 2 * kDAbox;
    L.b_off = L.sfa_off + 2 * kDAtom;
    L.slot_bytes = (L.b_off + (a.phase == 1 ? kMxdHImage : kDBstage) + 1023) / 1024 * 1024;
    const size_t tail = (sizeof(MxdTail) + 255) / 256 * 256;
    const size_t fixed = kDAtom + tail;
    const size_t budget = 227 * 1024 - 1024;
    if (fixed >= budget) return cudaErrorInvalidValue;
    L.nslot = static_cast<int>((budget - fixed) / L.slot_bytes);
    if (L.nslot > kDMaxSlots) L.nslot = kDMaxSlots;
    if (L.nslot < 2) return cudaErrorInvalidValue;
    L.sfb_off = L.nslot * L.slot_bytes;
    L.tail_off = L.sfb_off + kDAtom;
    const size_t smem = 1024 + static_cast<size_t>(L.tail_off) + tail;
    if (!make_map_mxd_codes(&P.tmA, a.w, a.phase == 0 ? 2 : 1, a.K, a.R, a.E)) return cudaErrorInvalidValue;
    const int grid = num_sms < kMxdMaxCtas ? num_sms : kMxdMaxCtas;
    cudaError_t e;
    if (a.phase == 0) {
        e = ensure_smem(mxd_kernel<0>, smem);
        if (e != cudaSuccess) return e;
        return launch_pdl(mxd_kernel<0>, dim3(grid), dim3(kDThreads), smem, s, P);
    }
    e = ensure_smem(mxd_kernel<1>, smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(mxd_kernel<1>, dim3(grid), dim3(kDThreads), smem, s, P);
}

}  // namespace tsmoe

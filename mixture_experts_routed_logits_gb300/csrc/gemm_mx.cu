// gemm_mx.cu -- steps 4-5 of the routed-expert layer for MXFP4 experts and bf16 activations on
// the block-scaled tensor cores (tcgen05.mma kind::mxf8f6f4 with e8m0 block scales in TMEM).
//
// Source pages (docs.rs, turbospark-runtime 0.3.0):
//   gpt-oss routed-expert pass (src/families/gptoss/moe.rs), module header: the experts are
//     MXFP4 (e2m1 values, one e8m0 scale per 32), the clamped SwiGLU and the per-expert biases
//     ride inside the phase pair; phase 1 writes the 16-bit acts, phase 2 the down projection.
//   Gemma-4 batched routed prefill (src/families/gemma4/moe_batch.rs): one route list for the
//     micro-batch, a phase-1 / phase-2 pair of kernels over it.
//
// Design (GB300, one CTA per SM, persistent):
//   * A = e2m1 weights straight from HBM: the 4-bit TMA type spreads each 16 codes over 16 bytes
//     of shared memory (the operand layout of kind::mxf8f6f4), so no thread touches a weight;
//     their e8m0 scales arrive as pre-arranged 512-byte atoms (one 1-D bulk copy) and reach TMEM
//     with tcgen05.cp.  Each weight byte crosses HBM once per route tile.
//   * B = activations split exactly into two e4m3 terms under e8m0 block scales: a bf16 value v
//     of a 32-block with max |v| = m is v = 2^s (t1 + t2 / 16), s = floor(log2 m) - 7, t1 the
//     e4m3 rounding of v / 2^s and t2 that of 16 (v / 2^s - t1); both are exact for every
//     |v| >= m 2^-14 (a bf16 significand has 8 bits, each term carries 4), and smaller values
//     keep an error below m 2^-23.  The two terms of a tile's routes are stacked as 2 nb columns
//     of B with scales 2^s and 2^(s-4); the epilogue adds column n and column nb + n.  So the
//     tensor core computes sum_k w_k x_k with exact products and f32 accumulation, the same
//     quantity as the plain oracle, with no dequantisation on the ALUs.
//   * Work item = (expert, block of weight rows, tile of <= 56 routes, K part).  Swap-AB: weights
//     are the MMA's M = 128 rows, the stacked routes its N = 2 nb columns.  Phase 1: gate and up
//     of the same rows (two accumulators); phase 2: two 128-row blocks of down.  Two
//     accumulator sets alternate per item so an item's epilogue overlaps the next one's MMAs.
//   * Phase-1 epilogue: bias, activation, h rounded to bf16, then split into the two e4m3 terms
//     for phase 2 (a warp holds 32 consecutive rows of h = one 32-block: the block max is a warp
//     max).  Phase-2 epilogue: bias, e in f32 by route id for the slot-ordered combine.
//   * Every stage is three copies: 16 KB of weight codes in ONE tensor copy (gate and up of 128
//     rows side by side in the blob, or 256 rows of down), their two scale atoms in one 1 KB bulk
//     copy, and the tile's activations (both term planes) in one tensor copy.  A TMA
//     instruction holds its issuing thread for ~140 clocks whatever its size (measured on
//     GB300), so the copies are few, large, and issued from two warps.
//   * Warps: 0 weight producer, 7 scale + activation producer (each also prefetches its share
//     of a later stage into L2), 1 MMA issuer (one thread, only MMAs: ~88 clocks each for this
//     kind up to N = 128), 2-5 and 8-11 epilogue (two per TMEM lane quarter, alternate groups
//     of 8 route columns), 6 builds the activation
//     scale atoms and copies every stage's scale atoms into TMEM (tcgen05.cp, committed to the
//     stage's scale barrier).  Every mbarrier wait is bounded.
//   * Above 64 routes one cooperative launch runs both phases (gate/up, bias, clamped SwiGLU and
//     down fused): the CTAs draw items from one counter, every phase-0 item before any phase-1
//     item, so CTAs that finish early take more (measured: the per-CTA end times of a static
//     round-robin spread over ~50 us); a phase-0 item counts the h slices it writes per
//     (expert, route tile) and a phase-1 item's readers wait (acquire, bounded) for the full
//     count before their first read of that h.  Warp 0 draws the items and publishes them in a
//     small shared-memory queue that the other roles read in order.  Fewer routes split K
//     (parked partials) and keep one launch per phase.
#include "mx_common.cuh"

namespace tsmoe {

namespace {

constexpr int kMxBM = 128;            // weight rows per accumulator
constexpr int kMxBK = 128;            // K per stage: one 128-byte swizzle row of 8-bit operand
constexpr int kMxAbox = 16384;        // shared bytes of one A box (128 rows x 128 padded codes)
constexpr int kMxAtx = 8192;          // transaction bytes of one A box (the packed codes)
constexpr int kMxAtom = 512;          // scale atom: 128 rows x 4 blocks
constexpr int kMxNbMax = 56;          // routes per tile with two accumulator sets
constexpr int kMxNbMax1 = 112;        // routes per tile with one accumulator set
constexpr int kMxEpiWarps = 8;        // epilogue warps: 2-5 and 8.., kMxEpiWarps / 4 per lane quarter
constexpr int kMxThreads = (kMxEpiWarps + 4) * 32;   // see the roles in the file header
static_assert(kMxEpiWarps % 4 == 0, "whole TMEM lane quarters");
constexpr int kMxMaxSlots = 6;
constexpr int kMxQ = 8;               // item queue entries (two-phase launch)
constexpr int kMxQReaders = 3 + kMxEpiWarps;   // roles reading each entry: warps 7, 6, 1, epilogue

struct MxLayout {
    int nb;               // routes per tile at most (multiple of 8); the MMA's N is 2 nb
    int nsets;            // accumulator sets (2 when 4 * 2nb <= 448)
    int sf_col0;          // first TMEM column of the stage scale factors (16 per slot)
    int nslot;
    int slot_bytes;       // A0, A1, B (2 nb rows), SFA0, SFA1
    int b_off, sfa_off;   // offsets inside a slot
    int S[2];             // K parts per phase
};

struct MxParams {
    // per phase: weight codes, 4-bit: phase 0 {128, R, 2, KG, E} box {128, 128, 2, 1, 1};
    // phase 1 {128, R, KG, E} box {128, 256, 1, 1}; activation planes {K, rows_in, 2} u8, box
    // {128, 8 (q + 1), 2}
    CUtensorMap tmA[2];
    CUtensorMap tmB[2][kMxNbMax / 8];
    MxArgs a[2];
    MxLayout ly;
    int p0, p1;           // the launch runs phases p0 .. p1 - 1
    int* hrdy;            // both phases: per (touched expert, route tile) count of finished h slices
    int* work;            // both phases: items handed out so far (over the grid)
};

struct MxTail {
    uint64_t full[kMxMaxSlots];       // TMA of a slot landed
    uint64_t sfull[kMxMaxSlots];      // activation scale atom of a slot written
    uint64_t empty[kMxMaxSlots];      // MMAs reading a slot done
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t qfull[kMxQ];             // two-phase launch: item entry published
    uint64_t qempty[kMxQ];            // every reader has taken the entry
    int qitem[kMxQ];
    uint32_t tmem_base;
    volatile int abort_flag;
    int nt;
    int touched[kMaxExperts];
    int cnt[kMaxExperts];
    int bnj[kMaxExperts];
    int tbase[kMaxExperts + 1];       // first route tile of each touched expert
    int ioff[2][kMaxExperts + 1];     // first item of each touched expert, per phase
};

// A phase as a type (phase-specialised code inside generic lambdas).
template <int V>
struct PhaseTag {
    static constexpr int value = V;
};

// One phase's geometry.
struct MxGeo {
    int ph, G, rpi, R, K, MB, KG, S, kbp;
    const uint8_t* sfa_base;
};

__device__ __forceinline__ MxGeo mx_geo(const MxParams& P, int ph) {
    const MxArgs& a = P.a[ph];
    MxGeo g;
    g.ph = ph;
    g.G = ph == 0 ? 2 : 1;                            // matrices of the blob (gate + up, or down)
    g.rpi = ph == 0 ? kMxBM : 2 * kMxBM;              // weight rows per item
    g.R = a.R;
    g.K = a.K;
    g.MB = mx_units(g.G, g.R);                        // row blocks of rpi rows
    g.KG = mx_kg(g.K);
    g.S = P.ly.S[ph];
    g.kbp = (g.KG + g.S - 1) / g.S;
    g.sfa_base = a.w + mx_sf_offset(g.G, a.E, g.R, g.K);
    return g;
}

// P0, P1: the phases the launch runs (P0 .. P1 - 1; P.p0 and P.p1 hold the same).
template <int P0, int P1>
__global__ void __launch_bounds__(kMxThreads, 1) tc_mx_kernel(const __grid_constant__ MxParams P) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const MxLayout& Ly = P.ly;
    unsigned char* base = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    unsigned char* ring = base;
    unsigned char* sfb_atoms = ring + static_cast<size_t>(Ly.nslot) * Ly.slot_bytes;
    MxTail* tl = reinterpret_cast<MxTail*>(sfb_atoms + kMxMaxSlots * kMxAtom);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_wait();
    pdl_launch_dependents();
    constexpr int p0 = P0, p1 = P1;
    const MxArgs& a0 = P.a[p0];                       // the fields both phases share
    int* status = a0.status;
    // the two phases' geometry, selected by value (a runtime-indexed array would live in local
    // memory); a phase the launch does not run is never read
    const MxGeo gA = mx_geo(P, p0), gB = mx_geo(P, p1 - 1);
    auto geo = [&](int ph) { return ph == p0 ? gA : gB; };
    const int NS = Ly.nslot;
    const int NMAX = 2 * Ly.nb;                       // accumulator columns per matrix
    const int Tk = a0.rows_in;
    const int hdone = P.hrdy ? gA.MB * kMxEpiWarps : 0;   // phase-0 slices of one (expert, tile)

    if (threadIdx.x == 0) {
        int nt = 0, acc0 = 0, acc1 = 0, tacc = 0;
        for (int e = 0; e < a0.E; ++e) {
            const int n = a0.off[e + 1] - a0.off[e];
            if (n > 0) {
                // the expert's routes in equal tiles (multiples of 8), not full tiles + a tail
                const int ntl0 = (n + Ly.nb - 1) / Ly.nb;
                const int bnj = min(Ly.nb, ((n + ntl0 - 1) / ntl0 + 7) & ~7);
                const int ntl = (n + bnj - 1) / bnj;
                tl->touched[nt] = e;
                tl->cnt[nt] = n;
                tl->bnj[nt] = bnj;
                tl->tbase[nt] = tacc;
                tl->ioff[0][nt] = acc0;
                tl->ioff[1][nt] = acc1;
                tacc += ntl;
                if (p0 == 0) acc0 += gA.MB * ntl * gA.S;
                if (p1 == 2) acc1 += gB.MB * ntl * gB.S;
                ++nt;
            }
        }
        tl->tbase[nt] = tacc;
        tl->ioff[0][nt] = acc0;
        tl->ioff[1][nt] = acc1;
        tl->nt = nt;
        tl->abort_flag = 0;
        for (int s = 0; s < NS; ++s) {
            mbar_init(&tl->full[s], 1);
            mbar_init(&tl->sfull[s], 1);
            mbar_init(&tl->empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tl->tfull[b], 1);
            mbar_init(&tl->tempty[b], kMxEpiWarps);
        }
        for (int q = 0; q < kMxQ; ++q) {
            mbar_init(&tl->qfull[q], 1);
            mbar_init(&tl->qempty[q], kMxQReaders);
        }
        fence_mbar_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(
                         smem_u32(&tl->tmem_base))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tl->tmem_base;
    const int nt = tl->nt;
    auto items = [&](int ph) { return tl->ioff[ph][nt]; };

    // item i of phase ph -> touched expert j, row block mb, route tile, K part kp (kp fastest)
    auto decode = [&](const MxGeo& g, int i, int& j, int& mb, int& tile, int& kp) {
        const int* io = tl->ioff[g.ph];
        j = 0;
        while (j + 1 < nt && i >= io[j + 1]) ++j;
        const int ntl = (tl->cnt[j] + tl->bnj[j] - 1) / tl->bnj[j];
        const int local = i - io[j];
        kp = local % g.S;
        const int rest = local / g.S;
        tile = rest % ntl;
        mb = rest / ntl;
    };
    // routes of item: first route-list position p0, valid routes nv, tile width tw (the
    // expert's tile size, a multiple of 8).  A tile is loaded and multiplied tw routes wide: its
    // two term planes land at rows [0, tw) and [tw, 2 tw) of the B operand, N = 2 tw.
    auto tile_of = [&](int j, int tile, int& q0, int& nv, int& tw) {
        tw = tl->bnj[j];
        q0 = a0.off[tl->touched[j]] + tile * tw;
        nv = min(tw, tl->cnt[j] - tile * tw);
    };
    // The items of this CTA, in order: a single-phase launch takes items blockIdx.x, +
    // gridDim.x, ...; the two-phase launch takes them as they come from one counter over the
    // grid (phase 0's items first, then phase 1's), so CTAs that finish early take more.  Warp 0
    // draws them (the draw for the next item is in flight while it issues this one's copies)
    // and publishes each in a small queue the other roles read in the same order.
    constexpr bool kFused = P0 == 0 && P1 == 2;
    const int total = kFused ? items(0) + items(1) : items(p0);
    auto item_of = [&](int gi, int& ph, int& i) {
        ph = kFused ? (gi < items(0) ? 0 : 1) : p0;
        i = kFused && ph == 1 ? gi - items(0) : gi;
    };
    // the n-th item (a reader role: one thread per warp calls this); total on a timeout
    auto read_item = [&](int n) {
        if (!kFused) return static_cast<int>(blockIdx.x) + n * static_cast<int>(gridDim.x);
        const int slot = n % kMxQ;
        if (!mbar_wait_bounded(&tl->qfull[slot], (n / kMxQ) & 1)) {
            tl->abort_flag = 1;
            report_error(status, DEV_ERR_TIMEOUT);
            return total;
        }
        const int gi = tl->qitem[slot];
        mbar_arrive(&tl->qempty[slot]);
        return gi;
    };
    // the same for a whole warp (lane 0 reads, every lane gets the item)
    auto read_item_warp = [&](int n) {
        int gi = 0;
        if (lane == 0) gi = read_item(n);
        return __shfl_sync(0xffffffffu, gi, 0);
    };
    // warp 0's draw of the n-th item (n = 0, 1, ... in order): publishes it, then starts the draw
    // of the next
    int draw_next = 0;
    auto draw_item = [&](int n) {
        if (!kFused) return static_cast<int>(blockIdx.x) + n * static_cast<int>(gridDim.x);
        const int gi = n == 0 ? atomicAdd(P.work, 1) : draw_next;
        const int slot = n % kMxQ;
        if (n >= kMxQ && !mbar_wait_bounded(&tl->qempty[slot], ((n / kMxQ) - 1) & 1)) {
            tl->abort_flag = 1;
            report_error(status, DEV_ERR_TIMEOUT);
            return total;
        }
        tl->qitem[slot] = gi;
        mbar_arrive(&tl->qfull[slot]);
        draw_next = gi < total ? atomicAdd(P.work, 1) : total;
        return gi;
    };
    // The stage sequence: each item's K stages in order.  Walked by the copy roles.
    struct Stage { int n, ph, i, kb, kb1, e, j, tile, mb, q0, tw; };
    auto first_stage = [&](Stage& c) {
        c.n = -1;
        c.kb1 = 0;
    };
    // moves c to the next stage (the next item from get(n)); false at the end
    auto next_stage = [&](Stage& c, auto&& get) -> bool {
        if (c.kb1 > 0 && c.kb + 1 < c.kb1) { ++c.kb; return true; }
        const int gi = get(++c.n);
        if (gi >= total) {
            c.kb1 = 0;
            c.n = 1 << 30;               // stays at the end
            return false;
        }
        item_of(gi, c.ph, c.i);
        const MxGeo g = geo(c.ph);
        int kp, nv;
        decode(g, c.i, c.j, c.mb, c.tile, kp);
        tile_of(c.j, c.tile, c.q0, nv, c.tw);
        c.e = tl->touched[c.j];
        c.kb = kp * g.kbp;
        c.kb1 = min(g.KG, c.kb + g.kbp);
        return true;
    };
    // the look-ahead cursors of the single-phase launch see the same static sequence
    auto static_item = [&](int n) { return static_cast<int>(blockIdx.x) + n * static_cast<int>(gridDim.x); };
    // one stage's weights: 16 KB of codes (gate and up of 128 rows, or 256 rows of down) in ONE
    // tensor copy, and their two scale atoms in one 1 KB bulk copy
    auto a_load = [&](const Stage& c, void* dst, uint64_t* bar) {
        if (c.ph == 0) tma_load_5d(dst, &P.tmA[0], 0, c.mb * kMxBM, 0, c.kb, c.e, bar);
        else tma_load_4d(dst, &P.tmA[1], 0, c.mb * 2 * kMxBM, c.kb, c.e, bar);
    };
    auto a_prefetch = [&](const Stage& c) {
        if (c.ph == 0) tma_prefetch_5d(&P.tmA[0], 0, c.mb * kMxBM, 0, c.kb, c.e);
        else tma_prefetch_4d(&P.tmA[1], 0, c.mb * 2 * kMxBM, c.kb, c.e);
    };
    auto sfa_src = [&](const Stage& c) {
        const MxGeo g = geo(c.ph);
        return g.sfa_base + ((static_cast<size_t>(c.e) * g.MB + c.mb) * g.KG + c.kb) * (2 * kMxAtom);
    };
    // Both phases in one launch: a phase-1 stage reads the h of its (expert, route tile), which
    // phase-0 items of any CTA write; they count their finished slices, and the readers wait
    // (acquire, bounded) for the full count before their first read of that h.  Every CTA
    // takes all its phase-0 items before any phase-1 item and the launch is cooperative, so
    // every count completes.
    auto h_key = [&](const Stage& c) { return tl->tbase[c.j] + c.tile; };
    auto wait_h = [&](int key) {
        const long long t0 = clock64();
        while (ld_acquire_gpu_s32(P.hrdy + key) < hdone) {
            if (tl->abort_flag || clock64() - t0 > (1ll << 31)) return false;
            __nanosleep(128);
        }
        return true;
    };
    // The copies of one stage come from two warps (a TMA instruction holds its issuing thread
    // for ~140 clocks whatever its size): warp 0 the weights, warp 7 their scales and the
    // activations; each also prefetches into L2 its share of the stage kPrefetch stages ahead,
    // so that more bytes are on their way from HBM than the ring holds.
    constexpr int kPrefetch = 6;

    if (warp == 0 || warp == 7) {
        if (lane == 0) {
            // ============================== TMA producers =====================================
            const bool wts = warp == 0;
            // (the two-phase launch draws its items as it goes: no look-ahead there)
            Stage look;
            first_stage(look);
            bool look_ok = !kFused;
            for (int q = 0; q < kPrefetch && look_ok; ++q)
                if ((look_ok = next_stage(look, static_item))) {
                    if (wts) a_prefetch(look);
                    else bulk_prefetch_l2(sfa_src(look), 2 * kMxAtom);
                }
            int it = 0;
            int issued[kMxMaxSlots];
            for (int q = 0; q < kMxMaxSlots; ++q) issued[q] = -1;
            int hkey = -1;                      // warp 7: the (expert, tile) whose h is complete
            Stage c;
            first_stage(c);
            while (wts ? next_stage(c, draw_item) : next_stage(c, read_item)) {
                const int s = it % NS;
                if (tl->abort_flag || !mbar_wait_bounded(&tl->empty[s], ((it / NS) & 1) ^ 1)) {
                    tl->abort_flag = 1;
                    report_error(status, DEV_ERR_TIMEOUT);
                    break;
                }
                unsigned char* st = ring + static_cast<size_t>(s) * Ly.slot_bytes;
                if (wts) {
                    // arms the stage barrier for every byte of the stage (the other producer's
                    // copies may complete before this; the count may go below zero meanwhile)
                    mbar_arrive_expect_tx(&tl->full[s], kMxAtx * 2 + 2 * kMxAtom + 2u * c.tw * 128u);
                    a_load(c, st, &tl->full[s]);
                } else {
                    if (c.ph == 1 && P.hrdy && h_key(c) != hkey) {
                        if (!wait_h(h_key(c))) {
                            // (warp 0 armed this barrier: its bytes still land; the consumers'
                            // bounded waits on it run out)
                            tl->abort_flag = 1;
                            report_error(status, DEV_ERR_TIMEOUT);
                            break;
                        }
                        asm volatile("fence.proxy.async.global;" ::: "memory");
                        hkey = h_key(c);
                    }
                    bulk_g2s(st + Ly.sfa_off, sfa_src(c), 2 * kMxAtom, &tl->full[s]);
                    // the tile's two term planes in one box: rows [0, tw) and [tw, 2 tw)
                    tma_load_3d(st + Ly.b_off, &P.tmB[c.ph][c.tw / 8 - 1], c.kb * kMxBK, c.q0, 0, &tl->full[s]);
                }
                issued[s] = it;
                ++it;
                if (look_ok && (look_ok = next_stage(look, static_item))) {
                    if (wts) a_prefetch(look);
                    else bulk_prefetch_l2(sfa_src(look), 2 * kMxAtom);
                }
            }
            // drain: every copy this thread issued must land before the CTA may exit (a stage
            // warp 7 left unissued after an error never completes: its wait runs out)
            for (int q = 0; q < NS; ++q)
                if (issued[q] >= 0) mbar_wait_bounded(&tl->full[q], (issued[q] / NS) & 1);
        }
    } else if (warp == 6) {
        // ============ activation scale atoms, and every stage's scales into TMEM ===============
        // The scale words of stage kb sit in a row of the transposed scale array ([k group]
        // [route], 4 block scales per word), so a tile's words are coalesced loads; the words of
        // the next stage are loaded while this stage waits for its slot (unless they are h
        // scales still to be waited for: then after this stage's commit).  Lane 0 then copies
        // the stage's weight and activation scale atoms into the slot's TMEM columns and
        // commits the copies to the slot's scale barrier, which the MMA issuer waits on.
        constexpr int kW = (2 * kMxNbMax + 31) / 32;          // words per lane and stage
        // (h scales written in this launch are read past L1, one branch per stage; the rest
        // through the read-only path.  The code for the waits exists only in the two-phase
        // kernel: a branch in this loop measured ~7 % slower single-phase kernels.)
        constexpr bool kFused = P0 == 0 && P1 == 2;
        const uint32_t* bsf0 = reinterpret_cast<const uint32_t*>(P.a[p0].bsf);
        const uint32_t* bsf1 = reinterpret_cast<const uint32_t*>(P.a[p1 - 1].bsf);
        auto load_words = [&](const Stage& c, uint32_t (&w)[kW]) {
            const uint32_t* bsfw = (c.ph == p0 ? bsf0 : bsf1) + static_cast<size_t>(c.kb) * Tk;
            if (kFused && c.ph == 1) {
#pragma unroll
                for (int q = 0; q < kW; ++q) {
                    const int n = lane + 32 * q;
                    const int p = c.q0 + (n < c.tw ? n : n - c.tw);
                    w[q] = (n < 2 * c.tw && p < Tk) ? __ldcg(bsfw + p) : 0x7F7F7F7Fu;
                }
            } else {
#pragma unroll
                for (int q = 0; q < kW; ++q) {
                    const int n = lane + 32 * q;
                    const int p = c.q0 + (n < c.tw ? n : n - c.tw);
                    w[q] = 0x7F7F7F7Fu;
                    if (n < 2 * c.tw && p < Tk) w[q] = __ldg(bsfw + p);
                }
            }
        };
        int hkey = -1;
        // h scales of stage c may be read (waits once per (expert, tile)); false on timeout
        auto h_ready = [&](const Stage& c) {
            if (!kFused || c.ph != 1 || h_key(c) == hkey) return true;
            int ok = 1;
            if (lane == 0) ok = wait_h(h_key(c));
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (ok) (void)ld_acquire_gpu_s32(P.hrdy + h_key(c));     // every lane acquires
            hkey = h_key(c);
            return ok != 0;
        };
        auto must_wait = [&](const Stage& c) { return kFused && c.ph == 1 && h_key(c) != hkey; };
        Stage cur, nxt;
        first_stage(nxt);
        uint32_t wcur[kW];
        bool have = next_stage(nxt, read_item_warp);
        bool fail = false;
        if (have) {
            if (!h_ready(nxt)) fail = true;
            else load_words(nxt, wcur);
        }
        for (int it = 0; have && !fail; ++it) {
            if (__shfl_sync(0xffffffffu, tl->abort_flag, 0)) break;
            cur = nxt;
            const int s = it % NS;
            uint32_t wnext[kW];
            const bool more = next_stage(nxt, read_item_warp);
            const bool defer = more && must_wait(nxt);
            if (more && !defer) load_words(nxt, wnext);
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(&tl->empty[s], ((it / NS) & 1) ^ 1))) {
                fail = true;
                break;
            }
            unsigned char* atom = sfb_atoms + s * kMxAtom;
            // column n < tw: first term of route q0 + n (scale 2^s); tw + n: second (2^(s-4))
#pragma unroll
            for (int q = 0; q < kW; ++q) {
                const int n = lane + 32 * q;
                if (n < 2 * cur.tw)
                    *reinterpret_cast<uint32_t*>(atom + 16 * (n & 31) + 4 * (n >> 5)) =
                        n < cur.tw ? wcur[q] : wcur[q] - 0x04040404u;
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            int ok = 1;
            if (lane == 0) {
                // the weight scale atoms come with the slot's copies
                ok = mbar_wait_bounded(&tl->full[s], (it / NS) & 1);
                if (ok) {
                    tc_fence_after();
                    const unsigned char* st = ring + static_cast<size_t>(s) * Ly.slot_bytes;
                    const uint32_t tsf = tmem + static_cast<uint32_t>(Ly.sf_col0 + 16 * s);
                    tmem_cp_atom(tsf, st + Ly.sfa_off);
                    tmem_cp_atom(tsf + 4, st + Ly.sfa_off + kMxAtom);
                    tmem_cp_atom(tsf + 8, atom);
                    umma_commit(&tl->sfull[s]);
                }
            }
            if (!__shfl_sync(0xffffffffu, ok, 0)) {
                fail = true;
                break;
            }
            if (defer) {
                if (!h_ready(nxt)) {
                    fail = true;
                    break;
                }
                load_words(nxt, wnext);
            }
#pragma unroll
            for (int q = 0; q < kW; ++q) wcur[q] = wnext[q];
            have = more;
        }
        if (fail && lane == 0) {
            tl->abort_flag = 1;
            report_error(status, DEV_ERR_TIMEOUT);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ================================= MMA issuer ====================================
            int it = 0, n_item = 0;
            bool ok = true;
            // one item (phase-specialised code, as for the epilogue); false on a timeout
            auto mma_item = [&](auto tag, int i) -> bool {
                constexpr int ph = decltype(tag)::value;
                const MxGeo g = ph == 0 ? gA : gB;
                {
                    const int my = n_item++;
                    int j, mb, tile, kp, q0, nv, tw;
                    decode(g, i, j, mb, tile, kp);
                    tile_of(j, tile, q0, nv, tw);
                    const bool has1 = ph == 0 || mb * g.rpi + kMxBM < g.R;
                    const int N = 2 * tw;
                    const int kb0 = kp * g.kbp, kb1 = min(g.KG, kb0 + g.kbp);
                    const int tb = my % Ly.nsets, tuse = my / Ly.nsets;
                    const uint32_t acc0 = tmem + static_cast<uint32_t>(tb * 2 * NMAX);
                    const uint32_t acc1 = acc0 + static_cast<uint32_t>(NMAX);
                    if (!mbar_wait_bounded(&tl->tempty[tb], (tuse & 1) ^ 1)) {
                        tl->abort_flag = 1;
                        report_error(status, DEV_ERR_TIMEOUT);
                        return false;
                    }
                    tc_fence_after();
                    bool okk = true;
                    for (int kb = kb0; kb < kb1; ++kb, ++it) {
                        const int s = it % NS;
                        if (!mbar_wait_bounded(&tl->full[s], (it / NS) & 1) ||
                            !mbar_wait_bounded(&tl->sfull[s], (it / NS) & 1)) {
                            tl->abort_flag = 1;
                            report_error(status, DEV_ERR_TIMEOUT);
                            okk = false;
                            break;
                        }
                        tc_fence_after();
                        const unsigned char* st = ring + static_cast<size_t>(s) * Ly.slot_bytes;
                        const uint32_t tsf = tmem + static_cast<uint32_t>(Ly.sf_col0 + 16 * s);
                        const uint64_t dA0 = sdesc_sw128(smem_u32(st));
                        const uint64_t dA1 = sdesc_sw128(smem_u32(st + kMxAbox));
                        const uint64_t dB = sdesc_sw128(smem_u32(st + Ly.b_off));
#pragma unroll
                        for (int ks = 0; ks < kMxBK / 32; ++ks) {
                            const uint32_t acc = (kb > kb0 || ks > 0) ? 1u : 0u;
                            const uint32_t idesc = idesc_mx(N, ks);
                            umma_mx(acc0, dA0 + 2 * ks, dB + 2 * ks, idesc, tsf, tsf + 8, acc);
                            if (has1) umma_mx(acc1, dA1 + 2 * ks, dB + 2 * ks, idesc, tsf + 4, tsf + 8, acc);
                        }
                        umma_commit(&tl->empty[s]);
                    }
                    if (!okk) return false;
                    umma_commit(&tl->tfull[tb]);
                }
                return true;
            };
            for (int n = 0; ok && !tl->abort_flag; ++n) {
                const int gi = read_item(n);
                if (gi >= total) break;
                int ph, i;
                item_of(gi, ph, i);
                if (P0 == 0 && ph == 0) ok = mma_item(PhaseTag<0>{}, i);
                else if (P1 == 2) ok = mma_item(PhaseTag<1>{}, i);
            }
        }
    } else {
        // =================================== epilogue ==========================================
        const int q = warp & 3;                     // TMEM lane quarter of this warp
        // nh warps per quarter (2-5, 8-11, ...) take groups of 8 route columns in turn
        constexpr int nh = kMxEpiWarps / 4;
        const int hw = warp < 8 ? 0 : (warp - 4) >> 2;
        const uint32_t tq = tmem + (static_cast<uint32_t>(32 * q) << 16);
        int n_item = 0;
        bool stop = false;
        // one item; false when the call is stopping
        auto epi_item = [&](auto tag, int i) -> bool {
            constexpr int ph = decltype(tag)::value;
            const MxGeo g = ph == 0 ? gA : gB;
            const MxArgs& a = P.a[ph];
            const int R = g.R, S = g.S;
            {
                const int my = n_item++;
                int j, mb, tile, kp, q0, nv, tw;
                decode(g, i, j, mb, tile, kp);
                tile_of(j, tile, q0, nv, tw);
                const int e = tl->touched[j];
                const int tb = my % Ly.nsets, tuse = my / Ly.nsets;
                const uint32_t t0 = tq + static_cast<uint32_t>(tb * 2 * NMAX);
                const uint32_t t1 = t0 + static_cast<uint32_t>(NMAX);
                const bool go = __shfl_sync(0xffffffffu, tl->abort_flag, 0) == 0;
                const bool ok = __all_sync(0xffffffffu, go && mbar_wait_bounded(&tl->tfull[tb], tuse & 1));
                if (!ok) {
                    if (lane == 0) {
                        tl->abort_flag = 1;
                        report_error(status, DEV_ERR_TIMEOUT);
                    }
                    return false;
                }
                tc_fence_after();
                // this lane's rows: phase 0 row ra of gate/up; phase 1 rows ra and ra + 128 of down
                const int ra = mb * g.rpi + 32 * q + lane;
                const int rb = ph == 0 ? ra : ra + kMxBM;
                const bool slice_a = mb * g.rpi + 32 * q < R;     // whole warp: R % 32 == 0
                const bool slice_b = ph == 0 ? slice_a : (mb * g.rpi + kMxBM + 32 * q < R);
                float bg = 0.0f, bu = 0.0f;
                if (ph == 0) {
                    const size_t bi = static_cast<size_t>(e) * R + (slice_a ? ra : 0);
                    if (a.b0) bg = __bfloat162float(__ushort_as_bfloat16(a.b0[bi]));
                    if (a.b1) bu = __bfloat162float(__ushort_as_bfloat16(a.b1[bi]));
                } else if (a.b0) {
                    if (slice_a) bg = __bfloat162float(__ushort_as_bfloat16(a.b0[static_cast<size_t>(e) * R + ra]));
                    if (slice_b) bu = __bfloat162float(__ushort_as_bfloat16(a.b0[static_cast<size_t>(e) * R + rb]));
                }
                // phase 0 finish of one route column: bias, activation, bf16 h, split for phase 2
                auto finish0 = [&](int n, float gv, float uv) {
                    const int p = q0 + n;
                    if (!slice_a) {
                        // rows past the matrix: the block's scale must still be a finite e8m0
                        if (lane == 0) a.hsf[(static_cast<size_t>(ra >> 7) * Tk + p) * 4 + ((ra >> 5) & 3)] = 127;
                        return;
                    }
                    const float h = act_fn(a.act, gv + bg, uv + bu, a.limit, a.alpha);
                    const float hb = __bfloat162float(__float2bfloat16_rn(h));
                    const int se = mx_scale_exp(warp_max(fabsf(hb)));
                    const float inv = __uint_as_float(static_cast<uint32_t>(127 - se) << 23);
                    // pair lanes (l, l ^ 1) so each conversion handles two values
                    const float other = __shfl_xor_sync(0xffffffffu, hb, 1);
                    uint32_t c1, c2;
                    mx_split2(__fmul_rn((lane & 1) ? other : hb, inv), __fmul_rn((lane & 1) ? hb : other, inv), c1, c2);
                    const uint32_t b1 = (lane & 1) ? (c1 >> 8) & 0xFFu : c1 & 0xFFu;
                    const uint32_t b2 = (lane & 1) ? (c2 >> 8) & 0xFFu : c2 & 0xFFu;
                    a.hq[static_cast<size_t>(p) * R + ra] = static_cast<uint8_t>(b1);
                    a.hq[(static_cast<size_t>(Tk) + p) * R + ra] = static_cast<uint8_t>(b2);
                    if (lane == 0)
                        a.hsf[(static_cast<size_t>(ra >> 7) * Tk + p) * 4 + ((ra >> 5) & 3)] = static_cast<uint8_t>(se + 127);
                };
                auto finish1 = [&](int n, float x0, float x1) {
                    const size_t r = static_cast<size_t>(a.perm[q0 + n]);
                    if (slice_a) a.e_out[r * R + ra] = x0 + bg;
                    if (slice_b) a.e_out[r * R + rb] = x1 + bu;
                };
                // this warp's slice of h for (expert, tile) is written: count it (release; the
                // readers copy h with the tensor-memory engine, hence the proxy fence)
                auto h_written = [&]() {
                    if (ph != 0 || !P.hrdy) return;
                    __syncwarp();
                    if (lane == 0) {
                        __threadfence();
                        asm volatile("fence.proxy.async.global;" ::: "memory");
                        asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(P.hrdy + tl->tbase[j] + tile)
                                     : "memory");
                    }
                };
                if (S == 1) {
                    for (int c0 = 8 * hw; c0 < nv; c0 += 8 * nh) {
                        float d0[8], d0b[8], d1[8], d1b[8];
                        tmem_ld8x4(t0 + c0, t0 + tw + c0, t1 + c0, t1 + tw + c0, d0, d0b, d1, d1b);
#pragma unroll
                        for (int t = 0; t < 8; ++t) {
                            const int n = c0 + t;
                            if (n >= nv) break;
                            const float x0 = d0[t] + d0b[t], x1 = d1[t] + d1b[t];
                            if (ph == 0) finish0(n, x0, x1);
                            else finish1(n, x0, x1);
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&tl->tempty[tb]);
                    h_written();
                    return true;
                }
                // split K: park this part's sums, the group's last part finishes
                float* part = a.part;
                for (int c0 = 8 * hw; c0 < nv; c0 += 8 * nh) {
                    float d0[8], d0b[8], d1[8], d1b[8];
                    tmem_ld8x4(t0 + c0, t0 + tw + c0, t1 + c0, t1 + tw + c0, d0, d0b, d1, d1b);
#pragma unroll
                    for (int t = 0; t < 8; ++t) {
                        const int n = c0 + t;
                        if (n >= nv) break;
                        const size_t pr = (static_cast<size_t>(kp) * Tk + q0 + n) * 2;
                        if (slice_a) part[pr * R + ra] = d0[t] + d0b[t];
                        if (slice_b) part[(pr + 1) * R + rb] = d1[t] + d1b[t];
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tl->tempty[tb]);
                __threadfence();
                __syncwarp();
                int last = 0;
                if (lane == 0) {
                    const int slot = (i / S) * 4 + q;
                    const int prev = atomicAdd(a.cnt + slot, 1);
                    last = (prev + 1 == S * nh);            // every part's warps of the quarter
                    if (last) a.cnt[slot] = 0;               // ready for the next call
                }
                if (__shfl_sync(0xffffffffu, last, 0) == 0) return true;
                __threadfence();
                for (int n = 0; n < nv; ++n) {
                    float x0 = 0.0f, x1 = 0.0f;        // parts summed in K order
                    for (int kk = 0; kk < S; ++kk) {
                        const size_t pr = (static_cast<size_t>(kk) * Tk + q0 + n) * 2;
                        if (slice_a) x0 += __ldcg(part + pr * R + ra);
                        if (slice_b) x1 += __ldcg(part + (pr + 1) * R + rb);
                    }
                    if (ph == 0) finish0(n, x0, x1);
                    else finish1(n, x0, x1);
                }
                h_written();
            }
            return true;
        };
        for (int n = 0; !stop; ++n) {
            const int gi = read_item_warp(n);
            if (gi >= total) break;
            int ph, i;
            item_of(gi, ph, i);
            if (P0 == 0 && ph == 0) stop = !epi_item(PhaseTag<0>{}, i);
            else if (P1 == 2) stop = !epi_item(PhaseTag<1>{}, i);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
}

// Route-ordered bf16 rows split into two e4m3 planes and e8m0 block scales (see the file
// header): a thread converts 8 consecutive elements, four threads form a 32-block.  The scales
// are stored transposed, [group of 4 blocks][row] words, so that the words one stage of the
// GEMM needs (one group, a tile's rows) are contiguous.
__global__ void __launch_bounds__(128) mx_split_rows_kernel(const uint16_t* __restrict__ x,
                                                            const int32_t* __restrict__ perm, int k,
                                                            int K, int n, uint8_t* __restrict__ q,
                                                            uint8_t* __restrict__ sf, int* zero, int nzero) {
    pdl_wait();
    pdl_launch_dependents();
    // the counters the GEMM launch after this one counts with start at zero
    if (blockIdx.x == 0)
        for (int i = threadIdx.x; i < nzero; i += blockDim.x) zero[i] = 0;
    const int p = blockIdx.x;
    if (p >= n) return;
    const int row = perm ? perm[p] / k : p;
    const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(row) * K);
    const int nwords = mx_sf_row(K) / 4;      // scale words per row (4 blocks each)
    uint8_t* q1 = q + static_cast<size_t>(p) * K;
    uint8_t* q2 = q + (static_cast<size_t>(n) + p) * K;
    const int nv = K / 8;
    for (int i0 = 0; i0 < nv; i0 += 128) {
        const int i = i0 + threadIdx.x;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (i < nv) v = __ldg(src + i);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        float f[8];
        float mx = 0.0f;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            f[2 * h] = __bfloat162float(__ushort_as_bfloat16(static_cast<uint16_t>(w[h] & 0xFFFF)));
            f[2 * h + 1] = __bfloat162float(__ushort_as_bfloat16(static_cast<uint16_t>(w[h] >> 16)));
            mx = fmaxf(mx, fmaxf(fabsf(f[2 * h]), fabsf(f[2 * h + 1])));
        }
        // the four threads of a 32-block are lanes 4m..4m+3 (i0 is a multiple of 128)
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        if (i >= nv) continue;
        const int se = mx_scale_exp(mx);
        const float inv = __uint_as_float(static_cast<uint32_t>(127 - se) << 23);
        uint32_t o1[2] = {0u, 0u}, o2[2] = {0u, 0u};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            uint32_t a1, a2;
            mx_split2(__fmul_rn(f[2 * h], inv), __fmul_rn(f[2 * h + 1], inv), a1, a2);
            o1[h >> 1] |= (a1 & 0xFFFFu) << (16 * (h & 1));
            o2[h >> 1] |= (a2 & 0xFFFFu) << (16 * (h & 1));
        }
        *reinterpret_cast<uint2*>(q1 + 8 * i) = make_uint2(o1[0], o1[1]);
        *reinterpret_cast<uint2*>(q2 + 8 * i) = make_uint2(o2[0], o2[1]);
        if ((threadIdx.x & 3) == 0)
            sf[(static_cast<size_t>(i >> 4) * n + p) * 4 + ((i >> 2) & 3)] = static_cast<uint8_t>(se + 127);
    }
    // blocks past K in the last group of four: a finite scale over zero data
    for (int b = K / 32 + threadIdx.x; b < 4 * nwords; b += 128)
        sf[(static_cast<size_t>(b >> 2) * n + p) * 4 + (b & 3)] = 127;
}

// Canonical MXFP4 codes [nmat][R][K/2] + e8m0 scales [nmat][R][K/32] of one matrix (G = 1) or
// of gate and up (G = 2) -> the tensor-core blob (mx_blob_bytes, layout in internal.h).
__global__ void mx_pack_kernel(int G, int nmat, int R, int K, const uint8_t* __restrict__ codes0,
                               const uint8_t* __restrict__ scales0, const uint8_t* __restrict__ codes1,
                               const uint8_t* __restrict__ scales1, uint8_t* __restrict__ out) {
    const int KG = mx_kg(K), U = mx_units(G, R), nblk = K / 32;
    const size_t codes_total = mx_codes_bytes(G, nmat, R, K);
    const size_t sf0 = mx_sf_offset(G, nmat, R, K);
    const size_t total = mx_blob_bytes(G, nmat, R, K);
    for (size_t o = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; o < total;
         o += static_cast<size_t>(gridDim.x) * blockDim.x) {
        uint8_t v = 0;
        if (o < codes_total) {
            // ((e KG + kg) G + g) R + r, then 64 bytes of codes
            const int c = static_cast<int>(o % 64);
            size_t q = o / 64;
            const int r = static_cast<int>(q % R);
            q /= R;
            const int g = static_cast<int>(q % G);
            q /= G;
            const int kg = static_cast<int>(q % KG);
            const size_t e = q / KG;
            const int cb = kg * 64 + c;                     // byte of the canonical row
            const uint8_t* src = g == 0 ? codes0 : codes1;
            if (cb < K / 2) v = src[(e * R + r) * (K / 2) + cb];
        } else if (o >= sf0) {
            // atom ((e U + u) KG + kg) 2 + m: row r0 + 32 w of its 128 rows, block kb
            const size_t qo = o - sf0;
            const int b = static_cast<int>(qo % kMxAtom);
            size_t q = qo / kMxAtom;
            const int m = static_cast<int>(q % 2);
            q /= 2;
            const int kg = static_cast<int>(q % KG);
            q /= KG;
            const int u = static_cast<int>(q % U);
            const size_t e = q / U;
            const int rr = 32 * ((b % 16) / 4) + b / 16;
            const int row = G == 2 ? u * 128 + rr : u * 256 + m * 128 + rr;
            const int blk = kg * 4 + (b % 4);
            const uint8_t* sc = (G == 2 && m == 1) ? scales1 : scales0;
            v = (row < R && blk < nblk) ? sc[(e * R + row) * nblk + blk] : 127;
        }
        out[o] = v;
    }
}

// 4-bit tensor map of a blob's codes: G = 2 {128, R, 2, KG, E} with box {128, 128, 2, 1, 1}
// (gate and up of 128 rows and one k group: 16 KB of codes), G = 1 {128, R, KG, E} with box
// {128, 256, 1, 1} (256 rows of one k group).  Rows past R come back as zero codes.
inline bool make_map_mx_codes(CUtensorMap* m, const void* blob, int G, int K, int R, int E) {
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

inline bool make_map_mx_act(CUtensorMap* m, const void* q, int K, int rows, int box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows), 2};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(K) * rows};
    const cuuint32_t box[3] = {128, static_cast<cuuint32_t>(box_rows), 2};
    const cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(q), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

static MxLayout mx_layout(int Tk, size_t* smem) {
    MxLayout L{};
    L.nb = kMxNbMax;
    L.nsets = 2;
    // few routes: narrower tiles (less B traffic per stage, deeper ring)
    if (Tk <= 64) L.nb = 16;
    L.sf_col0 = (4 * L.nsets * L.nb + 15) / 16 * 16;
    L.b_off = 2 * kMxAbox;
    const int bbytes = (2 * L.nb * 128 + 1023) / 1024 * 1024;
    L.sfa_off = L.b_off + bbytes;
    L.slot_bytes = (L.sfa_off + 2 * kMxAtom + 1023) / 1024 * 1024;
    constexpr size_t kTail = (sizeof(MxTail) + 255) / 256 * 256;
    const size_t budget = 227 * 1024 - 1024 - kTail - kMxMaxSlots * kMxAtom;
    L.nslot = static_cast<int>(budget / L.slot_bytes);
    if (L.nslot > kMxMaxSlots) L.nslot = kMxMaxSlots;
    if (L.nslot > (512 - L.sf_col0) / 16) L.nslot = (512 - L.sf_col0) / 16;   // TMEM scale slots
    L.S[0] = L.S[1] = 1;
    *smem = 1024 + static_cast<size_t>(L.nslot) * L.slot_bytes + kMxMaxSlots * kMxAtom + kTail;
    return L;
}

// K parts of one phase: enough (expert, row block) tiles x parts for every SM when partials fit
static int mx_split(const MxArgs& a, int num_sms) {
    if (a.max_split <= 1) return 1;
    const int Tk = a.rows_in;
    const int rows_per_item = a.phase == 0 ? kMxBM : 2 * kMxBM;
    const int MB = (a.R + rows_per_item - 1) / rows_per_item;
    const int nkb = mx_kg(a.K);
    const int e_eff = a.E < Tk ? a.E : Tk;
    const long long tiles = static_cast<long long>(e_eff) * MB;
    int S = static_cast<int>((4LL * num_sms + tiles - 1) / tiles);
    if (S > a.max_split) S = a.max_split;
    if (S > nkb / 2) S = nkb / 2;
    if (S < 1) S = 1;
    // parts of ceil(nkb / S) stages; no part may be left without a stage
    const int kbp = (nkb + S - 1) / S;
    return (nkb + kbp - 1) / kbp;
}

// the maps of phase ph (codes of its blob, planes of its activations)
static bool mx_maps(MxParams& P, int ph) {
    const MxArgs& a = P.a[ph];
    if (!make_map_mx_codes(&P.tmA[ph], a.w, ph == 0 ? 2 : 1, a.K, a.R, a.E)) return false;
    for (int q = 0; q < P.ly.nb / 8; ++q)
        if (!make_map_mx_act(&P.tmB[ph][q], a.bq, a.K, a.rows_in, 8 * (q + 1))) return false;
    return true;
}

cudaError_t launch_mx_gemm(const MxArgs& a, int num_sms, cudaStream_t s) {
    if (a.phase != 0 && a.phase != 1) return cudaErrorInvalidValue;
    MxParams P;
    memset(&P, 0, sizeof(P));
    P.a[a.phase] = a;
    P.p0 = a.phase;
    P.p1 = a.phase + 1;
    size_t smem = 0;
    P.ly = mx_layout(a.rows_in, &smem);
    if (P.ly.nslot < 2) return cudaErrorInvalidValue;
    P.ly.S[a.phase] = mx_split(a, num_sms);
    if (!mx_maps(P, a.phase)) return cudaErrorInvalidValue;
    if (a.phase == 0) {
        cudaError_t e = ensure_smem(tc_mx_kernel<0, 1>, smem);
        if (e != cudaSuccess) return e;
        return launch_pdl(tc_mx_kernel<0, 1>, dim3(num_sms), dim3(kMxThreads), smem, s, P);
    }
    cudaError_t e = ensure_smem(tc_mx_kernel<1, 2>, smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(tc_mx_kernel<1, 2>, dim3(num_sms), dim3(kMxThreads), smem, s, P);
}

cudaError_t launch_mx_fused(const MxArgs& a0, const MxArgs& a1, int* hrdy, int num_sms, cudaStream_t s) {
    if (a0.phase != 0 || a1.phase != 1 || !hrdy || a0.max_split > 1 || a1.max_split > 1)
        return cudaErrorInvalidValue;
    MxParams P;
    memset(&P, 0, sizeof(P));
    P.a[0] = a0;
    P.a[1] = a1;
    P.p0 = 0;
    P.p1 = 2;
    P.hrdy = hrdy;
    P.work = hrdy + a0.rows_in;
    size_t smem = 0;
    P.ly = mx_layout(a0.rows_in, &smem);
    if (P.ly.nslot < 2) return cudaErrorInvalidValue;
    if (!mx_maps(P, 0) || !mx_maps(P, 1)) return cudaErrorInvalidValue;
    cudaError_t e = ensure_smem(tc_mx_kernel<0, 2>, smem);
    if (e != cudaSuccess) return e;
    // phase-1 items wait for phase-0 items of other CTAs: every CTA must be resident
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, tc_mx_kernel<0, 2>, kMxThreads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_sms);
    cfg.blockDim = dim3(kMxThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeCooperative;
    at[0].val.cooperative = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, tc_mx_kernel<0, 2>, P);
}

cudaError_t launch_mx_split_rows(const uint16_t* x, const int32_t* perm, int k, int K, int n,
                                 uint8_t* q, uint8_t* sf, int* zero, int nzero, cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    return launch_pdl(mx_split_rows_kernel, dim3(n), dim3(128), 0, s, x, perm, k, K, n, q, sf, zero, nzero);
}

cudaError_t launch_mx_pack(int G, int nmat, int R, int K, const uint8_t* codes0, const uint8_t* scales0,
                           const uint8_t* codes1, const uint8_t* scales1, uint8_t* blob, cudaStream_t s) {
    const size_t total = mx_blob_bytes(G, nmat, R, K);
    if (total == 0) return cudaSuccess;
    size_t blocks = (total + 255) / 256;
    if (blocks > 65535u * 16u) blocks = 65535u * 16u;
    mx_pack_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(G, nmat, R, K, codes0, scales0, codes1,
                                                                  scales1, blob);
    return cudaGetLastError();
}

}  // namespace tsmoe

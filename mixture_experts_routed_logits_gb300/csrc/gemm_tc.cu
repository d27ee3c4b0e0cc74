// gemm_tc.cu -- steps 4-5 of the routed-expert layer for many tokens (prefill): the per-expert
// gated FFN as a grouped GEMM on the 5th-generation tensor cores (tcgen05, accumulators in
// TMEM, operands staged by TMA).
//
// Source pages (docs.rs, turbospark-runtime 0.3.0):
//   Gemma-4 batched routed prefill (src/families/gemma4/moe_batch.rs): one route list for the
//     whole micro-batch, encode_moe_prefill_phase1 (gate/up + activation for every route) and
//     encode_moe_prefill_phase2_fused (down projection + combine), "bit-exact against M
//     sequential decode-pair calls".
//   gpt-oss routed-expert pass (src/families/gptoss/moe.rs): clamped SwiGLU and per-expert
//     biases inside the expert kernels.
//
// Design (GB300, one CTA per SM, persistent):
//   * Work item = (expert, block of weight rows, tile of <= 256 routes of that expert).  The
//     routes of an expert are contiguous in the expert-sorted route list, so the activation
//     tile is a plain 2-D TMA box of the sorted activations.
//   * Swap-AB: the weights are the MMA's M side (128 rows per accumulator), the routes its N
//     side (16..256, a multiple of 16, sized to the tile's real route count), so small experts
//     waste no tensor time on padding.
//   * Phase 1: two accumulators per item, gate and up of the same 128 rows, 2 x N TMEM columns;
//     epilogue adds the biases, applies the activation, rounds h to 16 bits and stores it in
//     route-list order.  Phase 2: two accumulators cover 256 rows of the down projection;
//     epilogue adds the bias and stores f32 expert outputs by route id for the combine.
//   * Warp roles: warp 0 = TMA producer (3-stage ring of 64 KB), warp 1 = MMA issuer (one
//     thread, tcgen05.mma kind::f16, 128B-swizzled K-major smem descriptors), the rest =
//     epilogue (tcgen05.ld of their TMEM lane quarter, warp w taking quarter w % 4): warps 2-25
//     for 16-bit weights, 2-5 for MXFP4.  Every mbarrier wait is bounded.
//   * MXFP4 weights (QUANT variant): the producer bulk-copies the packed e2m1 tiles (with their
//     e8m0 block scales) into a staging area of each stage; sixteen dequant warps turn them
//     into f16 (hardware e2m1x2 -> f16x2 convert, times the block scale, exact while the scale
//     is in [2^-23, 2^13]; outside it the device status reports TS_ERR_UNSUPPORTED) written
//     straight into the 128B-swizzled A tile (two A stages); the MMA waits on a
//     "dequantised" barrier instead of the copy barrier.  Activations enter as f16 with a
//     per-route power-of-two prescale that the epilogue undoes.  Each weight element crosses HBM
//     once per route tile, as packed bytes.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "tc_common.cuh"

namespace tsmoe {

namespace {

constexpr int kBM = 128;                         // weight rows per accumulator
constexpr int kBN = 256;                         // max routes per tile
constexpr int kBK = 64;                          // K elements per stage (128 bytes of 16-bit)
constexpr int kATile = kBM * kBK * 2;            // 16 KB
constexpr int kBBox = 64 * kBK * 2;              // 8 KB: one 64-row TMA box of activations
constexpr int kThreads = 192;
// 16-bit weights: 24 epilogue warps (six per TMEM lane quarter, 16-column chunks dealt in
// turn) drain the single accumulator set of a 256-route tile while the tensor pipe waits for
// it (the activation and the stores of 64K h values per gate/up item); measured on the
// Mixtral prefill chunk, gate/up launch: 4 warps 937 us, 8 782, 16 712, 24 685
constexpr int kEpiWarps16 = 24;
constexpr int kThreads16 = (2 + kEpiWarps16) * 32;
// QUANT variant: a packed slot holds the B boxes and two 8-row-tile x 2-block packed tiles
constexpr int kPackBlk = 272;
constexpr int kStaging = 2 * 8 * 2 * kPackBlk;             // 8704 B
constexpr int kDqWarps = 16;                                // dequant warps (8 or 16)
constexpr int kThreadsQ = kThreads + 32 * kDqWarps;
static_assert(kDqWarps == 8 || kDqWarps == 16, "the dequant split covers 32 blocks per stage");

struct TcLayout {        // host-chosen shape of one launch
    int bn;              // routes per tile (64, 128 or 256; <= 128 double-buffers TMEM)
    int nslot;           // stages (16-bit weights) or packed slots (MXFP4)
    int slot_bytes;      // bytes per stage / slot (multiple of 1024)
    int a_ring_bytes;    // MXFP4: two dequantised A stages (64 KB); else 0
    int S;               // K split into S parts (partials reduced by the group's last CTA)
};

struct TcParams {
    CUtensorMap tmA0;     // phase 1: gate [E][I][H]; phase 2: down [E][H][I]
    CUtensorMap tmA1;     // phase 1: up; phase 2: unused (down again)
    CUtensorMap tmB;      // sorted activations [Tk][K]
    GemmArgs a;
    TcLayout ly;
};

constexpr int kMaxSlots = 8;

struct SmemTail {
    uint64_t full[kMaxSlots];       // stage / packed slot loaded
    uint64_t empty[kMaxSlots];      // stage / packed slot consumed by the MMA
    uint64_t afull[2];              // QUANT: dequantised A stage written
    uint64_t aempty[2];             // QUANT: dequantised A stage consumed by the MMA
    uint64_t tfull[2];              // accumulator set b holds a finished item
    uint64_t tempty[2];             // accumulator set b read out by the epilogue
    uint32_t tmem_base;
    volatile int abort_flag;
    int nt;                         // touched experts
    int touched[kMaxExperts];
    int cnt[kMaxExperts];
    int bnj[kMaxExperts];           // routes per tile of each touched expert (<= bn)
    int ioff[kMaxExperts + 1];      // item prefix per touched expert
};

template <bool QUANT>
__global__ void __launch_bounds__(QUANT ? kThreadsQ : kThreads16, 1)
tc_gemm_kernel(const __grid_constant__ TcParams P) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const TcLayout& Ly = P.ly;
    unsigned char* base = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    unsigned char* ring = base + Ly.a_ring_bytes;           // stages (16-bit) / packed slots
    SmemTail* tl = reinterpret_cast<SmemTail*>(ring + static_cast<size_t>(Ly.nslot) * Ly.slot_bytes);
    const GemmArgs& a = P.a;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_wait();                 // inputs of this launch may come from the previous kernel
    pdl_launch_dependents();
    const int R = a.R, K = a.K;
    const int rows_per_item = a.phase == 0 ? kBM : 2 * kBM;
    const int MB = (R + rows_per_item - 1) / rows_per_item;
    const int nkb = K / kBK;
    const int NS = Ly.nslot, BN = Ly.bn, S = Ly.S;
    // Accumulator sets in the 512 TMEM columns: tiles of <= 128 routes use two sets of (gate,
    // up) or (rows, rows + 128) at columns 0 / 128 and 256 / 384, alternating per item, so the
    // MMAs of an item run while the epilogue drains the one before; wider tiles use one set at
    // columns 0 and 256.
    const int NB = BN <= 128 ? 2 : 1;
    const uint32_t acc1 = NB == 2 ? 128u : 256u;      // column of the second accumulator
    const int kbp = (nkb + S - 1) / S;                      // stages per K part
    const int bbytes = (BN / 64) * kBBox;                   // B area of a stage / slot

    if (threadIdx.x == 0) {
        int nt = 0, acc = 0;
        for (int e = 0; e < a.E; ++e) {
            const int n = a.off[e + 1] - a.off[e];
            if (n > 0) {
                // the expert's routes in equal tiles (multiples of 16), not full tiles + a tail
                const int ntl0 = (n + BN - 1) / BN;
                const int bnj = min(BN, ((n + ntl0 - 1) / ntl0 + 15) & ~15);
                tl->touched[nt] = e;
                tl->cnt[nt] = n;
                tl->bnj[nt] = bnj;
                tl->ioff[nt] = acc;
                acc += MB * ((n + bnj - 1) / bnj) * S;
                ++nt;
            }
        }
        tl->ioff[nt] = acc;
        tl->nt = nt;
        tl->abort_flag = 0;
        for (int s = 0; s < NS; ++s) {
            mbar_init(&tl->full[s], 1);
            mbar_init(&tl->empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&tl->afull[s], kDqWarps);
            mbar_init(&tl->aempty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tl->tfull[b], 1);
            mbar_init(&tl->tempty[b], QUANT ? 4 : kEpiWarps16);
        }
        fence_mbar_init();
    }
    if (warp == 1) {
        // 512 TMEM columns: one or two accumulator sets (see NB above)
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
    const int items = tl->ioff[nt];

    // item i -> touched expert j, row block mb, route tile, K part kp (kp fastest: the S parts
    // of one output tile are consecutive items, group = i / S)
    auto decode = [&](int i, int& j, int& mb, int& tile, int& kp) {
        j = 0;
        while (j + 1 < nt && i >= tl->ioff[j + 1]) ++j;
        const int ntl = (tl->cnt[j] + tl->bnj[j] - 1) / tl->bnj[j];
        const int local = i - tl->ioff[j];
        kp = local % S;
        const int rest = local / S;
        tile = rest % ntl;
        mb = rest / ntl;
    };

    if (warp == 0) {
        if (lane == 0) {
            // =============================== TMA producer ====================================
            int it = 0;
            for (int i = blockIdx.x; i < items && !tl->abort_flag; i += gridDim.x) {
                int j, mb, tile, kp;
                decode(i, j, mb, tile, kp);
                const int e = tl->touched[j];
                const int p0 = a.off[e] + tile * tl->bnj[j];
                const int n_valid = min(tl->bnj[j], tl->cnt[j] - tile * tl->bnj[j]);
                const int nbox = (n_valid + 63) / 64;
                const int r0 = mb * rows_per_item;
                const int r1 = a.phase == 0 ? r0 : r0 + kBM;
                const int kb0 = kp * kbp, kb1 = min(nkb, kb0 + kbp);
                const uint32_t bytes = (QUANT ? 2 * 8 * 2 * kPackBlk : 2 * kATile) + nbox * kBBox;
                for (int kb = kb0; kb < kb1; ++kb, ++it) {
                    const int s = it % NS;
                    if (!mbar_wait_bounded(&tl->empty[s], ((it / NS) & 1) ^ 1)) {
                        tl->abort_flag = 1;
                        report_error(a.status, DEV_ERR_TIMEOUT);
                        break;
                    }
                    unsigned char* st = ring + static_cast<size_t>(s) * Ly.slot_bytes;
                    mbar_arrive_expect_tx(&tl->full[s], bytes);
                    unsigned char* bdst;
                    if (QUANT) {
                        // slot = [B boxes | packed A0 (8 row tiles x 2 blocks) | packed A1];
                        // row tiles past the matrix come back zero-filled
                        unsigned char* stg = st + bbytes;
                        tma_load_3d(stg, &P.tmA0, 2 * kb * (kPackBlk / 4), r0 / kRowTile, e, &tl->full[s]);
                        tma_load_3d(stg + 8 * 2 * kPackBlk, a.phase == 0 ? &P.tmA1 : &P.tmA0,
                                    2 * kb * (kPackBlk / 4), r1 / kRowTile, e, &tl->full[s]);
                        bdst = st;
                    } else {
                        tma_load_3d(st, &P.tmA0, kb * kBK, r0, e, &tl->full[s]);
                        tma_load_3d(st + kATile, a.phase == 0 ? &P.tmA1 : &P.tmA0, kb * kBK, r1, e,
                                    &tl->full[s]);
                        bdst = st + 2 * kATile;
                    }
                    for (int q = 0; q < nbox; ++q)
                        tma_load_2d(bdst + q * kBBox, &P.tmB, kb * kBK, p0 + 64 * q, &tl->full[s]);
                }
            }
            // drain: the last slots' copies must land before the CTA may exit
            for (int q = (it > NS ? it - NS : 0); q < it; ++q)
                mbar_wait_bounded(&tl->full[q % NS], (q / NS) & 1);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ================================= MMA issuer ====================================
            int it = 0, n_item = 0;
            for (int i = blockIdx.x; i < items && !tl->abort_flag; i += gridDim.x, ++n_item) {
                int j, mb, tile, kp;
                decode(i, j, mb, tile, kp);
                const int n_valid = min(tl->bnj[j], tl->cnt[j] - tile * tl->bnj[j]);
                const int N = (n_valid + 15) & ~15;
                const uint32_t idesc = idesc_f16kind(a.ab_bf16, kBM, N);
                const int kb0 = kp * kbp, kb1 = min(nkb, kb0 + kbp);
                const int tb = n_item % NB, tuse = n_item / NB;
                const uint32_t tset = tmem + static_cast<uint32_t>(tb) * 256u;
                if (!mbar_wait_bounded(&tl->tempty[tb], (tuse & 1) ^ 1)) {
                    tl->abort_flag = 1;
                    report_error(a.status, DEV_ERR_TIMEOUT);
                    break;
                }
                tc_fence_after();
                bool ok = true;
                for (int kb = kb0; kb < kb1; ++kb, ++it) {
                    const int s = it % NS, sa = it & 1;
                    const bool got = QUANT ? mbar_wait_bounded(&tl->afull[sa], (it >> 1) & 1)
                                           : mbar_wait_bounded(&tl->full[s], (it / NS) & 1);
                    if (!got) {
                        tl->abort_flag = 1;
                        report_error(a.status, DEV_ERR_TIMEOUT);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const unsigned char* st = ring + static_cast<size_t>(s) * Ly.slot_bytes;
                    const uint32_t sa0 = smem_u32(QUANT ? base + sa * 2 * kATile : st);
                    const uint64_t d0 = sdesc_sw128(sa0);
                    const uint64_t d1 = sdesc_sw128(sa0 + kATile);
                    const uint64_t db = sdesc_sw128(smem_u32(QUANT ? st : st + 2 * kATile));
#pragma unroll
                    for (int ks = 0; ks < kBK / 16; ++ks) {
                        const uint32_t acc = (kb > kb0 || ks > 0) ? 1u : 0u;
                        umma(tset, d0 + 2 * ks, db + 2 * ks, idesc, acc);
                        umma(tset + acc1, d1 + 2 * ks, db + 2 * ks, idesc, acc);
                    }
                    umma_commit(&tl->empty[s]);         // frees the slot once these MMAs are done
                    if (QUANT) umma_commit(&tl->aempty[sa]);
                }
                if (!ok) break;
                umma_commit(&tl->tfull[tb]);            // accumulators ready for the epilogue
            }
        }
    } else if (QUANT && warp >= 6) {
        // ======================= dequant warps (QUANT): packed e2m1 -> f16 A tiles =============
        const int dw = warp - 6;
        const int gid = lane >> 2, tid = lane & 3;
        const int bb = dw & 1;
        // rows gid (+8) of a row tile: (row & 7) == gid, so the swizzled chunk is fixed per lane
        const int sw_off = gid * 128 + (((4 * bb + tid) ^ gid) << 4);
        int it = 0;
        bool bad_scale = false;
        const int RTm = R / kRowTile;               // 16-row tiles that exist per matrix
        for (int i = blockIdx.x; i < items && !tl->abort_flag; i += gridDim.x) {
            int j, mb, tile_i, kp;
            decode(i, j, mb, tile_i, kp);
            const int rt0 = (mb * rows_per_item) / kRowTile;
            const int rt1 = a.phase == 0 ? rt0 : rt0 + kBM / kRowTile;
            const int kb0 = kp * kbp, kb1 = min(nkb, kb0 + kbp);
            for (int kb = kb0; kb < kb1; ++kb, ++it) {
                const int s = it % NS, sa = it & 1;
                if (!mbar_wait_bounded(&tl->full[s], (it / NS) & 1) ||
                    !mbar_wait_bounded(&tl->aempty[sa], ((it >> 1) & 1) ^ 1)) {
                    if (lane == 0) {
                        tl->abort_flag = 1;
                        report_error(a.status, DEV_ERR_TIMEOUT);
                    }
                    break;
                }
                const unsigned char* stg = ring + static_cast<size_t>(s) * Ly.slot_bytes + bbytes;
                unsigned char* adst = base + sa * 2 * kATile;
                // this warp: block column bb = dw & 1 of row tiles (dw >> 1) + (kDqWarps / 2) * g
                // (g < 16 / kDqWarps) of both tiles; the 128B swizzle puts 16-byte chunk c of row
                // r at c ^ (r & 7)
                constexpr int kPer = 32 / kDqWarps;       // blocks per warp and stage
#pragma unroll
                for (int qi = 0; qi < kPer; ++qi) {
                    const int tile = qi / (kPer / 2);
                    const int rt = (dw >> 1) + (kDqWarps / 2) * (qi % (kPer / 2));
                    // row tiles past the matrix only feed output rows that are never stored
                    if ((tile == 0 ? rt0 : rt1) + rt >= RTm) continue;
                    const unsigned char* blk = stg + (tile * 8 + rt) * 2 * kPackBlk + bb * kPackBlk;
                    const uint2 cw = *reinterpret_cast<const uint2*>(blk + lane * 8);
                    const uint32_t sc = *reinterpret_cast<const uint16_t*>(blk + 256 + gid * 2);
                    const uint32_t e0 = sc & 0xFF, e1 = sc >> 8;
                    uint32_t s0, s1;            // f16x2 scales
                    if (__all_sync(0xffffffffu, e0 >= 113u && e0 <= 140u && e1 >= 113u && e1 <= 140u)) {
                        // normal f16 powers of two: exponent field e - 112, both halves at once
                        s0 = (e0 - 112u) * 0x04000400u;
                        s1 = (e1 - 112u) * 0x04000400u;
                    } else {
                        // scaled e2m1 values are exact f16 numbers only for scales 2^-23 .. 2^13
                        bad_scale |= (e0 < 104u) | (e0 > 140u) | (e1 < 104u) | (e1 > 140u);
                        const __half2 h0 = __half2half2(__float2half_rn(e8m0_to_float(e0)));
                        const __half2 h1 = __half2half2(__float2half_rn(e8m0_to_float(e1)));
                        s0 = *reinterpret_cast<const uint32_t*>(&h0);
                        s1 = *reinterpret_cast<const uint32_t*>(&h1);
                    }
                    uint32_t ra[4], rb[4], va[4], vb[4];
                    e2m1x8_to_f16x2x4(cw.x, ra);
                    e2m1x8_to_f16x2x4(cw.y, rb);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        __half2 ha = __hmul2(*reinterpret_cast<__half2*>(&ra[q]), *reinterpret_cast<const __half2*>(&s0));
                        __half2 hb = __hmul2(*reinterpret_cast<__half2*>(&rb[q]), *reinterpret_cast<const __half2*>(&s1));
                        va[q] = *reinterpret_cast<uint32_t*>(&ha);
                        vb[q] = *reinterpret_cast<uint32_t*>(&hb);
                    }
                    unsigned char* at = adst + tile * kATile + rt * (kRowTile * 128) + sw_off;
                    *reinterpret_cast<uint4*>(at) = make_uint4(va[0], va[1], va[2], va[3]);
                    *reinterpret_cast<uint4*>(at + 8 * 128) = make_uint4(vb[0], vb[1], vb[2], vb[3]);
                }
                // generic-proxy stores must be visible to the tensor core's async-proxy reads
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(&tl->afull[sa]);
            }
        }
        if (__any_sync(0xffffffffu, bad_scale) && lane == 0) report_error(a.status, DEV_ERR_UNSUPPORTED);
    } else {
        // =================================== epilogue ==========================================
        const int q = warp & 3;                     // TMEM lane quarter this warp may access
        const uint32_t tq = tmem + (static_cast<uint32_t>(32 * q) << 16);
        // warps per lane quarter, and which of them this is: 16-column chunks alternate
        const int nh = QUANT ? 1 : kEpiWarps16 / 4;
        const int hw = QUANT ? 0 : (warp - 2) >> 2;
        const int Tk = a.rows_in;
        int n_item = 0;
        for (int i = blockIdx.x; i < items; i += gridDim.x, ++n_item) {
            int j, mb, tile, kp;
            decode(i, j, mb, tile, kp);
            const int e = tl->touched[j];
            const int p0 = a.off[e] + tile * tl->bnj[j];
            const int n_valid = min(tl->bnj[j], tl->cnt[j] - tile * tl->bnj[j]);
            const int N = (n_valid + 15) & ~15;
            const int tb = n_item % NB, tuse = n_item / NB;
            const uint32_t tqs = tq + static_cast<uint32_t>(tb) * 256u;   // this item's set
            bool ok = !tl->abort_flag && mbar_wait_bounded(&tl->tfull[tb], tuse & 1);
            if (!ok) {
                if (lane == 0) {
                    tl->abort_flag = 1;
                    report_error(a.status, DEV_ERR_TIMEOUT);
                }
                break;
            }
            tc_fence_after();
            // rows of this thread: phase 0 gate/up row `ra`; phase 1 rows ra and ra + 128
            const int ra = mb * rows_per_item + 32 * q + lane;
            const int rb = a.phase == 0 ? ra : ra + kBM;
            const bool va = ra < R, vb = rb < R;
            float bg = 0.0f, bu = 0.0f;                 // biases of rows ra / rb (phase 1: b0 only)
            if (a.phase == 0) {
                const size_t bi = static_cast<size_t>(e) * R + (va ? ra : 0);
                if (a.b0) bg = __bfloat162float(__ushort_as_bfloat16(a.b0[bi]));
                if (a.b1) bu = __bfloat162float(__ushort_as_bfloat16(a.b1[bi]));
            } else if (a.b0) {
                if (va) bg = __bfloat162float(__ushort_as_bfloat16(a.b0[static_cast<size_t>(e) * R + ra]));
                if (vb) bu = __bfloat162float(__ushort_as_bfloat16(a.b0[static_cast<size_t>(e) * R + rb]));
            }
            uint16_t* hout = static_cast<uint16_t*>(a.out);
            float* eout = static_cast<float*>(a.out);
            if (S == 1) {
                for (int c0 = 16 * hw; c0 < N; c0 += 16 * nh) {
                    float d0[16], d1[16];
                    tmem_ld16_pair(tqs + c0, tqs + acc1 + c0, d0, d1);
                    if (a.phase == 0) {
#pragma unroll
                        for (int t = 0; t < 16; ++t) {
                            const int c = c0 + t;
                            if (va && c < n_valid) {
                                float gv = d0[t], uv = d1[t];
                                if (QUANT) {
                                    const float inv = a.col_scale[p0 + c];
                                    gv *= inv;
                                    uv *= inv;
                                }
                                const float h = act_fn(a.act, gv + bg, uv + bu, a.limit, a.alpha);
                                const uint16_t hb = float_to_adt_bits(h, a.adt);
                                hout[static_cast<size_t>(p0 + c) * R + ra] = hb;
                            }
                        }
                    } else {
#pragma unroll
                        for (int t = 0; t < 16; ++t) {
                            const int c = c0 + t;
                            if (c < n_valid) {
                                const size_t r = static_cast<size_t>(a.perm[p0 + c]);
                                const float inv = QUANT ? a.col_scale[p0 + c] : 1.0f;
                                if (va) eout[r * R + ra] = d0[t] * inv + bg;
                                if (vb) eout[r * R + rb] = d1[t] * inv + bu;
                            }
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tl->tempty[tb]);
                continue;
            }
            // split K: park this part's accumulators, the group's last part finishes
            float* part = a.part;
            for (int c0 = 16 * hw; c0 < N; c0 += 16 * nh) {
                float d0[16], d1[16];
                tmem_ld16_pair(tqs + c0, tqs + acc1 + c0, d0, d1);
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    const int c = c0 + t;
                    if (c >= n_valid) continue;
                    const size_t pr = (static_cast<size_t>(kp) * Tk + p0 + c) * 2;
                    if (va) part[pr * R + ra] = d0[t];
                    if (a.phase == 0 ? va : vb) part[(pr + 1) * R + (a.phase == 0 ? ra : rb)] = d1[t];
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tl->tempty[tb]);   // this set is free again
            // the warps of a lane quarter own its 32-row slice: one counter per (group, slice),
            // counting every part's warps, so no barrier between the epilogue warps is needed;
            // the last to arrive sums every column of the slice
            __threadfence();
            __syncwarp();
            int last = 0;
            if (lane == 0) {
                const int slot = (i / S) * 4 + q;
                const int prev = atomicAdd(a.cnt + slot, 1);
                last = (prev + 1 == S * nh);
                if (last) a.cnt[slot] = 0;               // ready for the next call
            }
            if (__shfl_sync(0xffffffffu, last, 0) == 0) continue;
            __threadfence();
            const int r1 = a.phase == 0 ? ra : rb;
            const bool v1 = a.phase == 0 ? va : vb;
            for (int c = 0; c < n_valid; ++c) {
                // parts summed in K order
                float x0 = 0.0f, x1 = 0.0f;
                for (int kk = 0; kk < S; ++kk) {
                    const size_t pr = (static_cast<size_t>(kk) * Tk + p0 + c) * 2;
                    if (va) x0 += __ldcg(part + pr * R + ra);
                    if (v1) x1 += __ldcg(part + (pr + 1) * R + r1);
                }
                const float inv = QUANT ? a.col_scale[p0 + c] : 1.0f;
                if (a.phase == 0) {
                    if (va) {
                        const float h = act_fn(a.act, x0 * inv + bg, x1 * inv + bu, a.limit, a.alpha);
                        hout[static_cast<size_t>(p0 + c) * R + ra] = float_to_adt_bits(h, a.adt);
                    }
                } else {
                    const size_t r = static_cast<size_t>(a.perm[p0 + c]);
                    if (va) eout[r * R + ra] = x0 * inv + bg;
                    if (vb) eout[r * R + rb] = x1 * inv + bu;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
}

// x rows in route-list order: xs[p] = x[perm[p] / k]
__global__ void __launch_bounds__(128) gather_rows_kernel(const uint16_t* __restrict__ x,
                                                          const int32_t* __restrict__ perm,
                                                          int k, int H, int n,
                                                          uint16_t* __restrict__ xs) {
    pdl_wait();
    pdl_launch_dependents();
    const int p = blockIdx.x;
    if (p >= n) return;
    const int t = perm[p] / k;
    const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * H);
    uint4* dst = reinterpret_cast<uint4*>(xs + static_cast<size_t>(p) * H);
    for (int i = threadIdx.x; i < H / 8; i += blockDim.x) dst[i] = src[i];
}

// Power-of-two prescale for an f16 operand: 2^ks with max|v| * 2^ks in [2^14, 2^15).
__device__ __forceinline__ void prescale_of(float mx, float& scl, float& inv) {
    scl = inv = 1.0f;
    if (mx > 0.0f && mx < 3.0e38f) {
        int ex;
        frexpf(mx, &ex);
        int ks = max(-120, min(120, 15 - ex));
        scl = __uint_as_float(static_cast<uint32_t>(ks + 127) << 23);
        inv = __uint_as_float(static_cast<uint32_t>(127 - ks) << 23);
    }
}

__device__ __forceinline__ float block_max128(float v, float* red) {
    v = warp_max(v);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    const float m = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    __syncthreads();
    return m;
}

// One row of n 16-bit values (n % 8 == 0, both pointers 16-byte aligned) to f16 times 2^ks with
// max |v| * 2^ks in [2^14, 2^15) (prescale_of); returns 2^-ks.  A 128-thread block moves the row
// in 16-byte pieces; rows of up to 128 * 8 * kRowV elements are read once and kept in registers
// between the max and the conversion, longer rows are read twice.
constexpr int kRowV = 4;
__device__ __forceinline__ float row_to_f16(const uint16_t* __restrict__ src, uint16_t* __restrict__ dst,
                                            int n, int adt, float* red) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint4* d4 = reinterpret_cast<uint4*>(dst);
    const int nv = n / 8;
    auto absmax8 = [&](const uint4& v) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        float m = 0.0f;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            m = fmaxf(m, fabsf(adt_bits_to_float(static_cast<uint16_t>(w[h] & 0xFFFF), adt)));
            m = fmaxf(m, fabsf(adt_bits_to_float(static_cast<uint16_t>(w[h] >> 16), adt)));
        }
        return m;
    };
    auto conv8 = [&](const uint4& v, float scl) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const uint32_t lo = __half_as_ushort(__float2half_rn(
                __fmul_rn(adt_bits_to_float(static_cast<uint16_t>(w[h] & 0xFFFF), adt), scl)));
            const uint32_t hi = __half_as_ushort(__float2half_rn(
                __fmul_rn(adt_bits_to_float(static_cast<uint16_t>(w[h] >> 16), adt), scl)));
            o[h] = lo | (hi << 16);
        }
        return make_uint4(o[0], o[1], o[2], o[3]);
    };
    float mx = 0.0f, scl, inv;
    if (nv <= kRowV * 128) {
        uint4 v[kRowV];
#pragma unroll
        for (int q = 0; q < kRowV; ++q) {
            const int i = threadIdx.x + 128 * q;
            v[q] = i < nv ? __ldg(s4 + i) : make_uint4(0u, 0u, 0u, 0u);
            mx = fmaxf(mx, absmax8(v[q]));
        }
        mx = block_max128(mx, red);
        prescale_of(mx, scl, inv);
#pragma unroll
        for (int q = 0; q < kRowV; ++q) {
            const int i = threadIdx.x + 128 * q;
            if (i < nv) d4[i] = conv8(v[q], scl);
        }
    } else {
        for (int i = threadIdx.x; i < nv; i += 128) mx = fmaxf(mx, absmax8(__ldg(s4 + i)));
        mx = block_max128(mx, red);
        prescale_of(mx, scl, inv);
        for (int i = threadIdx.x; i < nv; i += 128) d4[i] = conv8(__ldg(s4 + i), scl);
    }
    return inv;
}

// Route-ordered activations for the f16 tensor-core operand: xs[p] = f16(x[perm[p]/k] * 2^ks),
// inv[p] = 2^-ks.
__global__ void __launch_bounds__(128) gather_rows_f16_kernel(const uint16_t* __restrict__ x, int adt,
                                                              const int32_t* __restrict__ perm, int k,
                                                              int H, int n, uint16_t* __restrict__ xs,
                                                              float* __restrict__ inv_out) {
    __shared__ float red[4];
    pdl_wait();
    pdl_launch_dependents();
    const int p = blockIdx.x;
    if (p >= n) return;
    const float inv = row_to_f16(x + static_cast<size_t>(perm[p] / k) * H, xs + static_cast<size_t>(p) * H,
                                 H, adt, red);
    if (threadIdx.x == 0) inv_out[p] = inv;
}

// h (16-bit, route order) -> f16 with a per-route power-of-two prescale from max |h| of the row.
__global__ void __launch_bounds__(128) h_to_f16_kernel(const uint16_t* __restrict__ h, int adt, int I,
                                                       int n, uint16_t* __restrict__ h16,
                                                       float* __restrict__ inv_out) {
    __shared__ float red[4];
    pdl_wait();
    pdl_launch_dependents();
    const int p = blockIdx.x;
    if (p >= n) return;
    const float inv = row_to_f16(h + static_cast<size_t>(p) * I, h16 + static_cast<size_t>(p) * I, I, adt, red);
    if (threadIdx.x == 0) inv_out[p] = inv;
}

}  // namespace

cudaError_t launch_gather_rows(const uint16_t* x, const int32_t* perm, int k, int H, int n,
                               uint16_t* xs, cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    return launch_pdl(gather_rows_kernel, dim3(n), dim3(128), 0, s, x, perm, k, H, n, xs);
}

cudaError_t launch_gather_rows_f16(const uint16_t* x, int adt, const int32_t* perm, int k, int H,
                                   int n, uint16_t* xs, float* inv, cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    return launch_pdl(gather_rows_f16_kernel, dim3(n), dim3(128), 0, s, x, adt, perm, k, H, n, xs, inv);
}

cudaError_t launch_h_to_f16(const uint16_t* h, int adt, int I, int n, uint16_t* h16, float* inv,
                            cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    return launch_pdl(h_to_f16_kernel, dim3(n), dim3(128), 0, s, h, adt, I, n, h16, inv);
}

// Launch shape: routes per tile, ring depth and K split.  Decode-sized calls (few routes) use
// 64-route tiles, a deep ring and, when the workspace has room for partials, split K so that the
// few (expert, row block) tiles still spread over every SM.
static TcLayout tc_layout(const GemmArgs& a, int num_sms, size_t* smem) {
    TcLayout L{};
    const int Tk = a.rows_in;
    // MXFP4 calls take 128-route tiles: the epilogue of one item then overlaps the next item's
    // MMAs (two accumulator sets), which outweighs re-dequantising the weights of experts with
    // more than 128 routes
    L.bn = Tk <= 256 ? 64 : (a.quant ? 128 : kBN);
    // shared-memory tail (barriers and the item tables) plus 1 KB for aligning the base to 1024
    constexpr size_t kTailBytes = (sizeof(SmemTail) + 255) / 256 * 256;
    const size_t tail = kTailBytes + 1024;
    const size_t budget = 227 * 1024;
    const int bbytes = (L.bn / 64) * kBBox;
    if (a.quant) {
        L.a_ring_bytes = 2 * 2 * kATile;
        L.slot_bytes = (bbytes + kStaging + 1023) / 1024 * 1024;
    } else {
        L.a_ring_bytes = 0;
        L.slot_bytes = 2 * kATile + bbytes;
    }
    L.nslot = static_cast<int>((budget - tail - L.a_ring_bytes) / L.slot_bytes);
    if (L.nslot > kMaxSlots) L.nslot = kMaxSlots;
    const int rows_per_item = a.phase == 0 ? kBM : 2 * kBM;
    const int MB = (a.R + rows_per_item - 1) / rows_per_item;
    const int nkb = a.K / kBK;
    L.S = 1;
    if (a.max_split > 1) {
        const int e_eff = a.E < Tk ? a.E : Tk;
        const long long tiles = static_cast<long long>(e_eff) * MB;
        int S = static_cast<int>((4LL * num_sms + tiles - 1) / tiles);
        if (S > a.max_split) S = a.max_split;
        if (S > nkb / 4) S = nkb / 4;
        if (S < 1) S = 1;
        // parts of ceil(nkb / S) stages; no part may be left without a stage
        const int kbp = (nkb + S - 1) / S;
        L.S = (nkb + kbp - 1) / kbp;
    }
    *smem = 1024 + L.a_ring_bytes + static_cast<size_t>(L.nslot) * L.slot_bytes + kTailBytes;
    return L;
}

cudaError_t launch_tc_gemm(const GemmArgs& a, int num_sms, cudaStream_t s) {
    TcParams P;
    memset(&P, 0, sizeof(P));
    P.a = a;
    const int KA = a.K;                 // reduction length
    const int Rm = a.R;                 // rows per expert matrix
    size_t smem = 0;
    P.ly = tc_layout(a, num_sms, &smem);
    if (P.ly.nslot < 2) return cudaErrorInvalidValue;
    if (!a.quant) {
        if (!make_map_3d(&P.tmA0, a.w0, a.ab_bf16, KA, Rm, a.E, kBK, kBM)) return cudaErrorInvalidValue;
        if (!make_map_3d(&P.tmA1, a.phase == 0 ? a.w1 : a.w0, a.ab_bf16, KA, Rm, a.E, kBK, kBM))
            return cudaErrorInvalidValue;
    } else {
        if (!make_map_packed(&P.tmA0, a.w0, KA, Rm, a.E, kPackBlk)) return cudaErrorInvalidValue;
        if (!make_map_packed(&P.tmA1, a.phase == 0 ? a.w1 : a.w0, KA, Rm, a.E, kPackBlk))
            return cudaErrorInvalidValue;
    }
    if (!make_map_2d(&P.tmB, a.act_in, a.ab_bf16, KA, a.rows_in, kBK, 64)) return cudaErrorInvalidValue;
    cudaError_t e;
    if (a.quant) {
        e = ensure_smem(tc_gemm_kernel<true>, smem);
        if (e != cudaSuccess) return e;
        return launch_pdl(tc_gemm_kernel<true>, dim3(num_sms), dim3(kThreadsQ), smem, s, P);
    } else {
        e = ensure_smem(tc_gemm_kernel<false>, smem);
        if (e != cudaSuccess) return e;
        return launch_pdl(tc_gemm_kernel<false>, dim3(num_sms), dim3(kThreads16), smem, s, P);
    }
    return cudaGetLastError();
}

}  // namespace tsmoe

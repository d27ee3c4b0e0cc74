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
//   * Decode calls combine inside phase 2 (the CTA completing a row tile combines it for every
//     token); with the Gemma sandwich tail requested, the CTAs count the tiles they combined
//     over the grid, and CTA b, once the count is complete, runs the tail of tokens b, b + grid,
//     ... (its wait is bounded; it waits only for CTAs that are running or that get an SM as the
//     launch ahead of this one drains: one CTA per SM, grid = SM count).
#include "gemv_common.cuh"
#include "tail_common.cuh"

namespace tsmoe {

namespace {

constexpr int kNCW = 16;                      // consumer warps
constexpr int kReducers = 2;                  // reducer warps: unit n goes to reducer n % 2
constexpr int kThreads = (kNCW + 1 + kReducers) * 32;   // + one producer warp + the reducers

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
                         + (kMaxExperts + 1 + 2 * kMaxLocalRoutes) * 4        // in-kernel routes
                         + 32 * 4                                            // combine tile list
                         + 18 * 16;                                           // region padding
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
    int* misc;        // [8]: 0 = ntouched, 1 = abort flag, 2 = combine on, 3 = tiles listed now
    float* rinv;      // [2][8]: prescale inverses travelling with the partials
    uint64_t* rfull;  // [2]: partials of a unit written (16 compute warps arrive)
    uint64_t* rempty; // [2]: partial buffer read by the reducer
    int* off_s;       // [257]: route offsets built in the kernel
    int* perm_s;      // [512]: route list built in the kernel
    int* ctile;       // [32]: row tiles this CTA combines in the current round
    int* tok_s;       // [512]: token of each in-kernel route-list entry
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
    c.ctile = reinterpret_cast<int*>(take(32 * 4));
    c.tok_s = reinterpret_cast<int*>(take(kMaxLocalRoutes * 4));
    return c;
}

// Walks a CTA's units in order: unit u = RT * goff[j] + rt * ng + g (touched expert j, row
// tile rt, group g of the ng = goff[j+1] - goff[j] groups of that expert).  Only the first unit
// is decoded with a division; next() steps without any.
struct UnitCursor {
    int j, rt, g, ng;
    __device__ __forceinline__ void seek(int u, int RT, const int* goff, int nt) {
        j = 0;
        while (j + 1 < nt && u >= RT * goff[j + 1]) ++j;
        ng = goff[j + 1] - goff[j];
        const int local = u - RT * goff[j];
        rt = local / ng;
        g = local - rt * ng;
    }
    // call only while a next unit exists (goff[j + 2] is read when the expert changes)
    __device__ __forceinline__ void next(int RT, const int* goff) {
        if (++g == ng) {
            g = 0;
            if (++rt == RT) {
                rt = 0;
                ++j;
                ng = goff[j + 1] - goff[j];
            }
        }
    }
};

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

// Block slot of compute warp w (a permutation of 0..15): warps 0,4,8,12 (sub-partition 0, with
// the producer warp 16) -> 10..13; 1,5,9,13 (with reducer 17) -> 14,0,1,2; 2,6,10,14 (with
// reducer 18) -> 15,3,4,5; 3,7,11,15 -> 6..9.
static_assert(kNCW == 16 && kReducers == 2, "block slot table assumes 16 compute warps, 2 reducers");
__device__ __forceinline__ int block_slot(int w) {
    constexpr uint64_t kSlots = 0x952D841C730B6FEAull;   // nibble w = slot of warp w
    return static_cast<int>((kSlots >> (4 * w)) & 15u);
}

// TAIL: the phase-2 launch that also runs the Gemma sandwich tail (its code exists only in that
// instantiation: compiled into every launch it measured a few per cent slower everywhere).
template <int FMT, bool TAIL>
__global__ void __launch_bounds__(kThreads, 1) gemv_kernel(const __grid_constant__ KParams P) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const GemvArgs& a = P.a;
    const Plan& p = P.p;
    const int K = a.K, R = a.R;
    const int nblk = K / kBlockK;
    const int RT = R / kRowTile;
    const int nchunk = (nblk + p.nb - 1) / p.nb;
    const int tg = p.tg;
    constexpr bool kPacked = (FMT == FMT_MXFP4 || FMT == FMT_INT4);
    constexpr int BB = kPacked ? packed_block_bytes(FMT) : 0;
    constexpr bool kMmaBf16 = (FMT == FMT_BF16);
    const bool prescale = !kMmaBf16 && a.adt == 1;

    Carve c = carve(smem_raw, p, K);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Phase 2 starts before the launch ahead of it has finished: it begins only once every CTA
    // of that launch has passed its own wait, so the route data are final by then, and weights
    // are never written on the device.  The route tables and the weight ring fill at once; only
    // the warps that read the hidden rows (or the combine's inputs) wait.
    const bool early = a.phase == 1;
    if (!early) pdl_wait();     // inputs of this launch may come from the previous kernel
    pdl_launch_dependents();

    // ---- route list (built here for decode sizes), unit tables --------------------------------
    const int* OFF = a.off;
    const int* PERM = a.perm;
    if (a.idx) {
        OFF = c.off_s;
        PERM = c.perm_s;
    }
    // Phase 1 with at most tg tokens ("token mode"): every token's row is staged once (x is per
    // token and shared by every expert) and the units index it by token; otherwise rows are
    // staged per group of routes when the group changes.
    const bool tokmode = a.phase == 0 && a.T <= tg;
    const bool copy_bits = kMmaBf16 || a.adt == 0;
    if (warp == kNCW + 1) {
        // ---- route list (decode sizes) and unit tables, built by one warp --------------------
        build_route_tables(a, tg, lane, c.off_s, c.perm_s, c.tok_s, c.touched, c.cnt, c.goff, c.misc);
    } else if (warp == kNCW) {
        if (lane == 0) {
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
    } else if (tokmode && warp < 8) {
        // token mode: stage every token's row while the route tables are being built
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
    // the phase-1 launch clears the combine counters the phase-2 launch will count with (and,
    // after them, the count of combined tiles)
    if (a.cmb_mode == 1 && blockIdx.x == 0)
        for (int i = threadIdx.x; i <= a.cmb_n; i += blockDim.x) a.cmb_cnt[i] = 0;
    __syncthreads();
    const int nt = c.misc[0];
    // Phase 2 (one matrix) takes two 16-row tiles per unit, in the slots phase 1 uses for gate
    // and up, when there are units enough for four per CTA even so: half the units, so half the
    // per-unit hand-offs and reductions.
    const bool pair2 = a.phase == 1 && (RT % 2) == 0 && RT * c.goff[nt] >= 8 * static_cast<int>(gridDim.x);
    const int RTu = pair2 ? RT / 2 : RT;              // units per route group of an expert
    const int TR = pair2 ? 2 * kRowTile : kRowTile;   // output rows per unit
    const int nmat = (a.phase == 0 || pair2) ? 2 : 1;
    const int U = RTu * c.goff[nt];
    const int u0 = static_cast<int>((static_cast<long long>(U) * blockIdx.x) / gridDim.x);
    const int u1 = static_cast<int>((static_cast<long long>(U) * (blockIdx.x + 1)) / gridDim.x);
    constexpr int kCmbThreads = (kNCW + kReducers) * 32;   // compute + reducer warps
    constexpr bool tail_on = TAIL;

    // Gemma sandwich tail of tokens blockIdx.x, + gridDim.x, ...: the row's other inputs are
    // loaded, then the CTA waits (bounded) until every row tile of y is combined, then the compute
    // and reducer warps finish the row, staged as f32 in the idle weight ring.
    auto run_tail = [&](int tix) {
        for (int t = blockIdx.x; t < a.tail.T; t += gridDim.x) {
            auto ready = [&]() {
                if (tix == 0) {
                    int ok = 1;
                    const long long t0 = clock64();
                    while (ld_acquire_gpu_s32(a.tdone) < RTu) {
                        if (clock64() - t0 > (1ll << 31)) {
                            ok = 0;
                            report_error(a.status, DEV_ERR_TIMEOUT);
                            break;
                        }
                        __nanosleep(64);
                    }
                    c.misc[4] = ok;
                }
                named_bar(2, kCmbThreads);
                const bool ok = c.misc[4] != 0;
                if (ok) (void)ld_acquire_gpu_s32(a.tdone);   // each thread acquires the rows itself
                return ok;
            };
            if (!gemma_tail_rows_v8(a.tail, t, 1, reinterpret_cast<float*>(c.ring), c.red, tix, kCmbThreads, 2,
                                    ready))
                return;
        }
    };

    if (u0 >= u1) {
        if (early) pdl_wait();  // completes after the launch ahead of it, like every launch
        if (tail_on && warp != kNCW) run_tail(warp < kNCW ? threadIdx.x : threadIdx.x - 32);
        return;
    }

    // Fused combine (phase 2 of a routed decode call), run by the compute warps and the
    // reducer warps together once every unit of this CTA is stored: every unit bumps its row
    // tile's counter (TR rows, over all CTAs); the CTA that completes a tile's count runs the
    // slot-ordered combine of that tile.  Rounds of up to 32 units: the first reducer bumps 32
    // counters at once (one lane each) and lists the completed tiles, then all compute and
    // reducer warps combine them.
    auto fused_combine = [&]() {
        named_bar(2, kCmbThreads);                  // combine decision published
        const int tix = warp < kNCW ? threadIdx.x : threadIdx.x - 32;     // skip the producer warp
        if (!c.misc[2]) {
            if (tail_on) run_tail(tix);         // (its wait runs out: the call has failed)
            return;
        }
        int jl = 0, ncomb = 0;
        for (int ub = u0; ub < u1; ub += 32) {
            if (warp == kNCW + 1) {
                const int u = ub + lane;
                int rt = 0, last = 0;
                if (u < u1) {
                    int g;
                    decode_unit(u, RTu, c.goff, nt, jl, rt, g, c.cnt, tg);
                    last = count_tile_unit(a.cmb_cnt, rt, c.goff[nt]);
                }
                const unsigned lm = __ballot_sync(0xffffffffu, last);
                if (last) {
                    c.ctile[__popc(lm & ((1u << lane) - 1u))] = rt;
                    a.cmb_cnt[rt] = 0;                  // complete: ready for the next call
                }
                if (lane == 0) c.misc[3] = __popc(lm);
            }
            named_bar(2, kCmbThreads);              // tile list ready
            const int ntile = c.misc[3];
            combine_tiles(a, c.ctile, ntile, TR, tix, kCmbThreads);
            named_bar(2, kCmbThreads);              // tile list consumed
            ncomb += ntile;
        }
        if (tail_on) {
            // this CTA's combined rows are written (the barrier above): count them (release)
            if (tix == 0 && ncomb > 0) {
                __threadfence();
                asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(a.tdone), "r"(ncomb) : "memory");
            }
            run_tail(tix);
        }
    };

    if (warp > kNCW) {
        // ================================ reducer warps =====================================
        // Reducer r takes the units u0 + r, u0 + r + 2, ...: it sums the 16 compute warps'
        // partials of a unit in fixed warp order, applies the prescale inverse, bias and
        // activation and stores the unit's outputs.  Two of them, so that the reduction (a
        // serial chain sharing its SM sub-partition with four compute warps) keeps pace.
        // Every output this lane touches has row (lane & 15) of the tile, so the unit's biases
        // are fetched one unit ahead (lane l < 16: bias 0 of row l, lane 16 + l: bias 1) and
        // handed out with shuffles.
        if (early) pdl_wait();
        const int r = warp - kNCW - 1;
        const int row = lane & 15;
        UnitCursor cu, cb;              // the unit being reduced, the unit whose bias is fetched
        auto step = [&](UnitCursor& x, int from) {     // x at unit `from` -> unit from + kReducers
            for (int q = 1; q <= kReducers; ++q)
                if (from + q < u1) x.next(RTu, c.goff);
        };
        if (u0 + r < u1) {
            cu.seek(u0 + r, RTu, c.goff, nt);
            cb = cu;
        }
        auto fetch_bias = [&]() {
            // phase 1: lanes 0-15 gate bias, 16-31 up bias of row `row`; phase 2: the down bias of
            // row `row` of the unit's first (lanes 0-15) and, paired, second 16-row tile
            const uint16_t* bp = lane < 16 ? a.b0 : (a.phase == 0 ? a.b1 : (pair2 ? a.b0 : nullptr));
            if (!bp) return 0.0f;
            const int brow = cb.rt * TR + ((pair2 && lane >= 16) ? kRowTile : 0) + row;
            return __bfloat162float(__ushort_as_bfloat16(bp[static_cast<size_t>(c.touched[cb.j]) * R + brow]));
        };
        float bias_next = u0 + r < u1 ? fetch_bias() : 0.0f;
        for (int u = u0 + r; u < u1; u += kReducers) {
            if (u > u0 + r) step(cu, u - kReducers);
            const int j = cu.j, rt = cu.rt, g = cu.g;
            const int e = c.touched[j];
            const int cnt_g = min(tg, c.cnt[j] - g * tg);
            const int rbase = a.dense ? g * tg : OFF[e] + g * tg;
            const float bias_cur = bias_next;
            if (u + kReducers < u1) {
                step(cb, u);
                bias_next = fetch_bias();
            }
            const float bias0 = __shfl_sync(0xffffffffu, bias_cur, row);
            const float bias1 = __shfl_sync(0xffffffffu, bias_cur, 16 + row);
            const int nl = u - u0, b = nl & 1;
            const bool ok = c.misc[1] == 0 && mbar_wait_bounded(&c.rfull[b], (nl >> 1) & 1);
            if (!ok) {
                if (lane == 0 && c.misc[1] == 0) {
                    c.misc[1] = 1;
                    report_error(a.status, DEV_ERR_TIMEOUT);
                }
            } else {
                const float* redb = c.red + static_cast<size_t>(b) * kNCW * 2 * kRowTile * 8;
                const int orow = rt * TR + row;
                for (int n = lane >> 4; n < cnt_g; n += 2) {
                    const int rid = a.dense ? rbase + n : PERM[rbase + n];
                    float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
                    for (int w = 0; w < kNCW; ++w) {
                        s0 += redb[(w * 2 + 0) * kRowTile * 8 + row * 8 + n];
                        if (nmat == 2) s1 += redb[(w * 2 + 1) * kRowTile * 8 + row * 8 + n];
                    }
                    const float inv = c.rinv[b * 8 + n];
                    s0 = s0 * inv + bias0;
                    if (a.phase == 0) {
                        s1 = s1 * inv + bias1;
                        const float h = act_fn(a.act, s0, s1, a.limit, a.alpha);
                        static_cast<uint16_t*>(a.out)[static_cast<size_t>(rid) * R + orow] = float_to_adt_bits(h, a.adt);
                    } else {
                        static_cast<float*>(a.out)[static_cast<size_t>(rid) * R + orow] = s0;
                        if (pair2)
                            static_cast<float*>(a.out)[static_cast<size_t>(rid) * R + orow + kRowTile] = s1 * inv + bias1;
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&c.rempty[b]);
        }
        if (a.cmb_mode == 2) {
            // the counting atomics (after the CTA barrier in the combine) release these outputs
            if (r == 0 && lane == 0) c.misc[2] = c.misc[1] == 0;
            __syncwarp();
            fused_combine();
        }
        return;
    }

    if (warp == kNCW) {
        // ================================ producer warp =====================================
        int it = 0, slot = 0;
        uint32_t ph = 0;                // phase parity of the ring slot `slot`
        int issued[kMaxStages];         // lane 0: the last iteration copied into each slot
#pragma unroll
        for (int q = 0; q < kMaxStages; ++q) issued[q] = -1;
        UnitCursor cu;
        cu.seek(u0, RTu, c.goff, nt);
        int pj = -1, e = 0;
        for (int u = u0; u < u1; ++u) {
            if (u > u0) cu.next(RTu, c.goff);
            if (cu.j != pj) {
                pj = cu.j;
                e = c.touched[pj];
            }
            for (int m = 0; m < nmat; ++m) {
                // the m-th stream of the unit: gate / up (phase 1), or the m-th 16-row tile (phase 2)
                const uint8_t* wbase = ((m == 0 || pair2) ? a.w0 : a.w1) + static_cast<size_t>(e) * a.mat_bytes;
                const int rt = pair2 ? cu.rt * 2 + m : cu.rt;
                for (int ch = 0; ch < nchunk; ++ch, ++it) {
                    const int s = slot;
                    const uint32_t par = ph ^ 1;
                    if (++slot == p.nstages) {
                        slot = 0;
                        ph ^= 1;
                    }
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
                    // test setting: the first stage's copy is withheld, so the consumers'
                    // bounded wait on it runs out (reported as TS_ERR_TIMEOUT)
                    if (a.stall && it == 0) continue;
                    if (lane == 0) issued[s] = it;
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
        // if the consumers gave up, wait (bounded) for the copies still in flight: the last
        // copy issued into each slot (the slot's barrier has started no later phase)
        if (c.misc[1] && lane == 0) {
            for (int q = 0; q < p.nstages; ++q)
                if (issued[q] >= 0) mbar_wait_bounded(&c.full[q], (issued[q] / p.nstages) & 1);
        }
        return;
    }

    // ================================== consumer warps =========================================
    if (early) pdl_wait();
    const int gid = lane >> 2, tid = lane & 3;
    int it = 0, slot = 0;
    uint32_t ph = 0;                    // phase parity of the ring slot `slot`
    const uint16_t* in = a.in;
    // The route group's row mapping is looked up (and, outside token mode, its activations
    // staged) only when the group changes: consecutive units mostly share it, only the row tile
    // moves, so a unit's first fragment load does not wait on a chain of shared-memory lookups.
    int ckey = -1;                      // (j << 16) | g of the current group
    int brow = 0, xc0 = 0, xc1 = 0;     // activation row this lane feeds the mma; INT4 x-sum columns
    float my_rinv = 0.0f;               // warp 0, lane n < 8: inverse prescale of column n
    UnitCursor cu;
    cu.seek(u0, RTu, c.goff, nt);
    for (int u = u0; u < u1; ++u) {
        if (u > u0) cu.next(RTu, c.goff);
        const int key = (cu.j << 16) | cu.g;
        if (key != ckey) {
            const bool first = ckey < 0;
            ckey = key;
            const int j = cu.j, g = cu.g;
            const int e = c.touched[j];
            const int cnt_g = min(tg, c.cnt[j] - g * tg);
            const int rbase = a.dense ? g * tg : OFF[e] + g * tg;
            // staged row of each of the unit's columns (routes): the token in token mode
            auto row_of = [&](int n) {
                if (!tokmode) return n < tg ? n : 0;
                if (n >= cnt_g) return 0;
                if (a.dense) return rbase + n;
                return a.idx ? c.tok_s[rbase + n] : PERM[rbase + n] / a.k;
            };
            brow = row_of(gid);
            if (FMT == FMT_INT4) {
                xc0 = row_of(2 * tid);
                xc1 = row_of(2 * tid + 1);
            }
            // ---- stage this group's activations (f16 with prescale, or as-is) -------------
            if (!tokmode) {
                // every compute warp must be done with the previous group's activations
                if (!first) named_bar(1, kNCW * 32);
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
            if (warp == 0 && lane < 8) my_rinv = c.xinv[row_of(lane)];
        }

        // ---- stream the unit's weight chunks ---------------------------------------------------
        float acc[2][4];
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[m][q] = 0.0f;

        for (int m = 0; m < nmat; ++m) {
            for (int ch = 0; ch < nchunk; ++ch, ++it) {
                const int s = slot;
                const uint32_t par = ph;
                if (++slot == p.nstages) {
                    slot = 0;
                    ph ^= 1;
                }
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
                    // three blocks in flight per warp: independent fragments, interleavable; the
                    // ragged rest (at most two blocks) also in one round.  Warp w starts at block
                    // slot block_slot(w): when a stage splits unevenly, the warps that share an SM
                    // sub-partition with the producer (w % 4 == 0) or a reducer (w % 4 == 1, 2)
                    // get the highest slots, which have one block fewer.
                    int i = block_slot(warp);
                    for (; i + 2 * kNCW < nbc; i += 3 * kNCW) {
                        block(i);
                        block(i + kNCW);
                        block(i + 2 * kNCW);
                    }
                    if (i < nbc) {
                        block(i);
                        if (i + kNCW < nbc) block(i + kNCW);
                    }
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
            if (warp == 0 && lane < 8) c.rinv[b * 8 + lane] = my_rinv;
            __syncwarp();
            if (lane == 0) mbar_arrive(&c.rfull[b]);
        }
    }
    if (a.cmb_mode == 2) fused_combine();
}

}  // namespace

cudaError_t launch_gemv(const GemvArgs& a, int num_sms, cudaStream_t s) {
    KParams P;
    P.a = a;
    const int tmax = a.T;                   // tokens per expert never exceed T
    P.p = make_plan(a.fmt, a.K, tmax < 8 ? (tmax > 0 ? tmax : 1) : 8);
    if (P.p.tg < 1) return cudaErrorInvalidValue;
    const bool tail_on = a.cmb_mode == 2 && a.tail.T > 0;
    // the tail stages rows of H floats in the weight ring (at least one), 8 elements a thread
    if (tail_on && (a.tail.H > kTailMaxH || a.tail.H % 8 ||
                    static_cast<size_t>(a.tail.H) * 4 > static_cast<size_t>(P.p.nstages) * kStageBytes ||
                    a.tail.H > kTailV * (kNCW + kReducers) * 32 * 8 || !a.tdone))
        return cudaErrorInvalidValue;
    P.a.tg = P.p.tg;
    void (*kern)(const KParams);
    switch (a.fmt) {
        case FMT_F16: kern = tail_on ? gemv_kernel<FMT_F16, true> : gemv_kernel<FMT_F16, false>; break;
        case FMT_BF16: kern = tail_on ? gemv_kernel<FMT_BF16, true> : gemv_kernel<FMT_BF16, false>; break;
        case FMT_MXFP4: kern = tail_on ? gemv_kernel<FMT_MXFP4, true> : gemv_kernel<FMT_MXFP4, false>; break;
        default: kern = tail_on ? gemv_kernel<FMT_INT4, true> : gemv_kernel<FMT_INT4, false>; break;
    }
    const cudaError_t e = ensure_smem(kern, P.p.smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(num_sms), dim3(kThreads), P.p.smem, s, P);
}

}  // namespace tsmoe

// gemv_common.cuh -- device helpers of the decode GEMV (gemv.cu): the activation functions,
// activation-row staging, the in-kernel route list and the fused combine's tile helpers.
#pragma once

#include "common.cuh"

namespace tsmoe {
namespace {

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

constexpr int kMaxLocalRoutes = 512;          // route lists built inside the kernel up to this

// Route list for decode sizes (T*k <= 512, counting sort of the route ids by expert, ascending
// id inside an expert, built by one warp) and the unit tables: touched experts in ascending
// order, their route counts and the prefix of their route groups (groups of <= tg routes).
// The route offsets are the in-kernel list when a.idx is set, else a.off.  The
// global route data are read past L1 (ld.global.cg): a phase-2 launch reads them before its
// wait on the launch ahead of it.
__device__ __forceinline__ void build_route_tables(const GemvArgs& a, int tg, int lane, int* off_s,
                                                   int* perm_s, int* tok_s, int* touched, int* cnt,
                                                   int* goff, int* misc) {
    if (a.idx) {
        // counting sort of the route ids by expert, ascending id inside an expert: chunks of
        // 32 routes, experts of a chunk grouped with match_any, one counter update per group
        const int n = a.T * a.k;
        int ev[kMaxLocalRoutes / 32];
#pragma unroll
        for (int q = 0; q < kMaxLocalRoutes / 32; ++q) {
            const int r = q * 32 + lane;
            ev[q] = r < n ? __ldcg(a.idx + r) : -1;
        }
        for (int e = lane; e <= a.E; e += 32) off_s[e] = 0;
        __syncwarp();
#pragma unroll
        for (int q = 0; q < kMaxLocalRoutes / 32; ++q) {
            if (q * 32 >= n) break;
            const int r = q * 32 + lane;
            const bool valid = ev[q] >= 0 && ev[q] < a.E;
            if (r < n && !valid) report_error(a.status, DEV_ERR_INVALID);
            const unsigned peers = __match_any_sync(0xffffffffu, valid ? ev[q] : -1);
            if (valid && __ffs(peers) - 1 == lane) off_s[ev[q] + 1] += __popc(peers);
            __syncwarp();
        }
        // inclusive scan of the counts (off_s[1..E]) -> route offsets; lane l owns 8 entries
        {
            int loc[8], sum = 0;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int e = lane * 8 + q;
                loc[q] = e < a.E ? off_s[e + 1] : 0;
                sum += loc[q];
            }
            int incl = sum;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, d);
                if (lane >= d) incl += v;
            }
            int run = incl - sum;
            __syncwarp();
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int e = lane * 8 + q;
                run += loc[q];
                if (e < a.E) {
                    off_s[e + 1] = run;
                    cnt[e] = run - loc[q];          // placement cursor (cnt reused)
                }
            }
            __syncwarp();
        }
#pragma unroll
        for (int q = 0; q < kMaxLocalRoutes / 32; ++q) {
            if (q * 32 >= n) break;
            const int r = q * 32 + lane;
            const bool valid = ev[q] >= 0 && ev[q] < a.E;
            const unsigned peers = __match_any_sync(0xffffffffu, valid ? ev[q] : -1);
            if (valid) {
                const int pos = cnt[ev[q]] + __popc(peers & ((1u << lane) - 1u));
                perm_s[pos] = r;
                tok_s[pos] = r / a.k;
            }
            __syncwarp();
            if (valid && __ffs(peers) - 1 == lane) cnt[ev[q]] += __popc(peers);
            __syncwarp();
        }
    }
    // touched experts in ascending order with their route counts and group prefix
    int nt = 0, acc = 0;
    if (a.dense) {
        if (lane == 0) {
            touched[0] = 0;
            cnt[0] = a.T;
            goff[0] = 0;
        }
        acc = (a.T + tg - 1) / tg;
        nt = 1;
    } else {
        for (int e0 = 0; e0 < a.E; e0 += 32) {
            const int e = e0 + lane;
            int n = 0;
            if (e < a.E) n = a.idx ? off_s[e + 1] - off_s[e] : __ldcg(a.off + e + 1) - __ldcg(a.off + e);
            const unsigned m = __ballot_sync(0xffffffffu, n > 0);
            const int groups = n > 0 ? (n + tg - 1) / tg : 0;
            int incl = groups;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, d);
                if (lane >= d) incl += v;
            }
            __syncwarp();
            if (n > 0) {
                const int pos = nt + __popc(m & ((1u << lane) - 1u));
                touched[pos] = e;
                cnt[pos] = n;
                goff[pos] = acc + incl - groups;
            }
            __syncwarp();
            acc += __shfl_sync(0xffffffffu, incl, 31);
            nt += __popc(m);
        }
    }
    if (lane == 0) {
        goff[nt] = acc;
        misc[0] = nt;
        misc[1] = 0;
    }
}

// Counts one unit of row tile `tile` as done and says whether it was the tile's last (`need`
// units).  The add is acq_rel at GPU scope: it releases this CTA's outputs (stored before a CTA
// barrier that precedes the call) and, for the last unit, acquires every other CTA's.
__device__ __forceinline__ bool count_tile_unit(int* cnt, int tile, int need) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(cnt + tile) : "memory");
    return old + 1 == need;
}

// Slot-ordered combine of `ntile` completed row tiles of TR rows (tiles[i] * TR + 0..TR-1, every
// token): y[t][row] = seed[t][row] + sum over slots q of w[t*k + q] * e[t*k + q][row], each
// product rounded and then added in slot order.  A thread takes four consecutive rows of one
// token (16-byte loads and stores) and two such quads per round, with all their loads issued
// before any is used: the CTA that completes the last tiles does this alone, so its latency is
// the call's tail.  TR and R are multiples of 4; e and the seed sit in the 256-byte aligned
// workspace and y, y_f32 are 16-byte aligned (the entry point refuses them otherwise).
__device__ __forceinline__ void combine_tiles(const GemvArgs& a, const int* tiles, int ntile, int TR,
                                              int tix, int nthr) {
    constexpr int kU = 2;
    const int R = a.R, TQ = TR / 4;
    const int per = a.T * TQ, total = ntile * per;
    const float* ev = static_cast<const float*>(a.out);
    uint16_t* y = static_cast<uint16_t*>(a.y);
    auto ld4 = [](const float* p) { return __ldcg(reinterpret_cast<const float4*>(p)); };
    for (int o0 = tix; o0 < total; o0 += kU * nthr) {
        float4 acc[kU];
        size_t yo[kU];
        int orow[kU], rk[kU];
        bool v[kU];
#pragma unroll
        for (int i = 0; i < kU; ++i) {
            const int o = o0 + i * nthr;
            v[i] = o < total;
            const int oo = v[i] ? o : 0;
            const int tile = oo / per, rem = oo - tile * per;
            const int t = rem / TQ;
            orow[i] = tiles[tile] * TR + (rem - t * TQ) * 4;
            rk[i] = t * a.k;
            yo[i] = static_cast<size_t>(t) * R + orow[i];
            acc[i] = (v[i] && a.seed) ? ld4(a.seed + yo[i]) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        for (int q0 = 0; q0 < a.k; q0 += 4) {
            float4 ex[kU][4];
            float wq[kU][4];
#pragma unroll
            for (int i = 0; i < kU; ++i)
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const bool use = v[i] && q0 + q < a.k;
                    const int r = rk[i] + q0 + q;
                    wq[i][q] = use ? a.w[r] : 0.0f;
                    ex[i][q] = use ? ld4(ev + static_cast<size_t>(r) * R + orow[i]) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
            for (int i = 0; i < kU; ++i)
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    if (q0 + q >= a.k) continue;
                    acc[i].x = __fadd_rn(acc[i].x, __fmul_rn(wq[i][q], ex[i][q].x));
                    acc[i].y = __fadd_rn(acc[i].y, __fmul_rn(wq[i][q], ex[i][q].y));
                    acc[i].z = __fadd_rn(acc[i].z, __fmul_rn(wq[i][q], ex[i][q].z));
                    acc[i].w = __fadd_rn(acc[i].w, __fmul_rn(wq[i][q], ex[i][q].w));
                }
        }
#pragma unroll
        for (int i = 0; i < kU; ++i) {
            if (!v[i]) continue;
            const uint16_t b0 = float_to_adt_bits(acc[i].x, a.adt), b1 = float_to_adt_bits(acc[i].y, a.adt);
            const uint16_t b2 = float_to_adt_bits(acc[i].z, a.adt), b3 = float_to_adt_bits(acc[i].w, a.adt);
            if (a.y_f32) *reinterpret_cast<float4*>(a.y_f32 + yo[i]) = acc[i];
            *reinterpret_cast<uint2*>(y + yo[i]) =
                make_uint2(b0 | (static_cast<uint32_t>(b1) << 16), b2 | (static_cast<uint32_t>(b3) << 16));
        }
    }
}

}  // namespace
}  // namespace tsmoe

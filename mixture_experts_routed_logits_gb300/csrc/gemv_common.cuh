// gemv_common.cuh -- device helpers shared by the two decode GEMV kernels (gemv.cu: the
// 16-bit-weight kernel with a producer warp and reducer warps; gemv_sk.cu: the packed-weight
// kernel in which every warp streams its own range of chunks).
#pragma once

#include "common.cuh"

namespace tsmoe {
namespace {

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
// OFF is the route offsets to use (the in-kernel list when a.idx is set, else a.off).
__device__ __forceinline__ void build_route_tables(const GemvArgs& a, int tg, int lane, int* off_s,
                                                   int* perm_s, int* tok_s, int* touched, int* cnt,
                                                   int* goff, int* misc) {
    const int* OFF = a.idx ? off_s : a.off;
    if (a.idx) {
        // counting sort of the route ids by expert, ascending id inside an expert: chunks of
        // 32 routes, experts of a chunk grouped with match_any, one counter update per group
        const int n = a.T * a.k;
        int ev[kMaxLocalRoutes / 32];
#pragma unroll
        for (int q = 0; q < kMaxLocalRoutes / 32; ++q) {
            const int r = q * 32 + lane;
            ev[q] = r < n ? a.idx[r] : -1;
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
            const int n = e < a.E ? OFF[e + 1] - OFF[e] : 0;
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

}  // namespace
}  // namespace tsmoe

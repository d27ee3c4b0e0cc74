// misc.cu -- the slot-ordered combine (step 5) and the one-time weight packer.
//
// Source pages (docs.rs, turbospark-runtime 0.3.0):
//   gpt-oss routed-expert pass (src/families/gptoss/moe.rs), module header: the slot order is
//     the router's ranking and phase 2 reduces blob[slot] * routing_w[slot] in slot-index order
//     because FP addition is not associative; zero_hidden is the residual input, so
//     y = residual + sum(w * expert) is the routed sum alone.
//   Gemma-4 batched routed prefill (src/families/gemma4/moe_batch.rs): phase 2 seeded from
//     zeros ("0.0f + p"); the shared expert is a dense gated FFN added to the routed half.
//   The repack walk (moe_offsets_from_layout, named in the gpt-oss module header) is the
//     counterpart of ts_moe_pack: it lays the expert blobs out for the kernels once.
#include "common.cuh"

namespace tsmoe {

namespace {

// y[t] = adt(seed[t] + sum_s w[t][s] * e[t*k+s]) with one rounded multiply and one rounded
// add per slot, in slot order; the f32 sum is optionally returned.
__global__ void __launch_bounds__(256) combine_kernel(CombineArgs a) {
    pdl_wait();
    pdl_launch_dependents();
    const int t = blockIdx.y;
    const int j4 = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= a.T || j4 * 4 >= a.H) return;
    const size_t rowo = static_cast<size_t>(t) * a.H + static_cast<size_t>(j4) * 4;
    float4 acc = a.seed ? *reinterpret_cast<const float4*>(a.seed + rowo) : make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < a.k; ++s) {
        const size_t r = static_cast<size_t>(t) * a.k + s;
        const float wv = a.w[r];
        const float4 ev = *reinterpret_cast<const float4*>(a.e + r * a.H + static_cast<size_t>(j4) * 4);
        acc.x = __fadd_rn(acc.x, __fmul_rn(wv, ev.x));
        acc.y = __fadd_rn(acc.y, __fmul_rn(wv, ev.y));
        acc.z = __fadd_rn(acc.z, __fmul_rn(wv, ev.z));
        acc.w = __fadd_rn(acc.w, __fmul_rn(wv, ev.w));
    }
    if (a.y_f32) *reinterpret_cast<float4*>(a.y_f32 + rowo) = acc;
    uint16_t* y = static_cast<uint16_t*>(a.y) + rowo;
    const uint2 o = make_uint2(static_cast<uint32_t>(float_to_adt_bits(acc.x, a.adt)) |
                                   (static_cast<uint32_t>(float_to_adt_bits(acc.y, a.adt)) << 16),
                               static_cast<uint32_t>(float_to_adt_bits(acc.z, a.adt)) |
                                   (static_cast<uint32_t>(float_to_adt_bits(acc.w, a.adt)) << 16));
    *reinterpret_cast<uint2*>(y) = o;
}

// Packed layout, per matrix, per 16-row tile, per 32-column block (BB bytes):
//   bytes [0, 256): lane L = 4*gid + tid holds 8 bytes: the 4 code bytes of row gid covering
//                   columns 8*tid .. 8*tid+7 of the block, then the same for row gid+8;
//   MXFP4 [256, 272): for gid 0..7: e8m0 of row gid, e8m0 of row gid+8;
//   INT4  [256, 320): for gid 0..7: (scale, min) f16 pair of row gid, then of row gid+8.
__global__ void pack_kernel(int fmt, int nmat, int R, int K, const uint8_t* __restrict__ codes,
                            const uint8_t* __restrict__ scales, uint8_t* __restrict__ out,
                            size_t total) {
    const int BB = packed_block_bytes(fmt);
    const int nblk = K / kBlockK;
    const size_t tile = static_cast<size_t>(nblk) * BB;
    const size_t mat = static_cast<size_t>(R / kRowTile) * tile;
    for (size_t o = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; o < total;
         o += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const size_t m = o / mat;
        const size_t rem = o % mat;
        const int rt = static_cast<int>(rem / tile);
        const size_t rem2 = rem % tile;
        const int b = static_cast<int>(rem2 / BB);
        const int q = static_cast<int>(rem2 % BB);
        uint8_t v;
        if (q < 256) {
            const int L = q / 8, half = (q % 8) / 4, byte = q % 4;
            const int gid = L / 4, tid = L % 4;
            const size_t row = m * R + static_cast<size_t>(rt) * kRowTile + gid + 8 * half;
            v = codes[row * (K / 2) + static_cast<size_t>(b) * 16 + tid * 4 + byte];
        } else if (fmt == FMT_MXFP4) {
            const int q2 = q - 256;
            const int gid = q2 / 2, which = q2 % 2;
            const size_t row = m * R + static_cast<size_t>(rt) * kRowTile + gid + 8 * which;
            v = scales[row * nblk + b];
        } else {
            const int q2 = q - 256;
            const int gid = q2 / 8, which = (q2 % 8) / 4, byte = q2 % 4;
            const size_t row = m * R + static_cast<size_t>(rt) * kRowTile + gid + 8 * which;
            v = scales[(row * nblk + b) * 4 + byte];
        }
        out[o] = v;
    }
}

}  // namespace

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s) {
    if (a.T <= 0) return cudaSuccess;
    dim3 grid((a.H / 4 + 255) / 256, a.T);
    return launch_pdl(combine_kernel, grid, dim3(256), 0, s, a);
}

cudaError_t launch_pack(int fmt, int nmat, int R, int K, const uint8_t* codes,
                        const uint8_t* scales, uint8_t* packed, cudaStream_t s) {
    const size_t total = static_cast<size_t>(nmat) * (R / kRowTile) * (K / kBlockK) *
                         packed_block_bytes(fmt);
    if (total == 0) return cudaSuccess;
    size_t blocks = (total + 255) / 256;
    if (blocks > 65535u * 16u) blocks = 65535u * 16u;
    pack_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(fmt, nmat, R, K, codes, scales,
                                                                packed, total);
    return cudaGetLastError();
}

}  // namespace tsmoe

// api.cu -- host side of the C ABI declared in include/ts_moe.h: argument validation, the
// workspace layout and the launch sequence.  Every check runs before anything is launched;
// a request the kernels cannot serve is refused with a message, never degraded (the pages'
// convention: the Gemma-4 batched routed prefill returns Unsupported rather than quietly
// looping the per-token kernels).
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>

#include "../../include/ts_moe.h"

#include "internal.h"

using namespace tsmoe;

namespace {

thread_local std::string g_err;
thread_local cudaEvent_t g_phase_ev[8];
thread_local int g_phase_n = 0;
thread_local int g_wait_test = 0;   // ts_moe_set_wait_test: consumed by the next forward call

// records phase event i (if registered) on the stream; capture-safe
cudaError_t phase_mark(int i, cudaStream_t st) {
    if (i >= g_phase_n || !g_phase_ev[i]) return cudaSuccess;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(st, &cs);
    if (e != cudaSuccess) return e;
    if (cs == cudaStreamCaptureStatusActive)
        return cudaEventRecordWithFlags(g_phase_ev[i], st, cudaEventRecordExternal);
    return cudaEventRecord(g_phase_ev[i], st);
}

ts_status fail(ts_status st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_err = buf;
    return st;
}

ts_status cuda_fail(cudaError_t e, const char* what) {
    return fail(TS_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

inline bool aligned(const void* p, size_t a) {
    return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

int num_sms_current() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev] = n;
    }
    return cache[dev];
}

inline size_t round_up(size_t v, size_t m) { return (v + m - 1) / m * m; }

size_t matrix_bytes(int fmt, int R, int K) {
    if (fmt == FMT_F16 || fmt == FMT_BF16) return static_cast<size_t>(R) * K * 2;
    return static_cast<size_t>(R / kRowTile) * (K / kBlockK) * packed_block_bytes(fmt);
}

ts_status check_experts(const ts_moe_experts* ex, const char* what, int adt) {
    if (!ex) return fail(TS_ERR_INVALID_ARG, "%s: descriptor is NULL", what);
    if (ex->fmt < 0 || ex->fmt > 3) return fail(TS_ERR_INVALID_ARG, "%s: bad weight format %d", what, ex->fmt);
    if (ex->act < 0 || ex->act > 2) return fail(TS_ERR_INVALID_ARG, "%s: bad activation %d", what, ex->act);
    if (ex->E < 1 || ex->E > kMaxExperts)
        return fail(TS_ERR_UNSUPPORTED, "%s: E=%d outside 1..%d", what, ex->E, kMaxExperts);
    if (ex->H <= 0 || ex->I <= 0 || ex->H % kBlockK || ex->I % kBlockK)
        return fail(TS_ERR_UNSUPPORTED, "%s: H=%d and I=%d must be positive multiples of 32", what,
                    ex->H, ex->I);
    if (!ex->gate || !ex->up || !ex->down)
        return fail(TS_ERR_INVALID_ARG, "%s: gate/up/down weight pointer is NULL", what);
    if (!aligned(ex->gate, 16) || !aligned(ex->up, 16) || !aligned(ex->down, 16))
        return fail(TS_ERR_INVALID_ARG, "%s: weight pointers must be 16-byte aligned", what);
    if (!aligned(ex->gate_b, 2) || !aligned(ex->up_b, 2) || !aligned(ex->down_b, 2))
        return fail(TS_ERR_INVALID_ARG, "%s: bias pointers must be 2-byte aligned", what);
    if (!aligned(ex->gateup_mx, 256) || !aligned(ex->down_mx, 256))
        return fail(TS_ERR_INVALID_ARG, "%s: tensor-core MXFP4 blobs must be 256-byte aligned", what);
    if ((ex->gateup_mx || ex->down_mx) && (ex->fmt != FMT_MXFP4 || !ex->gateup_mx || !ex->down_mx))
        return fail(TS_ERR_INVALID_ARG, "%s: gateup_mx/down_mx are MXFP4 blobs, both or none", what);
    if (ex->fmt == FMT_BF16 && adt != TS_DT_BF16)
        return fail(TS_ERR_UNSUPPORTED,
                    "%s: bf16 weights need bf16 activations (f16 activations would be rounded)", what);
    return TS_OK;
}

struct WsLayout {
    size_t status, off, perm, inv, h, e, hs, s, xs, xinv, hinv, h16, cmb, part, tcnt, total;
    size_t xq, xsf, hq, hsf;   // block-scaled path: split activations and their scales
    size_t hrdy;               // block-scaled path, both phases in one launch: h-ready counters
    size_t dxs, dhs, dpart, dcnt, dcnt_bytes;   // block-scaled decode kernels (T <= 8)
    size_t tcnt_n;        // split-K group counters per phase
    int max_split;        // > 1 when the partials fit (decode sizes)
};

constexpr int kMaxSplit = 8;

WsLayout ws_layout(int T, int k, const ts_moe_experts* ex, const ts_moe_experts* sh) {
    WsLayout L{};
    size_t a = 0;
    auto take = [&](size_t bytes) {
        const size_t o = a;
        a = round_up(a + bytes, 256);
        return o;
    };
    const size_t Tk = static_cast<size_t>(T) * k;
    L.status = take(256);
    L.off = take(static_cast<size_t>(ex->E + 1) * 4);
    L.perm = take(Tk * 4);
    L.inv = take(Tk * 4);
    L.h = take(Tk * ex->I * 2);
    L.e = take(Tk * ex->H * 4);
    if (sh) {
        L.hs = take(static_cast<size_t>(T) * sh->I * 2);
        L.s = take(static_cast<size_t>(T) * ex->H * 4);
    }
    L.xs = take(Tk * ex->H * 2);   // activations in route-list order (tensor-core path)
    L.cmb = take(static_cast<size_t>(ex->H / kRowTile + 1) * 4);   // fused-combine counters + tiles done
    if (ex->fmt == FMT_MXFP4) {      // f16 operands of the MXFP4 tensor-core path
        L.xinv = take(Tk * 4);
        L.hinv = take(Tk * 4);
        L.h16 = take(Tk * ex->I * 2);
        // two e4m3 planes and the e8m0 scales of x and of h for the block-scaled path
        L.xq = take(2 * Tk * ex->H);
        L.xsf = take(Tk * mx_sf_row(ex->H));
        L.hq = take(2 * Tk * ex->I);
        L.hsf = take(Tk * mx_sf_row(ex->I));
        L.hrdy = take((Tk + 1) * 4);   // one per (touched expert, route tile) at most + the item count
        if (T <= kMxdTokens && Tk <= kMxdMaxTouched && k <= kMxdMaxK && ex->H <= kMxdMaxH) {
            // decode kernels: the split x and h images, stream-K partials, and the part /
            // row-block counters
            const size_t nt = static_cast<size_t>(ex->E) < Tk ? static_cast<size_t>(ex->E) : Tk;
            const size_t mb0 = (static_cast<size_t>(ex->I) + 127) / 128, mb1 = (static_cast<size_t>(ex->H) + 255) / 256;
            L.dxs = take(((static_cast<size_t>(ex->H) + 127) / 128) * kMxdBStage + 512);
            L.dhs = take(nt * mb0 * kMxdHImage);
            L.dpart = take(static_cast<size_t>(kMxdMaxCtas) * 2 * 2 * kMxdPartFloats * 4);
            L.dcnt_bytes = round_up((nt + nt * mb0 * 4 + nt * mb1 * 4 + mb1 * 4) * 4, 256);
            L.dcnt = take(L.dcnt_bytes);
        }
    }
    // split-K partials of the tensor-core path for decode-sized calls (few routes, so the few
    // (expert, row block) tiles are cut along K to reach every SM): [part][route][2][rows] f32
    // and one counter per (tile group, 32-row slice) and phase
    if (Tk > 0 && Tk <= 64) {
        const size_t rmax = ex->I > ex->H ? ex->I : ex->H;
        const size_t e_eff = static_cast<size_t>(ex->E) < Tk ? static_cast<size_t>(ex->E) : Tk;
        L.max_split = kMaxSplit;
        L.part = take(static_cast<size_t>(kMaxSplit) * Tk * 2 * rmax * 4);
        L.tcnt_n = ((rmax + 127) / 128) * (Tk / 16 + e_eff) * 4;
        L.tcnt = take(2 * L.tcnt_n * 4);
    }
    L.total = a;
    return L;
}

// Decode batches (T <= 8) with MXFP4 blobs and bf16 activations: block-scaled phase 1 (route
// tables, gate/up, activation -> h per touched expert), the shared expert if any, block-scaled
// phase 2 (down -> e, slot-ordered combine -> y).
ts_status forward_mxd(const void* x, int T, const ts_moe_experts* ex, const int32_t* idx,
                      const float* w, int k, const ts_moe_experts* shared, void* y, float* y_f32,
                      unsigned char* W, const WsLayout& L, cudaStream_t st, bool prep_done);

ts_status launch_gemv_checked(const GemvArgs& a, cudaStream_t st, const char* what) {
    const int sms = num_sms_current();
    if (sms <= 0) return fail(TS_ERR_CUDA, "%s: no CUDA device", what);
    cudaError_t e = launch_gemv(a, sms, st);
    if (e != cudaSuccess) return cuda_fail(e, what);
    return TS_OK;
}

ts_status forward_mxd(const void* x, int T, const ts_moe_experts* ex, const int32_t* idx,
                      const float* w, int k, const ts_moe_experts* shared, void* y, float* y_f32,
                      unsigned char* W, const WsLayout& L, cudaStream_t st, bool prep_done) {
    const int sms = num_sms_current();
    if (sms <= 0) return fail(TS_ERR_CUDA, "ts_moe_forward: no CUDA device");
    int* status = reinterpret_cast<int*>(W + L.status);
    MxdArgs M{};
    M.act = ex->act;
    M.limit = ex->swiglu_limit;
    M.alpha = ex->swiglu_alpha;
    M.wgu = static_cast<const uint8_t*>(ex->gateup_mx);
    M.wd = static_cast<const uint8_t*>(ex->down_mx);
    M.bg = static_cast<const uint16_t*>(ex->gate_b);
    M.bu = static_cast<const uint16_t*>(ex->up_b);
    M.bd = static_cast<const uint16_t*>(ex->down_b);
    M.H = ex->H;
    M.I = ex->I;
    M.E = ex->E;
    M.T = T;
    M.k = k;
    M.idx = idx;
    M.wr = w;
    M.x = static_cast<const uint16_t*>(x);
    M.xs = W + L.dxs;
    M.hs = W + L.dhs;
    M.e_out = reinterpret_cast<float*>(W + L.e);
    M.seed = shared ? reinterpret_cast<const float*>(W + L.s) : nullptr;
    M.y = y;
    M.y_f32 = y_f32;
    M.part = reinterpret_cast<float*>(W + L.dpart);
    // the counters (h slices per touched expert, parts per tile of each phase, finished tiles
    // per row block of phase 2): the prep kernel zeroes them (the kernels leave them zero; this
    // covers a call that stopped early)
    M.cnt = reinterpret_cast<int*>(W + L.dcnt);
    M.ncnt = static_cast<int>(L.dcnt_bytes / 4);
    M.status = status;
    M.stall = g_wait_test;
    g_wait_test = 0;
    // the prep launch (x image, counters), unless the router launch already did its work
    cudaError_t e = prep_done ? cudaSuccess : launch_mxd_prep(M, st);
    if (e == cudaSuccess) e = phase_mark(0, st);
    if (e != cudaSuccess) return cuda_fail(e, "ts_moe_forward: block-scaled decode prep");
    if (shared) {
        // the shared expert's output seeds the combine of the fused launch
        GemvArgs gs{};
        gs.fmt = shared->fmt;
        gs.act = shared->act;
        gs.limit = shared->swiglu_limit;
        gs.alpha = shared->swiglu_alpha;
        gs.adt = TS_DT_BF16;
        gs.T = T;
        gs.k = 1;
        gs.E = 1;
        gs.status = status;
        gs.phase = 0;
        gs.w0 = static_cast<const uint8_t*>(shared->gate);
        gs.w1 = static_cast<const uint8_t*>(shared->up);
        gs.b0 = static_cast<const uint16_t*>(shared->gate_b);
        gs.b1 = static_cast<const uint16_t*>(shared->up_b);
        gs.R = shared->I;
        gs.K = shared->H;
        gs.mat_bytes = matrix_bytes(shared->fmt, shared->I, shared->H);
        gs.in = static_cast<const uint16_t*>(x);
        gs.out = W + L.hs;
        gs.dense = 1;
        ts_status s = launch_gemv_checked(gs, st, "ts_moe_forward: shared expert phase 1");
        if (s != TS_OK) return s;
        if ((e = phase_mark(2, st)) != cudaSuccess) return cuda_fail(e, "ts_moe_forward: phase event");
        gs.phase = 1;
        gs.w0 = static_cast<const uint8_t*>(shared->down);
        gs.w1 = nullptr;
        gs.b0 = static_cast<const uint16_t*>(shared->down_b);
        gs.b1 = nullptr;
        gs.R = shared->H;
        gs.K = shared->I;
        gs.mat_bytes = matrix_bytes(shared->fmt, shared->H, shared->I);
        gs.in = reinterpret_cast<const uint16_t*>(W + L.hs);
        gs.out = W + L.s;
        if ((s = launch_gemv_checked(gs, st, "ts_moe_forward: shared expert phase 2")) != TS_OK) return s;
        if ((e = phase_mark(4, st)) != cudaSuccess) return cuda_fail(e, "ts_moe_forward: phase event");
    }
    e = launch_mxd(M, sms, st);
    if (e == cudaSuccess) e = phase_mark(1, st);
    if (e == cudaSuccess) e = phase_mark(3, st);
    if (e == cudaSuccess) e = phase_mark(5, st);
    if (e != cudaSuccess) return cuda_fail(e, "ts_moe_forward: block-scaled decode kernel");
    return TS_OK;
}

}  // namespace

namespace tsmoe {
// Lets other translation units of the library record a ts_last_error() message.
int record_error_code(int status, const char* msg) {
    g_err = msg;
    return status;
}
}  // namespace tsmoe

extern "C" {

const char* ts_last_error(void) { return g_err.c_str(); }

const char* ts_moe_version(void) { return "0.1.0"; }

size_t ts_moe_packed_bytes(int32_t fmt, int32_t nmat, int32_t R, int32_t K) {
    if ((fmt != TS_W_MXFP4 && fmt != TS_W_INT4_AFFINE) || nmat < 1 || R <= 0 || K <= 0 ||
        R % kRowTile || K % kBlockK)
        return 0;
    return static_cast<size_t>(nmat) * matrix_bytes(fmt, R, K);
}

ts_status ts_moe_pack(int32_t fmt, int32_t nmat, int32_t R, int32_t K, const void* codes,
                      const void* scales, void* packed, size_t packed_bytes, void* stream) {
    g_err.clear();
    const size_t need = ts_moe_packed_bytes(fmt, nmat, R, K);
    if (need == 0)
        return fail(TS_ERR_INVALID_ARG,
                    "ts_moe_pack: fmt must be MXFP4 or INT4_AFFINE, R %% 16 == 0, K %% 32 == 0 "
                    "(fmt=%d nmat=%d R=%d K=%d)", fmt, nmat, R, K);
    if (!codes || !scales || !packed) return fail(TS_ERR_INVALID_ARG, "ts_moe_pack: NULL pointer");
    if (!aligned(packed, 16)) return fail(TS_ERR_INVALID_ARG, "ts_moe_pack: packed must be 16-byte aligned");
    if (packed_bytes < need)
        return fail(TS_ERR_INVALID_ARG, "ts_moe_pack: packed_bytes %zu < %zu", packed_bytes, need);
    cudaError_t e = launch_pack(fmt, nmat, R, K, static_cast<const uint8_t*>(codes),
                                static_cast<const uint8_t*>(scales), static_cast<uint8_t*>(packed),
                                static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "ts_moe_pack");
    return TS_OK;
}

size_t ts_moe_packed_mx_bytes(int32_t pair, int32_t nmat, int32_t R, int32_t K) {
    if ((pair != 0 && pair != 1) || nmat < 1 || R <= 0 || K <= 0 || R % 32 || K % kBlockK) return 0;
    return mx_blob_bytes(1 + pair, nmat, R, K);
}

ts_status ts_moe_pack_mx(int32_t pair, int32_t nmat, int32_t R, int32_t K, const void* codes0,
                         const void* scales0, const void* codes1, const void* scales1, void* blob,
                         size_t blob_bytes, void* stream) {
    g_err.clear();
    const size_t need = ts_moe_packed_mx_bytes(pair, nmat, R, K);
    if (need == 0)
        return fail(TS_ERR_INVALID_ARG, "ts_moe_pack_mx: needs pair 0 or 1, nmat >= 1, R %% 32 == 0, "
                    "K %% 32 == 0 (pair=%d nmat=%d R=%d K=%d)", pair, nmat, R, K);
    if (!codes0 || !scales0 || !blob || (pair && (!codes1 || !scales1)))
        return fail(TS_ERR_INVALID_ARG, "ts_moe_pack_mx: NULL pointer");
    if (!aligned(blob, 256)) return fail(TS_ERR_INVALID_ARG, "ts_moe_pack_mx: blob must be 256-byte aligned");
    if (blob_bytes < need)
        return fail(TS_ERR_INVALID_ARG, "ts_moe_pack_mx: blob_bytes %zu < %zu", blob_bytes, need);
    cudaError_t e = launch_mx_pack(1 + pair, nmat, R, K, static_cast<const uint8_t*>(codes0),
                                   static_cast<const uint8_t*>(scales0), static_cast<const uint8_t*>(codes1),
                                   static_cast<const uint8_t*>(scales1), static_cast<uint8_t*>(blob),
                                   static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "ts_moe_pack_mx");
    return TS_OK;
}

// argument checks of the router's x / W_r path (ts_moe_router_route, ts_moe_route_forward)
static ts_status check_router_args(const RouteArgs& a, const char* what) {
    if (a.adt != TS_DT_F16 && a.adt != TS_DT_BF16) return fail(TS_ERR_INVALID_ARG, "%s: bad adt %d", what, a.adt);
    if (a.H <= 0 || a.H % kBlockK) return fail(TS_ERR_UNSUPPORTED, "%s: H=%d must be a positive multiple of 32", what, a.H);
    if (a.H > 12288) return fail(TS_ERR_UNSUPPORTED, "%s: H=%d above 12288", what, a.H);
    if (a.rmsnorm != 0 && a.rmsnorm != 1) return fail(TS_ERR_INVALID_ARG, "%s: rmsnorm must be 0 or 1", what);
    if (a.T > 0 && (!a.x || !a.Wr)) return fail(TS_ERR_INVALID_ARG, "%s: x or W_r is NULL", what);
    if (!aligned(a.Wr, 16)) return fail(TS_ERR_INVALID_ARG, "%s: W_r must be 16-byte aligned", what);
    if (a.T > 0 && a.rmsnorm && !a.xn_out) return fail(TS_ERR_INVALID_ARG, "%s: rmsnorm needs xn_out", what);
    if (!(a.eps >= 0.0f)) return fail(TS_ERR_INVALID_ARG, "%s: eps must be >= 0", what);
    if (a.T < 0) return fail(TS_ERR_INVALID_ARG, "%s: T=%d < 0", what, a.T);
    if (a.E < 1 || a.E > kMaxExperts)
        return fail(TS_ERR_UNSUPPORTED, "%s: E=%d outside 1..%d", what, a.E, kMaxExperts);
    if (a.k < 1 || a.k > a.E) return fail(TS_ERR_INVALID_ARG, "%s: k=%d outside 1..E=%d", what, a.k, a.E);
    if (a.mode < 0 || a.mode > 2) return fail(TS_ERR_INVALID_ARG, "%s: bad mode %d", what, a.mode);
    if (a.mode == MODE_SOFTMAX_K_SCALED && !a.scale)
        return fail(TS_ERR_INVALID_ARG, "%s: SOFTMAX_K_SCALED needs per_expert_scale", what);
    return TS_OK;
}

static ts_status route_common(RouteArgs& a, cudaStream_t st, const char* what) {
    if (a.T < 0) return fail(TS_ERR_INVALID_ARG, "%s: T=%d < 0", what, a.T);
    if (a.E < 1 || a.E > kMaxExperts)
        return fail(TS_ERR_UNSUPPORTED, "%s: E=%d outside 1..%d", what, a.E, kMaxExperts);
    if (a.k < 1 || a.k > a.E) return fail(TS_ERR_INVALID_ARG, "%s: k=%d outside 1..E=%d", what, a.k, a.E);
    if (a.mode < 0 || a.mode > 2) return fail(TS_ERR_INVALID_ARG, "%s: bad mode %d", what, a.mode);
    if (a.mode == MODE_SOFTMAX_K_SCALED && !a.scale)
        return fail(TS_ERR_INVALID_ARG, "%s: SOFTMAX_K_SCALED needs per_expert_scale", what);
    if (a.T == 0) return TS_OK;
    if (!a.idx || !a.w) return fail(TS_ERR_INVALID_ARG, "%s: idx/w output is NULL", what);
    cudaError_t e = launch_router(a, st);
    if (e == cudaSuccess) e = phase_mark(6, st);
    if (e != cudaSuccess) return cuda_fail(e, what);
    return TS_OK;
}

ts_status ts_moe_route(const float* logits, const float* router_bias,
                       const float* per_expert_scale, int32_t T, int32_t E, int32_t k,
                       int32_t mode, int32_t* idx, float* w, void* stream) {
    g_err.clear();
    RouteArgs a{};
    a.logits_in = logits;
    a.bias = router_bias;
    a.scale = per_expert_scale;
    a.idx = idx;
    a.w = w;
    a.T = T;
    a.E = E;
    a.k = k;
    a.mode = mode;
    if (T > 0 && !logits) return fail(TS_ERR_INVALID_ARG, "ts_moe_route: logits is NULL");
    return route_common(a, static_cast<cudaStream_t>(stream), "ts_moe_route");
}

ts_status ts_moe_router_route(const void* x, int32_t adt, int32_t T, int32_t H, const void* W_r,
                              int32_t E, int32_t rmsnorm, float eps, const float* router_bias,
                              const float* per_expert_scale, int32_t k, int32_t mode,
                              void* xn_out, float* logits_out, int32_t* idx, float* w,
                              void* stream) {
    g_err.clear();
    const char* what = "ts_moe_router_route";
    if (adt != TS_DT_F16 && adt != TS_DT_BF16) return fail(TS_ERR_INVALID_ARG, "%s: bad adt %d", what, adt);
    if (H <= 0 || H % kBlockK) return fail(TS_ERR_UNSUPPORTED, "%s: H=%d must be a positive multiple of 32", what, H);
    if (H > 12288) return fail(TS_ERR_UNSUPPORTED, "%s: H=%d above 12288", what, H);
    if (rmsnorm != 0 && rmsnorm != 1) return fail(TS_ERR_INVALID_ARG, "%s: rmsnorm must be 0 or 1", what);
    if (T > 0 && (!x || !W_r)) return fail(TS_ERR_INVALID_ARG, "%s: x or W_r is NULL", what);
    if (!aligned(W_r, 16)) return fail(TS_ERR_INVALID_ARG, "%s: W_r must be 16-byte aligned", what);
    if (T > 0 && rmsnorm && !xn_out) return fail(TS_ERR_INVALID_ARG, "%s: rmsnorm needs xn_out", what);
    if (!(eps >= 0.0f)) return fail(TS_ERR_INVALID_ARG, "%s: eps must be >= 0", what);
    RouteArgs a{};
    a.x = x;
    a.Wr = W_r;
    a.bias = router_bias;
    a.scale = per_expert_scale;
    a.xn_out = xn_out;
    a.logits_out = logits_out;
    a.idx = idx;
    a.w = w;
    a.T = T;
    a.H = H;
    a.E = E;
    a.k = k;
    a.mode = mode;
    a.adt = adt;
    a.rmsnorm = rmsnorm;
    a.eps = eps;
    return route_common(a, static_cast<cudaStream_t>(stream), what);
}

ts_status ts_moe_build_routes(const int32_t* idx, int32_t T, int32_t E, int32_t k, int32_t* off,
                              int32_t* perm, int32_t* inv, void* stream) {
    g_err.clear();
    const char* what = "ts_moe_build_routes";
    if (T < 0 || k < 1 || E < 1) return fail(TS_ERR_INVALID_ARG, "%s: bad T/E/k", what);
    if (E > kMaxExperts) return fail(TS_ERR_UNSUPPORTED, "%s: E=%d above %d", what, E, kMaxExperts);
    if (static_cast<long long>(T) * k > (1ll << 24))
        return fail(TS_ERR_UNSUPPORTED, "%s: T*k above 2^24", what);
    if (!off || (T > 0 && (!idx || !perm || !inv))) return fail(TS_ERR_INVALID_ARG, "%s: NULL pointer", what);
    cudaError_t e = launch_build_routes(idx, T, E, k, off, perm, inv, nullptr,
                                        static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, what);
    return TS_OK;
}

size_t ts_moe_workspace_size(int32_t T, int32_t k, const ts_moe_experts* ex,
                             const ts_moe_experts* shared) {
    if (!ex || T < 0 || k < 1 || ex->E < 1 || ex->H <= 0 || ex->I <= 0) return 0;
    if (shared && (shared->I <= 0)) return 0;
    // Decode-sized calls (T*k <= 64) also carry split-K partials, so a smaller batch can need
    // more than a larger one: the size returned serves every call with up to T tokens.
    size_t need = ws_layout(T, k, ex, shared).total;
    const int tsplit = 64 / k;
    if (T > tsplit && tsplit > 0) need = std::max(need, ws_layout(tsplit, k, ex, shared).total);
    const int tdec = std::min(tsplit, static_cast<int>(kMxdTokens));   // block-scaled decode kernels
    if (T > tdec && tdec > 0) need = std::max(need, ws_layout(tdec, k, ex, shared).total);
    return need;
}

// The forward; with `fold` (ts_moe_route_forward) the router runs first, and does the decode
// kernels' prep as well when they take the call.  With `tail` (ts_moe_forward_tail) the GEMV
// phase 2 with the fused combine also runs the Gemma sandwich tail (*tail_done set), else the
// caller launches it.
static ts_status forward_impl(const void* x, int32_t adt, int32_t T, const ts_moe_experts* ex,
                              const int32_t* idx, const float* w, int32_t k,
                              const ts_moe_experts* shared, void* y, float* y_f32, void* ws,
                              size_t ws_bytes, int32_t path, void* stream, RouteArgs* fold,
                              const TailArgs* tail = nullptr, bool* tail_done = nullptr) {
    const char* what = fold ? "ts_moe_route_forward" : tail ? "ts_moe_forward_tail" : "ts_moe_forward";
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (adt != TS_DT_F16 && adt != TS_DT_BF16) return fail(TS_ERR_INVALID_ARG, "%s: bad adt %d", what, adt);
    if (T < 0) return fail(TS_ERR_INVALID_ARG, "%s: T=%d < 0", what, T);
    ts_status s = check_experts(ex, "ts_moe_forward: experts", adt);
    if (s != TS_OK) return s;
    if (k < 1 || k > ex->E) return fail(TS_ERR_INVALID_ARG, "%s: k=%d outside 1..E=%d", what, k, ex->E);
    if (shared) {
        s = check_experts(shared, "ts_moe_forward: shared expert", adt);
        if (s != TS_OK) return s;
        if (shared->E != 1 || shared->H != ex->H)
            return fail(TS_ERR_INVALID_ARG, "%s: shared expert needs E=1 and H=%d", what, ex->H);
    }
    if (path < TS_PATH_AUTO || path > TS_PATH_GEMM_DEQUANT) return fail(TS_ERR_INVALID_ARG, "%s: bad path %d", what, path);
    if (static_cast<long long>(T) * k > (1ll << 24)) return fail(TS_ERR_UNSUPPORTED, "%s: T*k above 2^24", what);
    if (T == 0) return TS_OK;
    if (!x || !idx || !w || !y) return fail(TS_ERR_INVALID_ARG, "%s: x/idx/w/y is NULL", what);
    if (!aligned(x, 16) || !aligned(y, 16) || !aligned(y_f32, 16))
        return fail(TS_ERR_INVALID_ARG, "%s: x, y and y_f32 must be 16-byte aligned", what);
    const WsLayout L = ws_layout(T, k, ex, shared);
    if (!ws) return fail(TS_ERR_WORKSPACE, "%s: workspace is NULL", what);
    if (!aligned(ws, 256)) return fail(TS_ERR_WORKSPACE, "%s: workspace must be 256-byte aligned", what);
    if (ws_bytes < L.total) return fail(TS_ERR_WORKSPACE, "%s: workspace %zu bytes < %zu", what, ws_bytes, L.total);
    const bool gemm_fmt = (ex->fmt == FMT_BF16 && adt == TS_DT_BF16) ||
                          (ex->fmt == FMT_F16 && adt == TS_DT_F16);
    const bool gemm_shape = ex->H % 64 == 0 && ex->I % 64 == 0;
    const bool quant_gemm = ex->fmt == FMT_MXFP4;
    // block-scaled MMA: MXFP4 weights with their tensor-core blobs, bf16 activations (two e4m3
    // terms hold a bf16 value exactly; an f16 value needs more)
    const bool mx_ok = quant_gemm && adt == TS_DT_BF16 && ex->gateup_mx && ex->down_mx;
    if ((path == TS_PATH_GEMM && !mx_ok && !((gemm_fmt || quant_gemm) && gemm_shape)) ||
        (path == TS_PATH_GEMM_DEQUANT && !((gemm_fmt || quant_gemm) && gemm_shape)))
        return fail(TS_ERR_UNSUPPORTED,
                    "%s: the tensor-core path serves MXFP4 weights or 16-bit weights of the "
                    "activation type, with H %% 64 == 0 and I %% 64 == 0 (or MXFP4 with its "
                    "tensor-core blobs and bf16 activations) (fmt=%d adt=%d H=%d I=%d)",
                    what, ex->fmt, adt, ex->H, ex->I);
    // decode batches (T <= 8, their workspace regions present) take the block-scaled decode
    // kernels (route tables built inside, combine fused into the last) on "gemm", and on "auto"
    // from 3 tokens (measured on GB300 with the router in front: the streaming GEMV is faster at
    // T = 1, level at T = 2, slower from T = 4)
    const bool use_mxd = mx_ok && L.dcnt_bytes > 0 &&
                         (path == TS_PATH_GEMM || (path == TS_PATH_AUTO && T >= kMxdAutoMinT));
    const bool use_mx = mx_ok && (path == TS_PATH_GEMM || (path == TS_PATH_AUTO && T > 8));
    const bool use_gemm = use_mx || path == TS_PATH_GEMM || path == TS_PATH_GEMM_DEQUANT ||
                          (path == TS_PATH_AUTO && T > 8 && (gemm_fmt || quant_gemm) && gemm_shape);

    unsigned char* W = static_cast<unsigned char*>(ws);
    int* status = reinterpret_cast<int*>(W + L.status);
    int32_t* off = reinterpret_cast<int32_t*>(W + L.off);
    int32_t* perm = reinterpret_cast<int32_t*>(W + L.perm);
    int32_t* inv = reinterpret_cast<int32_t*>(W + L.inv);

    cudaError_t e = cudaSuccess;
    if (fold) {
        if (use_mxd) {
            // the router launch also does the decode kernels' prep
            fold->mxd_xs = W + L.dxs;
            fold->mxd_cnt = reinterpret_cast<int*>(W + L.dcnt);
            fold->mxd_ncnt = static_cast<int>(L.dcnt_bytes / 4);
        }
        s = route_common(*fold, st, "ts_moe_route_forward: router");
        if (s != TS_OK) return s;
    }
    if (use_mxd) return forward_mxd(x, T, ex, idx, w, k, shared, y, y_f32, W, L, st, fold != nullptr);
    if (use_gemm || static_cast<long long>(T) * k > 512)   // else built inside the GEMV kernels
        e = launch_build_routes(idx, T, ex->E, k, off, perm, inv, status, st);
    if (e == cudaSuccess) e = phase_mark(0, st);
    if (e != cudaSuccess) return cuda_fail(e, "ts_moe_forward: route list");

    if (use_mx) {
        const int sms = num_sms_current();
        if (sms <= 0) return fail(TS_ERR_CUDA, "%s: no CUDA device", what);
        const int Tk = T * k;
        uint8_t* xq = W + L.xq;
        uint8_t* xsf = W + L.xsf;
        // both phases in one launch unless K is split (decode-sized calls)
        const bool one_launch = L.max_split <= 1;
        int* hrdy = reinterpret_cast<int*>(W + L.hrdy);
        e = launch_mx_split_rows(static_cast<const uint16_t*>(x), perm, k, ex->H, Tk, xq, xsf, hrdy,
                                 one_launch ? Tk + 1 : 0, st);
        if (e == cudaSuccess) e = phase_mark(0, st);
        if (e != cudaSuccess) return cuda_fail(e, "ts_moe_forward: activation split");
        MxArgs M{};
        M.phase = 0;
        M.act = ex->act;
        M.limit = ex->swiglu_limit;
        M.alpha = ex->swiglu_alpha;
        M.w = static_cast<const uint8_t*>(ex->gateup_mx);
        M.b0 = static_cast<const uint16_t*>(ex->gate_b);
        M.b1 = static_cast<const uint16_t*>(ex->up_b);
        M.R = ex->I;
        M.K = ex->H;
        M.E = ex->E;
        M.bq = xq;
        M.bsf = xsf;
        M.rows_in = Tk;
        M.hq = W + L.hq;
        M.hsf = W + L.hsf;
        M.off = off;
        M.perm = perm;
        M.status = status;
        M.max_split = L.max_split;
        M.part = L.max_split > 1 ? reinterpret_cast<float*>(W + L.part) : nullptr;
        M.cnt = L.max_split > 1 ? reinterpret_cast<int*>(W + L.tcnt) : nullptr;
        MxArgs M1 = M;
        M1.phase = 1;
        M1.w = static_cast<const uint8_t*>(ex->down_mx);
        M1.b0 = static_cast<const uint16_t*>(ex->down_b);
        M1.b1 = nullptr;
        M1.R = ex->H;
        M1.K = ex->I;
        M1.bq = W + L.hq;
        M1.bsf = W + L.hsf;
        M1.hq = nullptr;
        M1.hsf = nullptr;
        M1.e_out = reinterpret_cast<float*>(W + L.e);
        if (L.max_split > 1) M1.cnt = reinterpret_cast<int*>(W + L.tcnt) + L.tcnt_n;
        if (one_launch) {
            e = launch_mx_fused(M, M1, hrdy, sms, st);
            if (e == cudaSuccess) e = phase_mark(1, st);
            if (e == cudaSuccess) e = phase_mark(3, st);
            if (e != cudaSuccess) return cuda_fail(e, "ts_moe_forward: block-scaled phases");
        } else {
            e = cudaMemsetAsync(W + L.tcnt, 0, 2 * L.tcnt_n * 4, st);
            if (e == cudaSuccess) e = launch_mx_gemm(M, sms, st);
            if (e == cudaSuccess) e = phase_mark(1, st);
            if (e != cudaSuccess) return cuda_fail(e, "ts_moe_forward: block-scaled phase 1");
            e = launch_mx_gemm(M1, sms, st);
            if (e == cudaSuccess) e = phase_mark(3, st);
            if (e != cudaSuccess) return cuda_fail(e, "ts_moe_forward: block-scaled phase 2");
        }
    } else if (use_gemm) {
        const int sms = num_sms_current();
        if (sms <= 0) return fail(TS_ERR_CUDA, "%s: no CUDA device", what);
        const int Tk = T * k;
        uint16_t* xs = reinterpret_cast<uint16_t*>(W + L.xs);
        float* xinv = quant_gemm ? reinterpret_cast<float*>(W + L.xinv) : nullptr;

        if (quant_gemm)
            e = launch_gather_rows_f16(static_cast<const uint16_t*>(x), adt, perm, k, ex->H, Tk, xs,
                                       xinv, st);
        else
            e = launch_gather_rows(static_cast<const uint16_t*>(x), perm, k, ex->H, Tk, xs, st);
        if (e == cudaSuccess) e = phase_mark(0, st);
        if (e != cudaSuccess) return cuda_fail(e, "ts_moe_forward: gather");
        GemmArgs G{};
        G.phase = 0;
        G.quant = quant_gemm ? 1 : 0;
        G.ab_bf16 = (!quant_gemm && adt == TS_DT_BF16) ? 1 : 0;
        G.act = ex->act;
        G.limit = ex->swiglu_limit;
        G.alpha = ex->swiglu_alpha;
        G.adt = adt;
        G.w0 = ex->gate;
        G.w1 = ex->up;
        G.mat_bytes = matrix_bytes(ex->fmt, ex->I, ex->H);
        G.b0 = static_cast<const uint16_t*>(ex->gate_b);
        G.b1 = static_cast<const uint16_t*>(ex->up_b);
        G.R = ex->I;
        G.K = ex->H;
        G.E = ex->E;
        G.act_in = xs;
        G.rows_in = Tk;
        G.out = W + L.h;
        G.off = off;
        G.perm = perm;
        G.status = status;
        G.col_scale = xinv;
        G.max_split = L.max_split;
        G.part = L.max_split > 1 ? reinterpret_cast<float*>(W + L.part) : nullptr;
        G.cnt = L.max_split > 1 ? reinterpret_cast<int*>(W + L.tcnt) : nullptr;
        if (L.max_split > 1) e = cudaMemsetAsync(W + L.tcnt, 0, 2 * L.tcnt_n * 4, st);
        if (e == cudaSuccess) e = launch_tc_gemm(G, sms, st);
        if (e == cudaSuccess) e = phase_mark(1, st);
        if (e != cudaSuccess) return cuda_fail(e, "ts_moe_forward: tensor-core phase 1");
        G.phase = 1;
        G.w0 = ex->down;
        G.w1 = nullptr;
        G.mat_bytes = matrix_bytes(ex->fmt, ex->H, ex->I);
        G.b0 = static_cast<const uint16_t*>(ex->down_b);
        G.b1 = nullptr;
        G.R = ex->H;
        G.K = ex->I;
        G.act_in = W + L.h;
        G.out = W + L.e;
        if (L.max_split > 1) G.cnt = reinterpret_cast<int*>(W + L.tcnt) + L.tcnt_n;
        if (quant_gemm) {
            uint16_t* h16 = reinterpret_cast<uint16_t*>(W + L.h16);
            float* hinv = reinterpret_cast<float*>(W + L.hinv);
            e = launch_h_to_f16(reinterpret_cast<const uint16_t*>(W + L.h), adt, ex->I, Tk, h16, hinv, st);
            if (e != cudaSuccess) return cuda_fail(e, "ts_moe_forward: h to f16");
            G.act_in = h16;
            G.col_scale = hinv;
        }
        e = launch_tc_gemm(G, sms, st);
        if (e == cudaSuccess) e = phase_mark(3, st);
        if (e != cudaSuccess) return cuda_fail(e, "ts_moe_forward: tensor-core phase 2");
    }

    // Decode-sized GEMV calls build the route list inside the expert kernels and fuse the
    // combine into phase 2 (fewer launches); the order is routed phase 1, shared phase 1,
    // shared phase 2 (the combine's seed), routed phase 2 (+ combine).
    const bool fused = !use_gemm && static_cast<long long>(T) * k <= 512;
    int* cmb = reinterpret_cast<int*>(W + L.cmb);
    GemvArgs g{};
    g.act = ex->act;
    g.limit = ex->swiglu_limit;
    g.alpha = ex->swiglu_alpha;
    g.adt = adt;
    g.T = T;
    g.k = k;
    g.E = ex->E;
    g.status = status;
    g.fmt = ex->fmt;
    g.phase = 0;
    g.w0 = static_cast<const uint8_t*>(ex->gate);
    g.w1 = static_cast<const uint8_t*>(ex->up);
    g.b0 = static_cast<const uint16_t*>(ex->gate_b);
    g.b1 = static_cast<const uint16_t*>(ex->up_b);
    g.R = ex->I;
    g.K = ex->H;
    g.mat_bytes = matrix_bytes(ex->fmt, ex->I, ex->H);
    g.in = static_cast<const uint16_t*>(x);
    g.out = W + L.h;
    g.off = fused ? nullptr : off;
    g.perm = fused ? nullptr : perm;
    g.idx = fused ? idx : nullptr;
    g.dense = 0;
    g.cmb_mode = fused ? 1 : 0;
    g.cmb_cnt = cmb;
    g.cmb_n = ex->H / kRowTile;
    g.stall = g_wait_test;
    g_wait_test = 0;
    if (!use_gemm) {
        if ((s = launch_gemv_checked(g, st, "ts_moe_forward: expert phase 1")) != TS_OK) return s;
        if ((e = phase_mark(1, st)) != cudaSuccess) return cuda_fail(e, "ts_moe_forward: phase event");
    }
    GemvArgs gs = g;
    if (shared) {
        gs.fmt = shared->fmt;
        gs.act = shared->act;
        gs.limit = shared->swiglu_limit;
        gs.alpha = shared->swiglu_alpha;
        gs.E = 1;
        gs.w0 = static_cast<const uint8_t*>(shared->gate);
        gs.w1 = static_cast<const uint8_t*>(shared->up);
        gs.b0 = static_cast<const uint16_t*>(shared->gate_b);
        gs.b1 = static_cast<const uint16_t*>(shared->up_b);
        gs.R = shared->I;
        gs.K = shared->H;
        gs.mat_bytes = matrix_bytes(shared->fmt, shared->I, shared->H);
        gs.out = W + L.hs;
        gs.off = nullptr;
        gs.perm = nullptr;
        gs.idx = nullptr;
        gs.dense = 1;
        gs.k = 1;
        gs.cmb_mode = 0;
        gs.stall = 0;
        if ((s = launch_gemv_checked(gs, st, "ts_moe_forward: shared expert phase 1")) != TS_OK) return s;
        if ((e = phase_mark(2, st)) != cudaSuccess) return cuda_fail(e, "ts_moe_forward: phase event");
        gs.phase = 1;
        gs.w0 = static_cast<const uint8_t*>(shared->down);
        gs.w1 = nullptr;
        gs.b0 = static_cast<const uint16_t*>(shared->down_b);
        gs.b1 = nullptr;
        gs.R = shared->H;
        gs.K = shared->I;
        gs.mat_bytes = matrix_bytes(shared->fmt, shared->H, shared->I);
        gs.in = reinterpret_cast<const uint16_t*>(W + L.hs);
        gs.out = W + L.s;
        if ((s = launch_gemv_checked(gs, st, "ts_moe_forward: shared expert phase 2")) != TS_OK) return s;
        if ((e = phase_mark(4, st)) != cudaSuccess) return cuda_fail(e, "ts_moe_forward: phase event");
    }
    // phase 2: down projection -> e (f32, by route id)
    g.phase = 1;
    g.w0 = static_cast<const uint8_t*>(ex->down);
    g.w1 = nullptr;
    g.b0 = static_cast<const uint16_t*>(ex->down_b);
    g.b1 = nullptr;
    g.R = ex->H;
    g.K = ex->I;
    g.mat_bytes = matrix_bytes(ex->fmt, ex->H, ex->I);
    g.in = reinterpret_cast<const uint16_t*>(W + L.h);
    g.out = W + L.e;
    g.cmb_mode = fused ? 2 : 0;
    g.stall = 0;
    g.w = w;
    g.seed = shared ? reinterpret_cast<const float*>(W + L.s) : nullptr;
    g.y = y;
    g.y_f32 = y_f32;
    // (the fused tail moves 8 elements at a time: its buffers must be 16-byte aligned)
    if (fused && tail && !use_gemm && aligned(tail->h1, 16) && aligned(tail->x, 16) &&
        aligned(tail->w_post2, 16) && aligned(tail->w_post, 16)) {
        g.tail = *tail;
        g.tail.y = static_cast<uint16_t*>(y);
        g.tdone = cmb + ex->H / kRowTile;
        if (tail_done) *tail_done = true;
    }
    if (!use_gemm) {
        if ((s = launch_gemv_checked(g, st, "ts_moe_forward: expert phase 2")) != TS_OK) return s;
        if ((e = phase_mark(3, st)) != cudaSuccess) return cuda_fail(e, "ts_moe_forward: phase event");
    }
    if (!fused) {
        CombineArgs c{};
        c.e = reinterpret_cast<const float*>(W + L.e);
        c.w = w;
        c.seed = shared ? reinterpret_cast<const float*>(W + L.s) : nullptr;
        c.y = y;
        c.y_f32 = y_f32;
        c.T = T;
        c.H = ex->H;
        c.k = k;
        c.adt = adt;
        e = launch_combine(c, st);
        if (e != cudaSuccess) return cuda_fail(e, "ts_moe_forward: combine");
    }
    if ((e = phase_mark(5, st)) != cudaSuccess) return cuda_fail(e, "ts_moe_forward: phase event");
    return TS_OK;
}

ts_status ts_moe_forward_path(const void* x, int32_t adt, int32_t T, const ts_moe_experts* ex,
                              const int32_t* idx, const float* w, int32_t k,
                              const ts_moe_experts* shared, void* y, float* y_f32, void* ws,
                              size_t ws_bytes, int32_t path, void* stream) {
    g_err.clear();
    return forward_impl(x, adt, T, ex, idx, w, k, shared, y, y_f32, ws, ws_bytes, path, stream, nullptr);
}

// argument checks of the sandwich tail (ts_moe_gemma_tail, ts_moe_forward_tail)
static ts_status check_tail_args(const TailArgs& a, const char* what) {
    if (a.adt != TS_DT_F16 && a.adt != TS_DT_BF16) return fail(TS_ERR_INVALID_ARG, "%s: bad adt %d", what, a.adt);
    if (a.T < 0 || a.H <= 0) return fail(TS_ERR_INVALID_ARG, "%s: bad T=%d / H=%d", what, a.T, a.H);
    if (a.H % 32 || a.H > kTailMaxH)
        return fail(TS_ERR_UNSUPPORTED, "%s: H=%d must be a multiple of 32 and at most %d", what, a.H, kTailMaxH);
    if (a.T == 0) return TS_OK;
    if (!a.y || !a.h1 || !a.x || !a.w_post2 || !a.w_post) return fail(TS_ERR_INVALID_ARG, "%s: NULL pointer", what);
    if (a.y == a.h1 || a.y == a.x || a.h1 == a.x)
        return fail(TS_ERR_INVALID_ARG, "%s: y, h1 and x must be distinct", what);
    if (!aligned(a.y, 2) || !aligned(a.h1, 2) || !aligned(a.x, 2) || !aligned(a.w_post2, 2) || !aligned(a.w_post, 2))
        return fail(TS_ERR_INVALID_ARG, "%s: pointers must be 2-byte aligned", what);
    return TS_OK;
}

ts_status ts_moe_forward_tail(const void* x, int32_t adt, int32_t T, const ts_moe_experts* ex,
                              const int32_t* idx, const float* w, int32_t k,
                              const ts_moe_experts* shared, void* y, float* y_f32, void* ws,
                              size_t ws_bytes, int32_t path, void* h1, void* xres,
                              const void* w_post2, const void* w_post, float layer_scalar, float eps,
                              void* stream) {
    g_err.clear();
    const char* what = "ts_moe_forward_tail";
    if (!ex) return fail(TS_ERR_INVALID_ARG, "%s: experts is NULL", what);
    TailArgs a{};
    a.y = static_cast<uint16_t*>(y);
    a.h1 = static_cast<uint16_t*>(h1);
    a.x = static_cast<uint16_t*>(xres);
    a.w_post2 = static_cast<const uint16_t*>(w_post2);
    a.w_post = static_cast<const uint16_t*>(w_post);
    a.layer_scalar = layer_scalar;
    a.eps = eps;
    a.adt = adt;
    a.T = T;
    a.H = ex->H;
    ts_status s = check_tail_args(a, what);
    if (s != TS_OK) return s;
    bool done = false;
    s = forward_impl(x, adt, T, ex, idx, w, k, shared, y, y_f32, ws, ws_bytes, path, stream, nullptr, &a, &done);
    if (s != TS_OK || done || T == 0) return s;
    cudaError_t e = launch_gemma_tail(a, static_cast<cudaStream_t>(stream));
    if (e == cudaSuccess) e = phase_mark(7, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, what);
    return TS_OK;
}

ts_status ts_moe_route_forward(const void* x, int32_t adt, int32_t T, const void* W_r,
                               int32_t rmsnorm, float eps, const float* router_bias,
                               const float* per_expert_scale, int32_t k, int32_t mode,
                               const ts_moe_experts* ex, const ts_moe_experts* shared,
                               void* xn_out, int32_t* idx, float* w, void* y, float* y_f32,
                               void* ws, size_t ws_bytes, int32_t path, void* stream) {
    g_err.clear();
    const char* what = "ts_moe_route_forward";
    if (!ex) return fail(TS_ERR_INVALID_ARG, "%s: experts is NULL", what);
    RouteArgs a{};
    a.x = x;
    a.Wr = W_r;
    a.bias = router_bias;
    a.scale = per_expert_scale;
    a.xn_out = xn_out;
    a.idx = idx;
    a.w = w;
    a.T = T;
    a.H = ex->H;
    a.E = ex->E;
    a.k = k;
    a.mode = mode;
    a.adt = adt;
    a.rmsnorm = rmsnorm;
    a.eps = eps;
    ts_status s = check_router_args(a, what);
    if (s != TS_OK) return s;
    if (T > 0 && (!idx || !w)) return fail(TS_ERR_INVALID_ARG, "%s: idx/w output is NULL", what);
    // the experts read the normalised rows when the router normalises
    return forward_impl(rmsnorm ? xn_out : x, adt, T, ex, idx, w, k, shared, y, y_f32, ws, ws_bytes,
                        path, stream, &a);
}

ts_status ts_moe_forward(const void* x, int32_t adt, int32_t T, const ts_moe_experts* ex,
                         const int32_t* idx, const float* w, int32_t k,
                         const ts_moe_experts* shared, void* y, float* y_f32, void* ws,
                         size_t ws_bytes, void* stream) {
    return ts_moe_forward_path(x, adt, T, ex, idx, w, k, shared, y, y_f32, ws, ws_bytes,
                               TS_PATH_AUTO, stream);
}

ts_status ts_moe_set_wait_test(int32_t mode) {
    g_err.clear();
    if (mode != 0 && mode != 1) return fail(TS_ERR_INVALID_ARG, "ts_moe_set_wait_test: mode=%d not 0 or 1", mode);
    g_wait_test = mode;
    return TS_OK;
}

ts_status ts_moe_set_phase_events(void* const* events, int32_t n) {
    g_err.clear();
    if (n < 0 || n > 8) return fail(TS_ERR_INVALID_ARG, "ts_moe_set_phase_events: n=%d outside 0..8", n);
    if (!events) n = 0;
    for (int i = 0; i < 8; ++i) g_phase_ev[i] = (i < n) ? static_cast<cudaEvent_t>(events[i]) : nullptr;
    g_phase_n = n;
    return TS_OK;
}

ts_status ts_moe_gemma_tail(void* y, void* h1, void* x, const void* w_post2, const void* w_post,
                            float layer_scalar, float eps, int32_t adt, int32_t T, int32_t H,
                            void* stream) {
    g_err.clear();
    const char* what = "ts_moe_gemma_tail";
    TailArgs a{};
    a.y = static_cast<uint16_t*>(y);
    a.h1 = static_cast<uint16_t*>(h1);
    a.x = static_cast<uint16_t*>(x);
    a.w_post2 = static_cast<const uint16_t*>(w_post2);
    a.w_post = static_cast<const uint16_t*>(w_post);
    a.layer_scalar = layer_scalar;
    a.eps = eps;
    a.adt = adt;
    a.T = T;
    a.H = H;
    ts_status s = check_tail_args(a, what);
    if (s != TS_OK || T == 0) return s;
    cudaError_t e = launch_gemma_tail(a, static_cast<cudaStream_t>(stream));
    if (e == cudaSuccess) e = phase_mark(7, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, what);
    return TS_OK;
}

ts_status ts_moe_device_status(void* ws, int32_t* code, void* stream) {
    g_err.clear();
    if (!ws || !code) return fail(TS_ERR_INVALID_ARG, "ts_moe_device_status: NULL pointer");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, ws, sizeof(v), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e == cudaSuccess) e = cudaMemsetAsync(ws, 0, sizeof(int32_t), st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "ts_moe_device_status");
    *code = v;
    return TS_OK;
}

}  // extern "C"

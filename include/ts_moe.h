/*
 * ts_moe.h -- C ABI of the GB300 (sm_103a) routed-expert (MoE) layer library, libts_moe.so.
 *
 * The layer (source pages: docs.rs, turbospark-runtime 0.3.0):
 *   1. router logits r = m @ router, per-expert router bias added to the logits
 *      (gpt-oss routed-expert pass, src/families/gptoss/moe.rs, module header;
 *       Llama/Mixtral decode flow, src/families/llama/mod.rs, module header "one decoder layer")
 *   2. top-k on the RAW biased logits, softmax over the selected k only, no renormalisation,
 *      optionally times per_expert_scale (gptoss/moe.rs module header: llama.cpp SOFTMAX_WEIGHT
 *      gating, router_topk_gemma4's contract); MiniMax: biased-sigmoid selection with unbiased
 *      weights (llama/mod.rs module header)
 *   3. route list: tokens grouped by expert (Gemma-4 batched routed prefill,
 *      src/families/gemma4/moe_batch.rs, module header and encode_routes)
 *   4. per-expert gated FFN over MXFP4, INT4-affine or f16/bf16 weights with optional per-expert
 *      biases and the clamped SwiGLU (gptoss/moe.rs module header "THE CLAMPED SwiGLU AND THE
 *      PER-EXPERT BIASES"; phase1/phase2 encoders)
 *   5. weighted sum of expert outputs in router-rank slot order, seeded with zeros or the
 *      shared expert (gptoss/moe.rs module header "slot order is the ROUTER'S RANKING",
 *      "zero_hidden is the residual input"; moe_batch.rs "Seed from ZEROS")
 *
 * Conventions shared by every entry point
 *   - Pointers marked "device" are CUDA device (or managed) addresses on the current device;
 *     "host" pointers are ordinary host memory.  The caller owns every buffer; the library
 *     keeps no pointer after a call returns and allocates no device memory per call (scratch
 *     lives in the caller's workspace, sized by ts_moe_workspace_size).
 *   - Calls taking a stream are asynchronous on that stream (a cudaStream_t; NULL = the legacy
 *     default stream): no host synchronisation, no device-to-host readback.  They may be
 *     captured into a CUDA graph.
 *   - Arguments are validated on the host before anything is launched.  A call that cannot be
 *     served returns TS_ERR_INVALID_ARG or TS_ERR_UNSUPPORTED and launches nothing (the layer
 *     refuses rather than falls back, as the Gemma-4 batched prefill refuses unsupported
 *     layouts).  ts_last_error() returns a message for the last failing call on this thread.
 *   - 16-bit activations (ts_dtype) are IEEE binary16 or bfloat16, row-major, rows contiguous.
 *   - Token t's k routes have ids r = t*k + s, s = 0..k-1; slot s holds the s-th ranked expert.
 */
#ifndef TS_MOE_H
#define TS_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TS_OK = 0,
    TS_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misaligned pointer, bad enum      */
    TS_ERR_UNSUPPORTED = 2,  /* valid request outside what the kernels serve (e.g. E>256) */
    TS_ERR_CUDA = 3,         /* a CUDA runtime call failed (message has the CUDA error)   */
    TS_ERR_TIMEOUT = 4,      /* a kernel gave up waiting (reported via ts_moe_device_status) */
    TS_ERR_WORKSPACE = 5     /* workspace null or smaller than ts_moe_workspace_size      */
} ts_status;

/* Routing modes (step 2). */
typedef enum {
    TS_ROUTE_SOFTMAX_K = 0,        /* key = logit + bias; w = softmax over the k selected keys */
    TS_ROUTE_SIGMOID_BIASED = 1,   /* s = sigmoid(logit); key = s + bias; w = s / sum_k s      */
    TS_ROUTE_SOFTMAX_K_SCALED = 2  /* as SOFTMAX_K, then w *= per_expert_scale[expert]         */
} ts_route_mode;

typedef enum { TS_DT_F16 = 0, TS_DT_BF16 = 1 } ts_dtype;

/* Expert weight formats.  Every matrix is output-major ("[rows][K]", K contiguous):
 * gate/up are [E][I][H], down is [E][H][I].
 *   TS_W_F16 / TS_W_BF16: 16-bit elements in that canonical layout, used directly.
 *   TS_W_MXFP4 / TS_W_INT4_AFFINE: the device-packed layout written by ts_moe_pack from
 *     the canonical codes + scales (see ts_moe_pack).                                      */
typedef enum { TS_W_F16 = 0, TS_W_BF16 = 1, TS_W_MXFP4 = 2, TS_W_INT4_AFFINE = 3 } ts_wfmt;

/* Gated-FFN activations, h = act(g) * u with g, u the gate/up projections (+ biases):
 *   SILU_GLU:       h = silu(g) * u                                    (use_silu, llama/mod.rs)
 *   GELU_TANH_GLU:  h = 0.5 g (1 + tanh(sqrt(2/pi)(g + 0.044715 g^3))) * u   (gelu-tanh)
 *   GPTOSS_SWIGLU:  g = min(g, limit); u = clamp(u, -limit, limit);
 *                   h = g * sigmoid(alpha * g) * (u + 1)                (Mxfp4Activation::GPT_OSS) */
typedef enum { TS_ACT_SILU_GLU = 0, TS_ACT_GELU_TANH_GLU = 1, TS_ACT_GPTOSS_SWIGLU = 2 } ts_act;

/* Path selection for ts_moe_forward_path. */
typedef enum {
    TS_PATH_AUTO = 0,  /* 3 <= T <= 8 tokens: the block-scaled decode kernels when they apply
                          (MXFP4 with its tensor-core blobs, bf16 activations, T*k <= 64,
                          k <= 8, H <= 4096), else (and for T <= 2) the GEMV path.  T > 8: the
                          tensor-core grouped GEMM
                          when the format has one (MXFP4, or f16/bf16 weights of the activation
                          type) and H, I are multiples of 64, else the GEMV path              */
    TS_PATH_GEMV = 1,  /* streaming GEMV kernels (any T)                                        */
    TS_PATH_GEMM = 2,  /* tcgen05 grouped GEMM.  MXFP4 weights with bf16 activations and the
                          tensor-core blobs present (gateup_mx/down_mx): block-scaled MMA
                          (kind::mxf8f6f4, e2m1 x e4m3 with e8m0 scales; activations split
                          exactly into two e4m3 terms), through the decode kernels (prep, gate/up,
                          down + combine; stream-K over every SM) when T <= 8 and they apply.
                          Otherwise as TS_PATH_GEMM_DEQUANT                                    */
    TS_PATH_GEMM_DEQUANT = 3  /* tcgen05 grouped GEMM on 16-bit operands: 16-bit weights of the
                          activation type as they are; MXFP4 weights dequantised to f16 in
                          shared memory, exact for e8m0 scales 2^-23..2^13 (a block outside
                          that range makes ts_moe_device_status report TS_ERR_UNSUPPORTED)    */
} ts_path;

/* One set of experts (routed experts, or the shared expert with E = 1).
 * Requirements: H, I multiples of 32 (and of 16 rows); 1 <= E <= 256.
 * gate_b/up_b ([E][I]) and down_b ([E][H]) are bfloat16 device arrays or NULL (no bias;
 * the pages derive has_bias from a non-zero bias offset).  swiglu_limit / swiglu_alpha are
 * read only for TS_ACT_GPTOSS_SWIGLU (gpt-oss: 7.0 and 1.702).
 * gateup_mx/down_mx: MXFP4 only, optional (NULL = absent): the same matrices in the
 * tensor-core layout written by ts_moe_pack_mx (256-byte aligned device blobs; gateup_mx holds
 * gate and up together, pair = 1); with them, bf16 activations take the block-scaled
 * tensor-core path for more than 8 tokens.                                                   */
typedef struct ts_moe_experts {
    int32_t fmt;   /* ts_wfmt */
    int32_t act;   /* ts_act  */
    int32_t E, H, I;
    const void* gate;  /* device */
    const void* up;    /* device */
    const void* down;  /* device */
    const void* gate_b;
    const void* up_b;
    const void* down_b;
    float swiglu_limit;
    float swiglu_alpha;
    const void* gateup_mx; /* device, ts_moe_pack_mx layout with pair = 1, or NULL */
    const void* down_mx;   /* device, ts_moe_pack_mx layout with pair = 0, or NULL */
} ts_moe_experts;

/* ------------------------------------------------------------------------------------------ */
/* Weight packing (one-time, untimed).                                                         */
/* ------------------------------------------------------------------------------------------ */

/* Bytes of the packed layout of `nmat` matrices of R rows x K columns in format fmt
 * (MXFP4 or INT4_AFFINE; R % 16 == 0, K % 32 == 0).  Returns 0 for unsupported arguments.
 * The repack walk of the gpt-oss pages (moe_offsets_from_layout) is the counterpart. */
size_t ts_moe_packed_bytes(int32_t fmt, int32_t nmat, int32_t R, int32_t K);

/* Packs canonical quantised weights into the device layout the kernels stream.
 *   codes  device uint8 [nmat][R][K/2]; element 2j in the low nibble of byte j, 2j+1 in the high.
 *          MXFP4: e2m1 codes (bit 3 sign).  INT4_AFFINE: unsigned q in 0..15.
 *   scales device.  MXFP4: uint8 e8m0 [nmat][R][K/32], value 2^(byte-127), one per 32
 *          consecutive K elements.  INT4_AFFINE: [nmat][R][K/32] pairs of binary16
 *          (scale, min), w = q*scale + min.
 *   packed device, packed_bytes >= ts_moe_packed_bytes(...), 16-byte aligned.
 * Async on `stream`.  Packed layout: per 16-row tile, per 32-column block, 256 code bytes
 * ordered for the GEMV fragments, then the block's 16 scale bytes (MXFP4) or 64 scale/min
 * bytes (INT4); tiles of one matrix are contiguous, matrices follow each other.          */
ts_status ts_moe_pack(int32_t fmt, int32_t nmat, int32_t R, int32_t K, const void* codes,
                      const void* scales, void* packed, size_t packed_bytes, void* stream);

/* Bytes of the tensor-core layout of `nmat` MXFP4 matrices of R rows x K columns (pair = 0),
 * or of `nmat` gate/up pairs (pair = 1); R % 32 == 0, K % 32 == 0.  0 for unsupported
 * arguments.                                                                                  */
size_t ts_moe_packed_mx_bytes(int32_t pair, int32_t nmat, int32_t R, int32_t K);

/* Writes the tensor-core layout of canonical MXFP4 weights (codes and e8m0 scales exactly as
 * ts_moe_pack takes them) for the block-scaled MMA path.  pair = 1: codes0/scales0 are the gate
 * matrices and codes1/scales1 the up matrices, stored together; pair = 0: one matrix set
 * (codes1/scales1 ignored).  G = 1 + pair matrices per expert.
 *   - codes [nmat][KG][G][R][64 bytes], KG = ceil(K / 128): for each group of 128 columns the
 *     128 codes of a row (canonical nibble order), gate and up of a row group side by side, so
 *     one tensor copy fetches a stage of both; zero codes past K;
 *   - at the next 256-byte boundary, the scales in 512-byte atoms [nmat][U][KG][2][512],
 *     U = ceil(R / 128) for pairs (atom pair = gate, up) or ceil(R / 256) otherwise (atom pair =
 *     the two 128-row halves of a 256-row block); row r and block b of an atom at byte
 *     16*(r%32) + 4*(r/32) + b (the order in which tcgen05.cp spreads them over TMEM); scales of
 *     rows or blocks past the matrix are 1.0.
 *   blob device, 256-byte aligned, blob_bytes >= ts_moe_packed_mx_bytes(...).  Async on
 * `stream`; one-time work (untimed), like the pages' repack walk.                            */
ts_status ts_moe_pack_mx(int32_t pair, int32_t nmat, int32_t R, int32_t K, const void* codes0,
                         const void* scales0, const void* codes1, const void* scales1, void* blob,
                         size_t blob_bytes, void* stream);

/* ------------------------------------------------------------------------------------------ */
/* Steps 1-2: routing.                                                                         */
/* ------------------------------------------------------------------------------------------ */

/* Top-k + weights from precomputed raw router logits (router_topk_gemma4's contract plus the
 * bias placement of the gpt-oss pass).
 *   logits           device f32 [T][E] (raw: no bias)
 *   router_bias      device f32 [E] or NULL; SOFTMAX modes: added to the logits before top-k;
 *                    SIGMOID_BIASED: added to sigmoid(logit) for selection only
 *   per_expert_scale device f32 [E]; required for SOFTMAX_K_SCALED, ignored otherwise
 *   idx              device int32 [T][k] out: experts in rank order (largest key first,
 *                    equal keys -> lower expert id)
 *   w                device f32 [T][k] out: routing weights in the same slot order
 * 1 <= k <= E <= 256, T >= 0 (T == 0 launches nothing).                                   */
ts_status ts_moe_route(const float* logits, const float* router_bias,
                       const float* per_expert_scale, int32_t T, int32_t E, int32_t k,
                       int32_t mode, int32_t* idx, float* w, void* stream);

/* Fused optional RMSNorm + router GEMV + bias + top-k + weights (steps 1-2 in one kernel).
 *   x        device adt [T][H]
 *   W_r      device adt [E][H] (router weights, output-major)
 *   rmsnorm  0 or 1: if 1, x is first normalised, xn = adt(x / sqrt(mean(x^2) + eps)), and xn
 *            (written to xn_out, required) feeds the router; the plainest reading of the
 *            Gemma configuration is that xn is also the experts' input
 *   logits_out device f32 [T][E] or NULL: raw logits (before bias)
 * The logit of (t, e) is a fixed-order f32 sum: lane l of a warp accumulates
 * fmaf(x[l+32j], W_r[e][l+32j], p) over j, then an xor butterfly (16,8,4,2,1) adds the lanes;
 * the bias is one further f32 add.  H % 32 == 0.  Other arguments as ts_moe_route.         */
ts_status ts_moe_router_route(const void* x, int32_t adt, int32_t T, int32_t H, const void* W_r,
                              int32_t E, int32_t rmsnorm, float eps, const float* router_bias,
                              const float* per_expert_scale, int32_t k, int32_t mode,
                              void* xn_out, float* logits_out, int32_t* idx, float* w,
                              void* stream);

/* ------------------------------------------------------------------------------------------ */
/* Step 3: route list.                                                                         */
/* ------------------------------------------------------------------------------------------ */

/* Groups the T*k routes by expert with a deterministic counting sort.
 *   idx   device int32 [T][k], every entry in 0..E-1
 *   off   device int32 [E+1] out: off[e] = number of routes to experts below e
 *   perm  device int32 [T*k] out: route ids grouped by expert, ascending id within an expert
 *   inv   device int32 [T*k] out: inv[r] = position of route r in perm
 * Bit-exact (integer work).  Rejects T*k > 2^24.
 * A route whose expert id lies outside 0..E-1 is left out (inv[r] = -1; inside
 * ts_moe_forward it also sets TS_ERR_INVALID_ARG in the device status word), and perm
 * positions off[E]..T*k-1 hold route id 0.  Whatever idx holds, even if it changes while the
 * kernel runs, every perm entry is a route id in 0..T*k-1, so the kernels that read the list
 * stay inside their buffers.                                                              */
ts_status ts_moe_build_routes(const int32_t* idx, int32_t T, int32_t E, int32_t k, int32_t* off,
                              int32_t* perm, int32_t* inv, void* stream);

/* ------------------------------------------------------------------------------------------ */
/* Steps 3-5: experts + combine.                                                               */
/* ------------------------------------------------------------------------------------------ */

/* Workspace bytes ts_moe_forward needs for up to T tokens, k routes per token, these experts
 * and (optional, may be NULL) shared expert: a workspace of this size serves every call with
 * T or fewer tokens (a small batch can need more than a larger one, since decode-sized calls
 * keep split-K partials).  Returns 0 for invalid arguments.                               */
size_t ts_moe_workspace_size(int32_t T, int32_t k, const ts_moe_experts* ex,
                             const ts_moe_experts* shared);

/* The expert half of the layer:
 *   y[t] = adt( seed[t] + sum_{s=0..k-1} w[t][s] * expert_{idx[t][s]}(x[t]) )
 * with the sum taken in f32 in slot order (acc = acc + w*e, one rounded multiply and one
 * rounded add per slot), seed = shared expert output (f32) or zeros.  Each expert output is
 *   e = W_d (h) + b_d,   h = adt( act(W_g x + b_g, W_u x + b_u) )
 * with f32 accumulation; h is rounded to the activation type (the pages' acts buffer is
 * 16-bit) before the down projection.
 *   x       device adt [T][H]
 *   ex      host pointer to the routed experts' descriptor (device weight pointers inside)
 *   idx, w  device int32 / f32 [T][k] (e.g. from ts_moe_route / ts_moe_router_route)
 *   shared  host pointer to a dense shared expert (E = 1, same H) or NULL
 *   y       device adt [T][H] out
 *   y_f32   device f32 [T][H] out or NULL: the f32 sum before the final rounding
 *   ws      device workspace, 256-byte aligned, ws_bytes >= ts_moe_workspace_size(...)
 * Deterministic: the same inputs give the same bits run to run.  T == 0 launches nothing. */
ts_status ts_moe_forward(const void* x, int32_t adt, int32_t T, const ts_moe_experts* ex,
                         const int32_t* idx, const float* w, int32_t k,
                         const ts_moe_experts* shared, void* y, float* y_f32, void* ws,
                         size_t ws_bytes, void* stream);

/* As ts_moe_forward with an explicit path (ts_path).  TS_PATH_GEMM with a format that has no
 * tensor-core kernel returns TS_ERR_UNSUPPORTED.                                            */
ts_status ts_moe_forward_path(const void* x, int32_t adt, int32_t T, const ts_moe_experts* ex,
                              const int32_t* idx, const float* w, int32_t k,
                              const ts_moe_experts* shared, void* y, float* y_f32, void* ws,
                              size_t ws_bytes, int32_t path, void* stream);

/* The whole routed layer from x: ts_moe_router_route, then ts_moe_forward_path on its idx / w
 * (and on xn when rmsnorm is 1), with the same arguments, meaning and results: idx and w are
 * written as ts_moe_router_route writes them, y as ts_moe_forward writes it.  When the
 * block-scaled decode kernels take the call (MXFP4 experts, bf16, T <= 8; see TS_PATH_AUTO /
 * TS_PATH_GEMM), the router launch also does their prep (the x rows, after the RMSNorm when
 * on, split into the kernels' e4m3 image; their counters zeroed), so the layer without a
 * shared expert is two launches; otherwise the router launch is followed by the forward's.
 * H and E come from the experts; x is H columns wide.  T == 0 launches nothing.          */
ts_status ts_moe_route_forward(const void* x, int32_t adt, int32_t T, const void* W_r,
                               int32_t rmsnorm, float eps, const float* router_bias,
                               const float* per_expert_scale, int32_t k, int32_t mode,
                               const ts_moe_experts* ex, const ts_moe_experts* shared,
                               void* xn_out, int32_t* idx, float* w, void* y, float* y_f32,
                               void* ws, size_t ws_bytes, int32_t path, void* stream);

/* As ts_moe_forward (automatic path), for callers that cannot allocate device memory: instead
 * of a caller-provided workspace it uses a scratch array that lives in the library's own device
 * memory (16 MiB per GPU, held until the process exits).  The source pages have no counterpart;
 * it exists because some callers own all device memory themselves or must not allocate while
 * they run.  It calls no allocator (no cudaMalloc, no cudaFree).
 *   - Calls that need more scratch than 16 MiB (ts_moe_workspace_size) return
 *     TS_ERR_WORKSPACE and launch nothing.
 *   - The first call on each device (and the first after a device reset) looks up the
 *     scratch's device address (cudaGetSymbolAddress) and caches it for the current CUDA
 *     context; make that first call before any stream capture.
 *   - Every call on a device shares the one scratch array and it keeps the last call's
 *     contents; the call clears what must start at zero (the device status word) itself.
 *     Calls that overlap on the GPU (different streams, no ordering between them) race on the
 *     scratch and produce wrong results: order them on one stream or use ts_moe_forward.
 *   - Device-side failures of the call (a bounded wait that expired, an expert id outside
 *     0..E-1, an MXFP4 scale outside the tensor-core path's range) are reported through the
 *     scratch's status word: read them with ts_moe_noalloc_device_status.
 * Other arguments as ts_moe_forward.                                                        */
ts_status ts_moe_forward_noalloc(const void* x, int32_t adt, int32_t T, const ts_moe_experts* ex,
                                 const int32_t* idx, const float* w, int32_t k,
                                 const ts_moe_experts* shared, void* y, float* y_f32,
                                 void* stream);

/* Reads (synchronously, on `stream`) and clears the device status word of the scratch that
 * ts_moe_forward_noalloc uses on the current device: *code = 0 when the last such call (every
 * call clears the word when it starts) reported nothing, else a TS_ERR_* value.  The source
 * pages have no counterpart; it is the status read of ts_moe_device_status for callers that
 * hold no workspace.                                                                        */
ts_status ts_moe_noalloc_device_status(int32_t* code, void* stream);

/* ------------------------------------------------------------------------------------------ */
/* After step 5 (Gemma layers): the sandwich tail.                                             */
/* ------------------------------------------------------------------------------------------ */

/* The per-token tail that the Gemma-4 batched routed prefill (src/families/gemma4/moe_batch.rs)
 * encodes after the fused phase 2, in place on three 16-bit [T][H] buffers:
 *   y  <- adt(rms(y)  * w_post2)   rms(v) = v * (1 / sqrt(mean(v^2) + eps)), w bf16
 *   h1 <- adt(h1 + y)              the dense branch plus the normalised routed output
 *   f   = adt(rms(h1) * w_post)
 *   x  <- adt(adt(x + f) * layer_scalar)
 * Every step is one rounded f32 op (the weight multiply reads as (v * r) * w); the sum of
 * squares takes the fixed order of ts_moe_router_route's RMSNorm, so the result is bit-exact.
 *   y, h1, x          device adt [T][H], read and written (three distinct buffers)
 *   w_post2, w_post   device bf16 [H]
 *   adt               TS_DT_F16 or TS_DT_BF16
 * H must be a multiple of 32 and at most 8192 (TS_ERR_UNSUPPORTED otherwise).  T == 0 launches
 * nothing.                                                                                  */
ts_status ts_moe_gemma_tail(void* y, void* h1, void* x, const void* w_post2, const void* w_post,
                            float layer_scalar, float eps, int32_t adt, int32_t T, int32_t H,
                            void* stream);

/* ------------------------------------------------------------------------------------------ */
/* Diagnostics.                                                                                */
/* ------------------------------------------------------------------------------------------ */

/* ts_moe_forward_path followed by ts_moe_gemma_tail(y, h1, xres, w_post2, w_post,
 * layer_scalar, eps, adt, T, H) in one call, with the same arguments, meaning and results (every
 * output bit-exact against the two calls; y ends normalised, y_f32 keeps the f32 sum before the
 * final rounding).  When the streaming GEMV with its fused combine takes the call (decode sizes,
 * T * k <= 512), the tail runs inside that launch: once every row tile of y is combined, CTA b
 * runs the tail of tokens b, b + grid, ... (the Gemma-4 batched routed prefill page encodes the
 * tail right after the fused phase 2).  Otherwise the tail is a launch of its own after the forward.  xres
 * is the residual stream x of the tail;
 * checks as ts_moe_forward_path and ts_moe_gemma_tail (H from the experts).               */
ts_status ts_moe_forward_tail(const void* x, int32_t adt, int32_t T, const ts_moe_experts* ex,
                              const int32_t* idx, const float* w, int32_t k,
                              const ts_moe_experts* shared, void* y, float* y_f32, void* ws,
                              size_t ws_bytes, int32_t path, void* h1, void* xres,
                              const void* w_post2, const void* w_post, float layer_scalar, float eps,
                              void* stream);

/* Message of the last failing call on this thread ("" if none).  Valid until the next call. */
const char* ts_last_error(void);

/* Reads (synchronously, on `stream`) and clears the device status word that kernels of
 * ts_moe_forward set when a bounded wait expires or a device-side check fails.
 * *code = 0 when nothing was reported; otherwise a TS_ERR_* value.                          */
ts_status ts_moe_device_status(void* ws, int32_t* code, void* stream);

/* Exercises the bounded waits (test use; the pages' counterpart is the refusal convention:
 * fail with a status, never hang or degrade).  mode 1: the next ts_moe_forward* call on this
 * thread that runs the streaming GEMV expert path or the block-scaled decode kernels withholds
 * the first weight copy of its phase-1 launch, so that launch's consumer warps wait on a copy
 * that never arrives; their bounded wait (about 2^31 SM clocks, a second) runs out, they
 * report TS_ERR_TIMEOUT through the device status word (ts_moe_device_status), the launch
 * drains the copies it did issue and returns, and the call's outputs are meaningless.  The
 * setting is consumed by the next forward call whichever path it takes.  mode 0 clears it.  */
ts_status ts_moe_set_wait_test(int32_t mode);

/* Per-phase timing (the counterpart of the pages' PhaseCounters / per-command-buffer GPU
 * time).  Registers, for the calling thread, up to 8 cudaEvent_t handles (host array, copied;
 * n == 0 or events == NULL clears).  While set, ts_moe_forward* records events[i] on its
 * stream right after launching phase i, for the phases that exist:
 *   0 route list, 1 expert phase 1 (gate/up + activation), 2 shared-expert phase 1,
 *   3 expert phase 2 (down), 4 shared-expert phase 2, 5 combine;
 * ts_moe_route / ts_moe_router_route record events[6] after the router kernel and
 * ts_moe_gemma_tail records events[7] after the tail.
 * On a capturing stream the events become graph event-record nodes, so graph replays record
 * them too.  The caller owns the events.                                                     */
ts_status ts_moe_set_phase_events(void* const* events, int32_t n);

/* Library version as "major.minor.patch". */
const char* ts_moe_version(void);

#ifdef __cplusplus
}
#endif
#endif /* TS_MOE_H */

// internal.h -- launchers and parameter blocks shared between the host API (api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace tsmoe {

enum { FMT_F16 = 0, FMT_BF16 = 1, FMT_MXFP4 = 2, FMT_INT4 = 3 };
enum { ACT_SILU = 0, ACT_GELU = 1, ACT_GPTOSS = 2 };
enum { MODE_SOFTMAX_K = 0, MODE_SIGMOID_BIASED = 1, MODE_SOFTMAX_K_SCALED = 2 };

// error codes written to the device status word (match ts_status)
enum { DEV_ERR_INVALID = 1, DEV_ERR_UNSUPPORTED = 2, DEV_ERR_TIMEOUT = 4 };

constexpr int kMaxExperts = 256;
constexpr int kRowTile = 16;   // rows per GEMV unit (the mma M)
constexpr int kBlockK = 32;    // K elements per quantisation block / GEMV block

// bytes of one packed 16-row x 32-column block: 256 code bytes + scale bytes
__host__ __device__ constexpr int packed_block_bytes(int fmt) {
    return fmt == FMT_MXFP4 ? 256 + 16 : 256 + 64;
}

// ------------------------------------------------------------------------------------------
// routing
// ------------------------------------------------------------------------------------------
struct RouteArgs {
    const void* x;          // [T][H] adt (router_route) or nullptr
    const void* Wr;         // [E][H] adt
    const float* logits_in; // [T][E] (route from logits) or nullptr
    const float* bias;      // [E] or nullptr
    const float* scale;     // [E] or nullptr
    void* xn_out;           // [T][H] adt or nullptr
    float* logits_out;      // [T][E] or nullptr
    int32_t* idx;           // [T][k]
    float* w;               // [T][k]
    int T, H, E, k, mode, adt, rmsnorm;
    float eps;
    // the block-scaled decode kernels' prep, folded into the router launch (nullptr: none): the
    // token rows (after the RMSNorm, when on) split into their x image, rows T..7 zeroed, and the
    // decode counters zeroed (T <= 8, bf16, H <= 4096)
    uint8_t* mxd_xs;
    int* mxd_cnt;
    int mxd_ncnt;
};
cudaError_t launch_router(const RouteArgs& a, cudaStream_t s);
cudaError_t launch_build_routes(const int32_t* idx, int T, int E, int k, int32_t* off,
                                int32_t* perm, int32_t* inv, int* status, cudaStream_t s);

// the Gemma sandwich tail (tail.cu): in place on y, h1, x [T][H] 16-bit
constexpr int kTailMaxH = 8192;
struct TailArgs {
    uint16_t* y;            // routed output -> normalised routed output
    uint16_t* h1;           // dense branch -> h1 + normalised routed output
    uint16_t* x;            // residual stream -> (x + normalised h1) * layer_scalar
    const uint16_t* w_post2;   // [H] bf16 post_feedforward_layernorm_2
    const uint16_t* w_post;    // [H] bf16 post_feedforward_layernorm
    float layer_scalar, eps;
    int adt, T, H;
};
cudaError_t launch_gemma_tail(const TailArgs& a, cudaStream_t s);

// ------------------------------------------------------------------------------------------
// streaming GEMV (decode) path
// ------------------------------------------------------------------------------------------
struct GemvArgs {
    int fmt, phase;               // phase 0: gate/up + act -> h ; 1: down -> e (f32)
    int act;
    float limit, alpha;
    const uint8_t* w0;            // gate (phase 0) or down (phase 1), expert 0
    const uint8_t* w1;            // up (phase 0) or nullptr
    size_t mat_bytes;             // bytes per expert matrix
    const uint16_t* b0;           // bias of w0 ([E][R] bf16) or nullptr
    const uint16_t* b1;           // bias of w1 or nullptr
    int R, K;                     // rows per expert matrix, reduction length
    int E;
    const uint16_t* in;           // phase 0: x [T][K]; phase 1: h [T*k][K] (by route id)
    int adt;
    void* out;                    // phase 0: h [T*k][R] adt ; phase 1: e [T*k][R] f32
    const int32_t* off;           // [E+1] (routed) or nullptr (dense)
    const int32_t* perm;          // [T*k] (routed) or nullptr
    int T, k;                     // tokens, routes per token (dense: k = 1)
    int dense;                    // 1: every token routed to expert 0 (shared expert)
    int tg;                       // tokens per unit group (1..8)
    int* status;
    const int32_t* idx;           // [T][k]: build the route list in the kernel (T*k <= 512), or
                                  // nullptr: use off/perm
    int cmb_mode;                 // 0 none; 1 (phase 1) clear cmb_cnt; 2 (phase 2) fused combine
    int* cmb_cnt;                 // per-row-tile unit counters of phase 2 (H / 16 of them)
    int cmb_n;                    // number of counters (H / 16)
    const float* w;               // combine: routing weights [T][k]
    const float* seed;            // combine: shared-expert output [T][H] or nullptr
    void* y;                      // combine: [T][H] adt
    float* y_f32;                 // combine: [T][H] or nullptr
    int stall;                    // test setting: withhold the first weight copy (see api.cu)
    // the Gemma sandwich tail inside phase 2's fused combine (tail.T > 0; tail.y = y): once
    // tdone (counted over the grid) reaches the tile count, CTA b runs the tail of tokens b,
    // b + grid, ...
    TailArgs tail;
    int* tdone;                   // row tiles combined (cleared by phase 1 with the counters)
};
cudaError_t launch_gemv(const GemvArgs& a, int num_sms, cudaStream_t s);

struct CombineArgs {
    const float* e;        // [T*k][H] f32 by route id
    const float* w;        // [T][k]
    const float* seed;     // [T][H] f32 or nullptr
    void* y;               // [T][H] adt
    float* y_f32;          // [T][H] or nullptr
    int T, H, k, adt;
};
cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s);


// ------------------------------------------------------------------------------------------
// tensor-core grouped GEMM (prefill) path
// ------------------------------------------------------------------------------------------
struct GemmArgs {
    int phase;                    // 0: gate/up + act -> h (route-list order); 1: down -> e
    int ab_bf16;                  // mma operand type: 1 bf16, 0 f16
    int act;
    float limit, alpha;
    int adt;
    const void* w0;               // canonical 16-bit weights: phase 0 gate, phase 1 down
    const void* w1;               // phase 0 up
    const uint16_t* b0;           // bias of w0 ([E][R] bf16) or nullptr
    const uint16_t* b1;           // bias of w1 or nullptr
    int R, K, E;                  // rows per expert matrix, reduction length, experts
    const void* act_in;           // activations in route-list order [rows_in][K]
    int rows_in;                  // T*k
    void* out;                    // phase 0: h [T*k][R] (route-list order); 1: e [T*k][R] by id
    const int32_t* off;           // [E+1]
    const int32_t* perm;          // [T*k]
    int* status;
    int quant;                    // 1: w0/w1 are packed MXFP4 (dequantised to f16 in smem)
    size_t mat_bytes;             // packed bytes per expert matrix (quant)
    const float* col_scale;       // quant: per route-list position, undoes the f16 prescale
    int max_split;                // > 1: K may be split in up to this many parts (needs part/cnt)
    float* part;                  // split-K partials [max_split][rows_in][2][R] f32
    int* cnt;                     // split-K group counters (zero before the launch)
};
cudaError_t launch_tc_gemm(const GemmArgs& a, int num_sms, cudaStream_t s);
cudaError_t launch_gather_rows(const uint16_t* x, const int32_t* perm, int k, int H, int n,
                               uint16_t* xs, cudaStream_t s);
cudaError_t launch_gather_rows_f16(const uint16_t* x, int adt, const int32_t* perm, int k, int H,
                                   int n, uint16_t* xs, float* inv, cudaStream_t s);
cudaError_t launch_h_to_f16(const uint16_t* h, int adt, int I, int n,
                            uint16_t* h16, float* inv, cudaStream_t s);

// ------------------------------------------------------------------------------------------
// block-scaled tensor-core path for MXFP4 weights and bf16 activations (gemm_mx.cu)
// ------------------------------------------------------------------------------------------
// Tensor-core MXFP4 blob of one group of expert matrices [E][R][K]: G = 2 for gate and up of
// the same rows (phase 1 uses them together), G = 1 for down.
//   codes  [E][KG][G][R][64 B], KG = ceil(K / 128): the 128 codes of one row and one group of
//          128 columns (64 bytes), zero codes past K;
//   scales at the next 256-byte boundary: [E][U][KG][2][512 B] atoms, U = ceil(R / 128) for
//          G = 2 (atom pair = gate, up) and U = ceil(R / 256) for G = 1 (atom pair = the two
//          128-row halves of a 256-row block); row r and block b of an atom at byte
//          16 (r % 32) + 4 (r / 32) + b, 1.0 (127) for rows or blocks past the matrix.
__host__ __device__ inline int mx_kg(int K) { return (K + 127) / 128; }
__host__ __device__ inline int mx_units(int G, int R) { return G == 2 ? (R + 127) / 128 : (R + 255) / 256; }
__host__ __device__ inline size_t mx_codes_bytes(int G, int E, int R, int K) {
    return static_cast<size_t>(E) * mx_kg(K) * G * R * 64;
}
__host__ __device__ inline size_t mx_sf_offset(int G, int E, int R, int K) {
    return (mx_codes_bytes(G, E, R, K) + 255) / 256 * 256;
}
__host__ __device__ inline size_t mx_blob_bytes(int G, int E, int R, int K) {
    return mx_sf_offset(G, E, R, K) + static_cast<size_t>(E) * mx_units(G, R) * mx_kg(K) * 1024;
}
// bytes per row of an activation scale array: one e8m0 per 32 columns, rows padded to whole
// groups of four blocks
__host__ __device__ inline int mx_sf_row(int K) { return mx_kg(K) * 4; }

struct MxArgs {
    int phase;                    // 0: gate/up + act -> h (split); 1: down -> e (f32 by route id)
    int act;
    float limit, alpha;
    const uint8_t* w;             // phase 0: gate + up blob (G = 2); phase 1: down blob (G = 1)
    const uint16_t* b0;           // phase 0 gate bias / phase 1 down bias ([E][R] bf16) or nullptr
    const uint16_t* b1;           // phase 0 up bias or nullptr
    int R, K, E;                  // rows per expert matrix, reduction length, experts
    const uint8_t* bq;            // activations, route-list order: two e4m3 planes [2][rows_in][K]
    const uint8_t* bsf;           // their e8m0 block scales (of the first plane), transposed:
                                  // word [g][p] holds the scales of blocks 4g..4g+3 of row p
    int rows_in;                  // T*k
    uint8_t* hq;                  // phase 0 out: h split into two e4m3 planes [2][rows_in][R]
    uint8_t* hsf;                 // phase 0 out: scales of h, transposed like bsf
    float* e_out;                 // phase 1 out: e [T*k][R] by route id
    const int32_t* off;           // [E+1]
    const int32_t* perm;          // [T*k]
    int* status;
    int max_split;                // > 1: K may be split (needs part/cnt)
    float* part;                  // split-K partials [max_split][rows_in][2][R] f32
    int* cnt;                     // split-K group counters (zero before the launch)
};
cudaError_t launch_mx_gemm(const MxArgs& a, int num_sms, cudaStream_t s);
// both phases in one cooperative launch (a0.phase 0, a1.phase 1, no split K): the CTAs draw
// items from one counter (hrdy[rows_in]); phase-1 items wait for the h of their (touched expert,
// route tile), counted in hrdy[0 .. rows_in) (all rows_in + 1 zero before the launch)
cudaError_t launch_mx_fused(const MxArgs& a0, const MxArgs& a1, int* hrdy, int num_sms, cudaStream_t s);
// bf16 rows (route-list order, row p = x[perm[p] / k]; perm nullptr: row p = x[p]) split into two
// e4m3 planes [2][n][K] and e8m0 block scales, words [mx_sf_row(K) / 4][n] of four blocks; block
// 0 also zeroes zero[0 .. nzero)
cudaError_t launch_mx_split_rows(const uint16_t* x, const int32_t* perm, int k, int K, int n,
                                 uint8_t* q, uint8_t* sf, int* zero, int nzero, cudaStream_t s);
// canonical codes / scales of one matrix (G = 1) or of gate and up (G = 2: codes1/scales1 = up)
cudaError_t launch_mx_pack(int G, int nmat, int R, int K, const uint8_t* codes0, const uint8_t* scales0,
                           const uint8_t* codes1, const uint8_t* scales1, uint8_t* blob, cudaStream_t s);

// Decode batches (T <= 8) with MXFP4 experts and bf16 activations (gemm_mxd.cu): a prep launch
// (x split, counters zeroed), then one persistent cooperative launch running both phases over
// the touched experts, every touched expert's weights streamed once.
constexpr int kMxdTokens = 8;        // token rows per term plane
constexpr int kMxdMaxTouched = 64;   // touched experts <= min(E, T*k) <= 64
constexpr int kMxdMaxCtas = 256;     // stream-K partial slots
constexpr int kMxdMaxK = 8;          // routes per token
constexpr int kMxdAutoMinT = 3;      // TS_PATH_AUTO takes the decode kernels from this many tokens
constexpr int kMxdMaxH = 4096;       // the prep kernel takes a token row per 256 threads x 16
constexpr int kMxdBStage = 2 * kMxdTokens * 128;        // one K stage of B: 16 rows x 128 bytes
constexpr int kMxdHImage = kMxdBStage + 512;            // + its scale atom
constexpr size_t kMxdPartFloats = 2 * 128 * 8;          // one parked part: 2 x 128 rows x 8 tokens
struct MxdArgs {
    int act;
    float limit, alpha;
    const uint8_t* wgu;           // tensor-core blob of gate + up (G = 2)
    const uint8_t* wd;            // tensor-core blob of down (G = 1)
    const uint16_t* bg;           // biases [E][I], [E][I], [E][H] bf16, or nullptr
    const uint16_t* bu;
    const uint16_t* bd;
    int H, I, E, T, k;            // hidden, intermediate, experts, tokens, routes per token
    const int32_t* idx;           // [T][k]
    const float* wr;              // routing weights [T][k]
    const uint16_t* x;            // prep: [T][H] bf16
    uint8_t* xs;                  // x image: [ceil(H/128)][16][128 B] + a 512 B scale atom
    uint8_t* hs;                  // h images: [min(E, T*k)][ceil(I/128)][kMxdHImage]
    float* e_out;                 // e [T*k][H] f32 by route id
    const float* seed;            // combine seed [T][H] f32 or nullptr
    void* y;                      // [T][H] bf16
    float* y_f32;                 // [T][H] or nullptr
    float* part;                  // stream-K partials [kMxdMaxCtas][2 phases][2][kMxdPartFloats]
    int* cnt;                     // counters, zero on entry (the prep kernel zeroes ncnt of them):
    int ncnt;                     //   [hcnt: nt][tcnt0: nt*MB0*4][tcnt1: nt*MB1*4][rbcnt: MB1*4]
    int* status;
    int stall;                    // test setting: the first stage's copies are withheld
};
cudaError_t launch_mxd(const MxdArgs& a, int num_sms, cudaStream_t s);
cudaError_t launch_mxd_prep(const MxdArgs& a, cudaStream_t s);

// records the thread's ts_last_error() message (defined in api.cu); returns `status`
int record_error_code(int status, const char* msg);

cudaError_t launch_pack(int fmt, int nmat, int R, int K, const uint8_t* codes,
                        const uint8_t* scales, uint8_t* packed, cudaStream_t s);

}  // namespace tsmoe

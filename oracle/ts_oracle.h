/*
 * ts_oracle.h -- plain, slow CPU oracle for the routed-expert (MoE) layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this code: only tests/, __graft_entry__.smoke() and bench.py's
 * cpu_baseline / --impl reference legs use it.  It shares no code, header,
 * table or constant with the CUDA library under
 * mixture_experts_routed_logits_gb300/csrc.
 *
 * Source pages (docs.rs, turbospark-runtime 0.3.0):
 *   [gptoss/moe.rs]    src/families/gptoss/moe.rs        (module header; encode_gpt_oss_layer_moe)
 *   [gemma4/moe_batch] src/families/gemma4/moe_batch.rs  (module header; encode_gemma4_layer_routed_moe_batched)
 *   [llama/mod.rs]     src/families/llama/mod.rs         (module header "one decoder layer")
 *
 * Canonical layouts (the oracle reads only these):
 *   activations  x[T][H] 16-bit (adt: 0 = f16, 1 = bf16), raw IEEE bits
 *   router       W_r[E][H] in adt, logits[T][E] f32
 *   weights      "output-major": gate/up [E][I][H], down [E][H][I], K contiguous
 *     fmt 0 F16 / 1 BF16 : 16-bit elements
 *     fmt 2 MXFP4        : codes uint8 [E][R][K/2], element 2j in the low nibble,
 *                          element 2j+1 in the high nibble; one e8m0 scale byte per
 *                          32 consecutive K elements: scales uint8 [E][R][K/32]
 *     fmt 3 INT4_AFFINE  : codes uint8 [E][R][K/2] (same nibble order, q in 0..15);
 *                          per 32 consecutive K elements one (scale, min) pair of
 *                          f16 bits: sm uint16 [E][R][K/32][2]; w = q*scale + min
 *   biases       bf16 [E][R] or NULL
 */
#ifndef TS_ORACLE_H
#define TS_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { OR_F16 = 0, OR_BF16 = 1, OR_MXFP4 = 2, OR_INT4 = 3 };
enum { OR_ACT_SILU = 0, OR_ACT_GELU_TANH = 1, OR_ACT_GPTOSS = 2 };
enum { OR_MODE_SOFTMAX_K = 0, OR_MODE_SIGMOID_BIASED = 1, OR_MODE_SOFTMAX_K_SCALED = 2 };

typedef struct {
    int fmt, act, E, H, I;
    const void *gate, *up, *down;          /* codes or 16-bit elements      */
    const void *gate_s, *up_s, *down_s;    /* scales (quantised fmts only)  */
    const uint16_t *gate_b, *up_b, *down_b; /* bf16 biases or NULL          */
    float limit, alpha;                    /* clamped SwiGLU constants       */
} or_experts;

/* scalar format helpers (exposed so the tests can pin them directly) */
double or_f16_to_double(uint16_t b);
double or_bf16_to_double(uint16_t b);
uint16_t or_double_to_f16(double v);   /* round to nearest even */
uint16_t or_double_to_bf16(double v);  /* round to nearest even */
double or_e2m1_value(int code);        /* 4-bit e2m1 code -> value */
double or_e8m0_value(int byte);        /* e8m0 byte -> 2^(byte-127)  */
double or_weight(const or_experts* X, int mat, int e, int row, int col);
float or_dot32f(const float* a, const float* b, int n);
double or_act(int act, double g, double u, float limit, float alpha);

int or_rmsnorm(const uint16_t* x, int T, int H, int adt, float eps, uint16_t* xn);
int or_gemma_tail(uint16_t* y, uint16_t* h1, uint16_t* x, const uint16_t* w_post2,
                  const uint16_t* w_post, float layer_scalar, float eps, int T, int H, int adt);
int or_router_logits(const uint16_t* x, const uint16_t* Wr, int T, int H, int E, int adt,
                     float* logits);
int or_route(const float* logits, const float* bias, const float* scale, int T, int E, int k,
             int mode, int32_t* idx, float* w);
int or_build_routes(const int32_t* idx, int T, int E, int k, int32_t* off, int32_t* perm,
                    int32_t* inv);
int or_expert_ffn(const or_experts* X, int e, const double* xin, int adt, double* h_out,
                  float* e_out);
int or_expert_pre(const or_experts* X, int e, const double* xin, double* g_out, double* u_out,
                  double* sg_out, double* su_out);
void or_act_n(int act, const double* g, const double* u, int n, float limit, float alpha,
              double* out);
int or_moe_forward(const uint16_t* x, int adt, int T, const or_experts* X, const int32_t* idx,
                   const float* w, int k, const or_experts* shared, const int32_t* tokens,
                   int ntok, uint16_t* y, float* y_f32, float* e_routes, int nthreads);

#ifdef __cplusplus
}
#endif
#endif

/*
 * ts_oracle.c -- plain, slow CPU oracle for the routed-expert (MoE) layer.
 *
 * TEST INFRASTRUCTURE ONLY (see ts_oracle.h).  Built with
 *   gcc -std=c11 -O2 -ffp-contract=off [-fopenmp] -shared -fPIC
 * so that every float operation below is one correctly rounded IEEE-754 op.
 *
 * The layer, step by step, as the source pages state it:
 *   a0  optional pre-routing RMSNorm, eps 1e-6     [gemma4/moe_batch] RMS_EPS; [llama/mod.rs] "m = rms_norm(x, ...)"
 *   a1  router logits r = m @ router               [llama/mod.rs] "r = family_topk(m @ router)"
 *   a2  bias added to the logits BEFORE top-k, top-k on the raw biased logits,
 *       softmax over the selected k only, no renormalisation, optionally times
 *       per_expert_scale                           [gptoss/moe.rs] module header, "THE BIAS, BEFORE THE TOP-K"
 *       MiniMax: select on biased sigmoid scores, weight with unbiased ones
 *                                                  [llama/mod.rs] module header
 *   a3  route list (tokens grouped by expert)      [gemma4/moe_batch] encode_routes / route-list kernels
 *   a4  per-expert gated FFN, phase 1, 16-bit acts [gptoss/moe.rs] phase1; [gemma4/moe_batch] acts offset *2 bytes
 *   a5  phase 2 down projection                    [gptoss/moe.rs] phase2
 *   a7  y = residual + sum_slot w[slot]*expert_slot, reduced in slot-index
 *       (= router rank) order, residual = zeros or shared expert
 *                                                  [gptoss/moe.rs] module header "slot order is the ROUTER'S RANKING",
 *                                                  "zero_hidden is the residual input"
 * Where the pages are silent this file takes these readings: top-k ties go to the lower
 * expert id; a logit is lane l's fmaf chain over x[l+32j]*W[e][l+32j] followed by an xor
 * butterfly (16, 8, 4, 2, 1), plus the bias as one more f32 add; the softmax runs over the k
 * selected only; routing weights stay f32; per_expert_scale multiplies the weight, not the
 * selection; the clamped SwiGLU adds the biases before the clamp; h is rounded to the
 * activation type before the down projection, e stays f32, and the combine is f32 in slot
 * order.
 */
#include "ts_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ */
/* 16-bit float formats (IEEE binary16 and bfloat16), written from the */
/* format definitions.                                                  */
/* ------------------------------------------------------------------ */

double or_f16_to_double(uint16_t b) {
    int s = (b >> 15) & 1, e = (b >> 10) & 31, m = b & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);             /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25); /* (1 + m/1024) * 2^(e-15) */
    return s ? -v : v;
}

double or_bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* Round v to a binary format with p significant bits, minimum normal
 * exponent emin, round-half-to-even. */
static double rne_quantize(double v, int p, int emin) {
    if (v == 0.0 || !isfinite(v)) return v;
    int e = ilogb(v);
    if (e < emin) e = emin;
    double q = ldexp(1.0, e - (p - 1));
    return nearbyint(v / q) * q;
}

uint16_t or_double_to_f16(double v) {
    if (isnan(v)) return 0x7E00;
    double r = rne_quantize(v, 11, -14);
    uint16_t s = signbit(r) ? 0x8000 : 0;
    double a = fabs(r);
    if (a > 65504.0) return s | 0x7C00;
    if (a == 0.0) return s;
    if (a < ldexp(1.0, -14)) return s | (uint16_t)(a / ldexp(1.0, -24));
    int e = ilogb(a);
    uint16_t m = (uint16_t)((a / ldexp(1.0, e) - 1.0) * 1024.0);
    return s | (uint16_t)((e + 15) << 10) | m;
}

uint16_t or_double_to_bf16(double v) {
    if (isnan(v)) return 0x7FC0;
    double r = rne_quantize(v, 8, -126);
    /* largest finite bf16 = (2 - 2^-7) * 2^127 */
    if (fabs(r) > ldexp(255.0, 120)) return signbit(r) ? 0xFF80 : 0x7F80;
    float f = (float)r; /* exact: r has <= 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

static double adt_to_double(uint16_t b, int adt) {
    return adt == 0 ? or_f16_to_double(b) : or_bf16_to_double(b);
}
static uint16_t double_to_adt(double v, int adt) {
    return adt == 0 ? or_double_to_f16(v) : or_double_to_bf16(v);
}

/* ------------------------------------------------------------------ */
/* Quantised weight formats.                                            */
/* ------------------------------------------------------------------ */

/* e2m1 (OCP microscaling FP4): bit 3 sign, bits 2..1 exponent (bias 1),
 * bit 0 mantissa.  E == 0 is subnormal: M * 0.5. */
double or_e2m1_value(int code) {
    int s = (code >> 3) & 1, E = (code >> 1) & 3, M = code & 1;
    double mag = (E == 0) ? 0.5 * M : ldexp(1.0 + 0.5 * M, E - 1);
    return s ? -mag : mag;
}

/* e8m0 shared block scale: 2^(byte - 127); 0xFF encodes NaN. */
double or_e8m0_value(int byte) {
    if (byte == 255) return NAN;
    return ldexp(1.0, byte - 127);
}

static const void* mat_codes(const or_experts* X, int mat) {
    return mat == 0 ? X->gate : mat == 1 ? X->up : X->down;
}
static const void* mat_scales(const or_experts* X, int mat) {
    return mat == 0 ? X->gate_s : mat == 1 ? X->up_s : X->down_s;
}
static void mat_dims(const or_experts* X, int mat, int* R, int* K) {
    if (mat == 2) { *R = X->H; *K = X->I; }
    else          { *R = X->I; *K = X->H; }
}

/* One dequantised weight W_mat[e][row][col], exactly, in double. */
double or_weight(const or_experts* X, int mat, int e, int row, int col) {
    int R, K;
    mat_dims(X, mat, &R, &K);
    size_t rowi = (size_t)e * R + row;
    if (X->fmt == OR_F16 || X->fmt == OR_BF16) {
        const uint16_t* w = (const uint16_t*)mat_codes(X, mat);
        return adt_to_double(w[rowi * K + col], X->fmt == OR_F16 ? 0 : 1);
    }
    const uint8_t* c = (const uint8_t*)mat_codes(X, mat);
    uint8_t byte = c[rowi * (K / 2) + col / 2];
    int q = (col & 1) ? (byte >> 4) : (byte & 15);
    size_t blk = rowi * (K / 32) + col / 32;
    if (X->fmt == OR_MXFP4) {
        const uint8_t* s = (const uint8_t*)mat_scales(X, mat);
        return or_e2m1_value(q) * or_e8m0_value(s[blk]);
    }
    /* INT4 affine */
    const uint16_t* sm = (const uint16_t*)mat_scales(X, mat);
    double scale = or_f16_to_double(sm[2 * blk]);
    double mn = or_f16_to_double(sm[2 * blk + 1]);
    return (double)q * scale + mn;
}

/* ------------------------------------------------------------------ */
/* Fixed-order f32 dot product used for the router logits and for the   */
/* RMSNorm sum of squares.  The order is a reading (the pages do not    */
/* state one) chosen so that a 32-lane GPU warp can reproduce it bit    */
/* for bit: lane l runs p = fmaf(a[l+32j], b[l+32j], p) for j = 0,1,..; */
/* then an xor butterfly over offsets 16, 8, 4, 2, 1 adds p_l + p_(l^o).*/
/* ------------------------------------------------------------------ */
float or_dot32f(const float* a, const float* b, int n) {
    float p[32], q[32];
    for (int l = 0; l < 32; ++l) {
        p[l] = 0.0f;
        for (int j = 0; l + 32 * j < n; ++j) p[l] = fmaf(a[l + 32 * j], b[l + 32 * j], p[l]);
    }
    for (int o = 16; o >= 1; o >>= 1) {
        for (int l = 0; l < 32; ++l) q[l] = p[l] + p[l ^ o];
        for (int l = 0; l < 32; ++l) p[l] = q[l];
    }
    return p[0];
}

/* a0: unweighted RMSNorm (RMS_EPS = 1e-6 on [gemma4/moe_batch]): r = 1/sqrt(mean(x^2)+eps),
 * xn = adt(x * r), every step one rounded f32 op. */
int or_rmsnorm(const uint16_t* x, int T, int H, int adt, float eps, uint16_t* xn) {
    if (H % 32) return -1;
    float* xf = (float*)malloc(sizeof(float) * H);
    if (!xf) return -2;
    for (int t = 0; t < T; ++t) {
        for (int j = 0; j < H; ++j) xf[j] = (float)adt_to_double(x[(size_t)t * H + j], adt);
        float ss = or_dot32f(xf, xf, H);
        float ms = ss / (float)H;
        float r = 1.0f / sqrtf(ms + eps);
        for (int j = 0; j < H; ++j) {
            float v = xf[j] * r;
            xn[(size_t)t * H + j] = double_to_adt((double)v, adt);
        }
    }
    free(xf);
    return 0;
}

/* Weighted RMSNorm of one row: out_j = adt((v_j * r) * w_j), r = 1/sqrt(mean(v^2) + eps) with
 * the fixed-order sum above, w bf16, every step one rounded f32 op. */
static void rms_weighted(const float* v, const uint16_t* w, int H, float eps, int adt, uint16_t* out) {
    float ss = or_dot32f(v, v, H);
    float ms = ss / (float)H;
    float r = 1.0f / sqrtf(ms + eps);
    for (int j = 0; j < H; ++j) {
        float a = v[j] * r;
        float b = a * (float)or_bf16_to_double(w[j]);
        out[j] = double_to_adt((double)b, adt);
    }
}

/* The Gemma sandwich tail that follows the routed phase 2 ([gemma4/moe_batch] routed prefill,
 * per token, in place on 16-bit buffers):
 *   y  <- rms_w(y, w_post2)            post_feedforward_layernorm_2
 *   h1 <- adt(h1 + y)                  the dense branch plus the normalised routed output
 *   f   = rms_w(h1, w_post)            post_feedforward_layernorm
 *   x  <- adt(x + f)                   the residual stream
 *   x  <- adt(x * layer_scalar)
 * The weight multiply reads plainly as v * r * w (the pages name the kernel "rms_norm_bf16w"
 * without its body). */
int or_gemma_tail(uint16_t* y, uint16_t* h1, uint16_t* x, const uint16_t* w_post2,
                  const uint16_t* w_post, float layer_scalar, float eps, int T, int H, int adt) {
    if (H % 32) return -1;
    float* v = (float*)malloc(sizeof(float) * H);
    uint16_t* f = (uint16_t*)malloc(sizeof(uint16_t) * H);
    if (!v || !f) { free(v); free(f); return -2; }
    for (int t = 0; t < T; ++t) {
        uint16_t* yt = y + (size_t)t * H;
        uint16_t* ht = h1 + (size_t)t * H;
        uint16_t* xt = x + (size_t)t * H;
        for (int j = 0; j < H; ++j) v[j] = (float)adt_to_double(yt[j], adt);
        rms_weighted(v, w_post2, H, eps, adt, yt);
        for (int j = 0; j < H; ++j) {
            float s = (float)adt_to_double(ht[j], adt) + (float)adt_to_double(yt[j], adt);
            ht[j] = double_to_adt((double)s, adt);
            v[j] = (float)adt_to_double(ht[j], adt);
        }
        rms_weighted(v, w_post, H, eps, adt, f);
        for (int j = 0; j < H; ++j) {
            float s = (float)adt_to_double(xt[j], adt) + (float)adt_to_double(f[j], adt);
            uint16_t xs = double_to_adt((double)s, adt);
            float m = (float)adt_to_double(xs, adt) * layer_scalar;
            xt[j] = double_to_adt((double)m, adt);
        }
    }
    free(v);
    free(f);
    return 0;
}

/* a1: raw router logits (no bias), r[t][e] = sum_h x[t][h] * W_r[e][h] in the fixed order. */
int or_router_logits(const uint16_t* x, const uint16_t* Wr, int T, int H, int E, int adt,
                     float* logits) {
    if (H % 32) return -1;
    float* xf = (float*)malloc(sizeof(float) * H);
    float* wf = (float*)malloc(sizeof(float) * H);
    if (!xf || !wf) { free(xf); free(wf); return -2; }
    for (int t = 0; t < T; ++t) {
        for (int j = 0; j < H; ++j) xf[j] = (float)adt_to_double(x[(size_t)t * H + j], adt);
        for (int e = 0; e < E; ++e) {
            for (int j = 0; j < H; ++j) wf[j] = (float)adt_to_double(Wr[(size_t)e * H + j], adt);
            logits[(size_t)t * E + e] = or_dot32f(xf, wf, H);
        }
    }
    free(xf);
    free(wf);
    return 0;
}

/* "a ranks before b": larger value first, equal values -> lower expert id. */
static int ranks_before(float va, int ia, float vb, int ib) {
    if (va > vb) return 1;
    if (va < vb) return 0;
    return ia < ib;
}

/* a2: selection + weights.
 *  SOFTMAX_K (+_SCALED): key_e = logit_e + bias_e (one f32 add; bias before top-k,
 *    [gptoss/moe.rs] "THE BIAS, BEFORE THE TOP-K"); top-k of the keys; weights are the softmax
 *    over the k selected keys only (no renormalisation), times per_expert_scale in the
 *    SCALED mode ([gemma4/moe_batch] router_topk_gemma4(.., &per_expert_scale)).
 *  SIGMOID_BIASED: s_e = sigmoid(logit_e) in f32, key_e = s_e + bias_e; top-k of the keys;
 *    weights are the unbiased s of the selected, normalised over the k ([llama/mod.rs]
 *    "biased sigmoid scores with unbiased weights").
 * Slot i holds the i-th ranked expert. */
int or_route(const float* logits, const float* bias, const float* scale, int T, int E, int k,
             int mode, int32_t* idx, float* w) {
    if (k < 1 || k > E) return -1;
    float* key = (float*)malloc(sizeof(float) * E);
    float* sg = (float*)malloc(sizeof(float) * E);
    char* taken = (char*)malloc(E);
    if (!key || !sg || !taken) { free(key); free(sg); free(taken); return -2; }
    int rc = 0;
    for (int t = 0; t < T && rc == 0; ++t) {
        const float* l = logits + (size_t)t * E;
        for (int e = 0; e < E; ++e) {
            if (isnan(l[e])) { rc = -3; break; }
            if (mode == OR_MODE_SIGMOID_BIASED) {
                sg[e] = 1.0f / (1.0f + expf(-l[e]));
                key[e] = bias ? sg[e] + bias[e] : sg[e];
            } else {
                key[e] = bias ? l[e] + bias[e] : l[e];
            }
            taken[e] = 0;
        }
        if (rc) break;
        /* top-k by repeated selection of the best remaining key */
        for (int s = 0; s < k; ++s) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || ranks_before(key[e], e, key[best], best)) best = e;
            }
            taken[best] = 1;
            idx[(size_t)t * k + s] = best;
        }
        const int32_t* sel = idx + (size_t)t * k;
        if (mode == OR_MODE_SIGMOID_BIASED) {
            double sum = 0.0;
            for (int s = 0; s < k; ++s) sum += (double)sg[sel[s]];
            for (int s = 0; s < k; ++s) w[(size_t)t * k + s] = (float)((double)sg[sel[s]] / sum);
        } else {
            double m = (double)key[sel[0]], sum = 0.0;
            for (int s = 0; s < k; ++s) sum += exp((double)key[sel[s]] - m);
            for (int s = 0; s < k; ++s) {
                double p = exp((double)key[sel[s]] - m) / sum;
                if (mode == OR_MODE_SOFTMAX_K_SCALED && scale) p *= (double)scale[sel[s]];
                w[(size_t)t * k + s] = (float)p;
            }
        }
    }
    free(key);
    free(sg);
    free(taken);
    return rc;
}

/* a3: route list.  Route id r = t*k + s.  off[e] = number of routes to experts < e;
 * perm lists route ids grouped by expert, ascending r inside each expert (stable);
 * inv[r] = position of r in perm. */
int or_build_routes(const int32_t* idx, int T, int E, int k, int32_t* off, int32_t* perm,
                    int32_t* inv) {
    int n = T * k;
    for (int e = 0; e <= E; ++e) off[e] = 0;
    for (int r = 0; r < n; ++r) {
        if (idx[r] < 0 || idx[r] >= E) return -1;
        off[idx[r] + 1] += 1;
    }
    for (int e = 0; e < E; ++e) off[e + 1] += off[e];
    int pos = 0;
    for (int e = 0; e < E; ++e)
        for (int r = 0; r < n; ++r)
            if (idx[r] == e) { perm[pos] = r; inv[r] = pos; ++pos; }
    return 0;
}

/* Activations of the gated FFN ([llama/mod.rs] use_silu = hidden_activation.contains("silu"),
 * otherwise gelu-tanh; [gptoss/moe.rs] Mxfp4Activation::GPT_OSS clamped SwiGLU). */
double or_act(int act, double g, double u, float limit, float alpha) {
    if (act == OR_ACT_SILU) return g / (1.0 + exp(-g)) * u;
    if (act == OR_ACT_GELU_TANH) {
        const double c = sqrt(2.0 / 3.14159265358979323846);
        return 0.5 * g * (1.0 + tanh(c * (g + 0.044715 * g * g * g))) * u;
    }
    /* gpt-oss: g = min(g, limit), u = clamp(u, -limit, limit), h = g*sigmoid(alpha*g)*(u+1) */
    double L = (double)limit;
    if (g > L) g = L;
    if (u > L) u = L;
    if (u < -L) u = -L;
    return g / (1.0 + exp(-(double)alpha * g)) * (u + 1.0);
}

/* a4 + a5 for one (token, expert) pair.  Weights dequantised exactly, sums in double,
 * biases added before the activation, h rounded to the 16-bit activation type
 * (the acts buffer is 16-bit), down projection accumulated in double from the rounded h
 * and rounded once to f32. */
int or_expert_ffn(const or_experts* X, int e, const double* xin, int adt, double* h_out,
                  float* e_out) {
    int H = X->H, I = X->I;
    for (int i = 0; i < I; ++i) {
        double g = 0.0, u = 0.0;
        for (int c = 0; c < H; ++c) {
            g += or_weight(X, 0, e, i, c) * xin[c];
            u += or_weight(X, 1, e, i, c) * xin[c];
        }
        if (X->gate_b) g += or_bf16_to_double(X->gate_b[(size_t)e * I + i]);
        if (X->up_b) u += or_bf16_to_double(X->up_b[(size_t)e * I + i]);
        double h = or_act(X->act, g, u, X->limit, X->alpha);
        h_out[i] = adt_to_double(double_to_adt(h, adt), adt);
    }
    for (int j = 0; j < H; ++j) {
        double acc = 0.0;
        for (int i = 0; i < I; ++i) acc += or_weight(X, 2, e, j, i) * h_out[i];
        if (X->down_b) acc += or_bf16_to_double(X->down_b[(size_t)e * H + j]);
        e_out[j] = (float)acc;
    }
    return 0;
}

/* The pre-activation sums of phase 1 for one (token, expert) pair, exposed so that the tests can
 * bound how far any f32 evaluation of them may fall from these exact values:
 *   g[i] = sum_c W_g[e][i][c] x[c] + b_g[e][i],   u[i] likewise with W_u, b_u   (double)
 *   sg[i] = sum_c |W_g[e][i][c] x[c]|,             su[i] likewise              (double)
 * The same dequantisation and double sums as or_expert_ffn; nothing is rounded. */
int or_expert_pre(const or_experts* X, int e, const double* xin, double* g_out, double* u_out,
                  double* sg_out, double* su_out) {
    int H = X->H, I = X->I;
    for (int i = 0; i < I; ++i) {
        double g = 0.0, u = 0.0, sg = 0.0, su = 0.0;
        for (int c = 0; c < H; ++c) {
            double pg = or_weight(X, 0, e, i, c) * xin[c];
            double pu = or_weight(X, 1, e, i, c) * xin[c];
            g += pg;
            u += pu;
            sg += fabs(pg);
            su += fabs(pu);
        }
        if (X->gate_b) g += or_bf16_to_double(X->gate_b[(size_t)e * I + i]);
        if (X->up_b) u += or_bf16_to_double(X->up_b[(size_t)e * I + i]);
        g_out[i] = g;
        u_out[i] = u;
        sg_out[i] = sg;
        su_out[i] = su;
    }
    return 0;
}

/* or_act over n pairs (g[i], u[i]) -> out[i], in double. */
void or_act_n(int act, const double* g, const double* u, int n, float limit, float alpha,
              double* out) {
    for (int i = 0; i < n; ++i) out[i] = or_act(act, g[i], u[i], limit, alpha);
}

/* a4..a7 for the tokens listed in `tokens` (all T if tokens == NULL).  Output row q of
 * y / y_f32 belongs to token tokens[q].  The combine runs in f32, slot by slot:
 * acc = seed; acc = acc + w[t][s] * e_s (a rounded multiply, then a rounded add);
 * seed = shared-expert output (f32) or +0.0f.  y = adt(acc).  If e_routes is given,
 * row q*k+s receives the f32 expert output of slot s. */
int or_moe_forward(const uint16_t* x, int adt, int T, const or_experts* X, const int32_t* idx,
                   const float* w, int k, const or_experts* shared, const int32_t* tokens,
                   int ntok, uint16_t* y, float* y_f32, float* e_routes, int nthreads) {
    int H = X->H;
    if (shared && (shared->H != H || shared->E != 1)) return -1;
    int n = tokens ? ntok : T;
    int rc = 0;
    (void)nthreads;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic) num_threads(nthreads > 0 ? nthreads : 1)
#endif
    for (int q = 0; q < n; ++q) {
        int t = tokens ? tokens[q] : q;
        int Imax = X->I > (shared ? shared->I : 0) ? X->I : shared->I;
        double* xin = (double*)malloc(sizeof(double) * H);
        double* h = (double*)malloc(sizeof(double) * Imax);
        float* eo = (float*)malloc(sizeof(float) * H);
        float* acc = (float*)malloc(sizeof(float) * H);
        if (!xin || !h || !eo || !acc || t < 0 || t >= T) {
            rc = -2;
        } else {
            for (int c = 0; c < H; ++c) xin[c] = adt_to_double(x[(size_t)t * H + c], adt);
            if (shared) {
                or_expert_ffn(shared, 0, xin, adt, h, eo);
                for (int j = 0; j < H; ++j) acc[j] = eo[j];
            } else {
                for (int j = 0; j < H; ++j) acc[j] = 0.0f;
            }
            for (int s = 0; s < k; ++s) {
                int e = idx[(size_t)t * k + s];
                float ws = w[(size_t)t * k + s];
                or_expert_ffn(X, e, xin, adt, h, eo);
                if (e_routes) memcpy(e_routes + ((size_t)q * k + s) * H, eo, sizeof(float) * H);
                for (int j = 0; j < H; ++j) {
                    float p = ws * eo[j];
                    acc[j] = acc[j] + p;
                }
            }
            for (int j = 0; j < H; ++j) {
                if (y_f32) y_f32[(size_t)q * H + j] = acc[j];
                if (y) y[(size_t)q * H + j] = double_to_adt((double)acc[j], adt);
            }
        }
        free(xin);
        free(h);
        free(eo);
        free(acc);
    }
    return rc;
}

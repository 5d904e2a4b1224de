/*
 * CPU oracle for one batch-1 decode step of the Higgs-Audio-style TTS backbone.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the tests, the package smoke check and
 * the benchmark's CPU-baseline leg, never by the product path.  It shares no
 * code with the CUDA library.
 *
 * Every function below is the plain definition of one step of the method,
 * evaluated in fp64 (OpenMP only splits independent output rows / heads).
 * Citations name the page and section the step comes from:
 *   [FlashRT header]   "Higgs Audio v3 TTS-4B on FlashRT (RTX 5090 / SM120)",
 *                      the model paragraph under the title.
 *   [FlashRT s5]       same page, section 5 "What runs under the hood".
 *   [FlashRT s4]       same page, section 4 "Python API", "Sampling policy".
 *   [FlashRT perf]     same page, "Performance" (FP8 W8A8 / BF16 W16A16).
 *   [FlashRT s8]       same page, section 8 "Notes & limitations" (FP8 scale is
 *                      amax/448).
 *   [SGLang arch]      "SGLang-Omni ... Higgs Audio v3 TTS" post, architecture
 *                      paragraph (8 codebooks, delay pattern, fused
 *                      multi-codebook embedding and head).
 * Readings the pages leave open (RoPE pairing, mask details, FP8 rounding
 * points) are stated where they are used.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Scalar formats                                                            */
/* ------------------------------------------------------------------------ */

double or_bf16_to_f64(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* Round x to the nearest bf16 value (8 significant bits), ties to even,
 * directly from fp64 (no intermediate fp32 rounding). */
uint16_t or_f64_to_bf16(double x) {
    if (isnan(x)) return 0x7fc0;
    double a = fabs(x);
    double q;
    if (a == 0.0) {
        q = 0.0;
    } else {
        int ex;
        frexp(a, &ex);            /* a = m * 2^ex, m in [0.5, 1) */
        int e = ex - 1;           /* floor(log2 a) */
        if (e < -126) e = -126;   /* subnormal range: fixed quantum 2^-133 */
        double quantum = ldexp(1.0, e - 7);
        q = nearbyint(a / quantum) * quantum;   /* a/quantum is exact */
    }
    float f = (float)(x < 0 ? -q : q);          /* q has <= 8 significant bits: exact */
    uint32_t u;
    memcpy(&u, &f, 4);
    if (isinf(f)) return (uint16_t)(u >> 16);
    return (uint16_t)(u >> 16);
}

uint16_t or_f32_to_bf16(float x) { return or_f64_to_bf16((double)x); }

/* OCP 8-bit floating point E4M3 ("fn" variant): 1 sign, 4 exponent bits with
 * bias 7, 3 mantissa bits; exponent field 0 is subnormal (m/8 * 2^-6); no
 * infinities; S.1111.111 is NaN; largest finite 1.75 * 2^8 = 448. */
double or_e4m3_decode(uint8_t b) {
    int s = b >> 7, e = (b >> 3) & 15, m = b & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m / 8.0, -6);
    else v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* Nearest E4M3 value to the fp32 input, ties to even mantissa, finite values
 * above 448 in magnitude saturate to 448 (the "satfinite" convention). */
uint8_t or_e4m3_encode(float xf) {
    double x = (double)xf;
    if (isnan(x)) return 0x7f;
    int s = signbit(x) ? 1 : 0;
    double a = fabs(x);
    int code;
    if (a >= 448.0) {
        code = (15 << 3) | 6;
    } else {
        int ex;
        frexp(a, &ex);
        int e = (a == 0.0) ? -6 : ex - 1;
        if (e < -6) e = -6;                    /* subnormal quantum is 2^-9 */
        double quantum = ldexp(1.0, e - 3);
        double q = nearbyint(a / quantum) * quantum;
        if (q > 448.0) q = 448.0;
        if (q < ldexp(1.0, -6)) {
            code = (int)(q / ldexp(1.0, -9));  /* exponent field 0 */
        } else {
            frexp(q, &ex);
            int qe = ex - 1;
            int m = (int)(q / ldexp(1.0, qe) * 8.0) - 8;
            code = ((qe + 7) << 3) | m;
        }
    }
    return (uint8_t)((s << 7) | code);
}

/* ------------------------------------------------------------------------ */
/* Building blocks                                                           */
/* ------------------------------------------------------------------------ */

/* RMSNorm [FlashRT s5 "rms_norm"; Qwen3 definition]:
 * y_i = x_i / sqrt(mean(x^2) + eps) * gamma_i. */
void or_rmsnorm(const double* x, const uint16_t* gamma, int n, double eps, double* y) {
    double ss = 0.0;
    for (int i = 0; i < n; ++i) ss += x[i] * x[i];
    double r = 1.0 / sqrt(ss / (double)n + eps);
    for (int i = 0; i < n; ++i) y[i] = x[i] * r * or_bf16_to_f64(gamma[i]);
}

/* y = W x, W bf16 [N][K] row-major [FlashRT s5 "M=1 GEMV"]. */
void or_linear_bf16(const uint16_t* W, int N, int K, const double* x, double* y) {
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n) {
        const uint16_t* row = W + (size_t)n * K;
        double acc = 0.0;
        for (int k = 0; k < K; ++k) acc += or_bf16_to_f64(row[k]) * x[k];
        y[n] = acc;
    }
}

/* Per-token dynamic activation quantisation [FlashRT s8: scale amax/448;
 * per-token dynamic form]: s = max(amax, 1e-12)/448 and q = e4m3(x/s).  The
 * decision is taken in fp32, the precision the method keeps activations in. */
void or_quant_act(const double* x, int n, uint8_t* q, float* scale) {
    float amax = 0.0f;
    for (int i = 0; i < n; ++i) {
        float a = fabsf((float)x[i]);
        if (a > amax) amax = a;
    }
    float s = (amax > 1e-12f ? amax : 1e-12f) / 448.0f;
    for (int i = 0; i < n; ++i) q[i] = or_e4m3_encode((float)x[i] / s);
    *scale = s;
}

/* Static activation scale [FlashRT perf "FP8 W8A8", s5 "quantize_fp8_static":
 * a per-tensor scale calibrated offline as amax / 448]: the same fp32
 * division and saturating encode as the per-token path, scale given. */
void or_quant_act_static(const double* x, int n, float scale, uint8_t* q) {
    for (int i = 0; i < n; ++i) q[i] = or_e4m3_encode((float)x[i] / scale);
}

/* One FP8 activation site (layer l, site 0..3 = QKV, O, gate/up, down input):
 * records the input's amax for calibration runs, then quantises with the
 * site's static scale if one is set, else per token. */
static void quant_site(const or_weights* w, or_state* st, int l, int site, const double* x, int n, uint8_t* q,
                       float* scale) {
    if (st->amax_acc) {
        float amax = 0.0f;
        for (int i = 0; i < n; ++i) {
            const float a = fabsf((float)x[i]);
            if (a > amax) amax = a;
        }
        if (amax > st->amax_acc[4 * l + site]) st->amax_acc[4 * l + site] = amax;
    }
    const float s = w->act_scales ? w->act_scales[4 * l + site] : 0.0f;
    if (s > 0.0f) {
        or_quant_act_static(x, n, s, q);
        *scale = s;
    } else {
        or_quant_act(x, n, q, scale);
    }
}

/* FP8 W8A8 projection [FlashRT perf "FP8 W8A8"; FlashRT s5 "M=1 FP8 GEMV"]:
 * acc = sum_k w8[n][k] * a8[k] (exact in fp64: every e4m3 product has at most
 * 8 significant bits and the exponent span fits in 53 bits), then the output
 * y = bf16(fp32(acc) * fp32(sa * sw[n])) in fp32 arithmetic. */
void or_linear_fp8(const uint8_t* W8, const float* sw, int N, int K,
                   const uint8_t* a8, float sa, double* y) {
    double dec[256];
    for (int i = 0; i < 256; ++i) dec[i] = or_e4m3_decode((uint8_t)i);
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n) {
        const uint8_t* row = W8 + (size_t)n * K;
        double acc = 0.0;
        for (int k = 0; k < K; ++k) acc += dec[row[k]] * dec[a8[k]];
        float sc = sa * sw[n];
        float v = (float)acc * sc;
        y[n] = or_bf16_to_f64(or_f32_to_bf16(v));
    }
}

/* Per-output-channel weight quantisation: sw[n] = max_k |W[n][k]| / 448 (1 if
 * the row is zero) and w8 = e4m3(W / sw), all in fp32. */
void or_quant_weight(const uint16_t* W, int N, int K, uint8_t* W8, float* sw) {
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n) {
        const uint16_t* row = W + (size_t)n * K;
        float amax = 0.0f;
        for (int k = 0; k < K; ++k) {
            float a = fabsf((float)or_bf16_to_f64(row[k]));
            if (a > amax) amax = a;
        }
        float s = amax > 0.0f ? amax / 448.0f : 1.0f;
        for (int k = 0; k < K; ++k) W8[(size_t)n * K + k] = or_e4m3_encode((float)or_bf16_to_f64(row[k]) / s);
        sw[n] = s;
    }
}

/* Rotary embedding, rotate-half pairing (i, i + D/2) as in Qwen3, with inverse
 * frequencies theta^(-2i/D) [FlashRT header "RoPE theta=1e6"]. */
void or_rope(double* x, int D, int pos, double theta) {
    int half = D / 2;
    for (int i = 0; i < half; ++i) {
        double inv_f = pow(theta, -2.0 * (double)i / (double)D);
        double ang = (double)pos * inv_f;
        double c = cos(ang), s = sin(ang);
        double a = x[i], b = x[i + half];
        x[i] = a * c - b * s;
        x[i + half] = b * c + a * s;
    }
}

/* SwiGLU activation [FlashRT header "SwiGLU"]: silu(z) = z / (1 + e^-z). */
double or_silu(double z) { return z / (1.0 + exp(-z)); }

/* Grouped-query attention over positions [0, len) of one layer's cache
 * [FlashRT header "GQA 32q/8kv"; FlashRT s5 "FA2"]: q head h reads kv head
 * h / (n_q/n_kv); scores q.K/sqrt(D); softmax with the maximum subtracted;
 * output sum_t p_t V_t / sum_t p_t. */
void or_attention(const double* q, const uint16_t* Kc, const uint16_t* Vc,
                  int n_q, int n_kv, int D, int max_pos, int len, double* out) {
    int group = n_q / n_kv;
#pragma omp parallel for schedule(static)
    for (int h = 0; h < n_q; ++h) {
        int g = h / group;
        const uint16_t* Kh = Kc + (size_t)g * max_pos * D;
        const uint16_t* Vh = Vc + (size_t)g * max_pos * D;
        double* s = (double*)malloc(sizeof(double) * (size_t)(len > 0 ? len : 1));
        double scale = 1.0 / sqrt((double)D);
        double m = -INFINITY;
        for (int t = 0; t < len; ++t) {
            double acc = 0.0;
            for (int d = 0; d < D; ++d) acc += q[h * D + d] * or_bf16_to_f64(Kh[(size_t)t * D + d]);
            s[t] = acc * scale;
            if (s[t] > m) m = s[t];
        }
        double l = 0.0;
        for (int t = 0; t < len; ++t) { s[t] = exp(s[t] - m); l += s[t]; }
        for (int d = 0; d < D; ++d) {
            double acc = 0.0;
            for (int t = 0; t < len; ++t) acc += s[t] * or_bf16_to_f64(Vh[(size_t)t * D + d]);
            out[h * D + d] = len > 0 ? acc / l : 0.0;
        }
        free(s);
    }
}

/* Fused multi-codebook embedding [SGLang arch]: x = sum_k E_k[codes[k]]. */
void or_embed(const uint16_t* E, int n_cb, int V, int H, const int32_t* codes, double* x) {
    for (int i = 0; i < H; ++i) x[i] = 0.0;
    for (int k = 0; k < n_cb; ++k) {
        const uint16_t* row = E + ((size_t)k * V + (size_t)codes[k]) * H;
        for (int i = 0; i < H; ++i) x[i] += or_bf16_to_f64(row[i]);
    }
}

/* Greedy argmax; ties go to the lowest index. */
int or_argmax(const double* v, int n) {
    int best = 0;
    for (int i = 1; i < n; ++i)
        if (v[i] > v[best]) best = i;
    return best;
}

/* Philox4x32-10 [Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
 * easy as 1, 2, 3", SC'11]: ten rounds; a round multiplies words 0 and 2 by
 * the two Philox multipliers and recombines the high and low halves with
 * words 1 and 3 and the round key; the key advances by the two Weyl
 * constants (golden ratio and sqrt(3) - 1, scaled to 32 bits) per round. */
void or_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int r = 0; r < 10; ++r) {
        const uint64_t p0 = (uint64_t)0xD2511F53u * c0;
        const uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
        const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
        const uint32_t n1 = (uint32_t)p1;
        const uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
        const uint32_t n3 = (uint32_t)p0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* Temperature sampling [FlashRT s4 sampling policy: stable softmax, a
 * stateless categorical draw keyed by the request seed]: inverse CDF in index
 * order, fp64. */
int or_sample_code(const double* logits, int V, double T, uint64_t seed, int t, int k, double* margin) {
    const uint32_t ctr[4] = {(uint32_t)t, (uint32_t)k, 0u, 0u};
    const uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t r[4];
    or_philox4x32_10(ctr, key, r);
    const double u = (double)(r[0] >> 8) / 16777216.0;
    double mx = -INFINITY;
    for (int v = 0; v < V; ++v)
        if (logits[v] > mx) mx = logits[v];
    double total = 0.0;
    for (int v = 0; v < V; ++v) total += exp((logits[v] - mx) / T);
    const double target = u * total;
    double run = 0.0, best = INFINITY;
    int code = -1;
    for (int v = 0; v < V; ++v) {
        run += exp((logits[v] - mx) / T);
        const double dist = fabs(run - target);
        if (dist < best) best = dist;
        if (code < 0 && run > target) code = v;
    }
    if (code < 0) code = V - 1;
    if (margin) *margin = fabs(target) < INFINITY ? best / total : 0.0;
    return code;
}

/* Delay pattern [FlashRT header "delay pattern"; FlashRT s5 "BOC/EOC";
 * SGLang arch]: codebook k runs k frames behind codebook 0.  At frame t,
 * codebook k has not started while t < k and emits BOS-pad; once codebook 0
 * has emitted EOC at frame eoc, codebook k emits EOC from frame eoc + k on;
 * otherwise it emits its argmax.  The pages' codebooks have 1026 entries:
 * 1024 acoustic codes, then BOS-pad (1024) and EOC (1025).  For another
 * vocabulary size V the last two entries take those roles (V - 2, V - 1). */
int or_delay_code(int k, int t, int eoc, int argmax_code, int V) {
    if (t < k) return V - 2;
    if (eoc >= 0 && t >= eoc + k) return V - 1;
    return argmax_code;
}

/* ------------------------------------------------------------------------ */
/* The layer stack and the step                                              */
/* ------------------------------------------------------------------------ */

static int check_dims(const or_dims* d) {
    if (!d || d->n_layers < 1 || d->hidden < 1 || d->n_q < 1 || d->n_kv < 1 || d->head_dim < 2 ||
        (d->head_dim & 1) || d->n_q % d->n_kv || d->inter < 1 || d->n_cb < 1 || d->cb_vocab < 1 ||
        d->max_pos < 1)
        return -1;
    return 0;
}

static double round_bf16(double x) { return or_bf16_to_f64(or_f64_to_bf16(x)); }

/* One position through layers [l0, l1): h holds that layer's input
 * residual stream on entry and layer l1-1's output on exit.  Writes K/V of
 * those layers at `pos`. */
static void stack_layers(const or_dims* d, const or_weights* w, or_state* st, int pos,
                         double* h, int a16, int l0, int l1) {
    const int H = d->hidden, D = d->head_dim, NQ = d->n_q, NKV = d->n_kv, I = d->inter;
    const int QKV = (NQ + 2 * NKV) * D, A = NQ * D;
    const int fp8 = d->precision == 1;
    double* a = (double*)malloc(sizeof(double) * H);
    double* qkv = (double*)malloc(sizeof(double) * QKV);
    double* attn = (double*)malloc(sizeof(double) * A);
    double* o = (double*)malloc(sizeof(double) * H);
    double* gu = (double*)malloc(sizeof(double) * 2 * I);
    double* m = (double*)malloc(sizeof(double) * I);
    double* tmp = (double*)malloc(sizeof(double) * (D > H ? D : H));
    int maxv = H > A ? H : A;
    if (I > maxv) maxv = I;
    uint8_t* q8 = (uint8_t*)malloc((size_t)maxv);

    for (int l = l0; l < l1; ++l) {
        size_t cache_off = (size_t)l * NKV * d->max_pos * D;
        uint16_t* Kl = st->k + cache_off;
        uint16_t* Vl = st->v + cache_off;

        /* input RMSNorm, then the fused q/k/v projection [FlashRT s5] */
        or_rmsnorm(h, w->ln_in[l], H, d->rms_eps, a);
        if (fp8) {
            float s;
            quant_site(w, st, l, 0, a, H, q8, &s);
            or_linear_fp8(w->qqkv[l], w->sqkv[l], QKV, H, q8, s, qkv);
        } else {
            if (a16) for (int i = 0; i < H; ++i) a[i] = round_bf16(a[i]);
            or_linear_bf16(w->wqkv[l], QKV, H, a, qkv);
        }

        /* per-head q/k RMSNorm, then RoPE at `pos` [FlashRT s5 "fused q/k-norm + RoPE"] */
        for (int hq = 0; hq < NQ; ++hq) {
            or_rmsnorm(qkv + hq * D, w->q_norm[l], D, d->rms_eps, tmp);
            memcpy(qkv + hq * D, tmp, sizeof(double) * D);
            or_rope(qkv + hq * D, D, pos, d->rope_theta);
        }
        for (int j = 0; j < NKV; ++j) {
            double* kj = qkv + (NQ + j) * D;
            double* vj = qkv + (NQ + NKV + j) * D;
            or_rmsnorm(kj, w->k_norm[l], D, d->rms_eps, tmp);
            memcpy(kj, tmp, sizeof(double) * D);
            or_rope(kj, D, pos, d->rope_theta);
            /* bf16 KV-cache write [FlashRT s5 "KV-write"] */
            for (int i = 0; i < D; ++i) {
                Kl[((size_t)j * d->max_pos + pos) * D + i] = or_f64_to_bf16(kj[i]);
                Vl[((size_t)j * d->max_pos + pos) * D + i] = or_f64_to_bf16(vj[i]);
            }
        }

        /* attention over positions [0, pos] of the cache */
        or_attention(qkv, Kl, Vl, NQ, NKV, D, d->max_pos, pos + 1, attn);

        /* output projection with the residual add h += W_o attn */
        if (fp8) {
            float s;
            quant_site(w, st, l, 1, attn, A, q8, &s);
            or_linear_fp8(w->qo[l], w->so[l], H, A, q8, s, o);
        } else {
            if (a16) for (int i = 0; i < A; ++i) attn[i] = round_bf16(attn[i]);
            or_linear_bf16(w->wo[l], H, A, attn, o);
        }
        for (int i = 0; i < H; ++i) h[i] += o[i];

        /* post-attention RMSNorm, gate/up, SwiGLU */
        or_rmsnorm(h, w->ln_post[l], H, d->rms_eps, a);
        if (fp8) {
            float s;
            quant_site(w, st, l, 2, a, H, q8, &s);
            or_linear_fp8(w->qgu[l], w->sgu[l], 2 * I, H, q8, s, gu);
            for (int i = 0; i < I; ++i) m[i] = round_bf16(or_silu(gu[i]) * gu[I + i]);
        } else {
            if (a16) for (int i = 0; i < H; ++i) a[i] = round_bf16(a[i]);
            or_linear_bf16(w->wgu[l], 2 * I, H, a, gu);
            for (int i = 0; i < I; ++i) m[i] = or_silu(gu[i]) * gu[I + i];
        }

        /* down projection with the residual add h += W_d m */
        if (fp8) {
            float s;
            quant_site(w, st, l, 3, m, I, q8, &s);
            or_linear_fp8(w->qd[l], w->sd[l], H, I, q8, s, o);
        } else {
            if (a16) for (int i = 0; i < I; ++i) m[i] = round_bf16(m[i]);
            or_linear_bf16(w->wd[l], H, I, m, o);
        }
        for (int i = 0; i < H; ++i) h[i] += o[i];
    }
    free(a); free(qkv); free(attn); free(o); free(gu); free(m); free(tmp); free(q8);
}

static void layer_stack(const or_dims* d, const or_weights* w, or_state* st, int pos,
                        double* h, int a16) {
    stack_layers(d, w, st, pos, h, a16, 0, d->n_layers);
}

/* Final RMSNorm, fused codebook head and per-codebook greedy argmax under the
 * delay pattern at frame st->t (bf16 weights in both precisions, no
 * activation quantisation) [FlashRT s5 "fused 8-codebook head"; FlashRT s4,
 * s5 sampling].  Reads the state, changes nothing. */
static void head_codes(const or_dims* d, const or_weights* w, const or_state* st, const double* h,
                       int32_t* codes_out, double* logits, double* gaps) {
    const int H = d->hidden, V = d->cb_vocab, C = d->n_cb;
    double* f = (double*)malloc(sizeof(double) * H);
    double* lg = (double*)malloc(sizeof(double) * (size_t)C * V);
    or_rmsnorm(h, w->final_norm, H, d->rms_eps, f);
    or_linear_bf16(w->head, C * V, H, f, lg);
    int t = st->t, eoc = st->eoc;
    for (int k = 0; k < C; ++k) {
        const double* row = lg + (size_t)k * V;
        int am = or_argmax(row, V);
        if (gaps) {
            double second = -INFINITY;
            for (int v = 0; v < V; ++v)
                if (v != am && row[v] > second) second = row[v];
            gaps[k] = row[am] - second;
        }
        codes_out[k] = or_delay_code(k, t, eoc, am, V);
    }
    if (logits) memcpy(logits, lg, sizeof(double) * (size_t)C * V);
    free(f);
    free(lg);
}

int or_layer(const or_dims* d, const or_weights* w, or_state* st, int layer, int pos, double* h, int a16) {
    if (check_dims(d) || !w || !st || !h || layer < 0 || layer >= d->n_layers || pos < 0 || pos >= d->max_pos)
        return -1;
    stack_layers(d, w, st, pos, h, a16, layer, layer + 1);
    return 0;
}

int or_head(const or_dims* d, const or_weights* w, const or_state* st, const double* h,
            int32_t* codes_out, double* logits, double* gaps) {
    if (check_dims(d) || !w || !st || !h || !codes_out) return -1;
    head_codes(d, w, st, h, codes_out, logits, gaps);
    return 0;
}

int or_decode_step(const or_dims* d, const or_weights* w, or_state* st,
                   const int32_t* codes_in, int32_t* codes_out,
                   double* logits, double* gaps) {
    if (check_dims(d) || !w || !st || !codes_in || !codes_out) return -1;
    if (st->pos < 0 || st->pos >= d->max_pos) return -1;
    for (int k = 0; k < d->n_cb; ++k)
        if (codes_in[k] < 0 || codes_in[k] >= d->cb_vocab) return -1;
    const int H = d->hidden, V = d->cb_vocab, C = d->n_cb;
    double* h = (double*)malloc(sizeof(double) * H);
    or_embed(w->embed, C, V, H, codes_in, h);
    layer_stack(d, w, st, st->pos, h, 0);
    head_codes(d, w, st, h, codes_out, logits, gaps);
    if (st->eoc < 0 && codes_out[0] == V - 1) st->eoc = st->t;
    st->pos += 1;
    st->t += 1;
    free(h);
    return 0;
}

int or_prefill(const or_dims* d, const or_weights* w, or_state* st,
               const int32_t* codes, int P, int a16) {
    if (check_dims(d) || !w || !st || (P > 0 && !codes) || P < 0) return -1;
    if (st->pos < 0 || st->pos + P > d->max_pos) return -1;
    for (int i = 0; i < P * d->n_cb; ++i)
        if (codes[i] < 0 || codes[i] >= d->cb_vocab) return -1;
    double* h = (double*)malloc(sizeof(double) * d->hidden);
    for (int p = 0; p < P; ++p) {
        or_embed(w->embed, d->n_cb, d->cb_vocab, d->hidden, codes + (size_t)p * d->n_cb, h);
        layer_stack(d, w, st, st->pos, h, a16);
        st->pos += 1;
    }
    free(h);
    return 0;
}

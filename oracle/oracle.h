/*
 * CPU oracle for one batch-1 decode step of the Higgs-Audio-style TTS backbone.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The product path (the
 * CUDA library) shares no code, header, table or constant with it.
 *
 * Plain, slow, obviously correct: fp64 arithmetic throughout, except where the
 * method itself fixes a precision (the bf16 KV cache; FP8 quantisation and the
 * bf16 outputs of the FP8 projections, whose rounding decisions are taken in
 * fp32 exactly as the method states them).
 *
 * Sources ("Higgs Audio v3 TTS-4B on FlashRT"): the model description in the
 * page header (Qwen3-4B backbone: 36 layers, hidden 2560, GQA 32q/8kv,
 * head_dim 128, SwiGLU, RoPE theta 1e6; fused 8 x 1026 codebook head, delay
 * pattern); the decode chain in section 5 "What runs under the hood"; the
 * sampling policy in section 4 (greedy argmax + delay mask + embedding, or a
 * seeded categorical draw at a positive temperature); the
 * FP8 W8A8 description in the Performance section and section 8.  The fused
 * multi-codebook embedding (sum of 8 codebook embeddings) is from the
 * SGLang-Omni Higgs Audio v3 post, architecture paragraph.
 */
#ifndef AR_ORACLE_H
#define AR_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
    int n_layers, hidden, n_q, n_kv, head_dim, inter, n_cb, cb_vocab, max_pos;
    double rms_eps, rope_theta;
    int precision;            /* 0: bf16 weights, fp32-or-wider activations; 1: FP8 E4M3 W8A8 */
} or_dims;

typedef struct {
    const uint16_t* embed;       /* bf16 [n_cb][cb_vocab][hidden] */
    const uint16_t* head;        /* bf16 [n_cb*cb_vocab][hidden] */
    const uint16_t* final_norm;  /* bf16 [hidden] */
    const uint16_t* const* wqkv; /* per layer, bf16 [(n_q+2n_kv)*D][hidden]  (precision 0) */
    const uint16_t* const* wo;   /* bf16 [hidden][n_q*D] */
    const uint16_t* const* wgu;  /* bf16 [2*inter][hidden]: gate rows then up rows */
    const uint16_t* const* wd;   /* bf16 [hidden][inter] */
    const uint8_t* const* qqkv;  /* per layer, e4m3 images of the same matrices (precision 1) */
    const uint8_t* const* qo;
    const uint8_t* const* qgu;
    const uint8_t* const* qd;
    const float* const* sqkv;    /* per-output-row fp32 weight scales (precision 1) */
    const float* const* so;
    const float* const* sgu;
    const float* const* sd;
    const uint16_t* const* ln_in;   /* bf16 [hidden] */
    const uint16_t* const* ln_post; /* bf16 [hidden] */
    const uint16_t* const* q_norm;  /* bf16 [D] */
    const uint16_t* const* k_norm;  /* bf16 [D] */
    const float* act_scales;        /* precision 1, optional: static activation scales [n_layers][4]
                                       (QKV, O, gate/up, down inputs; a site <= 0, or NULL: per-token) */
} or_weights;

typedef struct {
    uint16_t* k;   /* bf16 [n_layers][n_kv][max_pos][D] */
    uint16_t* v;
    int pos;       /* next position to write */
    int t;         /* decode frame index since the last reset */
    int eoc;       /* frame at which codebook 0 first emitted EOC, -1 if none */
    float* amax_acc; /* precision 1, optional: [n_layers][4] raised to the largest input amax seen
                        at each activation site (calibration) */
} or_state;

/* ---- scalar formats ---- */
double   or_bf16_to_f64(uint16_t b);
uint16_t or_f64_to_bf16(double x);          /* round to nearest even, straight from fp64 */
uint16_t or_f32_to_bf16(float x);           /* round to nearest even from an fp32 value */
double   or_e4m3_decode(uint8_t b);         /* OCP E4M3 "fn": bias 7, no inf, 0x7f/0xff NaN */
uint8_t  or_e4m3_encode(float x);           /* nearest even, saturating to +-448 */

/* ---- building blocks ---- */
void   or_rmsnorm(const double* x, const uint16_t* gamma, int n, double eps, double* y);
void   or_linear_bf16(const uint16_t* W, int N, int K, const double* x, double* y);
void   or_quant_act(const double* x, int n, uint8_t* q, float* scale);
/* FP8 quantisation with a given (static, calibrated) scale: q = e4m3(x / scale)
 * in fp32, saturating beyond +-448. */
void   or_quant_act_static(const double* x, int n, float scale, uint8_t* q);
void   or_linear_fp8(const uint8_t* W8, const float* sw, int N, int K,
                     const uint8_t* a8, float sa, double* y);
void   or_quant_weight(const uint16_t* W, int N, int K, uint8_t* W8, float* sw);
void   or_rope(double* x, int D, int pos, double theta);
double or_silu(double z);
void   or_attention(const double* q, const uint16_t* Kc, const uint16_t* Vc,
                    int n_q, int n_kv, int D, int max_pos, int len, double* out);
void   or_embed(const uint16_t* E, int n_cb, int V, int H, const int32_t* codes, double* x);
int    or_argmax(const double* v, int n);
/* Philox4x32-10 (Salmon et al., SC'11): out = the 4 words for counter ctr
 * and key key. */
void   or_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);
/* Temperature sampling of one codebook (FlashRT section 4 sampling policy):
 * u = top 24 bits of the first Philox word for counter (t, k, 0, 0), key
 * seed, over 2^24; the first v whose running sum of exp((logit_v - max)/T)
 * exceeds u times the total (fp64).  Also writes, when margin != NULL, the
 * distance of u * total from the nearest running sum, relative to the total
 * (how far the draw is from flipping to a neighbouring code). */
int    or_sample_code(const double* logits, int V, double T, uint64_t seed, int t, int k, double* margin);
int    or_delay_code(int k, int t, int eoc, int argmax_code, int V);

/* ---- the step ---- */
/* One decode step at st->pos, frame st->t.  Writes K/V at st->pos, fills
 * logits[n_cb*cb_vocab] and gaps[n_cb] (top-1 minus top-2 logit per codebook,
 * either may be NULL), writes codes_out[n_cb], then advances pos and t.
 * Returns 0, or -1 on a bad argument. */
int or_decode_step(const or_dims* d, const or_weights* w, or_state* st,
                   const int32_t* codes_in, int32_t* codes_out,
                   double* logits, double* gaps);

/* One layer `layer` at position pos (layer-level checks): h holds the
 * layer's input residual stream on entry and its output on exit; writes that
 * layer's K/V at pos.  a16 as in or_prefill.  Changes neither pos nor t.
 * Returns 0 or -1. */
int or_layer(const or_dims* d, const or_weights* w, or_state* st, int layer, int pos, double* h, int a16);

/* The head of the step on a given final residual stream h: final RMSNorm,
 * codebook logits, argmax under the delay mask at frame st->t (codes_out,
 * logits and gaps as in or_decode_step).  Changes nothing.  Returns 0 or -1. */
int or_head(const or_dims* d, const or_weights* w, const or_state* st, const double* h,
            int32_t* codes_out, double* logits, double* gaps);

/* Prefill: runs the layer stack at positions st->pos .. st->pos+P-1 with the
 * given codes (row p = the n_cb codes of position p), writing K/V; no head.
 * a16 != 0 rounds the input of every projection to bf16 (the tensor-core
 * prefill's W16A16 arithmetic).  Leaves t and eoc unchanged. */
int or_prefill(const or_dims* d, const or_weights* w, or_state* st,
               const int32_t* codes, int P, int a16);

#ifdef __cplusplus
}
#endif
#endif

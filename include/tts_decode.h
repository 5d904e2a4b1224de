/*
 * tts_decode.h -- C ABI of the GB300 (sm_103a) batch-1 decode-step library for
 * a Higgs-Audio-style TTS backbone.
 *
 * The backbone is a dense Qwen3-4B-shaped decoder (36 layers, hidden 2560, GQA
 * 32 query / 8 key-value heads, head_dim 128, SwiGLU, RoPE theta 1e6, per-head
 * q/k RMSNorm), fed by a fused embedding of 8 codebooks under a delay pattern
 * and read out by a fused 8 x 1026 codebook head with a per-codebook greedy
 * argmax ("Higgs Audio v3 TTS-4B on FlashRT (RTX 5090 / SM120)", page header
 * and section 5 "What runs under the hood"; the SGLang-Omni Higgs Audio v3
 * post, architecture paragraph).
 *
 * Conventions for every entry point:
 *  - Return value: TTS_OK (0) or a negative TTS_ERR_* code.  On error the
 *    decode position is left unchanged.  tts_status_str() names a code.
 *  - "device" pointers are CUDA global-memory addresses on the current
 *    device; "host" pointers are ordinary CPU memory.  Pointers are borrowed:
 *    the library copies host arrays before returning and never frees caller
 *    memory.  Device weight buffers must stay valid until tts_shutdown().
 *  - All work runs on the stream given in tts_config (NULL = legacy default
 *    stream).  Entry points that return host results synchronise that stream.
 *  - One context per stream; a context is not thread-safe.
 *
 * Layouts (all row-major):
 *  - bf16 matrices are [out][in]; FP8 matrices are E4M3 bytes [out][in] with
 *    one fp32 scale per output row (value = byte_value * scale).
 *  - Wqkv rows: query heads (head*D + d), then key heads, then value heads.
 *  - Wgu rows: the gate matrix [inter][hidden] followed by the up matrix.
 *  - Codebook head rows: codebook k, code v at row k*cb_vocab + v.
 *  - KV cache: bf16 [n_layers][n_kv_heads][max_pos][head_dim], owned by the
 *    library.
 */
#ifndef TTS_DECODE_H
#define TTS_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
    TTS_OK = 0,
    TTS_ERR_ARG = -1,         /* NULL pointer, bad size, unsupported dimensions */
    TTS_ERR_CODE = -2,        /* an input code outside [0, cb_vocab) */
    TTS_ERR_FULL = -3,        /* the step would write at or past max_pos */
    TTS_ERR_CUDA = -4,        /* a CUDA runtime call failed */
    TTS_ERR_DEVICE = -5,      /* a kernel recorded a bounds or wait failure */
    TTS_ERR_STATE = -6,       /* context not initialised / already shut down */
    TTS_ERR_UNSUPPORTED = -7  /* valid request this build does not implement */
};

enum { TTS_BF16 = 0, TTS_FP8 = 1 };

/* tts_config.options bits (0 = the default decode and prefill paths). */
enum {
    /* Run each decode step as a graph of one kernel per projection, attention
     * and head (programmatic-dependent-launch edges) instead of the one
     * persistent step kernel.  Kept for per-projection timing; slower. */
    TTS_OPT_SEPARATE_KERNELS = 1,
    /* Prefill a prompt position by position through the decode step kernel
     * instead of the batched tensor-core pass. */
    TTS_OPT_PREFILL_STEPS = 2
};

typedef struct tts_ctx tts_ctx;

/* Model and run configuration.  Supported shapes: head_dim 128; n_q_heads a
 * multiple of n_kv_heads with 1, 2, 4 or 8 query heads per key-value head;
 * hidden, inter and n_q_heads*128 multiples of 256 and at most 12288 (for
 * TTS_FP8: multiples of 512);
 * n_codebooks 1..8; cb_vocab >= 2 (codes
 * cb_vocab-2 and cb_vocab-1 are BOS-pad and EOC, i.e. 1024 and 1025 for the
 * 1026-entry codebooks); 1 <= max_pos <= 65536. */
typedef struct {
    int n_layers;      /* 36 for the full backbone */
    int hidden;        /* 2560 */
    int n_q_heads;     /* 32 */
    int n_kv_heads;    /* 8 */
    int head_dim;      /* 128 */
    int inter;         /* 9728 */
    int n_codebooks;   /* 8 */
    int cb_vocab;      /* 1026 */
    int max_pos;       /* KV-cache capacity in positions */
    float rms_eps;     /* 1e-6 */
    float rope_theta;  /* 1e6 */
    int precision;     /* TTS_BF16 (W16, fp32 activations) or TTS_FP8 (E4M3 W8A8) */
    void* stream;      /* cudaStream_t; NULL = default stream */
    int options;       /* TTS_OPT_* bits; 0 for the default paths */
} tts_config;

/* Device pointers to the weights (borrowed).  The per-layer members are HOST
 * arrays of n_layers device pointers.  wqkv/wo/wgu/wd point to bf16 matrices
 * when precision == TTS_BF16 and to E4M3 matrices when precision == TTS_FP8;
 * sqkv/so/sgu/sd (fp32 per-output-row scales) are used only for TTS_FP8 and
 * may be NULL otherwise.  Norm gains are bf16.  The codebook embedding and
 * head are bf16 in both precisions. */
typedef struct {
    const void* embed;        /* bf16 [n_codebooks][cb_vocab][hidden] */
    const void* head;         /* bf16 [n_codebooks*cb_vocab][hidden] */
    const void* final_norm;   /* bf16 [hidden] */
    const void* const* wqkv;  /* [(n_q+2*n_kv)*head_dim][hidden] */
    const void* const* wo;    /* [hidden][n_q*head_dim] */
    const void* const* wgu;   /* [2*inter][hidden] */
    const void* const* wd;    /* [hidden][inter] */
    const float* const* sqkv; /* [(n_q+2*n_kv)*head_dim] */
    const float* const* so;   /* [hidden] */
    const float* const* sgu;  /* [2*inter] */
    const float* const* sd;   /* [hidden] */
    const void* const* ln_in;   /* [hidden]   input RMSNorm gain */
    const void* const* ln_post; /* [hidden]   post-attention RMSNorm gain */
    const void* const* q_norm;  /* [head_dim] per-head query RMSNorm gain */
    const void* const* k_norm;  /* [head_dim] per-head key RMSNorm gain */
} tts_weights;

/* Create a context: validates the configuration, allocates the KV cache, the
 * RoPE table and all step scratch, and captures the decode step as one CUDA
 * graph that reads the position from device memory (so it replays at any
 * position).  Position, frame and EOC state start at 0, 0, none.
 * Source: FlashRT page, Performance ("position-agnostic CUDA graph") and
 * section 7; the graph-lifetime rule (graph destroyed before memory is freed)
 * follows the TTS-Audio-Suite report on CUDA-graph teardown. */
int tts_init(const tts_config* cfg, const tts_weights* w, tts_ctx** out);

/* Destroy the graph, then free everything the library allocated.  NULL is a
 * no-op.  The context pointer is invalid afterwards. */
int tts_shutdown(tts_ctx* ctx);

/* Rewind: position 0, frame 0, no EOC.  KV contents are left stale (they are
 * overwritten as positions are re-filled). */
int tts_reset(tts_ctx* ctx);

/* Batched prefill of P positions (FlashRT page, section 7 "Prefill is one
 * batched M=P forward").  codes: HOST int32 [P][n_codebooks], each in
 * [0, cb_vocab).  Runs the layer stack for positions pos..pos+P-1 and writes
 * their K/V; no head, frame counter unchanged.  Afterwards the next decode
 * step's input is the all-BOS frame.  Errors: TTS_ERR_FULL if pos+P > max_pos.
 * Synchronises the stream. */
int tts_prefill(tts_ctx* ctx, const int32_t* codes, int P);

/* One decode step (FlashRT page, section 5).  codes_in: HOST int32
 * [n_codebooks], the frame fed to the embedding (NULL = use the codes the
 * previous step produced, or the all-BOS frame after a reset/prefill).
 * codes_out: HOST int32 [n_codebooks], the step's greedy codes under the
 * delay pattern (section 4, sampling policy).  Advances position and frame by
 * one.  Errors: TTS_ERR_CODE, TTS_ERR_FULL.  Synchronises the stream. */
int tts_decode_step(tts_ctx* ctx, const int32_t* codes_in, int32_t* codes_out);

/* n decode steps with device-side feedback: each step embeds the codes the
 * previous one produced, without a host round trip (SGLang-Omni post, "AR
 * backbone": one transfer per step batched away).  codes_out: HOST int32
 * [n][n_codebooks] (may be NULL), copied back once at the end.  Errors:
 * TTS_ERR_FULL if pos+n > max_pos.  Synchronises the stream. */
int tts_decode_steps(tts_ctx* ctx, int n, int32_t* codes_out);

/* Free-running decode with a one-frame lookahead (the pages' zero-sync host
 * loop: "Higgs Audio v3 TTS-4B on FlashRT", section 4 and the SGLang-Omni
 * post's AR backbone loop).  Frame f + 1 is queued on the GPU before the host
 * reads frame f's codes, which arrive by an asynchronous copy of the state
 * into a double-buffered pinned ring, so the GPU never waits on the host
 * between frames.  Stops after max_frames frames, at the end of the cache, or
 * after the frame in which the last codebook emits EOC (frame eoc +
 * n_codebooks - 1 of the delay pattern); a frame queued past the stop is
 * undone (the state returns to the one after the last reported frame; the
 * cache row it wrote lies past that position).  The first frame's input is
 * the device-resident codes, as in tts_decode_steps.  codes_out: HOST int32
 * [max_frames][n_codebooks] (may be NULL); *n_frames: frames produced.
 * Errors: TTS_ERR_FULL if the cache is already full, TTS_ERR_DEVICE if a
 * kernel recorded a failure (the frames before it are reported). */
int tts_decode_until_eoc(tts_ctx* ctx, int max_frames, int32_t* codes_out, int* n_frames);

/* Rewind to position pos (0 <= pos <= current position) and frame t, with no
 * EOC: cache positions [0, pos) are kept and later ones are overwritten as
 * decoding proceeds, so a prompt prefilled once can start many utterances
 * (FlashRT page, section 4: a shared preamble's KV is reused and only new
 * input is processed).  The next decode step's input is the all-BOS frame. */
int tts_rewind(tts_ctx* ctx, int pos, int t);

/* Set the input frame of the next decode step (the codes the embedding
 * reads) without running a step: teacher forcing for tts_decode_steps and
 * tts_decode_until_eoc.  codes: HOST int32 [n_codebooks], each in
 * [0, cb_vocab) (TTS_ERR_CODE otherwise, nothing changed).  Synchronises
 * the stream. */
int tts_set_input(tts_ctx* ctx, const int32_t* codes);

/* FP8 static activation scales (FlashRT page, FP8 W8A8 and section 5: the
 * production FP8 path quantises each projection input with a per-tensor
 * scale calibrated offline as amax / 448, instead of the per-token amax).
 * scales: HOST fp32 [n_layers][4] for the inputs of the QKV, O, gate/up and
 * down projections of each layer; a site set to 0 keeps the per-token
 * (dynamic) scale; NULL makes every site dynamic again.  With a static scale
 * s, x quantises to e4m3(x / s), values beyond 448 s saturating.  Applies to
 * every later decode step (and to prompts prefilled position by position,
 * TTS_OPT_PREFILL_STEPS); the batched prefill keeps per-token scales.
 * TTS_ERR_UNSUPPORTED for BF16 contexts or without the persistent step
 * kernel; TTS_ERR_ARG for a negative or non-finite scale. */
int tts_set_fp8_scales(tts_ctx* ctx, const float* scales);

/* FP8 calibration run: n_frames free-running decode frames from the current
 * state (as tts_decode_steps) with the current scales, recording for every
 * activation site the largest amax of its (normalised) input over the frames
 * into amax_out, HOST fp32 [n_layers][4] (same order as tts_set_fp8_scales;
 * the static scale is amax / 448).  The frames are then discarded: position,
 * frame, EOC frame and next input are restored (cache rows at and past the
 * position are left stale).  Errors as tts_set_fp8_scales, TTS_ERR_FULL if
 * the frames do not fit the cache. */
int tts_fp8_calibrate(tts_ctx* ctx, int n_frames, float* amax_out);

/* Prefix reuse (FlashRT page, section 4 and Performance "prompt prefill": a
 * resident system prompt's KV is kept and each request prefills only its own
 * suffix, bit-identically).  tts_prefix_save snapshots cache positions
 * [0, pos) of every layer and kv head into a library-owned device buffer,
 * together with the decode state (position, frame, EOC frame, next input
 * codes); tts_prefix_restore copies them back and restores that state, so a
 * later tts_prefill(suffix) continues exactly as right after the prefix --
 * also after a tts_rewind below the prefix or a tts_reset overwrote it.  One
 * snapshot per context; a new save replaces it.  Errors: TTS_ERR_ARG when
 * pos is 0 (nothing to save), TTS_ERR_STATE when restoring without a save. */
int tts_prefix_save(tts_ctx* ctx);
int tts_prefix_restore(tts_ctx* ctx);

/* Copy a KV prefix into the cache and set the position to len.  k, v: DEVICE
 * bf16 [n_layers][n_kv_heads][len_stride][head_dim] with len <= len_stride;
 * positions [0, len) are copied.  Frame and EOC state are not changed. */
int tts_set_kv(tts_ctx* ctx, const void* k, const void* v, int len, int len_stride);

/* Copy cache positions [p0, p1) of every layer and kv head to HOST bf16
 * buffers [n_layers][n_kv_heads][p1-p0][head_dim] (either may be NULL). */
int tts_get_kv(tts_ctx* ctx, void* k_host, void* v_host, int p0, int p1);

/* HOST fp32 [n_codebooks*cb_vocab]: the logits of the last decode step. */
int tts_get_logits(tts_ctx* ctx, float* logits_host);

/* HOST fp32 [hidden]: the residual stream after the last layer of the last
 * decode step (the input of the final RMSNorm), or of the last prompt row
 * of a position-by-position prefill; the batched prefill leaves it as it
 * was. */
int tts_get_hidden(tts_ctx* ctx, float* hidden_host);

/* Set the frame index and the EOC frame (-1 = none) used by the delay mask. */
int tts_set_frame(tts_ctx* ctx, int t, int eoc_frame);

/* Sampling head ("Higgs Audio v3 TTS-4B on FlashRT", section 4 sampling
 * policy).  temperature == 0 (the default) keeps the greedy argmax; a positive
 * temperature T replaces it, per codebook k at frame t, by a categorical draw
 * from softmax(logits_k / T) over all cb_vocab entries: with u the top 24 bits
 * of the first Philox4x32-10 word for counter (t, k, 0, 0) and key `seed`
 * (low word first), scaled to [0, 1), the code is the first v whose running
 * sum of exp((logit_v - max) / T) exceeds u times the total.  The delay mask
 * applies afterwards as in greedy decoding.  The same seed and frames give the
 * same draws.  The setting stays until changed (also across tts_reset and
 * tts_rewind) and applies to every later step, including tts_decode_steps.
 * Returns TTS_ERR_ARG for a negative or non-finite temperature. */
int tts_set_sampling(tts_ctx* ctx, float temperature, unsigned long long seed);

/* Read position, frame index and EOC frame (any pointer may be NULL). */
int tts_get_state(tts_ctx* ctx, int* pos, int* t, int* eoc_frame);

/* Device time of the last tts_decode_steps() call in milliseconds, measured
 * with CUDA events around the graph replays (inputs already resident). */
int tts_last_steps_ms(tts_ctx* ctx, float* ms);

/* Measurement hook (not part of the step): launch the GEMV of one projection
 * kind -- 0 QKV, 1 O-proj, 2 gate/up, 3 down-proj, 4 codebook head (logits
 * only, no argmax) -- once per layer's weights (the head n_layers times),
 * `reps` rounds back to back on the context's stream with the step's launch
 * configuration, and return the mean device time of one launch from CUDA
 * events.  Overwrites step scratch (not the KV cache or the state): call it
 * between steps.  Synchronises the stream. */
int tts_time_gemv(tts_ctx* ctx, int kind, int reps, float* ms_per_launch);

/* Measurement hook (not part of the product path): run one decode step of
 * the persistent step kernel with its phase trace enabled, outside the
 * graph, and copy the trace to `host_out` (uint64 nanosecond timestamps,
 * per CTA `stride` entries, followed by a per-ring-stage trace of two
 * consumer warps of CTA 0, 2 x 2048 stages x 4 entries: copy issued, consumer
 * start, consumer done (ns) and the stage's SM cycles; the layout is
 * documented with the kernel).
 * `capacity` is the number of uint64 the buffer holds; *stride and *n_cta
 * receive the shape.  The step advances the position like tts_decode_step
 * (input: the codes the previous step produced).  Returns TTS_ERR_UNSUPPORTED
 * when the context runs the step as separate kernels. */
int tts_trace_step(tts_ctx* ctx, uint64_t* host_out, int capacity, int* stride, int* n_cta);

/* Test hook (not part of the product path): one decode step like
 * tts_decode_step(ctx, codes_in, codes_out) (codes_in may be NULL: the
 * device's own codes; codes_out may be NULL), run by the traced variant of the step kernel, which also
 * records the fp32 residual stream after the embedding and after every layer
 * into `host_h` ([n_layers + 1][hidden], row 0 = the embedding; caller-owned,
 * `capacity` floats).  Lets a check start the CPU oracle's layer l from the
 * GPU's own input to that layer ("Higgs Audio v3 TTS-4B on FlashRT", section
 * 5, one layer of the chain).  Returns TTS_ERR_UNSUPPORTED when the step runs
 * as separate kernels, TTS_ERR_ARG if capacity is short; synchronises. */
int tts_debug_layer_states(tts_ctx* ctx, const int32_t* codes_in, int32_t* codes_out, float* host_h,
                           int capacity);

/* Test hook (not part of the product path): tts_prefill of P <= 512
 * positions on the batched path that also records the fp32 residual stream
 * of every prompt row after the embedding and after every layer into
 * `host_h` ([n_layers + 1][P][hidden], caller-owned, `capacity` floats), so a
 * check can start the CPU oracle's layer l from the GPU's input to it.
 * TTS_ERR_UNSUPPORTED when the context does not prefill on the batched path;
 * otherwise as tts_prefill.  Synchronises. */
int tts_debug_prefill_states(tts_ctx* ctx, const int32_t* codes, int P, float* host_h, long long capacity);

/* Test hook for failure detection (not part of the product path): one launch
 * of the persistent step kernel, outside the graph, whose embedding phase
 * stores nothing into its exchange buffer and whose waits give up after 1 ms
 * instead of 1 s.  The first layer's wait for the embedding runs out, the
 * kernel records the timeout in the device error word, every CTA leaves at
 * its next wait, the copies in flight land, and the launch ends; no spin is
 * left running.  Returns TTS_ERR_DEVICE (the error word is cleared again);
 * position, frame and cache are left as they were, so the next step runs
 * normally.  TTS_ERR_UNSUPPORTED when the step runs as separate kernels.
 * Synchronises the stream. */
int tts_debug_expire_wait(tts_ctx* ctx);

/* Stand-alone op: C = A . B^T on the tensor cores (tcgen05 MMA, TMEM
 * accumulators, TMA-staged operands), the GEMM of the batched prompt prefill
 * ("Higgs Audio v3 TTS-4B on FlashRT", Performance "BF16 W16A16" and section
 * 7: the prompt runs as one M = P pass over the weights).
 *   A: device bf16 [M][K] row-major (activations), B: device bf16 [N][K]
 *   (weights, one output feature per row), both borrowed, 16-byte aligned.
 *   epi 0: C = device fp32 [M][N], overwritten.
 *   epi 1: C = device fp32 [M][N], C += A . B^T.
 *   epi 2: SwiGLU: B = [gate rows; up rows], a [2N][K] matrix; C = device
 *          bf16 [M][N] = bf16(silu(A . gate^T) * (A . up^T)).
 * fp32 accumulation; K % 64 == 0, N a multiple of 64, 80, 128, 160 or 192
 * (epi 2: of 128), any M >= 1.  The tile (128 or 256 rows x one of those
 * widths) is chosen to fill the SMs; splits > 0 fixes how many CTAs share
 * the K range of a tile (1..4, epi 2: 1), splits <= 0 lets the library
 * choose.  Split sums are added in a fixed order: every result is
 * deterministic.  Enqueued on `stream` (NULL: the default stream); does not
 * synchronise.  Returns TTS_ERR_ARG for bad sizes, NULL or misaligned
 * pointers. */
int tts_gemm_bf16(const void* A, const void* B, void* C, int M, int N, int K, int epi, int splits, void* stream);

/* Stand-alone op: the FP8 W8A8 GEMM of the batched prefill of FP8 contexts
 * (FlashRT page, "FP8 W8A8": E4M3 weights with a per-row scale, E4M3
 * activations with a per-token scale), on the tensor cores
 * (tcgen05.mma kind::f8f6f4, fp32 accumulation in tensor memory).
 *   A8: device E4M3 [M][K] (activations), a_scale: device fp32 [M];
 *   B8: device E4M3 [N][K] (epi 2: [2N][K], gate rows then up rows),
 *   b_scale: device fp32 [N] (epi 2: [2N]); all borrowed.
 * Every product sum is turned into y = bf16(acc * (a_scale[m] * b_scale[n]))
 * (the FP8 projection's bf16 output), then epi 0: C fp32 [M][N] = y;
 * epi 1: C += y; epi 2: C bf16 [M][N] = bf16(silu(y_gate) * y_up).
 * K % 128 == 0, N as tts_gemm_bf16, any M >= 1; tile and K split chosen as
 * by tts_gemm_bf16.  Enqueued on `stream`; does not synchronise.
 * TTS_ERR_ARG for bad sizes, NULL or misaligned pointers (A8, B8, C
 * 16-byte aligned). */
int tts_gemm_fp8(const void* A8, const void* B8, const float* a_scale, const float* b_scale, void* C, int M, int N,
                 int K, int epi, void* stream);

/* Stand-alone op: tts_gemm_bf16 (fp8 = 0; a_scale, b_scale unused) or
 * tts_gemm_fp8 (fp8 = 1) with the tile fixed by the caller: tile_rows 128
 * or 256 (two 128-row accumulators sharing each weight tile), tile_cols
 * 64, 80, 128, 160 or 192 (epi 2: 128), the K range split over `splits`
 * CTAs of a cluster (1..4; epi 2: 1; at most the number of k-blocks).
 * TTS_ERR_ARG when the tile does not fit the shape; otherwise as those. */
int tts_gemm_tiled(const void* A, const void* B, const float* a_scale, const float* b_scale, void* C, int M, int N,
                   int K, int epi, int fp8, int tile_rows, int tile_cols, int splits, void* stream);

/* Per-output-row FP8 weight quantisation on the GPU (FlashRT page,
 * Performance "FP8 W8A8"; section 8, scale amax/448): for each row n,
 * s[n] = max_k |W[n][k]| / 448 (1 if the row is zero) and
 * W8[n][k] = E4M3(W[n][k] / s[n]) rounded to nearest even, saturating.
 * W: DEVICE bf16 [N][K]; W8: DEVICE uint8 [N][K]; s: DEVICE fp32 [N].
 * stream: cudaStream_t or NULL.  Asynchronous. */
int tts_quantize_fp8_weight(const void* W, int N, int K, void* W8, float* s, void* stream);

/* One layer's decode attention as a standalone call, outside a context: the
 * kernel the step uses ("Higgs Audio v3 TTS-4B on FlashRT", section 5: fused
 * q/k-norm + RoPE, KV write, attention).  For position pos it RMS-normalises
 * each query and key head over head_dim 128 (gains q_norm / k_norm), rotates
 * them (rotate-half RoPE, inverse frequencies rope_theta^(-2i/128)), writes the
 * key and value rows of pos to the caches in bf16, and attends the n_q query
 * heads over positions [0, pos] (query head h reads key-value head
 * h / (n_q/n_kv); scores scaled by 1/sqrt(128); softmax over positions).
 * qkv: DEVICE fp32 [(n_q + 2*n_kv)*128] (queries, keys, values);
 * q_norm, k_norm: DEVICE bf16 [128]; k_cache, v_cache: DEVICE bf16
 * [n_kv][max_pos][128] (row pos of each head is overwritten);
 * out: DEVICE fp32 [n_q*128].  n_q/n_kv in {1,2,4,8}; 0 <= pos < max_pos <=
 * 65536 (TTS_ERR_FULL otherwise).  Scratch for the split partials is taken
 * from the stream-ordered allocator and released before returning.
 * Synchronises the stream. */
int tts_attention_decode(const float* qkv, const void* q_norm, const void* k_norm, void* k_cache,
                         void* v_cache, float* out, int n_q, int n_kv, int max_pos, int pos, float eps,
                         float rope_theta, void* stream);

/* tts_attention_decode without any allocation, for callers that cannot
 * allocate device memory during the call: code running under another
 * runtime's fixed memory budget, host loops that must not block on or fail in
 * cudaMalloc, or processes that freeze allocation after start-up.  The paper
 * has no counterpart; this is a library-level variant.
 * Same arguments, layouts and result as tts_attention_decode (bit for bit:
 * the same kernel, split count and merge order).  Its scratch (the split
 * partials, tickets, a state word and the RoPE row) lives in one static
 * device array of 2 MiB per GPU.  Requests needing more (about
 * n_q * min(64, ceil(max_pos/16)) * 520 bytes) are rejected with
 * TTS_ERR_ARG and a message on stderr; nothing is launched.
 * Set-up: under lazy module loading (the CUDA default) the array is created
 * on a device when its module is first loaded there, which happens at the
 * first lookup of its address; the attention kernel's module loads on its
 * first launch.  Both may allocate device memory.  The first call of this
 * entry point on a device does both (and caches the address), and so does
 * tts_init for its device: make one of them part of start-up, while
 * allocation is still allowed.  A device reset unloads the module; do not
 * call this entry point on a device after resetting it.  The call
 * synchronises the stream.  Every call shares the one array; each call
 * clears the tickets and state word before launching, so calls that overlap
 * on the GPU (on different streams, or without ordering) race on it:
 * serialise them.  No cudaMalloc, cudaFree or other allocating routine is
 * called. */
int tts_attention_decode_noalloc(const float* qkv, const void* q_norm, const void* k_norm, void* k_cache,
                                 void* v_cache, float* out, int n_q, int n_kv, int max_pos, int pos,
                                 float eps, float rope_theta, void* stream);

/* Name of a status code (static string). */
const char* tts_status_str(int status);

#ifdef __cplusplus
}
#endif
#endif /* TTS_DECODE_H */

// Internal launch interface of the decode-step kernels.
#pragma once

#include "common.cuh"

namespace tts {

enum Prec { kBF16 = 0, kFP8 = 1 };
enum Pro { kProPlain = 0, kProRms = 1 };
enum Epi { kEpiStore = 0, kEpiResid = 1, kEpiSwiglu = 2, kEpiLogits = 3 };

// ---- weight-streaming geometry (host and device) ------------------------------
// A CTA = kConsumerWarps consumer warps + one producer warp.  Eight consumer
// warps keep the register budget at 168 per thread (nine warps: at most three
// per SM sub-partition).  A lane holds the activations of up to
// kMaxLaneChunks 16-byte weight chunks of its column segment and reduces them
// against up to four rows per ring stage at once.
#ifndef TTS_CONSUMER_WARPS
#define TTS_CONSUMER_WARPS 8
#endif
#ifndef TTS_MAX_LANE_CHUNKS
#define TTS_MAX_LANE_CHUNKS 10
#endif
constexpr int kConsumerWarps = TTS_CONSUMER_WARPS;
constexpr int kMaxLaneChunks = TTS_MAX_LANE_CHUNKS;
// FP8 projections run their stage loop on the tensor cores (E4M3 mma.sync,
// fp32 accumulation).  A stage holds R rows (R = 16, 8, 4 or 2, R x K bytes
// at most kStageTarget); each row is cut into P = 16 / R K-subranges and each
// subrange into kConsumerWarps pieces of whole 64-byte units, so that the 16
// MMA rows of a warp's tile are all (row, subrange) pairs of the stage.
constexpr int kFp8MmaRows = 16;
constexpr int kStageTarget = 40 * 1024;  // bytes per ring stage, at most (unless one row is longer)
constexpr int kMaxRmsK = 4096;            // persistent step: longest normalised activation (hidden)
constexpr int kMaxPlainK = 12288;         // longest plain activation (attention output, MLP activation)

// How one projection with inner dimension K is cut: each row is split into
// wpr column segments (one warp each), so kConsumerWarps / wpr rows are reduced
// side by side ("row slots"); a ring stage holds rs whole rows, 1, 2 or 4 per
// row slot (a warp reduces its rows of a stage together).  wpr is the smallest
// power of two whose segments fit a lane's registers and whose row slots fit
// one stage.
struct StageGeom {
    int rs, wpr;
    bool ok;  // segments fit the lane registers and every warp has a chunk
};
inline __host__ __device__ StageGeom stage_geom(int prec, int epi, int K) {
    if (prec != kBF16) {
        // tensor-core FP8: R rows per stage (a power of two, 2..16, R x K <=
        // kStageTarget), P = 16 / R subranges per row; a row's partial sums
        // are kept per (warp, subrange): wpr = kConsumerWarps x P.  SwiGLU
        // stages hold R / 2 gate and R / 2 up rows.
        int rs = kFp8MmaRows;
        while (rs > 2 && (long long)rs * K > kStageTarget) rs >>= 1;
        const int P = kFp8MmaRows / rs;
        return StageGeom{rs, kConsumerWarps * P, K % 512 == 0 && (long long)rs * K <= kStageTarget};
    }
    const int cpr = K / 8;
    const long long rowb = (long long)cpr * 16;
    auto lane_chunks = [&](int w) { return ((cpr + w - 1) / w + 31) / 32; };
    int wpr = 1;
    const int limit = kMaxLaneChunks;
    while (wpr < kConsumerWarps && lane_chunks(wpr) > limit) wpr *= 2;
    while (wpr < kConsumerWarps && (long long)(kConsumerWarps / wpr) * rowb > kStageTarget) wpr *= 2;
    const int slots = kConsumerWarps / wpr;
    int rs = slots;
    while (rs < 4 * slots && 2LL * rs * rowb <= kStageTarget) rs *= 2;  // up to four rows per warp and stage
    if (epi == kEpiSwiglu && rs < 2) rs = 2;
    return StageGeom{rs, wpr, K % 256 == 0 && cpr >= wpr && lane_chunks(wpr) <= limit};
}

// y = epilogue(W . prologue(x)) for one activation vector (M = 1).
struct GemvParams {
    const void* W;              // [rows][K], bf16 or E4M3 bytes, row-major
    const float* wscale;        // FP8: per-row fp32 scales
    const float* x;             // input activation, fp32 [K]
    const __nv_bfloat16* gamma; // kProRms: RMSNorm gain [K]
    float eps;
    float* y;                   // output [N] (kEpiResid: the residual stream, updated in place)
    int N;                      // outputs (kEpiSwiglu: inter; rows are gate [0,N) and up [N,2N))
    int K;
    // kEpiLogits only: last-CTA greedy argmax + delay mask + state advance
    DevState* st;
    unsigned* counter;          // zero on entry; the last CTA resets it
    int n_cb, cb_vocab;
    int* hist;                  // code history ring [hist_cap][n_cb]
    int hist_cap;
    int* err;                   // error word (DevState::err), may be NULL
    // L2 prefetch of the next projection's weights once this kernel's copies are out:
    // rows split over the grid like this kernel's; next_pf bytes per CTA (0 = none)
    const void* next_W;
    int next_N;
    size_t next_rowb;
    size_t next_pf;
    // ring geometry, filled in by launch_gemv
    int rs, wpr, nstages, part_bytes;
};

// Shared-memory geometry of one GEMV launch: rows per ring stage, ring stages,
// bytes of the per-(row, segment) partial sums, total dynamic smem.
struct GemvGeom {
    int rs, wpr, nstages, part_bytes, smem;
    bool ok;
};

struct LaunchCfg {
    int grid;
    int threads;
    bool pdl;
};

GemvGeom gemv_geom(int prec, int epi, int N, int K, int grid);
cudaError_t gemv_prepare();  // raise the dynamic shared-memory limit of every variant
cudaError_t launch_gemv(int prec, int pro, int epi, const GemvParams& p, const LaunchCfg& lc,
                        cudaStream_t s);

// Decode attention for one layer (q/k RMSNorm + RoPE + KV write fused in).
struct AttnParams {
    const float* qkv;            // [(n_q + 2 n_kv) * 128] fp32
    const __nv_bfloat16* q_norm; // [128]
    const __nv_bfloat16* k_norm; // [128]
    const float2* rope;          // [max_pos][64] (cos, sin), row pos used; or null when rope_row is set
    const float2* rope_row;      // if non-null: the (cos, sin) row [64] of this call's position itself
    __nv_bfloat16* kc;           // this layer's K cache [n_kv][max_pos][128]
    __nv_bfloat16* vc;
    float* out;                  // [n_q * 128] fp32
    float* part_o;               // [n_kv][S][G][128]
    float* part_ml;              // [n_kv][S][G][2]
    unsigned* counter;           // [n_kv], zero on entry; reset by the last CTA
    DevState* st;
    int pos_override;            // >= 0: use this position instead of st->pos (prefill rows)
    int n_q, n_kv, max_pos, S;
    float eps;
};
int attn_splits_for(int max_pos);
cudaError_t attention_prepare();  // load the attention kernels' module on the current device
cudaError_t launch_attention(const AttnParams& p, const LaunchCfg& lc, cudaStream_t s);
// Device address of the allocation-free attention entry point's static
// scratch on the current device (looked up once per device, then cached).
// Returns a TTS_* status.
int static_scratch_address(void** out);

// h = sum_k E_k[codes[k]], codes read from st->codes (or from `rows` when
// non-NULL: row st->prefill_row of a [P][n_cb] prompt).
struct EmbedParams {
    const __nv_bfloat16* E;  // [n_cb][cb_vocab][H]
    DevState* st;
    const int* rows;         // prompt codes or NULL
    float* h;
    int n_cb, cb_vocab, H;
};
cudaError_t launch_embed(const EmbedParams& p, const LaunchCfg& lc, cudaStream_t s);

// st->pos += 1, st->prefill_row += 1 (end of one prefill position).
cudaError_t launch_advance(DevState* st, const LaunchCfg& lc, cudaStream_t s);

// The persistent decode-step kernel (one launch per step or prefill position).
struct StepLayer {
    const void* wqkv;
    const void* wo;
    const void* wgu;
    const void* wd;
    const float* sqkv;
    const float* so;
    const float* sgu;
    const float* sd;
    const __nv_bfloat16* ln_in;
    const __nv_bfloat16* ln_post;
    const __nv_bfloat16* qn;
    const __nv_bfloat16* kn;
};

struct StepParams {
    const StepLayer* layers;  // device array [n_layers]
    int n_layers;
    const __nv_bfloat16* embed;
    const __nv_bfloat16* head;
    const __nv_bfloat16* final_norm;
    const float2* rope;
    __nv_bfloat16* kc;  // [n_layers][n_kv][max_pos][128]
    __nv_bfloat16* vc;
    DevState* st;
    const int* prompt;  // prefill rows [P][n_cb]
    int decode;         // 1: head + argmax + advance; 0: prefill position advance
    float *h, *qkv, *attn, *act, *logits;
    float *part_o, *part_ml;                  // attention split partials
    // the vectors the phases hand to each other, one buffer per layer and
    // kind, and the last-arriver tickets, every word 0xffffffff at launch
    // (the data exchange in gemv_core.cuh; layout: step_xch_words)
    float* xch;
    int* hist;
    int hist_cap;
    int hidden, n_q, n_kv, inter, n_cb, cb_vocab, max_pos;
    int S;  // attention splits per kv head (allocation stride), at most
    float eps;
    int rs[5];   // rows per ring stage: QKV, O, gate/up, down, head
    int wpr[5];  // column segments (warps) per row, same order
    int ns, slot_bytes, xs_bytes, part_bytes;
    unsigned ns_magic;  // floor(2^32 / ns) + 1 (ring_magic)
    int xf_off;  // FP8: byte offset in the activation scratch of the fp32 copy of a plain input
    int pf_stages;  // how many stages the L2 prefetch runs ahead of the ring copies
    int pf_max;     // ... and how far it may run ahead while the ring is full
    // FP8: static activation scales [n_layers][4] (QKV, O, gate/up, down
    // inputs; a site <= 0 is dynamic), and the calibration accumulators
    // (same layout; null outside calibration runs)
    const float* fp8_sa;
    float* fp8_calib;
    // optional phase trace: per CTA, trace_stride globaltimer stamps (ns)
    unsigned long long* trace;
    int trace_stride;
    // optional per-stage trace of CTA 0: for ring stage i, [4 i] copy issued,
    // [4 i + 1] data seen, [4 i + 2] released, [4 i + 3] SM cycles in between,
    // by consumer warp 0 (first stage_trace_stride entries) and by the last
    // consumer warp (next stage_trace_stride entries; no issue time)
    unsigned long long* stage_trace;
    int stage_trace_stride;
    // optional (traced launches): the residual stream after the embedding and
    // after every layer, [n_layers + 1][hidden] fp32
    float* hsnap;
    // bound on each wait for exchanged data in ns (0: kWaitLimitNs), and a
    // test hook: non-zero makes the embedding store nothing, so the first
    // layer's wait for it cannot complete and runs out (0 on the product path)
    unsigned long long wait_limit_ns;
    int fault_skip_embed;
};

// Layout of StepParams::xch in 4-byte words: [0, hidden) h after the
// embedding; then per layer l, from hidden + l * step_xch_layer_words: qkv
// [qkv_rows], attention output [attn_dim], h after the attention [hidden],
// MLP activation [inter], h after the MLP [hidden]; then the counters
// (unsigned): last-arriver tickets of the attention [n_layers][n_q] (one per
// unit slot: kv head, or q head) and of the head [1], then the arrival
// counters of the vectors: the embedding [1], then per layer the five vectors
// in the order above [n_layers][5].
__host__ __device__ inline size_t step_xch_layer_words(int hidden, int qkv_rows, int attn_dim, int inter) {
    return (size_t)qkv_rows + attn_dim + 2 * (size_t)hidden + inter;
}
inline size_t step_xch_words(int n_layers, int hidden, int qkv_rows, int attn_dim, int inter) {
    return (size_t)hidden + (size_t)n_layers * step_xch_layer_words(hidden, qkv_rows, attn_dim, inter) +
           (size_t)n_layers * (attn_dim / 128) + 1 + 1 + 5 * (size_t)n_layers;
}

// Phase-trace layout of the persistent kernel, per CTA (see step.cu):
//   [0] consumer start; [1 + 14 l + k] layer l, event k (after: 0 QKV norm,
//   1 QKV reduce, 3 attention, 5 O stage, 6 O reduce, 8 gate/up norm, 9
//   gate/up reduce, 11 down stage, 12 down reduce; 2, 4, 7, 10 and 13 repeat
//   the event before them: each staging includes its wait for the exchanged
//   input); [1 + 14 L + 0..2] head norm, reduce, tail;
//   [4 + 14 L + 5 l + k] producer: last copy of layer l's projection k issued
//   (k = 4: head), [4 + 19 L + 1] producer done; [8 + 19 L + 4 l + k] ns the
//   consumers waited for ring data in layer l's projection k; [8 + 23 L +
//   4 l + k] ns the producer waited for free slots (the head adds to the last
//   layer's down-proj slot); [8 + 27 L + 4 l + k] the attention unit of layer
//   l: k = 0 inputs loaded (queries and the new key/value row ready), 1
//   positions done, 2 warps merged, 3 splits merged (CTAs without a unit: 0).
inline int step_trace_stride(int n_layers) { return 8 + 31 * n_layers; }

cudaError_t step_prepare(int prec, int G, int smem);
int step_attn_scratch_bytes(int G);
int step_threads();
cudaError_t launch_step(const StepParams& p, int prec, int G, int grid, int smem, cudaStream_t s);

// C = A . B^T on the tensor cores (gemm_tc.cu): A [M][K] and B [N][K], bf16
// or E4M3, K-major, fp32 accumulation.  Epilogues: store fp32 C[M][ldc]; add
// into fp32 C (the residual stream; one writer per element, deterministic);
// SwiGLU: B = [gate rows; up rows] of a [2 n_half][K] matrix,
// out_bf16[M][ldc] = bf16(silu(gate) * up), N = n_half.
enum GemmEpi { kGemmStore = 0, kGemmAdd = 1, kGemmSwiglu = 2 };
struct GemmParams {
    float* C;
    __nv_bfloat16* out_bf16;
    int ldc;
    int M, N, K;
    int n_half;
    int kb_per_split;  // filled in by launch_gemm
    int* err;          // error word (kErrTimeout on an expired wait), may be NULL
    // E4M3 operands: per-row activation scales [M] and per-row weight scales
    // [N] (SwiGLU: [2 n_half]); every product sum becomes
    // bf16(acc * (a_scale[m] * b_scale[n])) before the epilogue's operation
    const float* a_scale;
    const float* b_scale;
};
// A CTA's tile: 128 mt rows (mt = 1 or 2 accumulators sharing each weight
// tile) x bn output columns (64, 80, 128, 160 or 192; SwiGLU: 128 gate + 128
// up), the K range cut over `splits` CTAs of a cluster whose partial sums are
// added in a fixed order.  mt = 0: chosen by gemm_pick (splits > 0 fixes the split).
struct GemmTile {
    int mt, bn, splits;
};
GemmTile gemm_pick(int M, int N, int K, int epi, bool fp8, int num_sms, int splits);
bool gemm_shape_ok(int N, int K, int epi, bool fp8);  // some tile covers N x K
cudaError_t launch_gemm(const void* A, const void* B, const GemmParams& p, int epi, bool fp8, GemmTile t,
                        int num_sms, cudaStream_t s);

// Batched prefill glue (prefill.cu): P rows at positions pos0 .. pos0+P-1.
cudaError_t launch_prefill_embed(const __nv_bfloat16* E, const int* codes, float* H, int P, int n_cb, int V,
                                 int hidden, cudaStream_t s);
cudaError_t launch_prefill_rmsnorm_fp8(const float* H, const __nv_bfloat16* gamma, uint8_t* out, float* scale, int P,
                                       int hidden, float eps, cudaStream_t s);
cudaError_t launch_prefill_quant_rows(const __nv_bfloat16* X, uint8_t* out, float* scale, int P, int n,
                                      cudaStream_t s);
cudaError_t launch_prefill_quant_rows_f32(const float* X, uint8_t* out, float* scale, int P, int n, cudaStream_t s);
cudaError_t launch_prefill_rmsnorm(const float* H, const __nv_bfloat16* gamma, __nv_bfloat16* out, int P,
                                   int hidden, float eps, cudaStream_t s);
cudaError_t launch_prefill_qk_rope_kv(const float* QKV, const __nv_bfloat16* qn, const __nv_bfloat16* kn,
                                      const float2* rope, float* Q, __nv_bfloat16* kc, __nv_bfloat16* vc, int pos0,
                                      int P, int n_q, int n_kv, int max_pos, float eps, cudaStream_t s);
cudaError_t launch_prefill_attention(const float* Q, const __nv_bfloat16* kc, const __nv_bfloat16* vc,
                                     __nv_bfloat16* out, int pos0, int P, int n_q, int n_kv, int max_pos,
                                     cudaStream_t s, float* out_f32 = nullptr);

// Per-row E4M3 weight quantisation.
cudaError_t launch_quantize_weight(const __nv_bfloat16* W, int N, int K, uint8_t* W8, float* s,
                                   cudaStream_t st);

}  // namespace tts

// Internal launch interface of the decode-step kernels.
#pragma once

#include "common.cuh"

namespace tts {

enum Prec { kBF16 = 0, kFP8 = 1 };
enum Pro { kProPlain = 0, kProRms = 1 };
enum Epi { kEpiStore = 0, kEpiResid = 1, kEpiSwiglu = 2, kEpiLogits = 3 };

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
    int rs, nstages, part_bytes;
};

// Shared-memory geometry of one GEMV launch: rows per ring stage, ring stages,
// bytes of the per-(row, segment) partial sums, total dynamic smem.
struct GemvGeom {
    int rs, nstages, part_bytes, smem;
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
    const float2* rope;          // [max_pos][64] (cos, sin)
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
cudaError_t launch_attention(const AttnParams& p, const LaunchCfg& lc, cudaStream_t s);

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

// Per-row E4M3 weight quantisation.
cudaError_t launch_quantize_weight(const __nv_bfloat16* W, int N, int K, uint8_t* W8, float* s,
                                   cudaStream_t st);

}  // namespace tts

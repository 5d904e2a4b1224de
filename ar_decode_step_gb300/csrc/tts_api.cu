// C ABI of the decode-step library: context lifetime, the position-agnostic
// CUDA graph of one decode step, prefill, and state/test accessors.
//
// The whole step (embedding, 36 x [QKV GEMV, fused q/k-norm+RoPE+KV-write
// attention, O-proj+residual, gate/up+SwiGLU, down+residual], head + argmax +
// delay mask) is captured once into a CUDA graph whose kernels read the
// position from device memory ("Higgs Audio v3 TTS-4B on FlashRT",
// Performance: "position-agnostic CUDA graph"; section 7: replayed at any
// position).  Kernels after the first are linked by programmatic dependent
// launch edges so each can start streaming its weights before its producer
// ends.  The graph is destroyed before any buffer it references is freed (the
// TTS-Audio-Suite report's CUDA-graph teardown hazard).
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <set>
#include <tuple>
#include <vector>

#include "kernels.h"
#include "tts_decode.h"

using namespace tts;

namespace {

struct LayerW {
    const void *wqkv, *wo, *wgu, *wd;
    const float *sqkv, *so, *sgu, *sd;
    const __nv_bfloat16 *ln_in, *ln_post, *qn, *kn;
};

}  // namespace

struct tts_ctx {
    tts_config cfg{};
    cudaStream_t stream = nullptr;  // caller's stream (may be the legacy default)
    cudaStream_t cap = nullptr;     // private stream used for graph capture
    int device = 0, num_sms = 0;
    int qkv_rows = 0, attn_dim = 0, G = 1, S = 1;
    bool pdl = true;
    float temperature = 0.f;     // sampling head: <= 0 greedy
    unsigned long long seed = 0;
    // saved prefix (tts_prefix_save): K/V rows [0, pre_len) of every layer and
    // kv head, packed [n_layers][n_kv][pre_len][128], and the state after them
    __nv_bfloat16 *pre_k = nullptr, *pre_v = nullptr;
    int pre_cap = 0, pre_len = 0;
    DevState pre_state{};
    // batched prefill chunks captured as graphs, by (first position, rows,
    // prompt row offset); a chunk shape runs directly the first time
    std::map<std::tuple<int, int, int>, cudaGraphExec_t> pf_graphs;
    std::set<std::tuple<int, int, int>> pf_seen;

    const __nv_bfloat16 *embed = nullptr, *head = nullptr, *final_norm = nullptr;
    std::vector<LayerW> L;

    std::vector<void*> allocs;
    __nv_bfloat16 *kc = nullptr, *vc = nullptr;
    float2* rope = nullptr;
    float *h = nullptr, *qkv = nullptr, *attn = nullptr, *act = nullptr, *logits = nullptr;
    float *part_o = nullptr, *part_ml = nullptr;
    unsigned* counters = nullptr;  // [n_kv] attention tickets, [n_kv] head ticket
    DevState* st = nullptr;
    int* hist = nullptr;
    int* prompt = nullptr;

    DevState* h_in = nullptr;   // pinned staging, host -> device
    DevState* h_out = nullptr;  // pinned staging, device -> host

    // persistent step kernel
    bool persistent = true;
    StepLayer* d_layers = nullptr;
    float* xch = nullptr;  // the persistent step's exchange buffers (StepParams::xch)
    size_t xch_bytes = 0;
    StepParams sp{};
    int step_smem = 0;

    cudaGraphExec_t step_exec = nullptr;     // one decode step
    cudaGraphExec_t prefill_exec = nullptr;  // one prefill position (no head)
    cudaEvent_t ev0 = nullptr, ev1 = nullptr;
    // lookahead loop (tts_decode_until_eoc): double-buffered pinned copies of
    // the state after each frame, and the events that mark them
    DevState* h_ring = nullptr;
    cudaEvent_t ev_ring[2] = {nullptr, nullptr};
    float last_ms = 0.f;
    int pos = 0;  // host shadow of st->pos

    // batched prefill scratch (allocated on first use, kPrefillChunk rows)
    float *pf_h = nullptr, *pf_qkv = nullptr, *pf_q = nullptr, *pf_sa = nullptr, *pf_attn_f = nullptr;
    uint8_t* pf_a8 = nullptr;  // FP8 prefill: the quantised projection input rows
    __nv_bfloat16 *pf_a = nullptr, *pf_attn = nullptr, *pf_m = nullptr;
    bool batched_prefill = true;
};

namespace {

int report(cudaError_t e, const char* what) {
    std::fprintf(stderr, "tts: %s failed: %s\n", what, cudaGetErrorString(e));
    return TTS_ERR_CUDA;
}

#define TTS_CK(call)                                      \
    do {                                                  \
        cudaError_t e_ = (call);                          \
        if (e_ != cudaSuccess) return report(e_, #call);  \
    } while (0)

bool aligned16(const void* p) { return p && ((uintptr_t)p & 15u) == 0; }

int validate(const tts_config* c, const tts_weights* w) {
    if (!c || !w) return TTS_ERR_ARG;
    if (c->n_layers < 1 || c->n_layers > 4096) return TTS_ERR_ARG;
    if (c->head_dim != kHeadDim) return TTS_ERR_ARG;
    if (c->n_kv_heads < 1 || c->n_q_heads < 1 || c->n_q_heads % c->n_kv_heads) return TTS_ERR_ARG;
    const int G = c->n_q_heads / c->n_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8) return TTS_ERR_ARG;
    // GEMV inputs are staged in 48 KB of shared memory as fp32: K <= 12288
    if (c->hidden < 256 || c->hidden % 256 || c->hidden > 12288) return TTS_ERR_ARG;
    if (c->inter < 256 || c->inter % 256 || c->inter > 12288) return TTS_ERR_ARG;
    if ((long long)c->n_q_heads * kHeadDim > 12288) return TTS_ERR_ARG;
    if (c->n_codebooks < 1 || c->n_codebooks > kMaxCodebooks) return TTS_ERR_ARG;
    if (c->cb_vocab < 2 || c->cb_vocab > (1 << 20)) return TTS_ERR_ARG;
    if (c->max_pos < 1 || c->max_pos > 65536) return TTS_ERR_ARG;
    if (!(c->rms_eps >= 0.f) || !(c->rope_theta > 0.f)) return TTS_ERR_ARG;
    if (c->precision != TTS_BF16 && c->precision != TTS_FP8) return TTS_ERR_ARG;
    if (c->options & ~(TTS_OPT_SEPARATE_KERNELS | TTS_OPT_PREFILL_STEPS)) return TTS_ERR_ARG;
    if (!aligned16(w->embed) || !aligned16(w->head) || !aligned16(w->final_norm)) return TTS_ERR_ARG;
    if (!w->wqkv || !w->wo || !w->wgu || !w->wd || !w->ln_in || !w->ln_post || !w->q_norm || !w->k_norm)
        return TTS_ERR_ARG;
    const bool fp8 = c->precision == TTS_FP8;
    if (fp8 && (!w->sqkv || !w->so || !w->sgu || !w->sd)) return TTS_ERR_ARG;
    // FP8 projections reduce whole 64-byte units of each row on the tensor
    // cores, in stages of at least 2 rows: K a multiple of 512, at most 20480
    if (fp8)
        for (const long long K : {(long long)c->hidden, (long long)c->inter, (long long)c->n_q_heads * kHeadDim})
            if (!stage_geom(kFP8, kEpiStore, (int)K).ok) return TTS_ERR_ARG;
    for (int l = 0; l < c->n_layers; ++l) {
        if (!aligned16(w->wqkv[l]) || !aligned16(w->wo[l]) || !aligned16(w->wgu[l]) || !aligned16(w->wd[l]))
            return TTS_ERR_ARG;
        if (!aligned16(w->ln_in[l]) || !aligned16(w->ln_post[l]) || !aligned16(w->q_norm[l]) ||
            !aligned16(w->k_norm[l]))
            return TTS_ERR_ARG;
        if (fp8 && (!aligned16(w->sqkv[l]) || !aligned16(w->so[l]) || !aligned16(w->sgu[l]) || !aligned16(w->sd[l])))
            return TTS_ERR_ARG;
    }
    return TTS_OK;
}

template <typename T>
int dalloc(tts_ctx* c, T** p, size_t count) {
    void* q = nullptr;
    TTS_CK(cudaMalloc(&q, count * sizeof(T) > 0 ? count * sizeof(T) : 16));
    c->allocs.push_back(q);
    *p = static_cast<T*>(q);
    return TTS_OK;
}

#define TTS_TRY(expr)              \
    do {                           \
        int r_ = (expr);           \
        if (r_ != TTS_OK) return r_; \
    } while (0)

LaunchCfg gemv_cfg(const tts_ctx* c, bool pdl) { return LaunchCfg{c->num_sms, 0, pdl}; }

enum Proj { kQKV = 0, kO = 1, kGU = 2, kDown = 3, kHead = 4 };

// Parameters of projection `kind` of layer l (kHead ignores l).
GemvParams proj_params(const tts_ctx* c, int kind, int l) {
    const tts_config& k = c->cfg;
    GemvParams g{};
    g.eps = k.rms_eps;
    g.err = &c->st->err;
    if (kind == kHead) {
        g.W = c->head; g.x = c->h; g.gamma = c->final_norm; g.y = c->logits;
        g.N = k.n_codebooks * k.cb_vocab; g.K = k.hidden;
        return g;
    }
    const LayerW& w = c->L[l];
    switch (kind) {
        case kQKV: g.W = w.wqkv; g.wscale = w.sqkv; g.x = c->h; g.gamma = w.ln_in; g.y = c->qkv;
                   g.N = c->qkv_rows; g.K = k.hidden; break;
        case kO:   g.W = w.wo; g.wscale = w.so; g.x = c->attn; g.y = c->h; g.N = k.hidden; g.K = c->attn_dim; break;
        case kGU:  g.W = w.wgu; g.wscale = w.sgu; g.x = c->h; g.gamma = w.ln_post; g.y = c->act;
                   g.N = k.inter; g.K = k.hidden; break;
        default:   g.W = w.wd; g.wscale = w.sd; g.x = c->act; g.y = c->h; g.N = k.hidden; g.K = k.inter; break;
    }
    return g;
}

// Point g's L2 prefetch at projection `kind` of layer l (the one launched next).
void set_next(const tts_ctx* c, GemvParams& g, int kind, int l, size_t pf_bytes) {
    const GemvParams n = proj_params(c, kind, l);
    const size_t wb = (kind == kHead || c->cfg.precision == TTS_BF16) ? 2 : 1;
    g.next_W = n.W;
    g.next_N = n.N;
    g.next_rowb = (size_t)n.K * wb;
    g.next_pf = pf_bytes;
}

// Separate-kernel mode: bytes of the next projection's weights each GEMV CTA
// asks L2 for once its own copies are out (after the QKV GEMV, for the
// attention kernel that follows: more, since attention streams no weights).
constexpr size_t kGemvPrefetchBytes = 96 * 1024;
constexpr size_t kGemvPrefetchAttnBytes = 160 * 1024;
// Persistent kernel: how many ring stages the L2 prefetch cursor runs ahead
// of the copies, and how far it may run ahead while the ring is full
// (measured: 4 and 12 stages).
constexpr int kStepPrefetchStages = 4;
constexpr int kStepPrefetchMax = 12;

// Every exchange word of the persistent step back to 0xffffffff (the unset
// sentinel, and the tickets' starting value): before every launch.
cudaError_t xch_reset(tts_ctx* c, cudaStream_t s) { return cudaMemsetAsync(c->xch, 0xFF, c->xch_bytes, s); }

// Persistent form: reset the exchange buffers, then one cooperative launch.
int record_step_persistent(tts_ctx* c, cudaStream_t s, bool decode) {
    StepParams p = c->sp;
    p.decode = decode ? 1 : 0;
    TTS_CK(xch_reset(c, s));
    const int prec = c->cfg.precision == TTS_FP8 ? kFP8 : kBF16;
    TTS_CK(launch_step(p, prec, c->G, c->num_sms, c->step_smem, s));
    return TTS_OK;
}

// Enqueue one position through the layer stack, then either the head (decode)
// or the prefill advance.
int record_step(tts_ctx* c, cudaStream_t s, bool decode) {
    if (c->persistent) return record_step_persistent(c, s, decode);
    const tts_config& k = c->cfg;
    const int prec = k.precision == TTS_FP8 ? kFP8 : kBF16;
    const size_t pf = kGemvPrefetchBytes, pf_attn = kGemvPrefetchAttnBytes;
    EmbedParams ep{c->embed, c->st, decode ? nullptr : c->prompt, c->h, k.n_codebooks, k.cb_vocab, k.hidden};
    TTS_CK(launch_embed(ep, LaunchCfg{0, 0, false}, s));
    for (int l = 0; l < k.n_layers; ++l) {
        const LayerW& w = c->L[l];
        const bool last = l + 1 == k.n_layers;
        // QKV: input RMSNorm (+ FP8 quant) fused in the prologue
        GemvParams g = proj_params(c, kQKV, l);
        set_next(c, g, kO, l, pf_attn);
        TTS_CK(launch_gemv(prec, kProRms, kEpiStore, g, gemv_cfg(c, c->pdl), s));
        // attention with q/k norm + RoPE + KV write
        AttnParams a{};
        a.qkv = c->qkv; a.q_norm = w.qn; a.k_norm = w.kn; a.rope = c->rope;
        const size_t lay = (size_t)l * k.n_kv_heads * k.max_pos * kHeadDim;
        a.kc = c->kc + lay; a.vc = c->vc + lay;
        a.out = c->attn; a.part_o = c->part_o; a.part_ml = c->part_ml; a.counter = c->counters;
        a.st = c->st; a.pos_override = -1;
        a.n_q = k.n_q_heads; a.n_kv = k.n_kv_heads; a.max_pos = k.max_pos; a.S = c->S; a.eps = k.rms_eps;
        TTS_CK(launch_attention(a, LaunchCfg{0, 0, c->pdl}, s));
        // O-proj with residual add into h
        g = proj_params(c, kO, l);
        set_next(c, g, kGU, l, pf);
        TTS_CK(launch_gemv(prec, kProPlain, kEpiResid, g, gemv_cfg(c, c->pdl), s));
        // post-attention RMSNorm + gate/up + SwiGLU
        g = proj_params(c, kGU, l);
        set_next(c, g, kDown, l, pf);
        TTS_CK(launch_gemv(prec, kProRms, kEpiSwiglu, g, gemv_cfg(c, c->pdl), s));
        // down-proj with residual add into h
        g = proj_params(c, kDown, l);
        if (!last) set_next(c, g, kQKV, l + 1, pf);
        else if (decode) set_next(c, g, kHead, 0, pf);
        TTS_CK(launch_gemv(prec, kProPlain, kEpiResid, g, gemv_cfg(c, c->pdl), s));
    }
    if (decode) {
        GemvParams g = proj_params(c, kHead, 0);
        set_next(c, g, kQKV, 0, pf);  // the next frame starts with layer 0's QKV
        g.st = c->st; g.counter = c->counters + k.n_kv_heads; g.n_cb = k.n_codebooks; g.cb_vocab = k.cb_vocab;
        g.hist = c->hist; g.hist_cap = k.max_pos;
        TTS_CK(launch_gemv(kBF16, kProRms, kEpiLogits, g, gemv_cfg(c, c->pdl), s));
    } else {
        TTS_CK(launch_advance(c->st, LaunchCfg{0, 0, c->pdl}, s));
    }
    return TTS_OK;
}

int capture(tts_ctx* c, bool decode, cudaGraphExec_t* out) {
    cudaGraph_t graph = nullptr;
    TTS_CK(cudaStreamBeginCapture(c->cap, cudaStreamCaptureModeThreadLocal));
    int rc = record_step(c, c->cap, decode);
    cudaError_t e = cudaStreamEndCapture(c->cap, &graph);
    if (rc != TTS_OK) {
        if (graph) cudaGraphDestroy(graph);
        return rc;
    }
    if (e != cudaSuccess) return report(e, "cudaStreamEndCapture");
    e = cudaGraphInstantiate(out, graph, 0);
    cudaGraphDestroy(graph);
    if (e != cudaSuccess) return report(e, "cudaGraphInstantiate");
    TTS_CK(cudaGraphUpload(*out, c->stream));
    return TTS_OK;
}

// Read the device state into h_out (synchronising) and check the error word.
int pull_state(tts_ctx* c) {
    TTS_CK(cudaMemcpyAsync(c->h_out, c->st, sizeof(DevState), cudaMemcpyDeviceToHost, c->stream));
    TTS_CK(cudaStreamSynchronize(c->stream));
    c->pos = c->h_out->pos;
    if (c->h_out->err) {
        const int zero = 0;
        cudaMemcpy(&c->st->err, &zero, sizeof(int), cudaMemcpyHostToDevice);
        return TTS_ERR_DEVICE;
    }
    return TTS_OK;
}

int push_state(tts_ctx* c, const DevState& s) {
    *c->h_in = s;
    c->h_in->temperature = c->temperature;  // the sampling settings outlive resets and rewinds
    c->h_in->seed = c->seed;
    TTS_CK(cudaMemcpyAsync(c->st, c->h_in, sizeof(DevState), cudaMemcpyHostToDevice, c->stream));
    TTS_CK(cudaStreamSynchronize(c->stream));
    c->pos = s.pos;
    return TTS_OK;
}

DevState bos_state(const tts_ctx* c, int pos, int t, int eoc) {
    DevState s{};
    s.pos = pos;
    s.t = t;
    s.eoc = eoc;
    for (int k = 0; k < kMaxCodebooks; ++k) s.codes[k] = c->cfg.cb_vocab - 2;
    return s;
}

int round128i(int x) { return (x + 127) & ~127; }

// Shared-memory geometry of the persistent step kernel and its parameter block.
int setup_persistent(tts_ctx* c) {
    const tts_config& k = c->cfg;
    const int prec = k.precision == TTS_FP8 ? kFP8 : kBF16;
    const int H = k.hidden, A = c->attn_dim, I = k.inter, grid = c->num_sms;
    struct KindShape { int N, K, prec, epi; };
    const KindShape kinds[5] = {{c->qkv_rows, H, prec, kEpiStore}, {H, A, prec, kEpiResid},
                                {I, H, prec, kEpiSwiglu},          {H, I, prec, kEpiResid},
                                {k.n_codebooks * k.cb_vocab, H, kBF16, kEpiStore}};
    StepParams& p = c->sp;
    int slot = 0, part = 0;
    for (int i = 0; i < 5; ++i) {
        const KindShape& ks = kinds[i];
        const StageGeom g = stage_geom(ks.prec, ks.epi, ks.K);
        if (!g.ok) return TTS_ERR_ARG;  // segments must fit the lane registers
        if ((g.rs & (g.rs - 1)) || (g.wpr & (g.wpr - 1))) return TTS_ERR_ARG;  // the kernels shift, not divide
        const int rowb = ks.K / (ks.prec == kBF16 ? 8 : 16) * 16;
        p.rs[i] = g.rs;
        p.wpr[i] = g.wpr;
        slot = std::max(slot, g.rs * rowb);
        const int opst = ks.epi == kEpiSwiglu ? g.rs / 2 : g.rs;
        const int rows_max = (ks.N + grid - 1) / grid;
        part = std::max(part, (rows_max + opst - 1) / opst * g.rs * g.wpr * (int)sizeof(float));
    }
    // shared scratch: the staged activation vector, or the attention unit's state
    // bf16: plain inputs (attention output, MLP activation) are read into
    // registers directly, only RMSNorm inputs are staged (fp32, as is the
    // head's input in both precisions); FP8 stages all as E4M3 bytes, plain
    // inputs through an fp32 copy at xf_off
    const int xf_off = round128i(std::max({H, A, I}));
    int xs = prec == kBF16 ? std::max(H * 4, step_attn_scratch_bytes(c->G))
                           : std::max({H * 4, xf_off + 4 * std::max(A, I), step_attn_scratch_bytes(c->G)});
    xs = round128i(xs);
    part = round128i(part);
    const int budget = 225 * 1024;
    if ((H + grid - 1) / grid > 256) return TTS_ERR_ARG;           // rows of h per CTA kept in shared memory
    const int tbl = round128i(k.n_layers * (int)sizeof(StepLayer));  // per-layer pointer table
    int ns = (budget - 128 - tbl - xs - part) / slot;
    // ring depth: deeper rings measured slower (more bytes queued per SM for
    // the same L2-to-SM rate; the L2 prefetch keeps HBM busy instead):
    // BF16 4 slots (1.953 -> 1.929 ms per frame), FP8 3 (2.152 -> 2.108)
    ns = std::min(ns, prec == kBF16 ? 4 : 3);
    if (ns < 2) return TTS_ERR_ARG;
    c->step_smem = 128 + tbl + xs + part + ns * slot;
    p.ns = ns;
    p.ns_magic = 0xffffffffu / (unsigned)ns + 1u;
    p.slot_bytes = slot;
    p.xs_bytes = xs;
    p.part_bytes = part;
    p.xf_off = xf_off;

    std::vector<StepLayer> layers(k.n_layers);
    for (int l = 0; l < k.n_layers; ++l) {
        const LayerW& w = c->L[l];
        layers[l] = StepLayer{w.wqkv, w.wo, w.wgu, w.wd, w.sqkv, w.so, w.sgu, w.sd, w.ln_in, w.ln_post, w.qn, w.kn};
    }
    TTS_TRY(dalloc(c, &c->d_layers, (size_t)k.n_layers));
    TTS_CK(cudaMemcpy(c->d_layers, layers.data(), layers.size() * sizeof(StepLayer), cudaMemcpyHostToDevice));
    c->xch_bytes = 4 * step_xch_words(k.n_layers, H, c->qkv_rows, A, I);
    TTS_TRY(dalloc(c, &c->xch, c->xch_bytes / 4));
    p.fp8_sa = nullptr;
    p.fp8_calib = nullptr;
    if (prec == kFP8) {  // static activation scales, all dynamic until set
        float* sa = nullptr;
        TTS_TRY(dalloc(c, &sa, (size_t)k.n_layers * 4));
        TTS_CK(cudaMemset(sa, 0, sizeof(float) * (size_t)k.n_layers * 4));
        p.fp8_sa = sa;
    }
    TTS_CK(step_prepare(prec, c->G, c->step_smem));

    p.layers = c->d_layers;
    p.n_layers = k.n_layers;
    p.embed = c->embed;
    p.head = c->head;
    p.final_norm = c->final_norm;
    p.rope = c->rope;
    p.kc = c->kc;
    p.vc = c->vc;
    p.st = c->st;
    p.prompt = c->prompt;
    p.h = c->h; p.qkv = c->qkv; p.attn = c->attn; p.act = c->act; p.logits = c->logits;
    p.part_o = c->part_o; p.part_ml = c->part_ml;
    p.xch = c->xch;
    p.hist = c->hist;
    p.hist_cap = k.max_pos;
    p.hidden = H; p.n_q = k.n_q_heads; p.n_kv = k.n_kv_heads; p.inter = I;
    p.n_cb = k.n_codebooks; p.cb_vocab = k.cb_vocab; p.max_pos = k.max_pos;
    p.S = c->S;
    p.eps = k.rms_eps;
    // L2 prefetch lookahead in ring stages: steady state, and while the ring is full
    p.pf_stages = kStepPrefetchStages;
    p.pf_max = kStepPrefetchMax;
    return TTS_OK;
}

int init_impl(tts_ctx* c, const tts_config* cfg, const tts_weights* w) {
    c->cfg = *cfg;
    const tts_config& k = c->cfg;
    c->stream = static_cast<cudaStream_t>(cfg->stream);
    c->qkv_rows = (k.n_q_heads + 2 * k.n_kv_heads) * kHeadDim;
    c->attn_dim = k.n_q_heads * kHeadDim;
    c->G = k.n_q_heads / k.n_kv_heads;
    c->S = attn_splits_for(k.max_pos);

    TTS_CK(cudaGetDevice(&c->device));
    {
        // load the allocation-free attention entry point's modules (its static
        // scratch and its kernel) on this device now, while allocating is allowed
        void* scratch = nullptr;
        TTS_TRY(static_scratch_address(&scratch));
        TTS_CK(attention_prepare());
    }
    TTS_CK(gemv_prepare());
    TTS_CK(cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device));
    TTS_CK(cudaStreamCreateWithFlags(&c->cap, cudaStreamNonBlocking));
    TTS_CK(cudaEventCreate(&c->ev0));
    TTS_CK(cudaEventCreate(&c->ev1));
    for (auto& e : c->ev_ring) TTS_CK(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));

    c->embed = static_cast<const __nv_bfloat16*>(w->embed);
    c->head = static_cast<const __nv_bfloat16*>(w->head);
    c->final_norm = static_cast<const __nv_bfloat16*>(w->final_norm);
    const bool fp8 = k.precision == TTS_FP8;
    c->L.resize(k.n_layers);
    for (int l = 0; l < k.n_layers; ++l) {
        LayerW& x = c->L[l];
        x.wqkv = w->wqkv[l]; x.wo = w->wo[l]; x.wgu = w->wgu[l]; x.wd = w->wd[l];
        x.sqkv = fp8 ? w->sqkv[l] : nullptr; x.so = fp8 ? w->so[l] : nullptr;
        x.sgu = fp8 ? w->sgu[l] : nullptr; x.sd = fp8 ? w->sd[l] : nullptr;
        x.ln_in = static_cast<const __nv_bfloat16*>(w->ln_in[l]);
        x.ln_post = static_cast<const __nv_bfloat16*>(w->ln_post[l]);
        x.qn = static_cast<const __nv_bfloat16*>(w->q_norm[l]);
        x.kn = static_cast<const __nv_bfloat16*>(w->k_norm[l]);
    }

    const size_t kv = (size_t)k.n_layers * k.n_kv_heads * k.max_pos * kHeadDim;
    TTS_TRY(dalloc(c, &c->kc, kv));
    TTS_TRY(dalloc(c, &c->vc, kv));
    TTS_TRY(dalloc(c, &c->rope, (size_t)k.max_pos * (kHeadDim / 2)));
    TTS_TRY(dalloc(c, &c->h, k.hidden));
    TTS_TRY(dalloc(c, &c->qkv, c->qkv_rows));
    TTS_TRY(dalloc(c, &c->attn, c->attn_dim));
    TTS_TRY(dalloc(c, &c->act, k.inter));
    TTS_TRY(dalloc(c, &c->logits, (size_t)k.n_codebooks * k.cb_vocab));
    TTS_TRY(dalloc(c, &c->part_o, (size_t)k.n_kv_heads * c->S * c->G * kHeadDim));
    TTS_TRY(dalloc(c, &c->part_ml, (size_t)k.n_kv_heads * c->S * c->G * 2));
    TTS_TRY(dalloc(c, &c->counters, (size_t)2 * k.n_kv_heads));
    TTS_TRY(dalloc(c, &c->st, 1));
    TTS_TRY(dalloc(c, &c->hist, (size_t)k.max_pos * k.n_codebooks));
    TTS_TRY(dalloc(c, &c->prompt, (size_t)k.max_pos * k.n_codebooks));
    TTS_CK(cudaMemsetAsync(c->kc, 0, kv * sizeof(__nv_bfloat16), c->stream));
    TTS_CK(cudaMemsetAsync(c->vc, 0, kv * sizeof(__nv_bfloat16), c->stream));
    TTS_CK(cudaMemsetAsync(c->counters, 0, 2 * k.n_kv_heads * sizeof(unsigned), c->stream));
    TTS_CK(cudaMemsetAsync(c->h, 0, k.hidden * sizeof(float), c->stream));
    TTS_CK(cudaMemsetAsync(c->logits, 0, (size_t)k.n_codebooks * k.cb_vocab * sizeof(float), c->stream));
    TTS_CK(cudaHostAlloc((void**)&c->h_in, sizeof(DevState), cudaHostAllocDefault));
    TTS_CK(cudaHostAlloc((void**)&c->h_out, sizeof(DevState), cudaHostAllocDefault));
    TTS_CK(cudaHostAlloc((void**)&c->h_ring, 2 * sizeof(DevState), cudaHostAllocDefault));

    // RoPE table: inverse frequencies theta^(-2i/D), angle pos * inv_f in fp64,
    // cos/sin rounded to fp32.
    {
        std::vector<float2> tab((size_t)k.max_pos * (kHeadDim / 2));
        for (int p = 0; p < k.max_pos; ++p)
            for (int i = 0; i < kHeadDim / 2; ++i) {
                const double inv_f = std::pow((double)k.rope_theta, -2.0 * i / (double)kHeadDim);
                const double ang = (double)p * inv_f;
                tab[(size_t)p * (kHeadDim / 2) + i] = make_float2((float)std::cos(ang), (float)std::sin(ang));
            }
        TTS_CK(cudaMemcpy(c->rope, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice));
    }
    // options: the step as a graph of separate kernels instead of the
    // persistent kernel; prompts position by position through the decode step
    c->persistent = (k.options & TTS_OPT_SEPARATE_KERNELS) == 0;
    c->batched_prefill = (k.options & TTS_OPT_PREFILL_STEPS) == 0;
    // the persistent kernel stages a normalised activation from registers
    // (hidden <= kMaxRmsK) and plain ones through shared memory (<= kMaxPlainK):
    // larger models take the graph of kernels
    if (c->cfg.hidden > kMaxRmsK || c->attn_dim > kMaxPlainK || c->cfg.inter > kMaxPlainK) c->persistent = false;
    if (c->persistent) TTS_TRY(setup_persistent(c));
    TTS_TRY(push_state(c, bos_state(c, 0, 0, -1)));
    TTS_TRY(capture(c, true, &c->step_exec));
    TTS_TRY(capture(c, false, &c->prefill_exec));
    TTS_CK(cudaStreamSynchronize(c->stream));
    return TTS_OK;
}

constexpr int kPrefillChunk = 512;  // rows per batched pass (the prompt is split into chunks)

// Whether tts_prefill runs the batched tensor-core path: BF16 weights (the
// tensor-core GEMM takes bf16 operands), K and N multiples of the GEMM tiles.
bool batched_prefill_ok(const tts_ctx* c) {
    const tts_config& k = c->cfg;
    const int G = k.n_q_heads / k.n_kv_heads;
    const bool f8 = k.precision == TTS_FP8;
    return c->batched_prefill && k.head_dim == kHeadDim && gemm_shape_ok(c->qkv_rows, k.hidden, kGemmStore, f8) &&
           gemm_shape_ok(k.hidden, c->attn_dim, kGemmAdd, f8) && gemm_shape_ok(k.inter, k.hidden, kGemmSwiglu, f8) &&
           gemm_shape_ok(k.hidden, k.inter, kGemmAdd, f8) && (G == 1 || G == 2 || G == 4 || G == 8);
}

// P rows (codes already on the device at c->prompt) through every layer at
// positions pos0 .. pos0+P-1: W16A16 tensor-core GEMMs, fp32 residual stream,
// bf16 K/V written to the cache.  P <= kPrefillChunk.
// The batched prefill of an FP8 context: the same layer as prefill_chunk with
// W8A8 projections (per-token activation scales, per-row weight scales, bf16
// projection outputs; the SwiGLU of the bf16-rounded gate and up, rounded to
// bf16 before its own quantisation), as the FP8 decode step computes them.
int prefill_chunk_fp8(tts_ctx* c, const int* d_codes, int pos0, int P, float* snap) {
    const tts_config& k = c->cfg;
    const int H = k.hidden, I = k.inter, A = c->attn_dim, QD = c->qkv_rows;
    cudaStream_t s = c->stream;
    int* err = &c->st->err;
    TTS_CK(launch_prefill_embed(c->embed, d_codes, c->pf_h, P, k.n_codebooks, k.cb_vocab, H, s));
    const size_t rows_bytes = sizeof(float) * (size_t)P * H;
    if (snap) TTS_CK(cudaMemcpyAsync(snap, c->pf_h, rows_bytes, cudaMemcpyDeviceToDevice, s));
    for (int l = 0; l < k.n_layers; ++l) {
        const LayerW& w = c->L[l];
        const size_t coff = (size_t)l * k.n_kv_heads * k.max_pos * kHeadDim;
        GemmParams g{};
        g.M = P; g.err = err; g.a_scale = c->pf_sa;
        TTS_CK(launch_prefill_rmsnorm_fp8(c->pf_h, w.ln_in, c->pf_a8, c->pf_sa, P, H, k.rms_eps, s));
        g.C = c->pf_qkv; g.ldc = QD; g.N = QD; g.K = H; g.b_scale = w.sqkv;
        TTS_CK(launch_gemm(c->pf_a8, w.wqkv, g, kGemmStore, true, GemmTile{}, c->num_sms, s));
        TTS_CK(launch_prefill_qk_rope_kv(c->pf_qkv, w.qn, w.kn, c->rope, c->pf_q, c->kc + coff, c->vc + coff, pos0,
                                         P, k.n_q_heads, k.n_kv_heads, k.max_pos, k.rms_eps, s));
        // fp32 attention output, quantised per row next
        TTS_CK(launch_prefill_attention(c->pf_q, c->kc + coff, c->vc + coff, nullptr, pos0, P, k.n_q_heads,
                                        k.n_kv_heads, k.max_pos, s, c->pf_attn_f));
        TTS_CK(launch_prefill_quant_rows_f32(c->pf_attn_f, c->pf_a8, c->pf_sa, P, A, s));
        g.C = c->pf_h; g.ldc = H; g.N = H; g.K = A; g.b_scale = w.so;
        TTS_CK(launch_gemm(c->pf_a8, w.wo, g, kGemmAdd, true, GemmTile{}, c->num_sms, s));
        TTS_CK(launch_prefill_rmsnorm_fp8(c->pf_h, w.ln_post, c->pf_a8, c->pf_sa, P, H, k.rms_eps, s));
        g.C = nullptr; g.out_bf16 = c->pf_m; g.ldc = I; g.N = I; g.n_half = I; g.K = H; g.b_scale = w.sgu;
        TTS_CK(launch_gemm(c->pf_a8, w.wgu, g, kGemmSwiglu, true, GemmTile{}, c->num_sms, s));
        TTS_CK(launch_prefill_quant_rows(c->pf_m, c->pf_a8, c->pf_sa, P, I, s));
        g.out_bf16 = nullptr; g.C = c->pf_h; g.ldc = H; g.N = H; g.n_half = 0; g.K = I; g.b_scale = w.sd;
        TTS_CK(launch_gemm(c->pf_a8, w.wd, g, kGemmAdd, true, GemmTile{}, c->num_sms, s));
        if (snap)
            TTS_CK(cudaMemcpyAsync(snap + (size_t)(l + 1) * P * H, c->pf_h, rows_bytes, cudaMemcpyDeviceToDevice, s));
    }
    return TTS_OK;
}

int prefill_chunk(tts_ctx* c, const int* d_codes, int pos0, int P, float* snap = nullptr) {
    const tts_config& k = c->cfg;
    const int H = k.hidden, I = k.inter, A = c->attn_dim, QD = c->qkv_rows;
    cudaStream_t s = c->stream;
    if (!c->pf_h) {
        const size_t R = kPrefillChunk;
        TTS_TRY(dalloc(c, &c->pf_h, R * H));
        TTS_TRY(dalloc(c, &c->pf_qkv, R * QD));
        TTS_TRY(dalloc(c, &c->pf_q, R * A));
        TTS_TRY(dalloc(c, &c->pf_a, R * H));
        TTS_TRY(dalloc(c, &c->pf_attn, R * A));
        TTS_TRY(dalloc(c, &c->pf_m, R * I));
        if (k.precision == TTS_FP8) {
            TTS_TRY(dalloc(c, &c->pf_a8, R * (size_t)std::max({H, A, I})));
            TTS_TRY(dalloc(c, &c->pf_sa, R));
            TTS_TRY(dalloc(c, &c->pf_attn_f, R * A));
        }
    }
    if (k.precision == TTS_FP8) return prefill_chunk_fp8(c, d_codes, pos0, P, snap);
    int* err = &c->st->err;
    TTS_CK(launch_prefill_embed(c->embed, d_codes, c->pf_h, P, k.n_codebooks, k.cb_vocab, H, s));
    const size_t rows_bytes = sizeof(float) * (size_t)P * H;
    if (snap) TTS_CK(cudaMemcpyAsync(snap, c->pf_h, rows_bytes, cudaMemcpyDeviceToDevice, s));
    // each GEMM's tile and K split chosen to fill the SMs (gemm_pick); split
    // sums are added in a fixed order, so the residual stream is deterministic
    for (int l = 0; l < k.n_layers; ++l) {
        const LayerW& w = c->L[l];
        const size_t coff = (size_t)l * k.n_kv_heads * k.max_pos * kHeadDim;
        TTS_CK(launch_prefill_rmsnorm(c->pf_h, w.ln_in, c->pf_a, P, H, k.rms_eps, s));
        GemmParams g{};
        g.M = P; g.err = err;
        g.C = c->pf_qkv; g.ldc = QD; g.N = QD; g.K = H;
        TTS_CK(launch_gemm(c->pf_a, w.wqkv, g, kGemmStore, false, GemmTile{}, c->num_sms, s));
        TTS_CK(launch_prefill_qk_rope_kv(c->pf_qkv, w.qn, w.kn, c->rope, c->pf_q, c->kc + coff, c->vc + coff, pos0,
                                         P, k.n_q_heads, k.n_kv_heads, k.max_pos, k.rms_eps, s));
        TTS_CK(launch_prefill_attention(c->pf_q, c->kc + coff, c->vc + coff, c->pf_attn, pos0, P, k.n_q_heads,
                                        k.n_kv_heads, k.max_pos, s));
        g.C = c->pf_h; g.ldc = H; g.N = H; g.K = A;
        TTS_CK(launch_gemm(c->pf_attn, w.wo, g, kGemmAdd, false, GemmTile{}, c->num_sms, s));
        TTS_CK(launch_prefill_rmsnorm(c->pf_h, w.ln_post, c->pf_a, P, H, k.rms_eps, s));
        g.C = nullptr; g.out_bf16 = c->pf_m; g.ldc = I; g.N = I; g.n_half = I; g.K = H;
        TTS_CK(launch_gemm(c->pf_a, w.wgu, g, kGemmSwiglu, false, GemmTile{}, c->num_sms, s));
        g.out_bf16 = nullptr; g.C = c->pf_h; g.ldc = H; g.N = H; g.n_half = 0; g.K = I;
        TTS_CK(launch_gemm(c->pf_m, w.wd, g, kGemmAdd, false, GemmTile{}, c->num_sms, s));
        if (snap)
            TTS_CK(cudaMemcpyAsync(snap + (size_t)(l + 1) * P * H, c->pf_h, rows_bytes, cudaMemcpyDeviceToDevice, s));
    }
    return TTS_OK;
}

// One batched prefill chunk, replayed from a captured graph once its shape
// has run before (the first run also does the lazy set-up: buffers, kernel
// attributes): the ~290 launches of a 36-layer chunk then cost one.  At most
// kMaxPrefillGraphs graphs are kept; the record of shapes seen once is
// bounded too (cleared when full).
constexpr size_t kMaxPrefillGraphs = 16;
constexpr size_t kMaxPrefillSeen = 1024;
int run_prefill_chunk(tts_ctx* c, int r, int pos0, int rows) {
    const int* d_codes = c->prompt + (size_t)r * c->cfg.n_codebooks;
    const auto key = std::make_tuple(pos0, rows, r);
    auto it = c->pf_graphs.find(key);
    if (it != c->pf_graphs.end()) {
        TTS_CK(cudaGraphLaunch(it->second, c->stream));
        return TTS_OK;
    }
    if (!c->pf_seen.count(key) || c->pf_graphs.size() >= kMaxPrefillGraphs) {
        if (c->pf_seen.size() >= kMaxPrefillSeen) c->pf_seen.clear();
        c->pf_seen.insert(key);
        return prefill_chunk(c, d_codes, pos0, rows);
    }
    // captured on the context's own capture stream (the caller's may be the
    // legacy default stream, which cannot be captured)
    cudaGraph_t g = nullptr;
    cudaStream_t user = c->stream;
    TTS_CK(cudaStreamBeginCapture(c->cap, cudaStreamCaptureModeThreadLocal));
    c->stream = c->cap;
    const int rc = prefill_chunk(c, d_codes, pos0, rows);
    c->stream = user;
    const cudaError_t e = cudaStreamEndCapture(c->cap, &g);  // always: leaves the stream usable
    if (rc != TTS_OK || e != cudaSuccess) {
        if (g) cudaGraphDestroy(g);
        return rc != TTS_OK ? rc : report(e, "prefill capture");
    }
    cudaGraphExec_t exec = nullptr;
    const cudaError_t ei = cudaGraphInstantiate(&exec, g, 0);
    cudaGraphDestroy(g);
    if (ei != cudaSuccess) return report(ei, "prefill graph");
    c->pf_graphs[key] = exec;
    TTS_CK(cudaGraphLaunch(exec, c->stream));
    return TTS_OK;
}

void destroy(tts_ctx* c) {
    if (!c) return;
    if (c->stream) cudaStreamSynchronize(c->stream);
    else cudaDeviceSynchronize();
    // graphs first: they reference the buffers below
    if (c->step_exec) cudaGraphExecDestroy(c->step_exec);
    for (auto& kv : c->pf_graphs) cudaGraphExecDestroy(kv.second);
    if (c->prefill_exec) cudaGraphExecDestroy(c->prefill_exec);
    for (void* p : c->allocs) cudaFree(p);
    if (c->pre_k) cudaFree(c->pre_k);
    if (c->pre_v) cudaFree(c->pre_v);
    if (c->h_in) cudaFreeHost(c->h_in);
    if (c->h_out) cudaFreeHost(c->h_out);
    if (c->h_ring) cudaFreeHost(c->h_ring);
    for (auto& e : c->ev_ring)
        if (e) cudaEventDestroy(e);
    if (c->ev0) cudaEventDestroy(c->ev0);
    if (c->ev1) cudaEventDestroy(c->ev1);
    if (c->cap) cudaStreamDestroy(c->cap);
    delete c;
}

}  // namespace

extern "C" {

int tts_init(const tts_config* cfg, const tts_weights* w, tts_ctx** out) {
    if (!out) return TTS_ERR_ARG;
    *out = nullptr;
    int rc = validate(cfg, w);
    if (rc != TTS_OK) return rc;
    tts_ctx* c = new tts_ctx();
    rc = init_impl(c, cfg, w);
    if (rc != TTS_OK) {
        destroy(c);
        return rc;
    }
    *out = c;
    return TTS_OK;
}

int tts_shutdown(tts_ctx* ctx) {
    destroy(ctx);
    return TTS_OK;
}

int tts_reset(tts_ctx* ctx) {
    if (!ctx) return TTS_ERR_STATE;
    // tickets are zero after every complete step; clear them in case a step
    // was cut short by a device error
    TTS_CK(cudaMemsetAsync(ctx->counters, 0, 2 * ctx->cfg.n_kv_heads * sizeof(unsigned), ctx->stream));
    return push_state(ctx, bos_state(ctx, 0, 0, -1));
}

int tts_decode_step(tts_ctx* ctx, const int32_t* codes_in, int32_t* codes_out) {
    if (!ctx) return TTS_ERR_STATE;
    const tts_config& k = ctx->cfg;
    if (ctx->pos >= k.max_pos) return TTS_ERR_FULL;
    if (codes_in) {
        for (int i = 0; i < k.n_codebooks; ++i)
            if (codes_in[i] < 0 || codes_in[i] >= k.cb_vocab) return TTS_ERR_CODE;
        std::memcpy(ctx->h_in->codes, codes_in, sizeof(int32_t) * k.n_codebooks);
        TTS_CK(cudaMemcpyAsync(ctx->st->codes, ctx->h_in->codes, sizeof(int32_t) * k.n_codebooks,
                               cudaMemcpyHostToDevice, ctx->stream));
    }
    TTS_CK(cudaGraphLaunch(ctx->step_exec, ctx->stream));
    int rc = pull_state(ctx);
    if (rc != TTS_OK) return rc;
    if (codes_out) std::memcpy(codes_out, ctx->h_out->codes, sizeof(int32_t) * k.n_codebooks);
    return TTS_OK;
}

int tts_decode_steps(tts_ctx* ctx, int n, int32_t* codes_out) {
    if (!ctx) return TTS_ERR_STATE;
    if (n < 0) return TTS_ERR_ARG;
    const tts_config& k = ctx->cfg;
    if ((long long)ctx->pos + n > k.max_pos) return TTS_ERR_FULL;
    if (n == 0) return TTS_OK;
    const int zero = 0;
    TTS_CK(cudaMemcpyAsync(&ctx->st->hist_idx, &zero, sizeof(int), cudaMemcpyHostToDevice, ctx->stream));
    TTS_CK(cudaEventRecord(ctx->ev0, ctx->stream));
    for (int i = 0; i < n; ++i) TTS_CK(cudaGraphLaunch(ctx->step_exec, ctx->stream));
    TTS_CK(cudaEventRecord(ctx->ev1, ctx->stream));
    if (codes_out)
        TTS_CK(cudaMemcpyAsync(codes_out, ctx->hist, sizeof(int32_t) * (size_t)n * k.n_codebooks,
                               cudaMemcpyDeviceToHost, ctx->stream));
    int rc = pull_state(ctx);
    TTS_CK(cudaEventElapsedTime(&ctx->last_ms, ctx->ev0, ctx->ev1));
    return rc;
}

int tts_prefill(tts_ctx* ctx, const int32_t* codes, int P) {
    if (!ctx) return TTS_ERR_STATE;
    const tts_config& k = ctx->cfg;
    if (P < 0 || (P > 0 && !codes)) return TTS_ERR_ARG;
    if ((long long)ctx->pos + P > k.max_pos) return TTS_ERR_FULL;
    for (long long i = 0; i < (long long)P * k.n_codebooks; ++i)
        if (codes[i] < 0 || codes[i] >= k.cb_vocab) return TTS_ERR_CODE;
    if (P == 0) return TTS_OK;
    TTS_CK(cudaMemcpyAsync(ctx->prompt, codes, sizeof(int32_t) * (size_t)P * k.n_codebooks,
                           cudaMemcpyHostToDevice, ctx->stream));
    TTS_CK(cudaMemcpyAsync(ctx->h_out, ctx->st, sizeof(DevState), cudaMemcpyDeviceToHost, ctx->stream));
    TTS_CK(cudaStreamSynchronize(ctx->stream));
    if (batched_prefill_ok(ctx)) {
        // the whole prompt as M = P tensor-core passes, kPrefillChunk rows at a time
        DevState s = *ctx->h_out;
        for (int r = 0; r < P; r += kPrefillChunk)
            TTS_TRY(run_prefill_chunk(ctx, r, s.pos + r, std::min(kPrefillChunk, P - r)));
        TTS_CK(cudaStreamSynchronize(ctx->stream));
        int rc = pull_state(ctx);  // reports a GEMM wait that expired (device error word)
        if (rc != TTS_OK) return rc;
        s.pos += P;
        s.prefill_row = 0;
        for (int i = 0; i < kMaxCodebooks; ++i) s.codes[i] = k.cb_vocab - 2;  // next input: all-BOS frame
        return push_state(ctx, s);
    }
    DevState s = *ctx->h_out;
    s.prefill_row = 0;
    TTS_TRY(push_state(ctx, s));
    for (int p = 0; p < P; ++p) TTS_CK(cudaGraphLaunch(ctx->prefill_exec, ctx->stream));
    int rc = pull_state(ctx);
    if (rc != TTS_OK) return rc;
    DevState after = *ctx->h_out;
    for (int i = 0; i < kMaxCodebooks; ++i) after.codes[i] = k.cb_vocab - 2;  // next input: all-BOS frame
    return push_state(ctx, after);
}

int tts_decode_until_eoc(tts_ctx* ctx, int max_frames, int32_t* codes_out, int* n_frames) {
    if (!ctx) return TTS_ERR_STATE;
    if (max_frames < 0 || !n_frames) return TTS_ERR_ARG;
    const tts_config& k = ctx->cfg;
    *n_frames = 0;
    const int room = k.max_pos - ctx->pos;  // frames that fit the cache
    if (max_frames > room) max_frames = room;
    if (max_frames == 0) return room == 0 ? TTS_ERR_FULL : TTS_OK;
    // queue frame f: one graph replay, then the state it leaves into ring slot f & 1
    auto queue = [&](int f) -> int {
        TTS_CK(cudaGraphLaunch(ctx->step_exec, ctx->stream));
        TTS_CK(cudaMemcpyAsync(ctx->h_ring + (f & 1), ctx->st, sizeof(DevState), cudaMemcpyDeviceToHost,
                               ctx->stream));
        TTS_CK(cudaEventRecord(ctx->ev_ring[f & 1], ctx->stream));
        return TTS_OK;
    };
    TTS_TRY(queue(0));
    int rc = TTS_OK;
    for (int f = 0; f < max_frames; ++f) {
        const bool ahead = f + 1 < max_frames;
        if (ahead) TTS_TRY(queue(f + 1));  // the GPU runs frame f + 1 while the host reads frame f
        TTS_CK(cudaEventSynchronize(ctx->ev_ring[f & 1]));
        const DevState s = ctx->h_ring[f & 1];  // read before slot f & 1 is queued again
        if (s.err) {
            rc = TTS_ERR_DEVICE;
            break;
        }
        if (codes_out) std::memcpy(codes_out + (size_t)f * k.n_codebooks, s.codes, sizeof(int32_t) * k.n_codebooks);
        *n_frames = f + 1;
        // stop once the last codebook has emitted EOC (delay pattern: frame eoc + n_cb - 1)
        const int frame = s.t - 1;
        if (s.eoc >= 0 && frame >= s.eoc + k.n_codebooks - 1) {
            if (ahead) {  // undo the frame queued past the stop: back to the state after frame f
                TTS_CK(cudaStreamSynchronize(ctx->stream));
                return push_state(ctx, s);
            }
            break;
        }
    }
    const int prc = pull_state(ctx);
    return rc != TTS_OK ? rc : prc;
}

int tts_set_input(tts_ctx* ctx, const int32_t* codes) {
    if (!ctx) return TTS_ERR_STATE;
    if (!codes) return TTS_ERR_ARG;
    const tts_config& k = ctx->cfg;
    for (int i = 0; i < k.n_codebooks; ++i)
        if (codes[i] < 0 || codes[i] >= k.cb_vocab) return TTS_ERR_CODE;
    std::memcpy(ctx->h_in->codes, codes, sizeof(int32_t) * k.n_codebooks);
    TTS_CK(cudaMemcpyAsync(ctx->st->codes, ctx->h_in->codes, sizeof(int32_t) * k.n_codebooks,
                           cudaMemcpyHostToDevice, ctx->stream));
    TTS_CK(cudaStreamSynchronize(ctx->stream));
    return TTS_OK;
}

int tts_rewind(tts_ctx* ctx, int pos, int t) {
    if (!ctx) return TTS_ERR_STATE;
    if (pos < 0 || pos > ctx->pos || t < 0) return TTS_ERR_ARG;
    return push_state(ctx, bos_state(ctx, pos, t, -1));
}

int tts_prefix_save(tts_ctx* ctx) {
    if (!ctx) return TTS_ERR_STATE;
    const tts_config& k = ctx->cfg;
    TTS_CK(cudaMemcpyAsync(ctx->h_out, ctx->st, sizeof(DevState), cudaMemcpyDeviceToHost, ctx->stream));
    TTS_CK(cudaStreamSynchronize(ctx->stream));
    const DevState s = *ctx->h_out;
    const int P = s.pos;
    if (P <= 0) return TTS_ERR_ARG;
    const size_t rows = (size_t)k.n_layers * k.n_kv_heads;
    if (P > ctx->pre_cap) {
        if (ctx->pre_k) cudaFree(ctx->pre_k);
        if (ctx->pre_v) cudaFree(ctx->pre_v);
        ctx->pre_k = ctx->pre_v = nullptr;
        ctx->pre_cap = ctx->pre_len = 0;
        const size_t bytes = rows * P * kHeadDim * sizeof(__nv_bfloat16);
        TTS_CK(cudaMalloc(&ctx->pre_k, bytes));
        TTS_CK(cudaMalloc(&ctx->pre_v, bytes));
        ctx->pre_cap = P;
    }
    const size_t row = (size_t)P * kHeadDim * sizeof(__nv_bfloat16);
    const size_t cpitch = (size_t)k.max_pos * kHeadDim * sizeof(__nv_bfloat16);
    TTS_CK(cudaMemcpy2DAsync(ctx->pre_k, row, ctx->kc, cpitch, row, rows, cudaMemcpyDeviceToDevice, ctx->stream));
    TTS_CK(cudaMemcpy2DAsync(ctx->pre_v, row, ctx->vc, cpitch, row, rows, cudaMemcpyDeviceToDevice, ctx->stream));
    TTS_CK(cudaStreamSynchronize(ctx->stream));
    ctx->pre_len = P;
    ctx->pre_state = s;
    return TTS_OK;
}

int tts_prefix_restore(tts_ctx* ctx) {
    if (!ctx) return TTS_ERR_STATE;
    if (ctx->pre_len <= 0) return TTS_ERR_STATE;
    const tts_config& k = ctx->cfg;
    const size_t rows = (size_t)k.n_layers * k.n_kv_heads;
    const size_t row = (size_t)ctx->pre_len * kHeadDim * sizeof(__nv_bfloat16);
    const size_t cpitch = (size_t)k.max_pos * kHeadDim * sizeof(__nv_bfloat16);
    TTS_CK(cudaMemcpy2DAsync(ctx->kc, cpitch, ctx->pre_k, row, row, rows, cudaMemcpyDeviceToDevice, ctx->stream));
    TTS_CK(cudaMemcpy2DAsync(ctx->vc, cpitch, ctx->pre_v, row, row, rows, cudaMemcpyDeviceToDevice, ctx->stream));
    DevState s = ctx->pre_state;
    s.err = 0;
    s.hist_idx = 0;
    return push_state(ctx, s);
}

int tts_set_fp8_scales(tts_ctx* ctx, const float* scales) {
    if (!ctx) return TTS_ERR_STATE;
    const tts_config& k = ctx->cfg;
    if (k.precision != TTS_FP8 || !ctx->persistent || !ctx->sp.fp8_sa) return TTS_ERR_UNSUPPORTED;
    const size_t n = (size_t)k.n_layers * 4;
    std::vector<float> h(n, 0.f);
    if (scales)
        for (size_t i = 0; i < n; ++i) {
            if (!(scales[i] >= 0.f) || !std::isfinite(scales[i])) return TTS_ERR_ARG;
            h[i] = scales[i];
        }
    TTS_CK(cudaMemcpyAsync(const_cast<float*>(ctx->sp.fp8_sa), h.data(), n * sizeof(float), cudaMemcpyHostToDevice,
                           ctx->stream));
    TTS_CK(cudaStreamSynchronize(ctx->stream));
    return TTS_OK;
}

int tts_fp8_calibrate(tts_ctx* ctx, int n_frames, float* amax_out) {
    if (!ctx) return TTS_ERR_STATE;
    const tts_config& k = ctx->cfg;
    if (k.precision != TTS_FP8 || !ctx->persistent) return TTS_ERR_UNSUPPORTED;
    if (n_frames < 1 || !amax_out) return TTS_ERR_ARG;
    if (ctx->pos + n_frames > k.max_pos) return TTS_ERR_FULL;
    const size_t n = (size_t)k.n_layers * 4;
    TTS_CK(cudaMemcpyAsync(ctx->h_out, ctx->st, sizeof(DevState), cudaMemcpyDeviceToHost, ctx->stream));
    TTS_CK(cudaStreamSynchronize(ctx->stream));
    const DevState saved = *ctx->h_out;
    float* cal = nullptr;
    TTS_CK(cudaMalloc(&cal, n * sizeof(float)));
    cudaError_t e = cudaMemsetAsync(cal, 0, n * sizeof(float), ctx->stream);
    StepParams p = ctx->sp;
    p.decode = 1;
    p.fp8_calib = cal;
    for (int f = 0; f < n_frames && e == cudaSuccess; ++f) {
        e = xch_reset(ctx, ctx->stream);
        if (e == cudaSuccess) e = launch_step(p, kFP8, ctx->G, ctx->num_sms, ctx->step_smem, ctx->stream);
    }
    if (e == cudaSuccess) e = cudaMemcpyAsync(amax_out, cal, n * sizeof(float), cudaMemcpyDeviceToHost, ctx->stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(ctx->stream);
    cudaFree(cal);
    if (e != cudaSuccess) return report(e, "tts_fp8_calibrate");
    TTS_TRY(pull_state(ctx));  // reports a device error of the calibration frames
    return push_state(ctx, saved);  // the frames are discarded: back to the state before them
}

int tts_set_kv(tts_ctx* ctx, const void* kd, const void* vd, int len, int len_stride) {
    if (!ctx) return TTS_ERR_STATE;
    const tts_config& k = ctx->cfg;
    if (!kd || !vd || len < 0 || len > k.max_pos || len_stride < len) return TTS_ERR_ARG;
    if (len > 0) {
        const size_t row = (size_t)len * kHeadDim * sizeof(__nv_bfloat16);
        const size_t spitch = (size_t)len_stride * kHeadDim * sizeof(__nv_bfloat16);
        const size_t dpitch = (size_t)k.max_pos * kHeadDim * sizeof(__nv_bfloat16);
        const size_t rows = (size_t)k.n_layers * k.n_kv_heads;
        TTS_CK(cudaMemcpy2DAsync(ctx->kc, dpitch, kd, spitch, row, rows, cudaMemcpyDeviceToDevice, ctx->stream));
        TTS_CK(cudaMemcpy2DAsync(ctx->vc, dpitch, vd, spitch, row, rows, cudaMemcpyDeviceToDevice, ctx->stream));
    }
    TTS_CK(cudaMemcpyAsync(ctx->h_out, ctx->st, sizeof(DevState), cudaMemcpyDeviceToHost, ctx->stream));
    TTS_CK(cudaStreamSynchronize(ctx->stream));
    DevState s = *ctx->h_out;
    s.pos = len;
    return push_state(ctx, s);
}

int tts_get_kv(tts_ctx* ctx, void* k_host, void* v_host, int p0, int p1) {
    if (!ctx) return TTS_ERR_STATE;
    const tts_config& k = ctx->cfg;
    if (p0 < 0 || p1 < p0 || p1 > k.max_pos) return TTS_ERR_ARG;
    if (p1 == p0) return TTS_OK;
    const size_t row = (size_t)(p1 - p0) * kHeadDim * sizeof(__nv_bfloat16);
    const size_t spitch = (size_t)k.max_pos * kHeadDim * sizeof(__nv_bfloat16);
    const size_t rows = (size_t)k.n_layers * k.n_kv_heads;
    const size_t off = (size_t)p0 * kHeadDim;
    if (k_host) TTS_CK(cudaMemcpy2DAsync(k_host, row, ctx->kc + off, spitch, row, rows, cudaMemcpyDeviceToHost, ctx->stream));
    if (v_host) TTS_CK(cudaMemcpy2DAsync(v_host, row, ctx->vc + off, spitch, row, rows, cudaMemcpyDeviceToHost, ctx->stream));
    TTS_CK(cudaStreamSynchronize(ctx->stream));
    return TTS_OK;
}

int tts_get_logits(tts_ctx* ctx, float* out) {
    if (!ctx) return TTS_ERR_STATE;
    if (!out) return TTS_ERR_ARG;
    const size_t n = (size_t)ctx->cfg.n_codebooks * ctx->cfg.cb_vocab;
    TTS_CK(cudaMemcpyAsync(out, ctx->logits, n * sizeof(float), cudaMemcpyDeviceToHost, ctx->stream));
    TTS_CK(cudaStreamSynchronize(ctx->stream));
    return TTS_OK;
}

int tts_get_hidden(tts_ctx* ctx, float* out) {
    if (!ctx) return TTS_ERR_STATE;
    if (!out) return TTS_ERR_ARG;
    TTS_CK(cudaMemcpyAsync(out, ctx->h, (size_t)ctx->cfg.hidden * sizeof(float), cudaMemcpyDeviceToHost, ctx->stream));
    TTS_CK(cudaStreamSynchronize(ctx->stream));
    return TTS_OK;
}

int tts_set_frame(tts_ctx* ctx, int t, int eoc_frame) {
    if (!ctx) return TTS_ERR_STATE;
    if (t < 0 || eoc_frame < -1) return TTS_ERR_ARG;
    TTS_CK(cudaMemcpyAsync(ctx->h_out, ctx->st, sizeof(DevState), cudaMemcpyDeviceToHost, ctx->stream));
    TTS_CK(cudaStreamSynchronize(ctx->stream));
    DevState s = *ctx->h_out;
    s.t = t;
    s.eoc = eoc_frame;
    return push_state(ctx, s);
}

int tts_set_sampling(tts_ctx* ctx, float temperature, unsigned long long seed) {
    if (!ctx) return TTS_ERR_STATE;
    if (!(temperature >= 0.f) || !std::isfinite(temperature)) return TTS_ERR_ARG;
    TTS_CK(cudaMemcpyAsync(ctx->h_out, ctx->st, sizeof(DevState), cudaMemcpyDeviceToHost, ctx->stream));
    TTS_CK(cudaStreamSynchronize(ctx->stream));
    ctx->temperature = temperature;
    ctx->seed = seed;
    return push_state(ctx, *ctx->h_out);
}

int tts_get_state(tts_ctx* ctx, int* pos, int* t, int* eoc) {
    if (!ctx) return TTS_ERR_STATE;
    TTS_CK(cudaMemcpyAsync(ctx->h_out, ctx->st, sizeof(DevState), cudaMemcpyDeviceToHost, ctx->stream));
    TTS_CK(cudaStreamSynchronize(ctx->stream));
    if (pos) *pos = ctx->h_out->pos;
    if (t) *t = ctx->h_out->t;
    if (eoc) *eoc = ctx->h_out->eoc;
    return TTS_OK;
}

int tts_last_steps_ms(tts_ctx* ctx, float* ms) {
    if (!ctx) return TTS_ERR_STATE;
    if (!ms) return TTS_ERR_ARG;
    *ms = ctx->last_ms;
    return TTS_OK;
}

int tts_time_gemv(tts_ctx* ctx, int kind, int reps, float* ms_per_launch) {
    if (!ctx) return TTS_ERR_STATE;
    if (kind < 0 || kind > 4 || reps < 1 || !ms_per_launch) return TTS_ERR_ARG;
    const tts_config& k = ctx->cfg;
    const int prec = (kind == kHead || k.precision == TTS_BF16) ? kBF16 : kFP8;
    const int pro = (kind == kO || kind == kDown) ? kProPlain : kProRms;
    const int epi = kind == kGU ? kEpiSwiglu : ((kind == kO || kind == kDown) ? kEpiResid : kEpiStore);
    const size_t pf = kGemvPrefetchBytes;
    TTS_CK(cudaEventRecord(ctx->ev0, ctx->stream));
    for (int r = 0; r < reps; ++r)
        for (int l = 0; l < k.n_layers; ++l) {
            GemvParams g = proj_params(ctx, kind, l);
            set_next(ctx, g, kind, (l + 1) % k.n_layers, pf);
            TTS_CK(launch_gemv(prec, pro, epi, g, gemv_cfg(ctx, ctx->pdl && (r | l)), ctx->stream));
        }
    TTS_CK(cudaEventRecord(ctx->ev1, ctx->stream));
    TTS_CK(cudaEventSynchronize(ctx->ev1));
    float ms = 0.f;
    TTS_CK(cudaEventElapsedTime(&ms, ctx->ev0, ctx->ev1));
    *ms_per_launch = ms / (float)(reps * k.n_layers);
    return TTS_OK;
}

int tts_trace_step(tts_ctx* ctx, uint64_t* host_out, int capacity, int* stride, int* n_cta) {
    if (!ctx) return TTS_ERR_STATE;
    if (!ctx->persistent) return TTS_ERR_UNSUPPORTED;
    const tts_config& k = ctx->cfg;
    const int st = step_trace_stride(k.n_layers);
    const size_t n = (size_t)st * ctx->num_sms;
    if (!host_out || capacity < (long long)(n + 2 * 4 * 2048)) return TTS_ERR_ARG;
    if (ctx->pos >= k.max_pos) return TTS_ERR_FULL;
    unsigned long long* d = nullptr;
    const int sstride = 4 * 2048;  // per-stage trace of two warps of CTA 0 (first 2048 stages)
    const size_t ntot = n + 2 * (size_t)sstride;
    TTS_CK(cudaMalloc(&d, ntot * sizeof(unsigned long long)));
    TTS_CK(cudaMemsetAsync(d, 0, ntot * sizeof(unsigned long long), ctx->stream));
    StepParams p = ctx->sp;
    p.decode = 1;
    p.trace = d;
    p.trace_stride = st;
    p.stage_trace = d + n;
    p.stage_trace_stride = sstride;
    const int prec = k.precision == TTS_FP8 ? kFP8 : kBF16;
    cudaError_t e = xch_reset(ctx, ctx->stream);
    if (e == cudaSuccess) e = launch_step(p, prec, ctx->G, ctx->num_sms, ctx->step_smem, ctx->stream);
    if (e == cudaSuccess) e = cudaMemcpyAsync(host_out, d, ntot * sizeof(unsigned long long), cudaMemcpyDeviceToHost, ctx->stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(ctx->stream);
    cudaFree(d);
    if (e != cudaSuccess) return report(e, "tts_trace_step");
    if (stride) *stride = st;
    if (n_cta) *n_cta = ctx->num_sms;
    return pull_state(ctx);
}

int tts_debug_layer_states(tts_ctx* ctx, const int32_t* codes_in, int32_t* codes_out, float* host_h,
                           int capacity) {
    if (!ctx) return TTS_ERR_STATE;
    if (!ctx->persistent) return TTS_ERR_UNSUPPORTED;
    const tts_config& k = ctx->cfg;
    const size_t nh = (size_t)(k.n_layers + 1) * k.hidden;
    if (!host_h || capacity < (long long)nh) return TTS_ERR_ARG;
    if (ctx->pos >= k.max_pos) return TTS_ERR_FULL;
    if (codes_in) {
        for (int i = 0; i < k.n_codebooks; ++i)
            if (codes_in[i] < 0 || codes_in[i] >= k.cb_vocab) return TTS_ERR_CODE;
        std::memcpy(ctx->h_in->codes, codes_in, sizeof(int32_t) * k.n_codebooks);
        TTS_CK(cudaMemcpyAsync(ctx->st->codes, ctx->h_in->codes, sizeof(int32_t) * k.n_codebooks,
                               cudaMemcpyHostToDevice, ctx->stream));
    }
    const int st = step_trace_stride(k.n_layers);
    const size_t nt = (size_t)st * ctx->num_sms;
    unsigned long long* d = nullptr;
    float* hs = nullptr;
    TTS_CK(cudaMalloc(&d, nt * sizeof(unsigned long long)));
    cudaError_t e = cudaMalloc(&hs, nh * sizeof(float));
    if (e == cudaSuccess) e = cudaMemsetAsync(hs, 0, nh * sizeof(float), ctx->stream);
    StepParams p = ctx->sp;
    p.decode = 1;
    p.trace = d;
    p.trace_stride = st;
    p.stage_trace = nullptr;
    p.stage_trace_stride = 0;
    p.hsnap = hs;
    const int prec = k.precision == TTS_FP8 ? kFP8 : kBF16;
    if (e == cudaSuccess) e = xch_reset(ctx, ctx->stream);
    if (e == cudaSuccess) e = launch_step(p, prec, ctx->G, ctx->num_sms, ctx->step_smem, ctx->stream);
    if (e == cudaSuccess) e = cudaMemcpyAsync(host_h, hs, nh * sizeof(float), cudaMemcpyDeviceToHost, ctx->stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(ctx->stream);
    cudaFree(d);
    if (hs) cudaFree(hs);
    if (e != cudaSuccess) return report(e, "tts_debug_layer_states");
    const int rc = pull_state(ctx);
    if (rc == TTS_OK && codes_out) std::memcpy(codes_out, ctx->h_out->codes, sizeof(int32_t) * k.n_codebooks);
    return rc;
}

int tts_debug_prefill_states(tts_ctx* ctx, const int32_t* codes, int P, float* host_h, long long capacity) {
    if (!ctx) return TTS_ERR_STATE;
    const tts_config& k = ctx->cfg;
    if (!codes || P < 1 || P > kPrefillChunk || !host_h) return TTS_ERR_ARG;
    if (!batched_prefill_ok(ctx)) return TTS_ERR_UNSUPPORTED;
    const size_t n = (size_t)(k.n_layers + 1) * P * k.hidden;
    if (capacity < (long long)n) return TTS_ERR_ARG;
    if ((long long)ctx->pos + P > k.max_pos) return TTS_ERR_FULL;
    for (long long i = 0; i < (long long)P * k.n_codebooks; ++i)
        if (codes[i] < 0 || codes[i] >= k.cb_vocab) return TTS_ERR_CODE;
    TTS_CK(cudaMemcpyAsync(ctx->prompt, codes, sizeof(int32_t) * (size_t)P * k.n_codebooks,
                           cudaMemcpyHostToDevice, ctx->stream));
    TTS_CK(cudaMemcpyAsync(ctx->h_out, ctx->st, sizeof(DevState), cudaMemcpyDeviceToHost, ctx->stream));
    TTS_CK(cudaStreamSynchronize(ctx->stream));
    DevState s = *ctx->h_out;
    float* snap = nullptr;
    TTS_CK(cudaMalloc(&snap, n * sizeof(float)));
    int rc = prefill_chunk(ctx, ctx->prompt, s.pos, P, snap);
    cudaError_t e = cudaSuccess;
    if (rc == TTS_OK) e = cudaMemcpyAsync(host_h, snap, n * sizeof(float), cudaMemcpyDeviceToHost, ctx->stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(ctx->stream);
    cudaFree(snap);
    if (rc != TTS_OK) return rc;
    if (e != cudaSuccess) return report(e, "tts_debug_prefill_states");
    rc = pull_state(ctx);
    if (rc != TTS_OK) return rc;
    s.pos += P;
    s.prefill_row = 0;
    for (int i = 0; i < kMaxCodebooks; ++i) s.codes[i] = k.cb_vocab - 2;
    return push_state(ctx, s);
}

int tts_debug_expire_wait(tts_ctx* ctx) {
    if (!ctx) return TTS_ERR_STATE;
    if (!ctx->persistent) return TTS_ERR_UNSUPPORTED;
    const tts_config& k = ctx->cfg;
    if (ctx->pos >= k.max_pos) return TTS_ERR_FULL;
    StepParams p = ctx->sp;
    p.decode = 1;
    p.wait_limit_ns = 1000ull * 1000ull;  // 1 ms
    p.fault_skip_embed = 1;               // the first layer waits for an embedding never stored
    const int prec = k.precision == TTS_FP8 ? kFP8 : kBF16;
    TTS_CK(xch_reset(ctx, ctx->stream));
    TTS_CK(launch_step(p, prec, ctx->G, ctx->num_sms, ctx->step_smem, ctx->stream));
    return pull_state(ctx);
}

int tts_quantize_fp8_weight(const void* W, int N, int K, void* W8, float* s, void* stream) {
    if (!W || !W8 || !s || N <= 0 || K <= 0) return TTS_ERR_ARG;
    TTS_CK(launch_quantize_weight(static_cast<const __nv_bfloat16*>(W), N, K, static_cast<uint8_t*>(W8), s,
                                  static_cast<cudaStream_t>(stream)));
    return TTS_OK;
}

const char* tts_status_str(int status) {
    switch (status) {
        case TTS_OK: return "ok";
        case TTS_ERR_ARG: return "bad argument";
        case TTS_ERR_CODE: return "code out of range";
        case TTS_ERR_FULL: return "context full";
        case TTS_ERR_CUDA: return "CUDA error";
        case TTS_ERR_DEVICE: return "device error flag set";
        case TTS_ERR_STATE: return "not initialised";
        case TTS_ERR_UNSUPPORTED: return "unsupported";
        default: return "unknown status";
    }
}

}  // extern "C"

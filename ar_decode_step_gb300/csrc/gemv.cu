// M = 1 weight-streaming GEMV, one projection per launch (sm_103a).
//
// Every projection of the step ("Higgs Audio v3 TTS-4B on FlashRT", section 5:
// QKV, O-proj with fused residual, gate/up with SwiGLU, down-proj with fused
// residual, fused codebook head) as its own kernel, built from the shared
// blocks in gemv_core.cuh: a producer warp streams the CTA's row range of
// the weights through a ring of 32-40 KB shared-memory stages (one bulk copy
// each, TMA engine, L2 evict-first) and eight consumer warps reduce them
// against the staged activation vector.  The producer starts before
// griddepcontrol.wait (weights do not depend on the previous kernel) and,
// once its own copies are out, warms L2 with the leading part of the next
// projection's weights.  Consumers wait, stage the activations (optional
// RMSNorm; FP8: per-token E4M3 quantisation, scale amax/448, computed by
// every CTA so there is no grid-wide dependency), reduce, and apply the
// epilogue: store, residual add, SwiGLU, or codebook logits + last-CTA greedy
// argmax under the delay mask.
//
// The persistent step kernel (step.cu) runs the same blocks for all
// projections of a step in one launch; this per-launch form serves the
// kernel-level measurements and the graph of separate kernels.
#include "gemv_core.cuh"

namespace tts {

namespace {

using namespace core;

constexpr int kSmemBudget = 220 * 1024;  // one CTA per SM
constexpr uint32_t kPrefetchPiece = 32 * 1024;

int round128(int x) { return (x + 127) & ~127; }

template <int PREC, int PRO, int EPI>
__global__ void __launch_bounds__(kThreads, 1) gemv_kernel(const GemvParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ float red[32];
    __shared__ int s_last;
    __shared__ int s_codes[kMaxCodebooks];
    __shared__ volatile int s_abort;

    constexpr bool FP8 = PREC == kFP8;
    const int cpr = p.K / (FP8 ? 16 : 8);
    const int xbytes = p.K * (FP8 ? 1 : 4);
    Proj j{static_cast<const unsigned char*>(p.W), p.wscale, p.y, p.N, p.K, p.rs, p.wpr, FP8 ? 1 : 0,
           EPI == kEpiSwiglu ? 1 : 0, 0, 0};
    proj_split_rows(j);
    Ring ring{reinterpret_cast<uint64_t*>(smem), reinterpret_cast<uint64_t*>(smem) + p.nstages,
              smem + kBarrierBytes + xbytes + p.part_bytes, (uint32_t)(p.rs * cpr * 16), p.nstages,
              ring_magic(p.nstages)};
    unsigned char* xs = smem + kBarrierBytes;
    float* part = reinterpret_cast<float*>(xs + xbytes);

    if (threadIdx.x == 0) {
        ring_init(ring);
        s_abort = 0;
    }
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == kConsumerWarps) {  // producer warp
        pdl_trigger();
        if (lane == 0) {
            int it = 0;
            if (produce(j, ring, it, l2_evict_first_policy(), &s_abort, p.err)) {
                if (p.next_W && p.next_pf > 0) {
                    // warm L2 with the start of this CTA's share of the next projection
                    const int nr0 = (int)((long long)blockIdx.x * p.next_N / gridDim.x);
                    const int nr1 = (int)((long long)(blockIdx.x + 1) * p.next_N / gridDim.x);
                    const unsigned char* nb = static_cast<const unsigned char*>(p.next_W) + (size_t)nr0 * p.next_rowb;
                    size_t n = (size_t)(nr1 - nr0) * p.next_rowb;
                    if (n > p.next_pf) n = p.next_pf;
                    n &= ~(size_t)15;
                    for (size_t off = 0; off < n; off += kPrefetchPiece)
                        prefetch_l2_bulk(nb + off, (uint32_t)(n - off < kPrefetchPiece ? n - off : kPrefetchPiece));
                }
            } else {
                drain(ring, it);
            }
        }
        return;
    }

    pdl_wait();
    pdl_trigger();
    XSeg<FP8> xr;
    float sa = 1.0f;
    {
        int rslot, sg, c0, c1;
        proj_segment(j, warp, rslot, sg, c0, c1);
        if constexpr (!FP8 && PRO == kProPlain) {
            load_xseg_plain(p.x, c0, c1, xr);  // plain bf16 input: straight into registers
        } else {
            sa = stage_x<FP8, PRO == kProRms>(p.x, p.gamma, p.K, p.eps, xs, red);
            load_xseg_smem<FP8>(xs, cpr, c0, c1, xr);
        }
    }
    int it = 0;
    constexpr int CEPI = EPI == kEpiLogits ? kEpiStore : EPI;
    if (!consume<FP8, CEPI>(j, ring, it, xr, sa, part, &s_abort, p.err)) return;
    if constexpr (EPI == kEpiLogits)
        head_tail(p.y, p.n_cb, p.cb_vocab, p.st, p.counter, 0u, p.hist, p.hist_cap, &s_last, s_codes);
}

template <int PREC, int PRO, int EPI>
cudaError_t launch_one(const GemvParams& p, int smem, const LaunchCfg& lc, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(lc.grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = lc.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, gemv_kernel<PREC, PRO, EPI>, p);
}

template <int PREC, int PRO, int EPI>
cudaError_t prepare_one() {
    return cudaFuncSetAttribute(gemv_kernel<PREC, PRO, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kSmemBudget);
}

#define TTS_GEMV_VARIANTS(X)            \
    X(kBF16, kProRms, kEpiStore)        \
    X(kBF16, kProPlain, kEpiResid)      \
    X(kBF16, kProRms, kEpiSwiglu)       \
    X(kBF16, kProRms, kEpiLogits)       \
    X(kBF16, kProPlain, kEpiStore)      \
    X(kFP8, kProRms, kEpiStore)         \
    X(kFP8, kProPlain, kEpiResid)       \
    X(kFP8, kProRms, kEpiSwiglu)        \
    X(kFP8, kProPlain, kEpiStore)

}  // namespace

GemvGeom gemv_geom(int prec, int epi, int N, int K, int grid) {
    GemvGeom g{};
    const int cpr = K / (prec == kBF16 ? 8 : 16);
    const long long rowb = (long long)cpr * 16;
    const bool swiglu = epi == kEpiSwiglu;
    const StageGeom sg = stage_geom(prec, epi, K);
    g.rs = sg.rs;
    g.wpr = sg.wpr;
    const int opst = swiglu ? g.rs / 2 : g.rs;
    const long long rows_max = grid > 0 ? (N + grid - 1) / grid : N;
    const long long nst_max = (rows_max + opst - 1) / opst;
    g.part_bytes = round128((int)(nst_max * g.rs * g.wpr * (long long)sizeof(float)));
    const int xbytes = K * (prec == kBF16 ? 4 : 1);
    const long long stage = g.rs * rowb;
    long long ns = stage > 0 ? (kSmemBudget - kBarrierBytes - xbytes - g.part_bytes) / stage : 0;
    if (ns > kMaxStages) ns = kMaxStages;
    g.nstages = (int)ns;
    g.smem = (int)(kBarrierBytes + xbytes + g.part_bytes + ns * stage);
    g.ok = sg.ok && ns >= 2 && g.smem <= kSmemBudget && K <= kMaxPlainK;
    return g;
}

cudaError_t gemv_prepare() {
#define TTS_PREP(PR, PO, EP)                                  \
    {                                                         \
        cudaError_t e = prepare_one<PR, PO, EP>();            \
        if (e != cudaSuccess) return e;                       \
    }
    TTS_GEMV_VARIANTS(TTS_PREP)
#undef TTS_PREP
    return cudaSuccess;
}

cudaError_t launch_gemv(int prec, int pro, int epi, const GemvParams& p_in, const LaunchCfg& lc,
                        cudaStream_t s) {
    GemvParams p = p_in;
    const GemvGeom g = gemv_geom(prec, epi, p.N, p.K, lc.grid);
    if (!g.ok) return cudaErrorInvalidValue;
    p.rs = g.rs;
    p.wpr = g.wpr;
    p.nstages = g.nstages;
    p.part_bytes = g.part_bytes;
#define TTS_GEMV_CASE(PR, PO, EP) \
    if (prec == PR && pro == PO && epi == EP) return launch_one<PR, PO, EP>(p, g.smem, lc, s);
    TTS_GEMV_VARIANTS(TTS_GEMV_CASE)
#undef TTS_GEMV_CASE
    return cudaErrorInvalidValue;
}

}  // namespace tts

// M = 1 weight-streaming GEMV family for the decode step (sm_103a).
//
// One kernel template covers every projection of the step ("Higgs Audio v3
// TTS-4B on FlashRT", section 5: QKV, O-proj with fused residual, gate/up with
// SwiGLU, down-proj with fused residual, fused codebook head).
//
// Data movement.  Each CTA (one per SM) owns a contiguous, row-aligned range
// of output rows.  A producer warp streams it through a ring of shared-memory
// stages; a stage is a group of RS whole rows (RS a power of two, 32-40 KB),
// filled by one bulk copy on the TMA engine (two for a gate/up stage: RS/2
// gate rows and the matching RS/2 up rows), completion counted on mbarriers,
// L2 evict-first.  Large single copies are what keeps HBM near its peak.
// When its own copies are all issued, the producer asks L2 to prefetch the
// leading part of the next projection's weights, so HBM keeps streaming
// across the kernel boundary.
//
// Compute.  Sixteen consumer warps: warp w owns segment w % WPR of row slot
// w / WPR of every stage (WPR = 16 / RS warps per row), so all warps get the
// same bytes, x is indexed directly and each warp does one shuffle reduction
// per stage.  The per-(row, segment) partial sums are added in segment order
// at the end (deterministic), then the epilogue: store, residual add, SwiGLU
// over the gate/up pair, or the codebook logits followed by a last-CTA greedy
// argmax under the delay-pattern mask (section 4, sampling policy).
//
// Prologue.  Consumers wait for the producing kernel (griddepcontrol.wait),
// then stage the activation vector in shared memory: optional RMSNorm (fp32)
// and, for FP8, the per-token dynamic E4M3 quantisation (scale amax/448),
// computed redundantly by every CTA, so no separate norm/quant kernel and no
// grid-wide dependency exist.  FP8 activations are kept as f16 (exact for
// E4M3 values) and multiplied with the mixed-precision f16 x f16 + f32 FMA.
//
// Every wait on a shared-memory barrier is bounded (kWaitLimitNs); on expiry
// the kernel records kErrTimeout, lets its in-flight copies land and returns.
#include "kernels.h"

namespace tts {

namespace {

constexpr int kConsumerWarps = 16;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;  // + one producer warp
constexpr int kStageTarget = 40 * 1024;    // bytes per ring stage, at most
constexpr int kSmemBudget = 220 * 1024;    // one CTA per SM
constexpr int kBarrierBytes = 128;
constexpr int kMaxStages = 8;
constexpr uint32_t kPrefetchPiece = 32 * 1024;

template <int PREC>
struct Traits;
template <>
struct Traits<kBF16> {
    static constexpr int kElems = 8;   // weights per 16-byte chunk
    static constexpr int kXBytes = 4;  // bytes per staged activation (fp32)
};
template <>
struct Traits<kFP8> {
    static constexpr int kElems = 16;
    static constexpr int kXBytes = 2;  // f16
};

int round128(int x) { return (x + 127) & ~127; }

// ---- chunk dot products ------------------------------------------------------
// BF16: 8 weights x fp32 activations held as two float4 planes.
__device__ __forceinline__ float dot_bf16(const uint4 w, const float4 a, const float4 b, float acc) {
    acc = fmaf(bf16lo(w.x), a.x, acc);
    acc = fmaf(bf16hi(w.x), a.y, acc);
    acc = fmaf(bf16lo(w.y), a.z, acc);
    acc = fmaf(bf16hi(w.y), a.w, acc);
    acc = fmaf(bf16lo(w.z), b.x, acc);
    acc = fmaf(bf16hi(w.z), b.y, acc);
    acc = fmaf(bf16lo(w.w), b.z, acc);
    acc = fmaf(bf16hi(w.w), b.w, acc);
    return acc;
}

// Two E4M3 weights (low 16 bits of w) times two f16 activations, f32 accumulate.
__device__ __forceinline__ float fma2_e4m3_f16(uint32_t w16, uint32_t x2, float acc) {
    const __half2_raw wh = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w16 & 0xffffu), __NV_E4M3);
    const uint32_t w2 = (uint32_t)wh.x | ((uint32_t)wh.y << 16);
    asm("{\n\t.reg .f16 a0, a1, b0, b1;\n\t"
        "mov.b32 {a0, a1}, %1;\n\t"
        "mov.b32 {b0, b1}, %2;\n\t"
        "fma.rn.f32.f16 %0, a0, b0, %0;\n\t"
        "fma.rn.f32.f16 %0, a1, b1, %0;\n\t}"
        : "+f"(acc)
        : "r"(w2), "r"(x2));
    return acc;
}

// FP8: 16 weights x f16 activations held as two planes of 8 f16.
__device__ __forceinline__ float dot_fp8(const uint4 w, const uint4 a, const uint4 b, float acc) {
    acc = fma2_e4m3_f16(w.x, a.x, acc);
    acc = fma2_e4m3_f16(w.x >> 16, a.y, acc);
    acc = fma2_e4m3_f16(w.y, a.z, acc);
    acc = fma2_e4m3_f16(w.y >> 16, a.w, acc);
    acc = fma2_e4m3_f16(w.z, b.x, acc);
    acc = fma2_e4m3_f16(w.z >> 16, b.y, acc);
    acc = fma2_e4m3_f16(w.w, b.z, acc);
    acc = fma2_e4m3_f16(w.w >> 16, b.w, acc);
    return acc;
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

// Barrier among the consumer warps only (the producer warp does not take part).
__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory"); }

__device__ __forceinline__ float consumer_sum(float v, float* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = warp_sum(v);
    consumer_sync();
    if (lane == 0) red[warp] = v;
    consumer_sync();
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kConsumerWarps; ++i) s += red[i];  // fixed order: deterministic
    return s;
}
__device__ __forceinline__ float consumer_max(float v, float* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = warp_max(v);
    consumer_sync();
    if (lane == 0) red[warp] = v;
    consumer_sync();
    float s = red[0];
#pragma unroll
    for (int i = 1; i < kConsumerWarps; ++i) s = fmaxf(s, red[i]);
    return s;
}

template <int PREC, int PRO, int EPI>
__global__ void __launch_bounds__(kThreads, 1) gemv_kernel(const GemvParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ float red[32];
    __shared__ int s_last;
    __shared__ int s_codes[kMaxCodebooks];
    __shared__ volatile int s_abort;

    constexpr bool kSwiglu = EPI == kEpiSwiglu;
    constexpr int E = Traits<PREC>::kElems;
    const int K = p.K, CPR = K / E, RS = p.rs, NS = p.nstages;
    const int WPR = kConsumerWarps / RS;  // consumer warps per row
    const size_t rowb = (size_t)CPR * 16;
    const uint32_t stage_bytes = (uint32_t)(RS * rowb);
    const int xbytes = K * Traits<PREC>::kXBytes;

    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + NS;
    unsigned char* xs = smem + kBarrierBytes;
    float* part = reinterpret_cast<float*>(xs + xbytes);
    unsigned char* ring = reinterpret_cast<unsigned char*>(part) + p.part_bytes;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r0 = (int)((long long)blockIdx.x * p.N / gridDim.x);
    const int r1 = (int)((long long)(blockIdx.x + 1) * p.N / gridDim.x);
    const int nrows = r1 - r0;               // outputs of this CTA
    const int opst = kSwiglu ? RS / 2 : RS;  // outputs per stage
    const int nst = (nrows + opst - 1) / opst;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        fence_mbar_init();
        s_abort = 0;
    }
    __syncthreads();

    // ---- producer warp ------------------------------------------------------
    if (warp == kConsumerWarps) {
        pdl_trigger();
        if (lane == 0) {
            const unsigned char* W = static_cast<const unsigned char*>(p.W);
            const uint64_t pol = l2_evict_first_policy();
            int issued = 0;
            for (int s = 0; s < nst; ++s) {
                const int slot = s % NS;
                if (!mbar_wait(&empty[slot], ((s / NS) & 1) ^ 1)) {
                    if (p.err) atomicOr(p.err, kErrTimeout);
                    s_abort = 1;
                    break;
                }
                if (s_abort) break;
                const int o0 = r0 + s * opst;
                const int no = min(opst, r1 - o0);
                unsigned char* dst = ring + (size_t)slot * stage_bytes;
                if constexpr (kSwiglu) {
                    mbar_arrive_expect_tx(&full[slot], (uint32_t)(2 * no * rowb));
                    bulk_g2s(dst, W + (size_t)o0 * rowb, (uint32_t)(no * rowb), &full[slot], pol);
                    bulk_g2s(dst + (size_t)opst * rowb, W + ((size_t)p.N + o0) * rowb, (uint32_t)(no * rowb),
                             &full[slot], pol);
                } else {
                    mbar_arrive_expect_tx(&full[slot], (uint32_t)(no * rowb));
                    bulk_g2s(dst, W + (size_t)o0 * rowb, (uint32_t)(no * rowb), &full[slot], pol);
                }
                issued = s + 1;
            }
            if (s_abort) {
                // let the copies still in flight land before the CTA retires
                for (int i = issued > NS ? issued - NS : 0; i < issued; ++i)
                    mbar_wait(&full[i % NS], (i / NS) & 1);
            } else if (p.next_W && p.next_pf > 0) {
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
        }
        return;
    }

    // ---- consumer warps ---------------------------------------------------------
    pdl_wait();
    pdl_trigger();

    // prologue: activation vector -> shared memory, planar per 16-byte chunk
    const float4* x4 = reinterpret_cast<const float4*>(p.x);
    float scale_in = 1.0f;
    if constexpr (PRO == kProRms) {
        float ss = 0.f;
        for (int i = threadIdx.x; i < K / 4; i += kConsumers) {
            const float4 v = x4[i];
            ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
        }
        ss = consumer_sum(ss, red);
        scale_in = 1.0f / sqrtf(ss / (float)K + p.eps);
    }
    float sa = 1.0f;
    if constexpr (PREC == kBF16) {
        float4* xs4 = reinterpret_cast<float4*>(xs);
        for (int i = threadIdx.x; i < K / 4; i += kConsumers) {
            float4 v = x4[i];
            if constexpr (PRO == kProRms) {
                const uint2 g = *reinterpret_cast<const uint2*>(p.gamma + 4 * i);
                v.x = v.x * scale_in * bf16lo(g.x);
                v.y = v.y * scale_in * bf16hi(g.x);
                v.z = v.z * scale_in * bf16lo(g.y);
                v.w = v.w * scale_in * bf16hi(g.y);
            }
            const int e = 4 * i;  // chunk e/8, plane (e%8)/4
            xs4[((e & 7) >> 2) * CPR + (e >> 3)] = v;
        }
    } else {
        // normalise, then amax, then quantise; the normalised values are
        // recomputed in the second pass instead of being stored
        float amax = 0.f;
        for (int i = threadIdx.x; i < K / 4; i += kConsumers) {
            float4 v = x4[i];
            if constexpr (PRO == kProRms) {
                const uint2 g = *reinterpret_cast<const uint2*>(p.gamma + 4 * i);
                v.x = v.x * scale_in * bf16lo(g.x);
                v.y = v.y * scale_in * bf16hi(g.x);
                v.z = v.z * scale_in * bf16lo(g.y);
                v.w = v.w * scale_in * bf16hi(g.y);
            }
            amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
        }
        amax = consumer_max(amax, red);
        sa = __fdiv_rn(fmaxf(amax, 1e-12f), 448.0f);
        uint2* xs2 = reinterpret_cast<uint2*>(xs);  // 4 f16 per uint2
        for (int i = threadIdx.x; i < K / 4; i += kConsumers) {
            float4 v = x4[i];
            if constexpr (PRO == kProRms) {
                const uint2 g = *reinterpret_cast<const uint2*>(p.gamma + 4 * i);
                v.x = v.x * scale_in * bf16lo(g.x);
                v.y = v.y * scale_in * bf16hi(g.x);
                v.z = v.z * scale_in * bf16lo(g.y);
                v.w = v.w * scale_in * bf16hi(g.y);
            }
            const __half2 h01 = __floats2half2_rn(quant_e4m3(__fdiv_rn(v.x, sa)), quant_e4m3(__fdiv_rn(v.y, sa)));
            const __half2 h23 = __floats2half2_rn(quant_e4m3(__fdiv_rn(v.z, sa)), quant_e4m3(__fdiv_rn(v.w, sa)));
            const int e = 4 * i;  // chunk e/16, plane (e%16)/8, half (e%8)/4
            uint2 packed;
            packed.x = *reinterpret_cast<const uint32_t*>(&h01);
            packed.y = *reinterpret_cast<const uint32_t*>(&h23);
            xs2[(((e & 15) >> 3) * CPR + (e >> 4)) * 2 + ((e & 7) >> 2)] = packed;
        }
    }
    consumer_sync();

    // main loop: warp w reduces segment w % WPR of row slot w / WPR of each stage
    const int rslot = warp / WPR, sg = warp % WPR;
    const int c0 = (int)((long long)sg * CPR / WPR), c1 = (int)((long long)(sg + 1) * CPR / WPR);
    // row slot -> output within the stage, and whether it is an up row
    const int oslot = kSwiglu ? (rslot % (RS / 2)) : rslot;
    for (int s = 0; s < nst; ++s) {
        const int slot = s % NS;
        if (!mbar_wait(&full[slot], (s / NS) & 1)) {
            if (lane == 0 && p.err) atomicOr(p.err, kErrTimeout);
            s_abort = 1;
            break;
        }
        const int out = s * opst + oslot;  // local output index of this warp's row
        if (out < nrows) {
            const uint4* wrow = reinterpret_cast<const uint4*>(ring + (size_t)slot * stage_bytes + rslot * rowb);
            float acc0 = 0.f, acc1 = 0.f;
#pragma unroll 4
            for (int c = c0 + lane; c < c1; c += 64) {
                if constexpr (PREC == kBF16) {
                    const float4* xs4 = reinterpret_cast<const float4*>(xs);
                    acc0 = dot_bf16(wrow[c], xs4[c], xs4[CPR + c], acc0);
                    if (c + 32 < c1) acc1 = dot_bf16(wrow[c + 32], xs4[c + 32], xs4[CPR + c + 32], acc1);
                } else {
                    const uint4* xs8 = reinterpret_cast<const uint4*>(xs);
                    acc0 = dot_fp8(wrow[c], xs8[c], xs8[CPR + c], acc0);
                    if (c + 32 < c1) acc1 = dot_fp8(wrow[c + 32], xs8[c + 32], xs8[CPR + c + 32], acc1);
                }
            }
            const float v = warp_sum(acc0 + acc1);
            if (lane == 0) part[(s * RS + rslot) * WPR + sg] = v;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
    }
    consumer_sync();
    if (s_abort) return;

    // ---- per-row sums over segments (in segment order) and the epilogue ---------
    auto row_sum = [&](int s, int rs) {
        const float* pr = part + (s * RS + rs) * WPR;
        float acc = 0.f;
        for (int q = 0; q < WPR; ++q) acc += pr[q];
        return acc;
    };
    for (int r = threadIdx.x; r < nrows; r += kConsumers) {
        const int n = r0 + r;
        const int s = r / opst, j = r % opst;
        if constexpr (kSwiglu) {
            float g = row_sum(s, j), u = row_sum(s, RS / 2 + j);
            if constexpr (PREC == kFP8) {
                g = round_bf16(g * (sa * p.wscale[n]));
                u = round_bf16(u * (sa * p.wscale[p.N + n]));
                p.y[n] = round_bf16(silu(g) * u);
            } else {
                p.y[n] = silu(g) * u;
            }
        } else {
            float o = row_sum(s, j);
            if constexpr (PREC == kFP8) o = round_bf16(o * (sa * p.wscale[n]));
            if constexpr (EPI == kEpiResid) p.y[n] += o;
            else p.y[n] = o;
        }
    }

    // ---- codebook head: the last CTA takes the greedy argmax --------------------
    if constexpr (EPI == kEpiLogits) {
        __threadfence();
        consumer_sync();
        if (threadIdx.x == 0) s_last = (atomicAdd(p.counter, 1u) == gridDim.x - 1);
        consumer_sync();
        if (!s_last) return;
        __threadfence();
        const int Vc = p.cb_vocab;
        const int t = p.st->t, eoc = p.st->eoc;
        for (int k = warp; k < p.n_cb; k += kConsumerWarps) {
            float best = -INFINITY;
            int bi = 0x7fffffff;
            for (int v = lane; v < Vc; v += 32) {
                const float x = __ldcg(p.y + (size_t)k * Vc + v);
                if (x > best) { best = x; bi = v; }  // increasing v: first maximum kept
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ob = __shfl_xor_sync(0xffffffffu, best, o);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                if (ob > best || (ob == best && oi < bi)) { best = ob; bi = oi; }
            }
            if (bi == 0x7fffffff) bi = 0;  // all NaN: take code 0
            if (lane == 0) {
                // Delay pattern: codebook k starts k frames late (BOS-pad before)
                // and ends k frames after codebook 0 emitted EOC.
                int c = bi;
                if (t < k) c = Vc - 2;
                else if (eoc >= 0 && t >= eoc + k) c = Vc - 1;
                s_codes[k] = c;
            }
        }
        consumer_sync();
        if (threadIdx.x == 0) {
            DevState* st = p.st;
            if (eoc < 0 && s_codes[0] == Vc - 1) st->eoc = t;
            int* hrow = p.hist + (size_t)(st->hist_idx % p.hist_cap) * p.n_cb;
            for (int k = 0; k < p.n_cb; ++k) {
                st->codes[k] = s_codes[k];
                hrow[k] = s_codes[k];
            }
            st->hist_idx += 1;
            st->t = t + 1;
            st->pos += 1;
            *p.counter = 0u;
        }
    }
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
    const int elems = prec == kBF16 ? 8 : 16;
    const int cpr = K / elems;
    const long long rowb = (long long)cpr * 16;
    const bool swiglu = epi == kEpiSwiglu;
    int rs = kConsumerWarps;                               // rows per stage: power of two <= 16
    while (rs > (swiglu ? 2 : 1) && rs * rowb > kStageTarget) rs >>= 1;
    g.rs = rs;
    const int opst = swiglu ? rs / 2 : rs;
    const long long rows_max = grid > 0 ? (N + grid - 1) / grid : N;
    const long long nst_max = (rows_max + opst - 1) / opst;
    g.part_bytes = round128((int)(nst_max * kConsumerWarps * (long long)sizeof(float)));
    const int xbytes = K * (prec == kBF16 ? 4 : 2);
    const long long stage = rs * rowb;
    long long ns = stage > 0 ? (kSmemBudget - kBarrierBytes - xbytes - g.part_bytes) / stage : 0;
    if (ns > kMaxStages) ns = kMaxStages;
    g.nstages = (int)ns;
    g.smem = (int)(kBarrierBytes + xbytes + g.part_bytes + ns * stage);
    g.ok = K % 256 == 0 && ns >= 2 && rs * rowb <= (1ll << 20) && g.smem <= kSmemBudget &&
           cpr >= kConsumerWarps / rs;
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
    p.nstages = g.nstages;
    p.part_bytes = g.part_bytes;
#define TTS_GEMV_CASE(PR, PO, EP) \
    if (prec == PR && pro == PO && epi == EP) return launch_one<PR, PO, EP>(p, g.smem, lc, s);
    TTS_GEMV_VARIANTS(TTS_GEMV_CASE)
#undef TTS_GEMV_CASE
    return cudaErrorInvalidValue;
}

}  // namespace tts

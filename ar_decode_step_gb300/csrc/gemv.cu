// M = 1 weight-streaming GEMV family for the decode step (sm_103a).
//
// One kernel template covers every projection of the step ("Higgs Audio v3
// TTS-4B on FlashRT", section 5: QKV, O-proj with fused residual, gate/up with
// SwiGLU, down-proj with fused residual, fused codebook head):
//   prologue : x -> shared memory, optionally RMSNorm (fp32) and, for FP8, the
//              per-token dynamic E4M3 quantisation (scale = amax / 448),
//              computed redundantly by every CTA so no separate norm/quant
//              kernel and no grid-wide dependency exist;
//   main loop: each warp owns a contiguous range of output rows; lanes stream
//              16-byte weight chunks straight from HBM to registers (no L1
//              allocation), two rows in flight per warp, and reduce with warp
//              shuffles;
//   epilogue : store, residual add, SwiGLU over the gate/up row pair, or the
//              codebook-head logits followed by a last-CTA greedy argmax with
//              the delay-pattern mask (section 4, sampling policy).
// Before waiting on the producing kernel (programmatic dependent launch) each
// warp asks L2 to prefetch its first rows, so HBM keeps streaming across the
// kernel boundary.
#include "kernels.h"

namespace tts {

namespace {

constexpr int kUnroll = 4;  // 16-byte chunks per lane per row per iteration

template <int PREC>
struct ChunkTraits;
template <>
struct ChunkTraits<kBF16> {
    static constexpr int kElems = 8;   // bf16 per 16 bytes
    static constexpr int kBytes = 2;
};
template <>
struct ChunkTraits<kFP8> {
    static constexpr int kElems = 16;  // e4m3 per 16 bytes
    static constexpr int kBytes = 1;
};

// Dot product of one 16-byte weight chunk with its activations (fp32 in
// shared memory, stored as kElems/4 float4 planes).
template <int PREC>
__device__ __forceinline__ float chunk_dot(const uint4 w, const float4* xv, float acc) {
    if constexpr (PREC == kBF16) {
        acc = fmaf(bf16lo(w.x), xv[0].x, acc);
        acc = fmaf(bf16hi(w.x), xv[0].y, acc);
        acc = fmaf(bf16lo(w.y), xv[0].z, acc);
        acc = fmaf(bf16hi(w.y), xv[0].w, acc);
        acc = fmaf(bf16lo(w.z), xv[1].x, acc);
        acc = fmaf(bf16hi(w.z), xv[1].y, acc);
        acc = fmaf(bf16lo(w.w), xv[1].z, acc);
        acc = fmaf(bf16hi(w.w), xv[1].w, acc);
    } else {
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float a, b, c, d;
            e4m3x4_to_f32(ws[q], a, b, c, d);
            acc = fmaf(a, xv[q].x, acc);
            acc = fmaf(b, xv[q].y, acc);
            acc = fmaf(c, xv[q].z, acc);
            acc = fmaf(d, xv[q].w, acc);
        }
    }
    return acc;
}

// Dot products of NR weight rows with the shared activation vector.  Lane l
// handles chunks l, l+32, ...; the result is summed over the warp (every lane
// gets it).
template <int PREC, int NR>
__device__ __forceinline__ void dot_rows(const uint8_t* const* rows, const float4* xs4, int nch,
                                         int lane, float* out) {
    constexpr int Q = ChunkTraits<PREC>::kElems / 4;
    float acc[NR][2];
#pragma unroll
    for (int r = 0; r < NR; ++r) acc[r][0] = acc[r][1] = 0.f;
    for (int c0 = lane; c0 < nch; c0 += 32 * kUnroll) {
        uint4 w[NR][kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int c = c0 + 32 * u;
#pragma unroll
            for (int r = 0; r < NR; ++r)
                w[r][u] = (c < nch) ? ldg_stream16(rows[r] + (size_t)c * 16) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int c = c0 + 32 * u;
            if (c < nch) {
                float4 xv[Q];
#pragma unroll
                for (int q = 0; q < Q; ++q) xv[q] = xs4[q * nch + c];
#pragma unroll
                for (int r = 0; r < NR; ++r) acc[r][u & 1] = chunk_dot<PREC>(w[r][u], xv, acc[r][u & 1]);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < NR; ++r) out[r] = warp_sum(acc[r][0] + acc[r][1]);
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

template <int PREC, int PRO, int EPI>
__global__ void __launch_bounds__(256) gemv_kernel(const GemvParams p) {
    extern __shared__ float4 xs4[];  // [kElems/4][nch] activation planes
    __shared__ float red[32];
    __shared__ int s_last;
    __shared__ int s_codes[kMaxCodebooks];

    constexpr int E = ChunkTraits<PREC>::kElems;
    constexpr bool kSwiglu = EPI == kEpiSwiglu;
    const int K = p.K, nch = K / E;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarp = blockDim.x >> 5;
    const long long TW = (long long)gridDim.x * nwarp, gw = (long long)blockIdx.x * nwarp + warp;
    const int n0 = (int)(gw * p.N / TW), n1 = (int)((gw + 1) * p.N / TW);
    const size_t rowb = (size_t)K * ChunkTraits<PREC>::kBytes;
    const uint8_t* W = static_cast<const uint8_t*>(p.W);

    // Warm L2 with this warp's first rows while the producer finishes.
    {
        const int nrows = n1 - n0;
        const int npf = kSwiglu ? (nrows < 2 ? nrows : 2) : (nrows < 4 ? nrows : 4);
        if (lane < npf) prefetch_l2_bulk(W + (size_t)(n0 + lane) * rowb, (uint32_t)rowb);
        if (kSwiglu && lane >= 16 && lane - 16 < npf)
            prefetch_l2_bulk(W + (size_t)(p.N + n0 + lane - 16) * rowb, (uint32_t)rowb);
    }

    pdl_wait();
    pdl_trigger();

    // ---- prologue: activation vector -> shared memory -------------------
    const float4* x4 = reinterpret_cast<const float4*>(p.x);
    float scale_in = 1.0f;
    if constexpr (PRO == kProRms) {
        float ss = 0.f;
        for (int i = threadIdx.x; i < K / 4; i += blockDim.x) {
            float4 v = x4[i];
            ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
        }
        ss = block_sum(ss, red);
        scale_in = 1.0f / sqrtf(ss / (float)K + p.eps);
    }
    float amax = 0.f;
    for (int i = threadIdx.x; i < K / 4; i += blockDim.x) {
        float4 v = x4[i];
        if constexpr (PRO == kProRms) {
            const uint2 g = *reinterpret_cast<const uint2*>(p.gamma + 4 * i);
            v.x = v.x * scale_in * bf16lo(g.x);
            v.y = v.y * scale_in * bf16hi(g.x);
            v.z = v.z * scale_in * bf16lo(g.y);
            v.w = v.w * scale_in * bf16hi(g.y);
        }
        if constexpr (PREC == kFP8)
            amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
        const int e = 4 * i;
        xs4[((e % E) / 4) * nch + e / E] = v;
    }
    float sa = 1.0f;
    if constexpr (PREC == kFP8) {
        amax = block_max(amax, red);  // includes __syncthreads(): planes are complete
        sa = __fdiv_rn(fmaxf(amax, 1e-12f), 448.0f);
        for (int i = threadIdx.x; i < K / 4; i += blockDim.x) {
            const int e = 4 * i;
            float4& v = xs4[((e % E) / 4) * nch + e / E];
            v.x = quant_e4m3(__fdiv_rn(v.x, sa));
            v.y = quant_e4m3(__fdiv_rn(v.y, sa));
            v.z = quant_e4m3(__fdiv_rn(v.z, sa));
            v.w = quant_e4m3(__fdiv_rn(v.w, sa));
        }
    }
    __syncthreads();

    // ---- main loop ------------------------------------------------------------
    if constexpr (kSwiglu) {
        for (int n = n0; n < n1; ++n) {
            const uint8_t* rows[2] = {W + (size_t)n * rowb, W + (size_t)(p.N + n) * rowb};
            float r[2];
            dot_rows<PREC, 2>(rows, xs4, nch, lane, r);
            if (lane == 0) {
                float g = r[0], u = r[1];
                if constexpr (PREC == kFP8) {
                    g = round_bf16(g * (sa * p.wscale[n]));
                    u = round_bf16(u * (sa * p.wscale[p.N + n]));
                    p.y[n] = round_bf16(silu(g) * u);
                } else {
                    p.y[n] = silu(g) * u;
                }
            }
        }
    } else {
        int n = n0;
        for (; n + 1 < n1; n += 2) {
            const uint8_t* rows[2] = {W + (size_t)n * rowb, W + (size_t)(n + 1) * rowb};
            float r[2];
            dot_rows<PREC, 2>(rows, xs4, nch, lane, r);
            if (lane < 2) {
                const int nn = n + lane;
                float v = lane ? r[1] : r[0];
                if constexpr (PREC == kFP8) v = round_bf16(v * (sa * p.wscale[nn]));
                if constexpr (EPI == kEpiResid) p.y[nn] += v;
                else p.y[nn] = v;
            }
        }
        if (n < n1) {
            const uint8_t* rows[1] = {W + (size_t)n * rowb};
            float r[1];
            dot_rows<PREC, 1>(rows, xs4, nch, lane, r);
            if (lane == 0) {
                float v = r[0];
                if constexpr (PREC == kFP8) v = round_bf16(v * (sa * p.wscale[n]));
                if constexpr (EPI == kEpiResid) p.y[n] += v;
                else p.y[n] = v;
            }
        }
    }

    // ---- codebook head: last CTA takes the greedy argmax -----------------------
    if constexpr (EPI == kEpiLogits) {
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) s_last = (atomicAdd(p.counter, 1u) == gridDim.x - 1);
        __syncthreads();
        if (!s_last) return;
        __threadfence();
        const int V = p.cb_vocab;
        const int t = p.st->t, eoc = p.st->eoc;
        for (int k = warp; k < p.n_cb; k += nwarp) {
            float best = -INFINITY;
            int bi = 0x7fffffff;
            for (int v = lane; v < V; v += 32) {
                const float x = __ldcg(p.y + (size_t)k * V + v);
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
                // Delay pattern: codebook k starts k frames late (BOS-pad before),
                // and ends k frames after codebook 0 emitted EOC.
                int c = bi;
                if (t < k) c = V - 2;
                else if (eoc >= 0 && t >= eoc + k) c = V - 1;
                s_codes[k] = c;
            }
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            DevState* st = p.st;
            if (eoc < 0 && s_codes[0] == V - 1) st->eoc = t;
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
cudaError_t launch_one(const GemvParams& p, const LaunchCfg& lc, cudaStream_t s) {
    auto kern = gemv_kernel<PREC, PRO, EPI>;
    const int smem = gemv_smem_bytes(PREC, p.K);
    if (smem > 48 * 1024) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(lc.grid);
    cfg.blockDim = dim3(lc.threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = lc.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace

int gemv_smem_bytes(int prec, int K) { return K * (int)sizeof(float); }

cudaError_t launch_gemv(int prec, int pro, int epi, const GemvParams& p, const LaunchCfg& lc,
                        cudaStream_t s) {
#define TTS_GEMV_CASE(PR, PO, EP)                                   \
    if (prec == PR && pro == PO && epi == EP) return launch_one<PR, PO, EP>(p, lc, s);
    TTS_GEMV_CASE(kBF16, kProRms, kEpiStore)
    TTS_GEMV_CASE(kBF16, kProPlain, kEpiResid)
    TTS_GEMV_CASE(kBF16, kProRms, kEpiSwiglu)
    TTS_GEMV_CASE(kBF16, kProRms, kEpiLogits)
    TTS_GEMV_CASE(kBF16, kProPlain, kEpiStore)
    TTS_GEMV_CASE(kFP8, kProRms, kEpiStore)
    TTS_GEMV_CASE(kFP8, kProPlain, kEpiResid)
    TTS_GEMV_CASE(kFP8, kProRms, kEpiSwiglu)
    TTS_GEMV_CASE(kFP8, kProPlain, kEpiStore)
#undef TTS_GEMV_CASE
    return cudaErrorInvalidValue;
}

}  // namespace tts

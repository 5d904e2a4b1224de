// Split-K GQA decode attention with the per-head q/k RMSNorm, RoPE and the
// bf16 KV-cache write fused into its prologue (sm_103a).
//
// "Higgs Audio v3 TTS-4B on FlashRT", section 5: "fused q/k-norm + RoPE" then
// attention over the KV cache; page header: GQA 32q/8kv, head_dim 128, RoPE
// theta 1e6.  One CTA handles one key-value head and one contiguous range of
// positions (a split); the G = n_q/n_kv query heads of the group share every
// K/V row it loads.  The current position's key and value are normalised,
// rotated, rounded to bf16, written to the cache and used from shared memory
// by the CTA whose range ends at the position.  Partial results (running max,
// sum of exponentials, unnormalised output) of all splits of a head are merged
// by whichever CTA finishes last (atomic ticket, no waiting).
#include "kernels.h"

namespace tts {

namespace {

constexpr int kMinChunk = 16;   // positions per split, at least
constexpr int kMaxSplits = 64;  // splits per kv head, at most
constexpr int kWarps = 4;

template <int G>
__global__ void __launch_bounds__(kWarps * 32) attn_decode_kernel(const AttnParams p) {
    __shared__ float qs[G][kHeadDim];       // normalised, rotated, pre-scaled queries
    __shared__ float knew[kHeadDim], vnew[kHeadDim];
    __shared__ float wm[kWarps][G], wl[kWarps][G];
    __shared__ float wo[kWarps][G][kHeadDim];
    __shared__ int s_last;

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = blockIdx.x / p.S, split = blockIdx.x % p.S;

    pdl_wait();
    pdl_trigger();

    const int pos = p.pos_override >= 0 ? p.pos_override : p.st->pos;
    if (pos < 0 || pos >= p.max_pos) {
        if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(&p.st->err, kErrPos);
        return;
    }
    const int len = pos + 1;
    int chunk = (len + p.S - 1) / p.S;
    if (chunk < kMinChunk) chunk = kMinChunk;
    const int nsplit = (len + chunk - 1) / chunk;
    if (split >= nsplit) return;
    const int t0 = split * chunk;
    const int t1 = min(len, t0 + chunk);
    const bool has_new = (t1 == len);  // this split ends at the current position

    const float2* rope = p.rope_row ? p.rope_row : p.rope + (size_t)pos * (kHeadDim / 2);
    const float scale = 1.0f / sqrtf((float)kHeadDim);

    // q/k RMSNorm over head_dim then rotate-half RoPE: lane l holds dims
    // 4l..4l+3; its rotation partner dims (+-64) sit in lane l^16.
    auto norm_rope = [&](const float* src, const __nv_bfloat16* gamma, float* dst, float post) {
        float4 v = *reinterpret_cast<const float4*>(src + 4 * lane);
        float ss = warp_sum(v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w);
        const float r = 1.0f / sqrtf(ss / (float)kHeadDim + p.eps);
        const uint2 gb = *reinterpret_cast<const uint2*>(gamma + 4 * lane);
        float a[4] = {v.x * r * bf16lo(gb.x), v.y * r * bf16hi(gb.x), v.z * r * bf16lo(gb.y),
                      v.w * r * bf16hi(gb.y)};
        float o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float partner = __shfl_xor_sync(0xffffffffu, a[j], 16);
            const float2 cs = rope[(4 * lane + j) & 63];
            o[j] = lane < 16 ? a[j] * cs.x - partner * cs.y : a[j] * cs.x + partner * cs.y;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) dst[4 * lane + j] = o[j] * post;
    };

    for (int j = warp; j < G; j += kWarps)
        norm_rope(p.qkv + (size_t)(g * G + j) * kHeadDim, p.q_norm, qs[j], scale);
    if (has_new && warp == 0) {
        norm_rope(p.qkv + (size_t)(p.n_q + g) * kHeadDim, p.k_norm, knew, 1.0f);
        __syncwarp();
        const float* vsrc = p.qkv + (size_t)(p.n_q + p.n_kv + g) * kHeadDim;
        __nv_bfloat16* kd = p.kc + ((size_t)g * p.max_pos + pos) * kHeadDim;
        __nv_bfloat16* vd = p.vc + ((size_t)g * p.max_pos + pos) * kHeadDim;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int d = 4 * lane + j;
            const __nv_bfloat16 kb = __float2bfloat16_rn(knew[d]);
            const __nv_bfloat16 vb = __float2bfloat16_rn(vsrc[d]);
            kd[d] = kb;
            vd[d] = vb;
            knew[d] = __bfloat162float(kb);
            vnew[d] = __bfloat162float(vb);
        }
    }
    __syncthreads();

    // ---- scan the positions: online softmax per query head ------------------
    float m[G], l[G], o[G][4];
    float qr[G][4];
#pragma unroll
    for (int j = 0; j < G; ++j) {
        m[j] = -INFINITY;
        l[j] = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) { o[j][i] = 0.f; qr[j][i] = qs[j][4 * lane + i]; }
    }
    const __nv_bfloat16* kbase = p.kc + (size_t)g * p.max_pos * kHeadDim + 4 * lane;
    const __nv_bfloat16* vbase = p.vc + (size_t)g * p.max_pos * kHeadDim + 4 * lane;
    const int tcache_end = has_new ? t1 - 1 : t1;  // cached rows; the new row comes from smem

    auto consume = [&](const float* kv4, const float* vv4) {
        float s[G];
#pragma unroll
        for (int j = 0; j < G; ++j)
            s[j] = qr[j][0] * kv4[0] + qr[j][1] * kv4[1] + qr[j][2] * kv4[2] + qr[j][3] * kv4[3];
#pragma unroll
        for (int j = 0; j < G; ++j) s[j] = warp_sum(s[j]);
#pragma unroll
        for (int j = 0; j < G; ++j) {
            const float mn = fmaxf(m[j], s[j]);
            const float corr = __expf(m[j] - mn);
            const float pj = __expf(s[j] - mn);
            l[j] = l[j] * corr + pj;
#pragma unroll
            for (int i = 0; i < 4; ++i) o[j][i] = o[j][i] * corr + pj * vv4[i];
            m[j] = mn;
        }
    };

    int t = t0 + warp;
    for (; t + kWarps < tcache_end; t += 2 * kWarps) {
        const uint2 ka = *reinterpret_cast<const uint2*>(kbase + (size_t)t * kHeadDim);
        const uint2 va = *reinterpret_cast<const uint2*>(vbase + (size_t)t * kHeadDim);
        const uint2 kb = *reinterpret_cast<const uint2*>(kbase + (size_t)(t + kWarps) * kHeadDim);
        const uint2 vb = *reinterpret_cast<const uint2*>(vbase + (size_t)(t + kWarps) * kHeadDim);
        float k4[4] = {bf16lo(ka.x), bf16hi(ka.x), bf16lo(ka.y), bf16hi(ka.y)};
        float v4[4] = {bf16lo(va.x), bf16hi(va.x), bf16lo(va.y), bf16hi(va.y)};
        consume(k4, v4);
        float k4b[4] = {bf16lo(kb.x), bf16hi(kb.x), bf16lo(kb.y), bf16hi(kb.y)};
        float v4b[4] = {bf16lo(vb.x), bf16hi(vb.x), bf16lo(vb.y), bf16hi(vb.y)};
        consume(k4b, v4b);
    }
    for (; t < tcache_end; t += kWarps) {
        const uint2 ka = *reinterpret_cast<const uint2*>(kbase + (size_t)t * kHeadDim);
        const uint2 va = *reinterpret_cast<const uint2*>(vbase + (size_t)t * kHeadDim);
        float k4[4] = {bf16lo(ka.x), bf16hi(ka.x), bf16lo(ka.y), bf16hi(ka.y)};
        float v4[4] = {bf16lo(va.x), bf16hi(va.x), bf16lo(va.y), bf16hi(va.y)};
        consume(k4, v4);
    }
    if (has_new && warp == ((t1 - 1 - t0) % kWarps)) {
        float k4[4], v4[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) { k4[i] = knew[4 * lane + i]; v4[i] = vnew[4 * lane + i]; }
        consume(k4, v4);
    }

    // ---- merge the warps of this CTA ------------------------------------------
#pragma unroll
    for (int j = 0; j < G; ++j) {
        if (lane == 0) { wm[warp][j] = m[j]; wl[warp][j] = l[j]; }
#pragma unroll
        for (int i = 0; i < 4; ++i) wo[warp][j][4 * lane + i] = o[j][i];
    }
    __syncthreads();
    // thread -> (head j, dim d): G*128 outputs over 128 threads
    float* po = p.part_o + (((size_t)g * p.S + split) * G) * kHeadDim;
    float* pml = p.part_ml + (((size_t)g * p.S + split) * G) * 2;
    for (int idx = threadIdx.x; idx < G * kHeadDim; idx += blockDim.x) {
        const int j = idx / kHeadDim, d = idx % kHeadDim;
        float M = wm[0][j];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) M = fmaxf(M, wm[w][j]);
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float c = (wm[w][j] == -INFINITY) ? 0.f : __expf(wm[w][j] - M);
            L += wl[w][j] * c;
            O += wo[w][j][d] * c;
        }
        if (nsplit == 1) {
            p.out[(size_t)(g * G + j) * kHeadDim + d] = O / L;
        } else {
            po[idx] = O;
            if (d == 0) { pml[2 * j] = M; pml[2 * j + 1] = L; }
        }
    }
    if (nsplit == 1) return;

    // ---- last split of this kv head merges all splits ----------------------------
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = (atomicAdd(&p.counter[g], 1u) == (unsigned)(nsplit - 1));
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    const float* po0 = p.part_o + ((size_t)g * p.S * G) * kHeadDim;
    const float* pml0 = p.part_ml + ((size_t)g * p.S * G) * 2;
    for (int idx = threadIdx.x; idx < G * kHeadDim; idx += blockDim.x) {
        const int j = idx / kHeadDim, d = idx % kHeadDim;
        float M = -INFINITY;
        for (int s = 0; s < nsplit; ++s) M = fmaxf(M, __ldcg(pml0 + ((size_t)s * G + j) * 2));
        float L = 0.f, O = 0.f;
        for (int s = 0; s < nsplit; ++s) {
            const float c = __expf(__ldcg(pml0 + ((size_t)s * G + j) * 2) - M);
            L += __ldcg(pml0 + ((size_t)s * G + j) * 2 + 1) * c;
            O += __ldcg(po0 + ((size_t)s * G + j) * kHeadDim + d) * c;
        }
        p.out[(size_t)(g * G + j) * kHeadDim + d] = O / L;
    }
    if (threadIdx.x == 0) p.counter[g] = 0u;
}

}  // namespace

cudaError_t attention_prepare() {
    // querying a kernel's attributes loads its module on the current device
    cudaFuncAttributes a;
    cudaError_t e = cudaFuncGetAttributes(&a, attn_decode_kernel<1>);
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&a, attn_decode_kernel<2>);
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&a, attn_decode_kernel<4>);
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&a, attn_decode_kernel<8>);
    return e;
}

int attn_splits_for(int max_pos) {
    int s = (max_pos + kMinChunk - 1) / kMinChunk;
    return s < 1 ? 1 : (s > kMaxSplits ? kMaxSplits : s);
}

cudaError_t launch_attention(const AttnParams& p, const LaunchCfg& lc, cudaStream_t s) {
    const int G = p.n_q / p.n_kv;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.n_kv * p.S);
    cfg.blockDim = dim3(kWarps * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = lc.pdl ? 1 : 0;
    switch (G) {
        case 1: return cudaLaunchKernelEx(&cfg, attn_decode_kernel<1>, p);
        case 2: return cudaLaunchKernelEx(&cfg, attn_decode_kernel<2>, p);
        case 4: return cudaLaunchKernelEx(&cfg, attn_decode_kernel<4>, p);
        case 8: return cudaLaunchKernelEx(&cfg, attn_decode_kernel<8>, p);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace tts

// Small kernels of the decode step: the fused multi-codebook embedding, the
// prefill position advance, and per-row FP8 weight quantisation (sm_103a).
#include "kernels.h"

namespace tts {

namespace {

// x = sum_k E_k[c_k] (SGLang-Omni Higgs Audio v3 post, architecture: the 8
// codebook embeddings are summed into the backbone's hidden state).  Codes
// come from the device state (the previous step's greedy codes, or the frame
// the host wrote) or from one row of a prompt.
__global__ void embed_kernel(const EmbedParams p) {
    pdl_wait();
    pdl_trigger();
    __shared__ int codes[kMaxCodebooks];
    if (threadIdx.x < p.n_cb) {
        int c = p.rows ? p.rows[(size_t)p.st->prefill_row * p.n_cb + threadIdx.x] : p.st->codes[threadIdx.x];
        if (c < 0 || c >= p.cb_vocab) {
            atomicOr(&p.st->err, kErrCode);
            c = 0;
        }
        codes[threadIdx.x] = c;
    }
    __syncthreads();
    const int i4 = blockIdx.x * blockDim.x + threadIdx.x;  // 4 elements per thread
    if (4 * i4 >= p.H) return;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k = 0; k < p.n_cb; ++k) {
        const uint2 e = *reinterpret_cast<const uint2*>(
            p.E + ((size_t)k * p.cb_vocab + codes[k]) * p.H + 4 * i4);
        acc.x += bf16lo(e.x);
        acc.y += bf16hi(e.x);
        acc.z += bf16lo(e.y);
        acc.w += bf16hi(e.y);
    }
    reinterpret_cast<float4*>(p.h)[i4] = acc;
}

__global__ void advance_kernel(DevState* st) {
    pdl_wait();
    pdl_trigger();
    if (threadIdx.x == 0) {
        st->pos += 1;
        st->prefill_row += 1;
    }
}

// s[n] = max_k |W[n][k]| / 448 (1 for a zero row); W8 = E4M3(W / s[n]) with
// the quotient rounded as an IEEE fp32 division (div_rn_by), nearest-even
// rounding, saturation.  One CTA per row.
__global__ void quantize_weight_kernel(const __nv_bfloat16* W, int K, uint8_t* W8, float* s) {
    __shared__ float red[32];
    const size_t row = blockIdx.x;
    const __nv_bfloat16* w = W + row * K;
    float amax = 0.f;
    for (int k = threadIdx.x; k < K; k += blockDim.x) amax = fmaxf(amax, fabsf(__bfloat162float(w[k])));
    amax = block_max(amax, red);
    const float sc = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
    const float rsc = __frcp_rn(sc);
    for (int k = threadIdx.x; k < K; k += blockDim.x)
        W8[row * K + k] = __nv_cvt_float_to_fp8(div_rn_by(__bfloat162float(w[k]), sc, rsc), __NV_SATFINITE, __NV_E4M3);
    if (threadIdx.x == 0) s[row] = sc;
}

cudaLaunchConfig_t make_cfg(int grid, int threads, cudaStream_t s, bool pdl, cudaLaunchAttribute* attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cfg;
}

}  // namespace

cudaError_t launch_embed(const EmbedParams& p, const LaunchCfg& lc, cudaStream_t s) {
    cudaLaunchAttribute attr[1];
    const int threads = 128;
    const int grid = (p.H / 4 + threads - 1) / threads;
    cudaLaunchConfig_t cfg = make_cfg(grid, threads, s, lc.pdl, attr);
    return cudaLaunchKernelEx(&cfg, embed_kernel, p);
}

cudaError_t launch_advance(DevState* st, const LaunchCfg& lc, cudaStream_t s) {
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = make_cfg(1, 32, s, lc.pdl, attr);
    return cudaLaunchKernelEx(&cfg, advance_kernel, st);
}

cudaError_t launch_quantize_weight(const __nv_bfloat16* W, int N, int K, uint8_t* W8, float* s,
                                   cudaStream_t st) {
    if (N <= 0 || K <= 0) return cudaErrorInvalidValue;
    quantize_weight_kernel<<<N, 256, 0, st>>>(W, K, W8, s);
    return cudaGetLastError();
}

}  // namespace tts

// Batched prompt prefill: P positions through the layer stack at once
// ("Higgs Audio v3 TTS-4B on FlashRT", Performance "Prompt prefill", "BF16
// W16A16"; section 7: the prompt runs as one M = P pass that reads every
// weight once).  The projections are tensor-core GEMMs (gemm_tc.cu); the
// kernels here are the row-parallel glue between them and the causal
// attention over the prompt:
//   embed_rows        h[p] = sum_k E_k[codes[p][k]]
//   rmsnorm_rows      a[p] = bf16(RMSNorm(h[p]) * gamma)   (the GEMM's A operand)
//   qk_rope_kv_rows   per-head q/k RMSNorm + RoPE at position pos0 + p, q kept
//                     in fp32 (pre-scaled by 1/sqrt(128)), k and v written to
//                     the bf16 cache
//   attention_mma     causal GQA on the tensor cores: row p attends positions
//                     [0, pos0 + p]; output rounded to bf16 (the O-proj
//                     GEMM's A operand)
#include "kernels.h"

namespace tts {

namespace {

constexpr int kRowThreads = 256;

__global__ void __launch_bounds__(kRowThreads) embed_rows_kernel(const __nv_bfloat16* E, const int* codes,
                                                                 float* H, int n_cb, int V, int hidden) {
    const int p = blockIdx.x;
    const int* c = codes + (size_t)p * n_cb;
    for (int i = threadIdx.x; i < hidden; i += blockDim.x) {
        float acc = 0.f;
        for (int k = 0; k < n_cb; ++k) acc += __bfloat162float(E[((size_t)k * V + c[k]) * hidden + i]);
        H[(size_t)p * hidden + i] = acc;
    }
}

__global__ void __launch_bounds__(kRowThreads) rmsnorm_rows_kernel(const float* H, const __nv_bfloat16* gamma,
                                                                   __nv_bfloat16* out, int hidden, float eps) {
    __shared__ float red[32];
    const int p = blockIdx.x;
    const float* h = H + (size_t)p * hidden;
    float ss = 0.f;
    for (int i = threadIdx.x; i < hidden; i += blockDim.x) ss += h[i] * h[i];
    ss = block_sum(ss, red);
    const float r = 1.0f / sqrtf(ss / (float)hidden + eps);
    for (int i = threadIdx.x; i < hidden; i += blockDim.x)
        out[(size_t)p * hidden + i] = __float2bfloat16_rn(h[i] * r * __bfloat162float(gamma[i]));
}

// two floats as bf16 (nearest even), the first in the low half: 8-byte cache stores
__device__ __forceinline__ uint32_t pack_bf16x2_rows(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

__global__ void __launch_bounds__(kRowThreads) qk_rope_kv_rows_kernel(const float* QKV, const __nv_bfloat16* qn,
                                                                      const __nv_bfloat16* kn, const float2* rope,
                                                                      float* Q, __nv_bfloat16* kc,
                                                                      __nv_bfloat16* vc, int pos0, int n_q,
                                                                      int n_kv, int max_pos, float eps) {
    const int p = blockIdx.x, pos = pos0 + p;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qkv_dim = (n_q + 2 * n_kv) * kHeadDim;
    const float* x = QKV + (size_t)p * qkv_dim;
    const float2* rp = rope + (size_t)pos * (kHeadDim / 2);
    const float scale = 1.0f / sqrtf((float)kHeadDim);
    for (int hd = warp; hd < n_q + 2 * n_kv; hd += kRowThreads / 32) {
        const float4 v = reinterpret_cast<const float4*>(x + (size_t)hd * kHeadDim)[lane];
        if (hd >= n_q + n_kv) {  // v head: straight to the cache
            const int j = hd - n_q - n_kv;
            __nv_bfloat16* dst = vc + ((size_t)j * max_pos + pos) * kHeadDim + 4 * lane;
            *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16x2_rows(v.x, v.y), pack_bf16x2_rows(v.z, v.w));
            continue;
        }
        // RMSNorm over the head (gain q_norm / k_norm), then rotate-half RoPE:
        // lane l holds dims 4l..4l+3, their partners (+-64) sit in lane l ^ 16
        const __nv_bfloat16* g = hd < n_q ? qn : kn;
        const float ss = warp_sum(v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w);
        const float r = 1.0f / sqrtf(ss / (float)kHeadDim + eps);
        const float a[4] = {v.x * r * __bfloat162float(g[4 * lane]), v.y * r * __bfloat162float(g[4 * lane + 1]),
                            v.z * r * __bfloat162float(g[4 * lane + 2]), v.w * r * __bfloat162float(g[4 * lane + 3])};
        float o[4];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const float partner = __shfl_xor_sync(0xffffffffu, a[jj], 16);
            const float2 cs = rp[(4 * lane + jj) & 63];
            o[jj] = lane < 16 ? a[jj] * cs.x - partner * cs.y : a[jj] * cs.x + partner * cs.y;
        }
        if (hd < n_q) {
            reinterpret_cast<float4*>(Q + ((size_t)p * n_q + hd) * kHeadDim)[lane] =
                make_float4(o[0] * scale, o[1] * scale, o[2] * scale, o[3] * scale);
        } else {
            const int j = hd - n_q;
            __nv_bfloat16* dst = kc + ((size_t)j * max_pos + pos) * kHeadDim + 4 * lane;
            *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16x2_rows(o[0], o[1]), pack_bf16x2_rows(o[2], o[3]));
        }
    }
}

// RMSNorm rows, one warp per row held in registers (NV float4 per lane,
// hidden <= 128 NV, NV up to kRowVec): one read of h, warp reductions only.
constexpr int kRowVec = 32;
constexpr int kRowWarps = kRowThreads / 32;
template <int NV>
__global__ void __launch_bounds__(kRowThreads) rmsnorm_rows_warp_kernel(const float* H, const __nv_bfloat16* gamma,
                                                                        __nv_bfloat16* out, int P, int hidden,
                                                                        float eps) {
    const int row = blockIdx.x * kRowWarps + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (row >= P) return;
    const float4* h4 = reinterpret_cast<const float4*>(H + (size_t)row * hidden);
    const uint2* g4 = reinterpret_cast<const uint2*>(gamma);
    const int n4 = hidden / 4;
    float4 v[NV];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int j = lane + 32 * i;
        if (j < n4) {
            v[i] = h4[j];
            ss += v[i].x * v[i].x + v[i].y * v[i].y + v[i].z * v[i].z + v[i].w * v[i].w;
        }
    }
    ss = warp_sum(ss);
    const float r = 1.0f / sqrtf(ss / (float)hidden + eps);
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int j = lane + 32 * i;
        if (j < n4) {
            const uint2 g = g4[j];
            v[i] = make_float4(v[i].x * r * bf16lo(g.x), v[i].y * r * bf16hi(g.x), v[i].z * r * bf16lo(g.y),
                               v[i].w * r * bf16hi(g.y));
        }
    }
    uint2* o = reinterpret_cast<uint2*>(out + (size_t)row * hidden);
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int j = lane + 32 * i;
        if (j < n4) {
            const __nv_bfloat162 a = __floats2bfloat162_rn(v[i].x, v[i].y);
            const __nv_bfloat162 b = __floats2bfloat162_rn(v[i].z, v[i].w);
            o[j] = make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
        }
    }
}

// FP8 W8A8 rows: the projection inputs quantised per row (per token) as the
// decode step does ("Higgs Audio v3 TTS-4B on FlashRT", Performance "FP8
// W8A8"): s = max(amax, 1e-12) / 448, q = e4m3(x / s) with IEEE fp32 division,
// saturating.
__device__ __forceinline__ uint8_t e4m3_sat(float x) {
    return (uint8_t)__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
}

// a = RMSNorm(h) * gamma, then quantised (the QKV and gate/up inputs)
__global__ void __launch_bounds__(kRowThreads) rmsnorm_quant_rows_kernel(const float* H, const __nv_bfloat16* gamma,
                                                                         uint8_t* out, float* scale, int hidden,
                                                                         float eps) {
    __shared__ float red[32];
    const int p = blockIdx.x;
    const float* h = H + (size_t)p * hidden;
    float ss = 0.f;
    for (int i = threadIdx.x; i < hidden; i += blockDim.x) ss += h[i] * h[i];
    ss = block_sum(ss, red);
    const float r = 1.0f / sqrtf(ss / (float)hidden + eps);
    float am = 0.f;
    for (int i = threadIdx.x; i < hidden; i += blockDim.x)
        am = fmaxf(am, fabsf(h[i] * r * __bfloat162float(gamma[i])));
    am = block_max(am, red);
    const float sa = __fdiv_rn(fmaxf(am, 1e-12f), 448.0f), rsa = __frcp_rn(sa);
    for (int i = threadIdx.x; i < hidden; i += blockDim.x)
        out[(size_t)p * hidden + i] = e4m3_sat(div_rn_by(h[i] * r * __bfloat162float(gamma[i]), sa, rsa));
    if (threadIdx.x == 0) scale[p] = sa;
}

// rows quantised as they are: the attention output (fp32) and the MLP
// activation (bf16, already rounded as the FP8 SwiGLU defines it)
__device__ __forceinline__ float as_f32(float v) { return v; }
__device__ __forceinline__ float as_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T>
__global__ void __launch_bounds__(kRowThreads) quant_rows_kernel(const T* X, uint8_t* out, float* scale, int n) {
    __shared__ float red[32];
    const int p = blockIdx.x;
    const T* x = X + (size_t)p * n;
    float am = 0.f;
    for (int i = threadIdx.x; i < n; i += blockDim.x) am = fmaxf(am, fabsf(as_f32(x[i])));
    am = block_max(am, red);
    const float sa = __fdiv_rn(fmaxf(am, 1e-12f), 448.0f), rsa = __frcp_rn(sa);
    for (int i = threadIdx.x; i < n; i += blockDim.x)
        out[(size_t)p * n + i] = e4m3_sat(div_rn_by(as_f32(x[i]), sa, rsa));
    if (threadIdx.x == 0) scale[p] = sa;
}

// The same two quantisations with each row held in registers: one read of
// the row, 16-byte loads and 8-byte stores (8 elements per vector, NV
// vectors per thread); the arithmetic is that of the kernels above.
__device__ __forceinline__ void load8(const float* x, float (&v)[8]) {
    const float4 a = *reinterpret_cast<const float4*>(x), b = *reinterpret_cast<const float4*>(x + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void load8(const __nv_bfloat16* x, float (&v)[8]) {
    const uint4 w = *reinterpret_cast<const uint4*>(x);
    v[0] = bf16lo(w.x); v[1] = bf16hi(w.x); v[2] = bf16lo(w.y); v[3] = bf16hi(w.y);
    v[4] = bf16lo(w.z); v[5] = bf16hi(w.z); v[6] = bf16lo(w.w); v[7] = bf16hi(w.w);
}
__device__ __forceinline__ uint2 quant8(const float (&v)[8], float sa, float rsa) {
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        lo |= (uint32_t)e4m3_sat(div_rn_by(v[e], sa, rsa)) << (8 * e);
        hi |= (uint32_t)e4m3_sat(div_rn_by(v[e + 4], sa, rsa)) << (8 * e);
    }
    return make_uint2(lo, hi);
}

template <int NV>
__global__ void __launch_bounds__(kRowThreads) rmsnorm_quant_rows_reg_kernel(const float* H,
                                                                             const __nv_bfloat16* gamma, uint8_t* out,
                                                                             float* scale, int hidden, float eps) {
    __shared__ float red[32];
    const int p = blockIdx.x, n8 = hidden / 8;
    const float* h = H + (size_t)p * hidden;
    float v[NV][8];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int j = threadIdx.x + i * kRowThreads;
        if (j < n8) {
            load8(h + 8 * j, v[i]);
#pragma unroll
            for (int e = 0; e < 8; ++e) ss += v[i][e] * v[i][e];
        }
    }
    ss = block_sum(ss, red);
    const float r = 1.0f / sqrtf(ss / (float)hidden + eps);
    float am = 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int j = threadIdx.x + i * kRowThreads;
        if (j < n8) {
            float g[8];
            load8(gamma + 8 * j, g);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                v[i][e] = v[i][e] * r * g[e];
                am = fmaxf(am, fabsf(v[i][e]));
            }
        }
    }
    am = block_max(am, red);
    const float sa = __fdiv_rn(fmaxf(am, 1e-12f), 448.0f), rsa = __frcp_rn(sa);
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int j = threadIdx.x + i * kRowThreads;
        if (j < n8) *reinterpret_cast<uint2*>(out + (size_t)p * hidden + 8 * j) = quant8(v[i], sa, rsa);
    }
    if (threadIdx.x == 0) scale[p] = sa;
}

template <typename T, int NV>
__global__ void __launch_bounds__(kRowThreads) quant_rows_reg_kernel(const T* X, uint8_t* out, float* scale, int n) {
    __shared__ float red[32];
    const int p = blockIdx.x, n8 = n / 8;
    const T* x = X + (size_t)p * n;
    float v[NV][8];
    float am = 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int j = threadIdx.x + i * kRowThreads;
        if (j < n8) {
            load8(x + 8 * j, v[i]);
#pragma unroll
            for (int e = 0; e < 8; ++e) am = fmaxf(am, fabsf(v[i][e]));
        }
    }
    am = block_max(am, red);
    const float sa = __fdiv_rn(fmaxf(am, 1e-12f), 448.0f), rsa = __frcp_rn(sa);
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int j = threadIdx.x + i * kRowThreads;
        if (j < n8) *reinterpret_cast<uint2*>(out + (size_t)p * n + 8 * j) = quant8(v[i], sa, rsa);
    }
    if (threadIdx.x == 0) scale[p] = sa;
}

// ---- causal GQA attention on the tensor cores --------------------------------
// Rows [row0, row0 + 16) of the prompt against the G query heads of kv head g:
// warp w takes query head g*G + w for the 16 rows.  Per 64-key tile,
//   S = Q K^T      mma.sync m16n8k16, bf16 operands, fp32 accumulation
//                  (Q rounded to bf16 once, or carried as two bf16 terms for
//                  FP8 contexts; K straight from the bf16 cache)
//   online softmax in fp32 on the accumulator fragments (row max and the
//                  rescale of O); P rounded to bf16 (or two bf16 terms) and
//                  reused in registers as the A operand of
//   O += P V       mma.sync, V read transposed from shared memory.
// Row p attends positions [0, pos0 + p].  K/V tiles are double-buffered in
// shared memory (cp.async); the row sums are taken over the weights O is
// built from (the rounded P, or the fp32 P when split).
constexpr int kMmaRows = 16;
constexpr int kMmaKeys = 64;
constexpr int kMmaPad = kHeadDim + 8;  // bf16 per shared row: 272 B, the 8 rows of an ldmatrix on distinct banks
constexpr float kLog2e = 1.4426950408889634f;

template <int G>
constexpr int attention_mma_smem() {
    return 2 * 2 * kMmaKeys * kMmaPad * (int)sizeof(__nv_bfloat16);
}

__device__ __forceinline__ float bf16_round(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ void mma_bf16_16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldmatrix_x4(uint32_t* r, const void* smem_row) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(smem_row)));
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t* r, const void* smem_row) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(smem_row)));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// SPLIT (FP8 contexts): Q and the softmax weights P are each carried as two
// bf16 terms, hi = bf16(x) and lo = bf16(x - hi), so Q K^T and P V keep about
// 16 significant bits of the fp32 values (the K/V cache is bf16 exactly); the
// row sums are taken over the fp32 weights.  Without SPLIT, Q and P are
// rounded to bf16 once (the W16A16 prefill of BF16 contexts).
template <int G, bool SPLIT>
__global__ void __launch_bounds__(32 * G) attention_mma_kernel(const float* Q, const __nv_bfloat16* kc,
                                                               const __nv_bfloat16* vc, __nv_bfloat16* out,
                                                               float* out_f32, int pos0, int P, int n_q,
                                                               int max_pos) {
    extern __shared__ __align__(16) __nv_bfloat16 kvs[];  // [2 buffers][K, V][64 keys][kMmaPad]
    const int rb = gridDim.x - 1 - blockIdx.x;             // the longest rows first
    const int g = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gi = lane >> 2, ti = lane & 3;                // fragment row group, thread in group
    const int row0 = rb * kMmaRows;
    const int nrows = min(kMmaRows, P - row0);
    const int key_end = pos0 + row0 + nrows;                // keys [0, key_end) are read
    const int ntiles = (key_end + kMmaKeys - 1) / kMmaKeys;
    const size_t cache0 = (size_t)g * max_pos * kHeadDim;
    const int h = g * G + warp;

    auto load_tile = [&](int t, int buf) {
        __nv_bfloat16* Ks = kvs + (size_t)buf * 2 * kMmaKeys * kMmaPad;
        __nv_bfloat16* Vs = Ks + kMmaKeys * kMmaPad;
        for (int i = threadIdx.x; i < kMmaKeys * (kHeadDim / 8); i += 32 * G) {
            const int kr = i / (kHeadDim / 8), c8 = i % (kHeadDim / 8);
            const int key = t * kMmaKeys + kr;
            __nv_bfloat16* kd = Ks + kr * kMmaPad + 8 * c8;
            __nv_bfloat16* vd = Vs + kr * kMmaPad + 8 * c8;
            if (key < key_end) {
                cp_async16(kd, kc + cache0 + (size_t)key * kHeadDim + 8 * c8);
                cp_async16(vd, vc + cache0 + (size_t)key * kHeadDim + 8 * c8);
            } else {  // past the last key read: zeros (masked scores, zero weights)
                *reinterpret_cast<uint4*>(kd) = make_uint4(0u, 0u, 0u, 0u);
                *reinterpret_cast<uint4*>(vd) = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        cp_async_commit();
    };
    load_tile(0, 0);

    // this warp's Q (16 rows x 128 dims) as A fragments, one per 16-dim k-step
    // (SPLIT: qa = bf16(Q), ql = bf16(Q - qa))
    uint32_t qa[kHeadDim / 16][4];
    uint32_t ql[SPLIT ? kHeadDim / 16 : 1][4];
    {
        const bool v0 = gi < nrows, v1 = gi + 8 < nrows;
        const float* q0 = Q + ((size_t)(row0 + gi) * n_q + h) * kHeadDim;
        const float* q1 = Q + ((size_t)(row0 + gi + 8) * n_q + h) * kHeadDim;
#pragma unroll
        for (int ks = 0; ks < kHeadDim / 16; ++ks) {
            const int d = ks * 16 + 2 * ti;
            const float2 z = make_float2(0.f, 0.f);
            const float2 a00 = v0 ? *reinterpret_cast<const float2*>(q0 + d) : z;
            const float2 a01 = v0 ? *reinterpret_cast<const float2*>(q0 + d + 8) : z;
            const float2 a10 = v1 ? *reinterpret_cast<const float2*>(q1 + d) : z;
            const float2 a11 = v1 ? *reinterpret_cast<const float2*>(q1 + d + 8) : z;
            qa[ks][0] = pack_bf16x2(a00.x, a00.y);
            qa[ks][1] = pack_bf16x2(a10.x, a10.y);
            qa[ks][2] = pack_bf16x2(a01.x, a01.y);
            qa[ks][3] = pack_bf16x2(a11.x, a11.y);
            if constexpr (SPLIT) {
                ql[ks][0] = pack_bf16x2(a00.x - bf16_round(a00.x), a00.y - bf16_round(a00.y));
                ql[ks][1] = pack_bf16x2(a10.x - bf16_round(a10.x), a10.y - bf16_round(a10.y));
                ql[ks][2] = pack_bf16x2(a01.x - bf16_round(a01.x), a01.y - bf16_round(a01.y));
                ql[ks][3] = pack_bf16x2(a11.x - bf16_round(a11.x), a11.y - bf16_round(a11.y));
            }
        }
    }
    float o[kHeadDim / 8][4];
#pragma unroll
    for (int d = 0; d < kHeadDim / 8; ++d) o[d][0] = o[d][1] = o[d][2] = o[d][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // rows gi and gi + 8 (lane partial sums)
    const int qpos0 = pos0 + row0 + gi, qpos1 = qpos0 + 8;
    const int mat = lane >> 3, mrow = lane & 7;  // ldmatrix: this lane addresses row mrow of matrix mat

    for (int t = 0; t < ntiles; ++t) {
        if (t + 1 < ntiles) {
            load_tile(t + 1, (t + 1) & 1);
            cp_async_wait_group<1>();
        } else {
            cp_async_wait_group<0>();
        }
        __syncthreads();
        const __nv_bfloat16* Ks = kvs + (size_t)(t & 1) * 2 * kMmaKeys * kMmaPad;
        const __nv_bfloat16* Vs = Ks + kMmaKeys * kMmaPad;

        // S = Q K^T over the tile: 8 n-tiles of 8 keys
        float s[kMmaKeys / 8][4];
#pragma unroll
        for (int j = 0; j < kMmaKeys / 8; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
        for (int np = 0; np < kMmaKeys / 16; ++np) {
#pragma unroll
            for (int ks = 0; ks < kHeadDim / 16; ++ks) {
                uint32_t b[4];  // keys np*16 + {0..7 | 8..15} x dims ks*16 + {0..7 | 8..15}
                ldmatrix_x4(b, Ks + (np * 16 + (mat >> 1) * 8 + mrow) * kMmaPad + ks * 16 + (mat & 1) * 8);
                mma_bf16_16816(s[2 * np], qa[ks], b[0], b[1]);
                mma_bf16_16816(s[2 * np + 1], qa[ks], b[2], b[3]);
                if constexpr (SPLIT) {
                    mma_bf16_16816(s[2 * np], ql[ks], b[0], b[1]);
                    mma_bf16_16816(s[2 * np + 1], ql[ks], b[2], b[3]);
                }
            }
        }
        // causal mask: key > position of the row
        const int kbase = t * kMmaKeys;
        if (kbase + kMmaKeys - 1 > qpos0) {
#pragma unroll
            for (int j = 0; j < kMmaKeys / 8; ++j) {
                const int key = kbase + j * 8 + 2 * ti;
                if (key > qpos0) s[j][0] = -INFINITY;
                if (key + 1 > qpos0) s[j][1] = -INFINITY;
                if (key > qpos1) s[j][2] = -INFINITY;
                if (key + 1 > qpos1) s[j][3] = -INFINITY;
            }
        }
        // online softmax: the four lanes of a row group share rows gi and gi + 8
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int j = 0; j < kMmaKeys / 8; ++j) {
            mx0 = fmaxf(mx0, fmaxf(s[j][0], s[j][1]));
            mx1 = fmaxf(mx1, fmaxf(s[j][2], s[j][3]));
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        // a row with no key yet (only rows past the prompt) keeps zero weights
        const float e0 = mn0 == -INFINITY ? 0.f : mn0 * kLog2e;
        const float e1 = mn1 == -INFINITY ? 0.f : mn1 * kLog2e;
        const float c0 = exp2f(m0 * kLog2e - e0), c1 = exp2f(m1 * kLog2e - e1);
        m0 = mn0;
        m1 = mn1;
        l0 *= c0;
        l1 *= c1;
#pragma unroll
        for (int d = 0; d < kHeadDim / 8; ++d) {
            o[d][0] *= c0;
            o[d][1] *= c0;
            o[d][2] *= c1;
            o[d][3] *= c1;
        }
        uint32_t pa[kMmaKeys / 16][4];  // P as A fragments, one per 16-key k-step
        uint32_t pl[SPLIT ? kMmaKeys / 16 : 1][4];  // SPLIT: bf16(P - pa)
#pragma unroll
        for (int j = 0; j < kMmaKeys / 8; ++j) {
            const float q0 = exp2f(s[j][0] * kLog2e - e0), q1 = exp2f(s[j][1] * kLog2e - e0);
            const float q2 = exp2f(s[j][2] * kLog2e - e1), q3 = exp2f(s[j][3] * kLog2e - e1);
            const __nv_bfloat162 p01 = __floats2bfloat162_rn(q0, q1);
            const __nv_bfloat162 p23 = __floats2bfloat162_rn(q2, q3);
            if constexpr (SPLIT) {
                l0 += q0 + q1;
                l1 += q2 + q3;
                const __nv_bfloat162 r01 =
                    __floats2bfloat162_rn(q0 - __low2float(p01), q1 - __high2float(p01));
                const __nv_bfloat162 r23 =
                    __floats2bfloat162_rn(q2 - __low2float(p23), q3 - __high2float(p23));
                pl[j >> 1][(j & 1) * 2] = *reinterpret_cast<const uint32_t*>(&r01);
                pl[j >> 1][(j & 1) * 2 + 1] = *reinterpret_cast<const uint32_t*>(&r23);
            } else {
                l0 += __low2float(p01) + __high2float(p01);
                l1 += __low2float(p23) + __high2float(p23);
            }
            pa[j >> 1][(j & 1) * 2] = *reinterpret_cast<const uint32_t*>(&p01);
            pa[j >> 1][(j & 1) * 2 + 1] = *reinterpret_cast<const uint32_t*>(&p23);
        }
        // O += P V: 16 n-tiles of 8 dims, 4 k-steps of 16 keys
#pragma unroll
        for (int dp = 0; dp < kHeadDim / 16; ++dp) {
#pragma unroll
            for (int kk = 0; kk < kMmaKeys / 16; ++kk) {
                uint32_t b[4];  // keys kk*16 + {0..7 | 8..15} x dims dp*16 + {0..7 | 8..15}, transposed
                ldmatrix_x4_trans(b, Vs + (kk * 16 + (mat & 1) * 8 + mrow) * kMmaPad + dp * 16 + (mat >> 1) * 8);
                mma_bf16_16816(o[2 * dp], pa[kk], b[0], b[1]);
                mma_bf16_16816(o[2 * dp + 1], pa[kk], b[2], b[3]);
                if constexpr (SPLIT) {
                    mma_bf16_16816(o[2 * dp], pl[kk], b[0], b[1]);
                    mma_bf16_16816(o[2 * dp + 1], pl[kk], b[2], b[3]);
                }
            }
        }
        __syncthreads();  // this buffer is refilled two tiles on
    }
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    const float inv0 = 1.0f / l0, inv1 = 1.0f / l1;
#pragma unroll
    for (int d = 0; d < kHeadDim / 8; ++d) {
        const int col = d * 8 + 2 * ti;
        const size_t i0 = ((size_t)(row0 + gi) * n_q + h) * kHeadDim + col;
        const size_t i1 = ((size_t)(row0 + gi + 8) * n_q + h) * kHeadDim + col;
        if (out_f32) {  // FP8 contexts: fp32, quantised per row next (as the decode step does)
            if (gi < nrows) *reinterpret_cast<float2*>(out_f32 + i0) = make_float2(o[d][0] * inv0, o[d][1] * inv0);
            if (gi + 8 < nrows) *reinterpret_cast<float2*>(out_f32 + i1) = make_float2(o[d][2] * inv1, o[d][3] * inv1);
        } else {
            if (gi < nrows)
                *reinterpret_cast<__nv_bfloat162*>(out + i0) = __floats2bfloat162_rn(o[d][0] * inv0, o[d][1] * inv0);
            if (gi + 8 < nrows)
                *reinterpret_cast<__nv_bfloat162*>(out + i1) = __floats2bfloat162_rn(o[d][2] * inv1, o[d][3] * inv1);
        }
    }
}

template <int G, bool SPLIT>
cudaError_t launch_attention_rows_split(const float* Q, const __nv_bfloat16* kc, const __nv_bfloat16* vc,
                                        __nv_bfloat16* out, float* out_f32, int pos0, int P, int n_q, int n_kv,
                                        int max_pos, cudaStream_t s) {
    constexpr int smem = attention_mma_smem<G>();
    static bool attr = false;  // set once, on the first (uncaptured) run of a chunk shape
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(attention_mma_kernel<G, SPLIT>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    const dim3 grid((P + kMmaRows - 1) / kMmaRows, n_kv);
    attention_mma_kernel<G, SPLIT><<<grid, 32 * G, smem, s>>>(Q, kc, vc, out, out_f32, pos0, P, n_q, max_pos);
    return cudaGetLastError();
}

// FP8 contexts (fp32 output, quantised per row next) take the split-bf16
// operands; BF16 contexts the single bf16 rounding of their W16A16 prefill.
template <int G>
cudaError_t launch_attention_rows_t(const float* Q, const __nv_bfloat16* kc, const __nv_bfloat16* vc,
                                    __nv_bfloat16* out, float* out_f32, int pos0, int P, int n_q, int n_kv,
                                    int max_pos, cudaStream_t s) {
    return out_f32 ? launch_attention_rows_split<G, true>(Q, kc, vc, out, out_f32, pos0, P, n_q, n_kv, max_pos, s)
                   : launch_attention_rows_split<G, false>(Q, kc, vc, out, out_f32, pos0, P, n_q, n_kv, max_pos, s);
}

}  // namespace

cudaError_t launch_prefill_embed(const __nv_bfloat16* E, const int* codes, float* H, int P, int n_cb, int V,
                                 int hidden, cudaStream_t s) {
    embed_rows_kernel<<<P, kRowThreads, 0, s>>>(E, codes, H, n_cb, V, hidden);
    return cudaGetLastError();
}

// the smallest register row that holds `hidden` (a multiple of 4 floats per lane)
cudaError_t launch_rows_warp(const float* H, const __nv_bfloat16* gamma, __nv_bfloat16* out, int P, int hidden,
                             float eps, cudaStream_t s) {
    const dim3 grid((P + kRowWarps - 1) / kRowWarps);
    const int nv = (hidden / 4 + 31) / 32;
#define TTS_ROWS_NV(NV)                                                                                            \
    if (nv <= NV) {                                                                                                \
        rmsnorm_rows_warp_kernel<NV><<<grid, kRowThreads, 0, s>>>(H, gamma, out, P, hidden, eps);                 \
        return cudaGetLastError();                                                                                 \
    }
    TTS_ROWS_NV(4)
    TTS_ROWS_NV(8)
    TTS_ROWS_NV(16)
    TTS_ROWS_NV(20)
    TTS_ROWS_NV(24)
    TTS_ROWS_NV(32)
#undef TTS_ROWS_NV
    return cudaErrorInvalidValue;
}

cudaError_t launch_prefill_rmsnorm(const float* H, const __nv_bfloat16* gamma, __nv_bfloat16* out, int P,
                                   int hidden, float eps, cudaStream_t s) {
    if (hidden % 4 == 0 && hidden <= 128 * kRowVec)
        return launch_rows_warp(H, gamma, out, P, hidden, eps, s);
    else
        rmsnorm_rows_kernel<<<P, kRowThreads, 0, s>>>(H, gamma, out, hidden, eps);
    return cudaGetLastError();
}

cudaError_t launch_prefill_rmsnorm_fp8(const float* H, const __nv_bfloat16* gamma, uint8_t* out, float* scale, int P,
                                       int hidden, float eps, cudaStream_t s) {
    // a CTA per row: the IEEE divisions of the quantisation spread over all its threads
    const int nv = hidden % 8 == 0 ? (hidden / 8 + kRowThreads - 1) / kRowThreads : 0;
#define TTS_RQ_NV(NV)                                                                                        \
    if (nv >= 1 && nv <= NV) {                                                                               \
        rmsnorm_quant_rows_reg_kernel<NV><<<P, kRowThreads, 0, s>>>(H, gamma, out, scale, hidden, eps);      \
        return cudaGetLastError();                                                                           \
    }
    TTS_RQ_NV(2)
    TTS_RQ_NV(4)
    TTS_RQ_NV(6)
#undef TTS_RQ_NV
    rmsnorm_quant_rows_kernel<<<P, kRowThreads, 0, s>>>(H, gamma, out, scale, hidden, eps);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_quant_rows_t(const T* X, uint8_t* out, float* scale, int P, int n, cudaStream_t s) {
    const int nv = n % 8 == 0 ? (n / 8 + kRowThreads - 1) / kRowThreads : 0;
#define TTS_Q_NV(NV)                                                                 \
    if (nv >= 1 && nv <= NV) {                                                       \
        quant_rows_reg_kernel<T, NV><<<P, kRowThreads, 0, s>>>(X, out, scale, n);    \
        return cudaGetLastError();                                                   \
    }
    TTS_Q_NV(2)
    TTS_Q_NV(4)
    TTS_Q_NV(6)
#undef TTS_Q_NV
    quant_rows_kernel<T><<<P, kRowThreads, 0, s>>>(X, out, scale, n);
    return cudaGetLastError();
}
cudaError_t launch_prefill_quant_rows(const __nv_bfloat16* X, uint8_t* out, float* scale, int P, int n,
                                      cudaStream_t s) {
    return launch_quant_rows_t(X, out, scale, P, n, s);
}
cudaError_t launch_prefill_quant_rows_f32(const float* X, uint8_t* out, float* scale, int P, int n, cudaStream_t s) {
    return launch_quant_rows_t(X, out, scale, P, n, s);
}

cudaError_t launch_prefill_qk_rope_kv(const float* QKV, const __nv_bfloat16* qn, const __nv_bfloat16* kn,
                                      const float2* rope, float* Q, __nv_bfloat16* kc, __nv_bfloat16* vc, int pos0,
                                      int P, int n_q, int n_kv, int max_pos, float eps, cudaStream_t s) {
    qk_rope_kv_rows_kernel<<<P, kRowThreads, 0, s>>>(QKV, qn, kn, rope, Q, kc, vc, pos0, n_q, n_kv, max_pos, eps);
    return cudaGetLastError();
}

// The G query heads of a kv head share one CTA's K/V tiles: 64 (row, head) pairs.
cudaError_t launch_prefill_attention(const float* Q, const __nv_bfloat16* kc, const __nv_bfloat16* vc,
                                     __nv_bfloat16* out, int pos0, int P, int n_q, int n_kv, int max_pos,
                                     cudaStream_t s, float* out_f32) {
    const int G = n_q / n_kv;
    if (G == 4) return launch_attention_rows_t<4>(Q, kc, vc, out, out_f32, pos0, P, n_q, n_kv, max_pos, s);
    if (G == 8) return launch_attention_rows_t<8>(Q, kc, vc, out, out_f32, pos0, P, n_q, n_kv, max_pos, s);
    if (G == 2) return launch_attention_rows_t<2>(Q, kc, vc, out, out_f32, pos0, P, n_q, n_kv, max_pos, s);
    if (G == 1) return launch_attention_rows_t<1>(Q, kc, vc, out, out_f32, pos0, P, n_q, n_kv, max_pos, s);
    return cudaErrorInvalidValue;
}

}  // namespace tts

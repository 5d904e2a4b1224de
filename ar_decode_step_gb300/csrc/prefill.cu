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
//   attention_rows    causal GQA: row p attends positions [0, pos0 + p];
//                     output rounded to bf16 (the O-proj GEMM's A operand)
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
            dst[0] = __float2bfloat16_rn(v.x);
            dst[1] = __float2bfloat16_rn(v.y);
            dst[2] = __float2bfloat16_rn(v.z);
            dst[3] = __float2bfloat16_rn(v.w);
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
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) dst[jj] = __float2bfloat16_rn(o[jj]);
        }
    }
}

// Causal GQA attention over the cache for rows [rb*16, rb*16+16) of the
// prompt and the G query heads of kv head g: G*16 (row, head) pairs per CTA,
// 2G per warp (one head, consecutive rows).  Keys go through shared memory 64
// at a time (fp32, K rows padded against bank conflicts).  Register tiling:
// a lane scores its two keys against every pair of its warp (each K value
// loaded once for all pairs, the queries broadcast); the probabilities go
// through a per-warp shared tile, and for the output each lane keeps 4 dims
// of every pair (each V value loaded once for all pairs).  Online softmax in
// fp32.
constexpr int kAttRows = 16;
constexpr int kAttKeys = 64;
constexpr int kKPad = kHeadDim + 4;

template <int G>
constexpr int attention_rows_smem() {
    return (G * kAttRows * kHeadDim + kAttKeys * kKPad + kAttKeys * kHeadDim + G * kAttRows * kAttKeys) *
           (int)sizeof(float);
}

template <int G>
__global__ void __launch_bounds__(kRowThreads) attention_rows_kernel(const float* Q, const __nv_bfloat16* kc,
                                                                     const __nv_bfloat16* vc,
                                                                     __nv_bfloat16* out, int pos0, int P, int n_q,
                                                                     int max_pos) {
    extern __shared__ __align__(16) float sm[];
    constexpr int kPairs = G * kAttRows;
    constexpr int kPerWarp = kPairs / (kRowThreads / 32);
    float* Qs = sm;                                    // [pairs][128]
    float* Ks = Qs + kPairs * kHeadDim;                // [64][132]
    float* Vs = Ks + kAttKeys * kKPad;                 // [64][128]
    float* Ps = Vs + kAttKeys * kHeadDim;              // [pairs][64] probabilities
    const int rb = blockIdx.x, g = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row0 = rb * kAttRows;
    const int nrows = min(kAttRows, P - row0);
    const size_t cache0 = (size_t)g * max_pos * kHeadDim;

    // pair = head_local * 16 + row_local; warp w owns pairs [w * kPerWarp, (w+1) * kPerWarp)
    for (int i = threadIdx.x; i < kPairs * kHeadDim / 4; i += kRowThreads) {
        const int pair = i / (kHeadDim / 4), d4 = i % (kHeadDim / 4);
        const int hl = pair / kAttRows, rl = pair % kAttRows;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (rl < nrows) v = reinterpret_cast<const float4*>(Q + ((size_t)(row0 + rl) * n_q + g * G + hl) * kHeadDim)[d4];
        reinterpret_cast<float4*>(Qs)[i] = v;
    }
    const int pair0 = warp * kPerWarp;
    int qpos[kPerWarp];
    int qpos_max = -1;
#pragma unroll
    for (int i = 0; i < kPerWarp; ++i) {
        const int rl = (pair0 + i) % kAttRows;
        qpos[i] = rl < nrows ? pos0 + row0 + rl : -1;  // -1: no such row (never attends)
        qpos_max = max(qpos_max, qpos[i]);
    }
    float m[kPerWarp], l[kPerWarp], o[kPerWarp][4];
#pragma unroll
    for (int i = 0; i < kPerWarp; ++i) {
        m[i] = -INFINITY;
        l[i] = 0.f;
        o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    }
    float* pw = Ps + pair0 * kAttKeys;
    const int kmax = pos0 + row0 + nrows - 1;  // last key any row of this block sees
    for (int k0 = 0; k0 <= kmax; k0 += kAttKeys) {
        __syncthreads();  // previous tile consumed (and Qs written, first time)
        for (int i = threadIdx.x; i < kAttKeys * kHeadDim / 4; i += kRowThreads) {
            const int kr = i / (kHeadDim / 4), d4 = i % (kHeadDim / 4);
            const int key = k0 + kr;
            float4 kv = make_float4(0.f, 0.f, 0.f, 0.f), vv = kv;
            if (key <= kmax) {
                const uint2 kb = *reinterpret_cast<const uint2*>(kc + cache0 + (size_t)key * kHeadDim + 4 * d4);
                const uint2 vb = *reinterpret_cast<const uint2*>(vc + cache0 + (size_t)key * kHeadDim + 4 * d4);
                kv = make_float4(bf16lo(kb.x), bf16hi(kb.x), bf16lo(kb.y), bf16hi(kb.y));
                vv = make_float4(bf16lo(vb.x), bf16hi(vb.x), bf16lo(vb.y), bf16hi(vb.y));
            }
            *reinterpret_cast<float4*>(Ks + kr * kKPad + 4 * d4) = kv;
            *reinterpret_cast<float4*>(Vs + kr * kHeadDim + 4 * d4) = vv;
        }
        __syncthreads();
        if (k0 > qpos_max) continue;  // warp-uniform: no row of this warp reaches the tile

        // scores of keys k0 + lane and k0 + lane + 32 against every pair of the warp
        float s0[kPerWarp], s1[kPerWarp];
#pragma unroll
        for (int i = 0; i < kPerWarp; ++i) s0[i] = s1[i] = 0.f;
        const float* ka = Ks + lane * kKPad;
        const float* kb = Ks + (lane + 32) * kKPad;
        const float* qw = Qs + pair0 * kHeadDim;
#pragma unroll 2
        for (int d = 0; d < kHeadDim; d += 4) {
            const float4 a = *reinterpret_cast<const float4*>(ka + d);
            const float4 b = *reinterpret_cast<const float4*>(kb + d);
#pragma unroll
            for (int i = 0; i < kPerWarp; ++i) {
                const float4 qq = *reinterpret_cast<const float4*>(qw + i * kHeadDim + d);
                s0[i] = fmaf(qq.x, a.x, fmaf(qq.y, a.y, fmaf(qq.z, a.z, fmaf(qq.w, a.w, s0[i]))));
                s1[i] = fmaf(qq.x, b.x, fmaf(qq.y, b.y, fmaf(qq.z, b.z, fmaf(qq.w, b.w, s1[i]))));
            }
        }
        // online softmax per pair; probabilities to the warp's shared tile
#pragma unroll
        for (int i = 0; i < kPerWarp; ++i) {
            if (k0 + lane > qpos[i]) s0[i] = -INFINITY;
            if (k0 + lane + 32 > qpos[i]) s1[i] = -INFINITY;
            const float mx = warp_max(fmaxf(s0[i], s1[i]));
            const float mn = fmaxf(m[i], mx);
            // a pair with no key in this tile (mn = -inf) keeps its state
            const float corr = mn == -INFINITY ? 1.f : __expf(m[i] - mn);
            const float p0 = mn == -INFINITY ? 0.f : __expf(s0[i] - mn);
            const float p1 = mn == -INFINITY ? 0.f : __expf(s1[i] - mn);
            l[i] = l[i] * corr + warp_sum(p0 + p1);
            m[i] = mn;
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) o[i][jj] *= corr;
            pw[i * kAttKeys + lane] = p0;
            pw[i * kAttKeys + lane + 32] = p1;
        }
        __syncwarp();
        const int nk = min(kAttKeys, qpos_max - k0 + 1);
        for (int kk = 0; kk < nk; ++kk) {
            const float4 vv = *reinterpret_cast<const float4*>(Vs + kk * kHeadDim + 4 * lane);
#pragma unroll
            for (int i = 0; i < kPerWarp; ++i) {
                const float pk = pw[i * kAttKeys + kk];
                o[i][0] = fmaf(pk, vv.x, o[i][0]);
                o[i][1] = fmaf(pk, vv.y, o[i][1]);
                o[i][2] = fmaf(pk, vv.z, o[i][2]);
                o[i][3] = fmaf(pk, vv.w, o[i][3]);
            }
        }
        __syncwarp();
    }
#pragma unroll
    for (int i = 0; i < kPerWarp; ++i) {
        const int pair = pair0 + i;
        const int hl = pair / kAttRows, rl = pair % kAttRows;
        if (rl >= nrows) continue;
        const float inv = 1.0f / l[i];
        __nv_bfloat16* dst = out + ((size_t)(row0 + rl) * n_q + g * G + hl) * kHeadDim + 4 * lane;
        dst[0] = __float2bfloat16_rn(o[i][0] * inv);
        dst[1] = __float2bfloat16_rn(o[i][1] * inv);
        dst[2] = __float2bfloat16_rn(o[i][2] * inv);
        dst[3] = __float2bfloat16_rn(o[i][3] * inv);
    }
}

template <int G>
cudaError_t launch_attention_rows_t(const float* Q, const __nv_bfloat16* kc, const __nv_bfloat16* vc,
                                    __nv_bfloat16* out, int pos0, int P, int n_q, int n_kv, int max_pos,
                                    cudaStream_t s) {
    constexpr int smem = attention_rows_smem<G>();
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(attention_rows_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             smem);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    const dim3 grid((P + kAttRows - 1) / kAttRows, n_kv);
    attention_rows_kernel<G><<<grid, kRowThreads, smem, s>>>(Q, kc, vc, out, pos0, P, n_q, max_pos);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_embed(const __nv_bfloat16* E, const int* codes, float* H, int P, int n_cb, int V,
                                 int hidden, cudaStream_t s) {
    embed_rows_kernel<<<P, kRowThreads, 0, s>>>(E, codes, H, n_cb, V, hidden);
    return cudaGetLastError();
}

cudaError_t launch_prefill_rmsnorm(const float* H, const __nv_bfloat16* gamma, __nv_bfloat16* out, int P,
                                   int hidden, float eps, cudaStream_t s) {
    rmsnorm_rows_kernel<<<P, kRowThreads, 0, s>>>(H, gamma, out, hidden, eps);
    return cudaGetLastError();
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
                                     cudaStream_t s) {
    const int G = n_q / n_kv;
    if (G == 4) return launch_attention_rows_t<4>(Q, kc, vc, out, pos0, P, n_q, n_kv, max_pos, s);
    if (G == 8) return launch_attention_rows_t<8>(Q, kc, vc, out, pos0, P, n_q, n_kv, max_pos, s);
    if (G == 2) return launch_attention_rows_t<2>(Q, kc, vc, out, pos0, P, n_q, n_kv, max_pos, s);
    if (G == 1) return launch_attention_rows_t<1>(Q, kc, vc, out, pos0, P, n_q, n_kv, max_pos, s);
    return cudaErrorInvalidValue;
}

}  // namespace tts

// BF16 GEMM on the 5th-generation tensor cores (sm_103a): C = A . B^T with
// A [M][K] activations and B [N][K] weights, both K-major bf16, fp32
// accumulation in tensor memory.  The batched prefill's projections
// ("Higgs Audio v3 TTS-4B on FlashRT", Performance: "BF16 W16A16", prompt
// prefill; section 7: the prompt runs as one M = P pass, weights read once)
// are dense contractions of P rows against every weight matrix, so they run
// here rather than on the M = 1 weight-streaming path.
//
// One CTA per 128 x BN output tile (BN = 64 or 128; 256 for the fused gate/up tile):
//   warp 0 (one thread)  TMA producer: 128 x 64 A box and BN x 64 B box(es)
//                        per k-block into a ring of 4-8 stages (128-byte swizzle),
//                        completion counted on the stage's "full" mbarrier;
//   warp 1 (one thread)  MMA issuer: four tcgen05.mma (K = 16 each) per
//                        k-block into the TMEM accumulator, then
//                        tcgen05.commit frees the stage ("empty") and, after
//                        the last block, signals "done";
//   warp 2               allocates / frees the TMEM columns;
//   warps 0-3            epilogue: tcgen05.ld of their 32 accumulator lanes
//                        (one output row per thread), then store fp32, add
//                        into fp32 (residual, split-K), or SwiGLU -> bf16.
// Every wait is bounded; on expiry the kernel records an error, lets its
// copies and MMAs finish and frees its tensor memory before returning.
#include <cuda.h>

#include <cstdio>

#include "kernels.h"
#include "tts_decode.h"

namespace tts {

namespace {

constexpr int kBM = 128;          // rows of A per tile (MMA M)
constexpr int kBK = 64;           // k-block: 64 bf16 = one 128-byte swizzle row
// ring depth: as many stages as fit in shared memory (at most 8), so narrow
// tiles keep as many bytes in flight from L2 as wide ones
constexpr int kSmemRing = 225 * 1024;
template <int MMA_N>
constexpr int gemm_stages() {
    return kSmemRing / (int)(kBM * kBK * 2 + MMA_N * kBK * 2) < 8 ? kSmemRing / (int)(kBM * kBK * 2 + MMA_N * kBK * 2)
                                                                   : 8;
}
constexpr int kGemmThreads = 128;
constexpr uint32_t kATileBytes = kBM * kBK * 2;  // 16 KB

// ---- tcgen05 / TMA wrappers ---------------------------------------------------
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem desc] . B[smem desc]^T, kind::f16 (bf16 inputs, fp32 D)
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// arrive on `bar` once every tcgen05 operation this thread issued so far is complete
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}
// 16 consecutive fp32 columns of this warp's 32 accumulator lanes (one lane per thread)
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor of a K-major tile stored the way a TMA
// 128-byte-swizzled box lands: rows of 128 bytes, 8-row (1024-byte) swizzle
// atoms stacked along M/N.  Fields: start address >> 4 (bits 0-13), leading
// byte offset >> 4 (16-29; unused for swizzled K-major, 1), stride byte
// offset >> 4 (32-45: 1024 bytes between 8-row groups), descriptor version 1
// (46-47), base offset 0 (49-51, 1024-byte aligned tiles), layout type
// 128-byte swizzle = 2 (61-63).
__device__ __forceinline__ uint64_t smem_desc_sw128(const void* tile) {
    const uint64_t addr = smem_u32(tile);
    return ((addr >> 4) & 0x3fffull) | (1ull << 16) | ((1024ull >> 4) << 32) | (1ull << 46) | (2ull << 61);
}
// Instruction descriptor, kind::f16: fp32 D (bits 4-5 = 1), bf16 A and B
// (7-9 = 1, 10-12 = 1), both K-major (15, 16 = 0), N >> 3 (17-22), M >> 4 (24-28).
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// kind::f8f6f4 with E4M3 A and B (type code 0), fp32 D; same field layout
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void tc_mma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ float round_bf16f(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

// F8: E4M3 operands; a k-block is then 128 elements (still one 128-byte
// swizzle row), an MMA takes K = 32 (still 32 bytes), and every accumulator
// is scaled by its row's and column's scales and rounded to bf16 before the
// epilogue's operation.
template <int EPI, int MMA_N, bool F8>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_bf16_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const GemmParams p) {
    constexpr int kBKE = F8 ? 2 * kBK : kBK;  // elements per k-block
    extern __shared__ unsigned char smem_raw[];
    constexpr int kStages = gemm_stages<MMA_N>();
    __shared__ __align__(8) uint64_t full[kStages], empty[kStages], done;
    __shared__ uint32_t s_tmem;
    __shared__ int s_fail;
    __shared__ int s_never;  // abort flag of the epilogue wait: only the time limit ends it
    constexpr uint32_t kBTileBytes = MMA_N * kBK * 2;
    constexpr uint32_t kStageBytes = kATileBytes + kBTileBytes;
    // fp32 accumulator columns: the allocation is a power of two >= 32
    constexpr uint32_t kTmemCols = MMA_N <= 32 ? 32 : MMA_N <= 64 ? 64 : MMA_N <= 128 ? 128 : 256;
    // stage tiles 1024-byte aligned (swizzle atoms)
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // the M tiles of one N tile are adjacent in the grid: they run together
    // and share the weight tile through L2 (one DRAM read per weight)
    const int m0 = blockIdx.x * kBM;
    const int nt = EPI == kGemmSwiglu ? MMA_N / 2 : MMA_N;  // output columns of this tile
    const int n0 = blockIdx.y * nt;
    const int kb0 = blockIdx.z * p.kb_per_split;
    const int kb1 = min(p.K / kBKE, kb0 + p.kb_per_split);
    const int nkb = kb1 - kb0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(&done, 1);
        fence_mbar_init();
        s_fail = 0;
        s_never = 0;
    }
    if (warp == 2) tmem_alloc(&s_tmem, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_d = s_tmem;

    if (warp == 0) {
      if (lane == 0) {
        // TMA producer
        for (int i = 0; i < nkb; ++i) {
            const int s = i % kStages;
            if (!mbar_wait(&empty[s], ((i / kStages) & 1) ^ 1)) {
                s_fail = 1;
                break;
            }
            unsigned char* st = smem + (size_t)s * kStageBytes;
            mbar_arrive_expect_tx(&full[s], kStageBytes);
            const int kx = (kb0 + i) * kBKE;
            tma_load_2d(st, &tmA, kx, m0, &full[s]);
            if constexpr (EPI == kGemmSwiglu) {
                tma_load_2d(st + kATileBytes, &tmB, kx, n0, &full[s]);                     // gate rows
                tma_load_2d(st + kATileBytes + kBTileBytes / 2, &tmB, kx, p.n_half + n0, &full[s]);  // up rows
            } else {
                tma_load_2d(st + kATileBytes, &tmB, kx, n0, &full[s]);
            }
        }
      }
      __syncwarp();
    } else if (warp == 1) {
      if (lane == 0) {
        // MMA issuer
        constexpr uint32_t idesc = F8 ? idesc_e4m3(kBM, MMA_N) : idesc_bf16(kBM, MMA_N);
        int i = 0;
        for (; i < nkb; ++i) {
            const int s = i % kStages;
            if (!mbar_wait(&full[s], (i / kStages) & 1)) {
                s_fail = 1;
                break;
            }
            tc_fence_after();
            const unsigned char* st = smem + (size_t)s * kStageBytes;
            const uint64_t ad = smem_desc_sw128(st);
            const uint64_t bd = smem_desc_sw128(st + kATileBytes);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {  // 32 bytes per MMA (16 bf16 or 32 E4M3) = +2 in the address field
                if constexpr (F8) tc_mma_f8(tmem_d, ad + 2 * kk, bd + 2 * kk, idesc, (i > 0 || kk > 0) ? 1u : 0u);
                else tc_mma(tmem_d, ad + 2 * kk, bd + 2 * kk, idesc, (i > 0 || kk > 0) ? 1u : 0u);
            }
            tc_commit(&empty[s]);
        }
        tc_commit(&done);  // after every MMA issued above (also on failure: lets them drain)
      }
      __syncwarp();
    }

    // epilogue: all four warps, one accumulator lane (output row) per thread
    const bool ok = mbar_wait_or_abort(&done, 0, reinterpret_cast<volatile int*>(&s_never));
    tc_fence_after();
    __syncthreads();
    if (ok && !s_fail && nkb > 0) {
        const int row = m0 + warp * 32 + lane;
        const uint32_t tbase = tmem_d + ((uint32_t)(warp * 32) << 16);
        const float sa = F8 && row < p.M ? __ldg(p.a_scale + row) : 1.0f;
        for (int c = 0; c < nt; c += 16) {
            float v[16];
            tmem_ld16(tbase + c, v);
            if constexpr (F8) {  // the FP8 projection output: bf16(acc * (s_a * s_w[n]))
#pragma unroll
                for (int e = 0; e < 16; ++e) v[e] = round_bf16f(v[e] * (sa * __ldg(p.b_scale + n0 + c + e)));
            }
            if constexpr (EPI == kGemmSwiglu) {
                float u[16];
                tmem_ld16(tbase + nt + c, u);
                if constexpr (F8) {
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        u[e] = round_bf16f(u[e] * (sa * __ldg(p.b_scale + p.n_half + n0 + c + e)));
                }
                if (row < p.M) {
                    __nv_bfloat16* dst = p.out_bf16 + (size_t)row * p.ldc + n0 + c;
#pragma unroll
                    for (int e = 0; e < 16; e += 2) {
                        const float a = v[e] / (1.0f + expf(-v[e])) * u[e];
                        const float b = v[e + 1] / (1.0f + expf(-v[e + 1])) * u[e + 1];
                        *reinterpret_cast<__nv_bfloat162*>(dst + e) = __floats2bfloat162_rn(a, b);
                    }
                }
            } else if (row < p.M) {
                float* dst = p.C + (size_t)row * p.ldc + n0 + c;
                if constexpr (EPI == kGemmStore) {
#pragma unroll
                    for (int e = 0; e < 16; e += 4)
                        *reinterpret_cast<float4*>(dst + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
                } else if (p.atomic) {  // split-K partials: several CTAs add into the same tile
#pragma unroll
                    for (int e = 0; e < 16; ++e) atomicAdd(dst + e, v[e]);
                } else {  // the only writer of these elements: deterministic
#pragma unroll
                    for (int e = 0; e < 16; e += 4) {
                        float4 o = *reinterpret_cast<const float4*>(dst + e);
                        o.x += v[e];
                        o.y += v[e + 1];
                        o.z += v[e + 2];
                        o.w += v[e + 3];
                        *reinterpret_cast<float4*>(dst + e) = o;
                    }
                }
            }
        }
    }
    if ((!ok || s_fail) && threadIdx.x == 0 && p.err) atomicOr(p.err, kErrTimeout);
    tc_fence_before();
    __syncthreads();
    if (warp == 2) tmem_dealloc(tmem_d, kTmemCols);
}

// ---- host: tensor maps ---------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    }
    return fn;
}

// 2-D bf16 [rows][K] row-major tensor, box of box_rows x 64, 128-byte swizzle;
// rows past `rows` read as zeros.
bool make_map(CUtensorMap* m, const void* base, int rows, int K, int box_rows, bool e4m3 = false) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const int esz = e4m3 ? 1 : 2;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)K * esz};
    const cuuint32_t box[2] = {(cuuint32_t)(128 / esz), (cuuint32_t)box_rows};  // one 128-byte row per box row
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, e4m3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base),
              dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int EPI, int MMA_N>
constexpr int gemm_smem_bytes() {
    return gemm_stages<MMA_N>() * (int)(kATileBytes + MMA_N * kBK * 2) + 1024;
}

template <int EPI, int MMA_N, bool F8 = false>
cudaError_t launch_t(const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p, dim3 grid, cudaStream_t s) {
    constexpr int smem = gemm_smem_bytes<EPI, MMA_N>();
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(gemm_bf16_kernel<EPI, MMA_N, F8>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    gemm_bf16_kernel<EPI, MMA_N, F8><<<grid, kGemmThreads, smem, s>>>(a, b, p);
    return cudaGetLastError();
}

}  // namespace

bool gemm_shape_ok(int M, int N, int K, int epi, int bn) {
    const bool bn_ok = bn == 64 || bn == 80 || bn == 128 || bn == 192;
    return M > 0 && N > 0 && K > 0 && K % kBK == 0 && bn_ok && N % bn == 0 && (epi != kGemmSwiglu || bn == 128);
}

int gemm_pick_bn(int M, int N, int epi, int num_sms) {
    // the widest tile whose grid still fits one wave of CTAs (fewest idle SMs)
    if (epi == kGemmSwiglu) return 128;
    const int mt = (M + kBM - 1) / kBM;
    int best = 0;
    double best_eff = -1.0;
    for (int bn : {192, 128, 80, 64}) {
        if (N % bn) continue;
        const long long ctas = (long long)(N / bn) * mt;
        const long long waves = (ctas + num_sms - 1) / num_sms;
        const double eff = (double)ctas / (double)(waves * num_sms);  // busy fraction of the SM-waves
        if (eff > best_eff + 1e-9) {
            best_eff = eff;
            best = bn;
        }
    }
    return best ? best : 128;
}

bool gemm_shape_ok_fp8(int M, int N, int K, int epi, int bn) {
    return gemm_shape_ok(M, N, K, epi, bn) && K % (2 * kBK) == 0;
}

cudaError_t launch_gemm_fp8(const void* A8, const void* B8, const GemmParams& p_in, int epi, cudaStream_t s) {
    GemmParams p = p_in;
    if (p.bn == 0) p.bn = 128;
    if (!gemm_shape_ok_fp8(p.M, p.N, p.K, epi, p.bn) || !p.a_scale || !p.b_scale) return cudaErrorInvalidValue;
    p.kb_per_split = p.K / (2 * kBK);  // no split-K: one writer per element
    p.atomic = 0;
    CUtensorMap ma, mb;
    if (!make_map(&ma, A8, p.M, p.K, kBM, true)) return cudaErrorInvalidValue;
    const dim3 grid((p.M + kBM - 1) / kBM, p.N / p.bn, 1);
    if (epi == kGemmSwiglu) {
        if (!make_map(&mb, B8, 2 * p.n_half, p.K, 128, true)) return cudaErrorInvalidValue;
        return launch_t<kGemmSwiglu, 256, true>(ma, mb, p, grid, s);
    }
    if (!make_map(&mb, B8, p.N, p.K, p.bn, true)) return cudaErrorInvalidValue;
#define TTS_GEMM_BN8(EP)                                                     \
    switch (p.bn) {                                                          \
        case 64: return launch_t<EP, 64, true>(ma, mb, p, grid, s);          \
        case 80: return launch_t<EP, 80, true>(ma, mb, p, grid, s);          \
        case 192: return launch_t<EP, 192, true>(ma, mb, p, grid, s);        \
        default: return launch_t<EP, 128, true>(ma, mb, p, grid, s);         \
    }
    if (epi == kGemmStore) TTS_GEMM_BN8(kGemmStore)
    TTS_GEMM_BN8(kGemmAdd)
#undef TTS_GEMM_BN8
}

cudaError_t launch_gemm_bf16(const void* A, const void* B, const GemmParams& p_in, int epi, int splits,
                             cudaStream_t s) {
    GemmParams p = p_in;
    if (p.bn == 0) p.bn = 128;
    if (!gemm_shape_ok(p.M, p.N, p.K, epi, p.bn) || splits < 1) return cudaErrorInvalidValue;
    const int nkb = p.K / kBK;
    if (epi != kGemmAdd) splits = 1;  // only an additive epilogue can take split-K partials
    p.kb_per_split = (nkb + splits - 1) / splits;
    splits = (nkb + p.kb_per_split - 1) / p.kb_per_split;
    p.atomic = splits > 1 ? 1 : 0;
    CUtensorMap ma, mb;
    if (!make_map(&ma, A, p.M, p.K, kBM)) return cudaErrorInvalidValue;
    const dim3 grid((p.M + kBM - 1) / kBM, p.N / p.bn, splits);
    if (epi == kGemmSwiglu) {
        // B = [gate rows; up rows] of a [2 n_half][K] matrix; N = n_half output columns
        if (!make_map(&mb, B, 2 * p.n_half, p.K, 128)) return cudaErrorInvalidValue;
        return launch_t<kGemmSwiglu, 256>(ma, mb, p, grid, s);
    }
    if (!make_map(&mb, B, p.N, p.K, p.bn)) return cudaErrorInvalidValue;
#define TTS_GEMM_BN(EP)                                                      \
    switch (p.bn) {                                                          \
        case 64: return launch_t<EP, 64>(ma, mb, p, grid, s);                \
        case 80: return launch_t<EP, 80>(ma, mb, p, grid, s);                \
        case 192: return launch_t<EP, 192>(ma, mb, p, grid, s);              \
        default: return launch_t<EP, 128>(ma, mb, p, grid, s);               \
    }
    if (epi == kGemmStore) TTS_GEMM_BN(kGemmStore)
    TTS_GEMM_BN(kGemmAdd)
#undef TTS_GEMM_BN
}

}  // namespace tts

// ---- stand-alone entry point -------------------------------------------------------
extern "C" int tts_gemm_bf16(const void* A, const void* B, void* C, int M, int N, int K, int epi, int splits,
                             void* stream) {
    using namespace tts;
    if (!A || !B || !C || epi < kGemmStore || epi > kGemmSwiglu || splits < 1) return TTS_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) | reinterpret_cast<uintptr_t>(C)) & 15)
        return TTS_ERR_ARG;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return TTS_ERR_CUDA;
    const int bn = gemm_pick_bn(M, N, epi, sms);
    if (!gemm_shape_ok(M, N, K, epi, bn)) return TTS_ERR_ARG;
    GemmParams p{};
    p.bn = bn;
    p.M = M;
    p.N = N;
    p.K = K;
    p.ldc = N;
    if (epi == kGemmSwiglu) {
        p.n_half = N;
        p.out_bf16 = static_cast<__nv_bfloat16*>(C);
    } else {
        p.C = static_cast<float*>(C);
    }
    const cudaError_t e = launch_gemm_bf16(A, B, p, epi, splits, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        std::fprintf(stderr, "tts: tts_gemm_bf16 failed: %s\n", cudaGetErrorString(e));
        return TTS_ERR_CUDA;
    }
    return TTS_OK;
}

extern "C" int tts_gemm_fp8(const void* A8, const void* B8, const float* a_scale, const float* b_scale, void* C, int M,
                            int N, int K, int epi, void* stream) {
    using namespace tts;
    if (!A8 || !B8 || !a_scale || !b_scale || !C || epi < kGemmStore || epi > kGemmSwiglu) return TTS_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(A8) | reinterpret_cast<uintptr_t>(B8) | reinterpret_cast<uintptr_t>(C)) & 15)
        return TTS_ERR_ARG;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return TTS_ERR_CUDA;
    const int bn = gemm_pick_bn(M, N, epi, sms);
    if (!gemm_shape_ok_fp8(M, N, K, epi, bn)) return TTS_ERR_ARG;
    GemmParams p{};
    p.bn = bn;
    p.M = M;
    p.N = N;
    p.K = K;
    p.ldc = N;
    p.a_scale = a_scale;
    p.b_scale = b_scale;
    if (epi == kGemmSwiglu) {
        p.n_half = N;
        p.out_bf16 = static_cast<__nv_bfloat16*>(C);
    } else {
        p.C = static_cast<float*>(C);
    }
    const cudaError_t e = launch_gemm_fp8(A8, B8, p, epi, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        std::fprintf(stderr, "tts: tts_gemm_fp8 failed: %s\n", cudaGetErrorString(e));
        return TTS_ERR_CUDA;
    }
    return TTS_OK;
}

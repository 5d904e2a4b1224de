// GEMM on the 5th-generation tensor cores (sm_103a): C = A . B^T with
// A [M][K] activations and B [N][K] weights, both K-major bf16 (or both
// E4M3), fp32 accumulation in tensor memory.  The batched prefill's projections
// ("Higgs Audio v3 TTS-4B on FlashRT", Performance: "BF16 W16A16", prompt
// prefill; section 7: the prompt runs as one M = P pass, weights read once)
// are dense contractions of P rows against every weight matrix, so they run
// here rather than on the M = 1 weight-streaming path.
//
// One CTA per (128 MT) x BN output tile (MT = 1 or 2 accumulators of 128
// rows sharing each weight tile; BN = 64, 80, 128, 160 or 192; 128 gate +
// 128 up columns for the fused gate/up tile), optionally one of S <= 4 CTAs
// of a cluster that share the tile's K range:
//   warp 0 (one thread)  TMA producer: (128 MT) x 64 A box and BN x 64 B
//                        box(es) per k-block into a ring of 3-8 stages
//                        (128-byte swizzle), completion counted on the
//                        stage's "full" mbarrier;
//   warp 1 (one thread)  MMA issuer: 4 MT tcgen05.mma (K = 16 each) per
//                        k-block into the TMEM accumulators, then
//                        tcgen05.commit frees the stage ("empty") and, after
//                        the last block, signals "done";
//   warp 2               allocates / frees the TMEM columns;
//   warps 0-3            epilogue: tcgen05.ld of their 32 accumulator lanes
//                        (one output row per thread), staged in the freed
//                        ring and written by TMA (store, or add at the
//                        destination for the residual); SwiGLU -> bf16; with
//                        a K split, the partial rows are first gathered and
//                        added in rank order through distributed shared memory.
// Every wait is bounded; on expiry the kernel records an error, lets its
// copies and MMAs finish and frees its tensor memory before returning.
#include <cuda.h>

#include <cstdio>

#include "kernels.h"
#include "tts_decode.h"

namespace tts {

namespace {

constexpr int kBM = 128;          // rows of A per accumulator (MMA M)
constexpr int kBK = 64;           // k-block: 64 bf16 = one 128-byte swizzle row
// ring depth: as many stages as fit in shared memory (at most 8), so narrow
// tiles keep as many bytes in flight from L2 as wide ones
constexpr int kSmemRing = 225 * 1024;
template <int MT>
constexpr uint32_t gemm_a_tile() { return MT * kBM * 128; }  // bytes of A per k-block
template <int MT, int MMA_N>
constexpr int gemm_stages() {
    return kSmemRing / (int)(gemm_a_tile<MT>() + MMA_N * 128) < 8 ? kSmemRing / (int)(gemm_a_tile<MT>() + MMA_N * 128)
                                                                  : 8;
}
constexpr int kGemmThreads = 128;
// epilogue staging in the freed ring: boxes of 32 rows x 64 bytes, 2 KB each
// (1024-byte aligned)
constexpr int kEpiBoxBytes = 2048;

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
// 32 consecutive fp32 columns of this warp's 32 accumulator lanes; the load
// and its wait are one statement, so no use of the registers can be placed
// between them
#define TTS_R8(b) "=r"(r[b]), "=r"(r[b + 1]), "=r"(r[b + 2]), "=r"(r[b + 3]), "=r"(r[b + 4]), "=r"(r[b + 5]), \
                  "=r"(r[b + 6]), "=r"(r[b + 7])
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : TTS_R8(0), TTS_R8(8), TTS_R8(16), TTS_R8(24)
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
#undef TTS_R8

// generic-proxy writes to shared memory made visible to the TMA engine
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// box of the tensor map at (x, y) <- shared memory: plain store, or an
// element-wise add performed at the destination (reduce .add)
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int x, int y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(smem_u32(src))
                 : "memory");
}
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* map, const void* src, int x, int y) {
    asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(smem_u32(src))
                 : "memory");
}
__device__ __forceinline__ void bulk_commit_and_wait_all() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
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

// distributed shared memory of the cluster: this CTA's shared address `a`
// as seen in CTA `rank`, and a 16-byte load from there
__device__ __forceinline__ uint32_t dsmem_map(uint32_t a, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}
__device__ __forceinline__ void dsmem_st4(uint32_t a, float x, float y, float z, float w) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a), "f"(x), "f"(y), "f"(z), "f"(w)
                 : "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// every thread of every CTA of the cluster: release this CTA's shared-memory
// writes and wait for all the others'
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// fp32 x 4 added at the destination; the only writer of these elements, so
// the result is C + v whatever the order of other rows' additions
__device__ __forceinline__ void red_add4(float* dst, float4 v) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "f"(v.x), "f"(v.y), "f"(v.z),
                 "f"(v.w)
                 : "memory");
}

// One CTA computes a (128 MT) x nt output tile: MT accumulators of 128 rows
// share every weight (B) tile, which halves the bytes each SM takes in per
// MMA at MT = 2.  SPLIT: the K range is cut over the CTAs of a cluster (grid
// z = cluster size S <= 4); CTA r owns rows [r R / S, (r + 1) R / S) of the
// tile, receives those rows of every CTA's fp32 partial sums in its shared
// memory (distributed shared memory stores), adds them in rank order (a
// fixed order: deterministic) and writes them.
// F8: E4M3 operands; a k-block is then 128 elements (still one 128-byte
// swizzle row), an MMA takes K = 32 (still 32 bytes), and every product sum
// is scaled by its row's and column's scales and rounded to bf16 before the
// epilogue's operation.
template <int EPI, int MMA_N, bool F8, int MT, bool SPLIT>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmC, const GemmParams p) {
    static_assert(MT == 1 || MT == 2, "one or two 128-row accumulators");
    static_assert(!(SPLIT && EPI == kGemmSwiglu), "SwiGLU needs the whole sum");
    constexpr int kBKE = F8 ? 2 * kBK : kBK;  // elements per k-block (128 bytes per row)
    extern __shared__ unsigned char smem_raw[];
    constexpr int kStages = gemm_stages<MT, MMA_N>();
    constexpr uint32_t kATile = gemm_a_tile<MT>();
    constexpr uint32_t kBTile = MMA_N * 128;
    constexpr uint32_t kStageBytes = kATile + kBTile;
    constexpr uint32_t kRing = kStages * kStageBytes;
    // fp32 accumulator columns per 128-row accumulator: a power of two >= 32
    constexpr uint32_t kAccCols = MMA_N <= 32 ? 32 : MMA_N <= 64 ? 64 : MMA_N <= 128 ? 128 : 256;
    constexpr uint32_t kTmemCols = MT * kAccCols;
    static_assert(kTmemCols <= 512, "tensor memory holds 512 columns");
    constexpr int nt = EPI == kGemmSwiglu ? MMA_N / 2 : MMA_N;  // output columns of this tile
    constexpr int kBoxCols = EPI == kGemmSwiglu ? 32 : 16;      // 64 bytes of output per staged box row
    constexpr int kEpiWarp = MT * (nt / kBoxCols) * kEpiBoxBytes;
    static_assert(SPLIT || 4 * kEpiWarp <= (int)kRing, "epilogue staging must fit in the ring");
    constexpr int kPld = nt + 4;  // partial-tile row stride (floats): odd multiple of 16 bytes, conflict-free
    // S slots of ceil(R / S) rows each: at most R + S - 1 rows (S <= 4)
    static_assert(!SPLIT || (MT * kBM + 3) * kPld * 4 <= (int)kRing, "the partial rows must fit in the ring");

    __shared__ __align__(8) uint64_t full[kStages], empty[kStages], done;
    __shared__ uint32_t s_tmem;
    __shared__ int s_fail;
    __shared__ int s_never;       // abort flag of the epilogue wait: only the time limit ends it
    __shared__ float s_bsc[256];  // E4M3: the tile's column scales (gate, then up)
    // stage tiles 1024-byte aligned (swizzle atoms)
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // the M tiles of one N tile are adjacent in the grid: they run together
    // and share the weight tile through L2 (one DRAM read per weight)
    const int m0 = blockIdx.x * (kBM * MT);
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
    if constexpr (F8) {
        for (int i = threadIdx.x; i < nt; i += kGemmThreads) {
            s_bsc[i] = __ldg(p.b_scale + n0 + i);
            if constexpr (EPI == kGemmSwiglu) s_bsc[nt + i] = __ldg(p.b_scale + p.n_half + n0 + i);
        }
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
            tma_load_2d(st, &tmA, kx, m0, &full[s]);  // 128 MT rows in one box
            if constexpr (EPI == kGemmSwiglu) {
                tma_load_2d(st + kATile, &tmB, kx, n0, &full[s]);                         // gate rows
                tma_load_2d(st + kATile + kBTile / 2, &tmB, kx, p.n_half + n0, &full[s]);  // up rows
            } else {
                tma_load_2d(st + kATile, &tmB, kx, n0, &full[s]);
            }
        }
      }
      __syncwarp();
    } else if (warp == 1) {
      if (lane == 0) {
        // MMA issuer
        constexpr uint32_t idesc = F8 ? idesc_e4m3(kBM, MMA_N) : idesc_bf16(kBM, MMA_N);
        for (int i = 0; i < nkb; ++i) {
            const int s = i % kStages;
            if (!mbar_wait(&full[s], (i / kStages) & 1)) {
                s_fail = 1;
                break;
            }
            tc_fence_after();
            const unsigned char* st = smem + (size_t)s * kStageBytes;
            const uint64_t ad = smem_desc_sw128(st);
            const uint64_t bd = smem_desc_sw128(st + kATile);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {  // 32 bytes per MMA (16 bf16 or 32 E4M3) = +2 in the address field
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {  // rows 128 mt.. of A start 16 KB (+1024 in the field) further
                    const uint64_t a_k = ad + (uint64_t)(mt * (kBM * 128 >> 4)) + 2 * kk;
                    const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
                    if constexpr (F8) tc_mma_f8(tmem_d + mt * kAccCols, a_k, bd + 2 * kk, idesc, acc);
                    else tc_mma(tmem_d + mt * kAccCols, a_k, bd + 2 * kk, idesc, acc);
                }
            }
            tc_commit(&empty[s]);
        }
        tc_commit(&done);  // after every MMA issued above (also on failure: lets them drain)
      }
      __syncwarp();
    }

    // epilogue: all four warps; warp w reads accumulator lanes 32w..32w+31
    // (one output row per thread) of each of the MT accumulators
    const bool ok = mbar_wait_or_abort(&done, 0, reinterpret_cast<volatile int*>(&s_never));
    tc_fence_after();
    __syncthreads();
    const bool have = ok && !s_fail && nkb > 0;
    if constexpr (!SPLIT) {
        // Each warp converts its rows a box of columns at a time into the
        // freed ring (64-byte-swizzled rows, the layout the store's tensor
        // map expects: conflict-free 16-byte writes); one lane then hands
        // the boxes to the TMA engine, which writes them (store) or adds
        // them into C at the destination (residual).
        unsigned char* stg = smem + (size_t)warp * kEpiWarp;
        const uint32_t swz = (uint32_t)((lane >> 1) & 3);  // 64-byte swizzle: 16-byte chunk j lands at j ^ swz
        constexpr int kBoxes = nt / kBoxCols;
#pragma unroll 1
        for (int mt = 0; mt < MT; ++mt) {
            const int row = m0 + mt * kBM + warp * 32 + lane;
            if (!have || m0 + mt * kBM + warp * 32 >= p.M) continue;  // warp-uniform
            const uint32_t tbase = tmem_d + mt * kAccCols + ((uint32_t)(warp * 32) << 16);
            const float sa = F8 && row < p.M ? __ldg(p.a_scale + row) : 1.0f;
            unsigned char* stm = stg + mt * kBoxes * kEpiBoxBytes;
            if constexpr (EPI == kGemmSwiglu) {
                for (int g = 0; g < kBoxes; ++g) {
                    float v[32], u[32];
                    tmem_ld32(tbase + g * 32, v);
                    tmem_ld32(tbase + nt + g * 32, u);
                    unsigned char* box = stm + g * kEpiBoxBytes + lane * 64;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint32_t w[4];
#pragma unroll
                        for (int e2 = 0; e2 < 4; ++e2) {
                            float o[2];
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                const int e = 8 * j + 2 * e2 + h;
                                float gv = v[e], uv = u[e];
                                if constexpr (F8) {  // the FP8 projection outputs: bf16(acc * (s_a * s_w[n]))
                                    gv = round_bf16f(gv * (sa * s_bsc[g * 32 + e]));
                                    uv = round_bf16f(uv * (sa * s_bsc[nt + g * 32 + e]));
                                }
                                // fast exponential and division: the product is rounded to bf16
                                o[h] = __fdividef(gv, 1.0f + __expf(-gv)) * uv;
                            }
                            const __nv_bfloat162 b2 = __floats2bfloat162_rn(o[0], o[1]);
                            w[e2] = *reinterpret_cast<const uint32_t*>(&b2);
                        }
                        *reinterpret_cast<uint4*>(box + ((j ^ swz) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            } else {
                for (int c = 0; c < nt; c += 32) {
                    float v[32];
                    tmem_ld32(tbase + c, v);  // columns past nt (a tile of 80 or 160) are read, not staged
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        if (c + 16 * h >= nt) break;
                        unsigned char* box = stm + ((c >> 4) + h) * kEpiBoxBytes + lane * 64;
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            float4 q;
                            float* qe = reinterpret_cast<float*>(&q);
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const int e = 16 * h + 4 * j + i;
                                qe[i] = F8 ? round_bf16f(v[e] * (sa * s_bsc[c + e])) : v[e];
                            }
                            *reinterpret_cast<float4*>(box + ((j ^ swz) << 4)) = q;
                        }
                    }
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                for (int g = 0; g < kBoxes; ++g) {
                    const void* src = stm + g * kEpiBoxBytes;
                    const int y = m0 + mt * kBM + warp * 32;
                    if constexpr (EPI == kGemmAdd) tma_reduce_add_2d(&tmC, src, n0 + g * kBoxCols, y);
                    else tma_store_2d(&tmC, src, n0 + g * kBoxCols, y);
                }
            }
        }
        if (lane == 0) bulk_commit_and_wait_all();
        __syncwarp();
    } else {
        // Rows [r0_q, r0_{q+1}) of the tile belong to CTA q of the cluster
        // (r0_q = q R / S).  Each CTA writes the rows of its partial tile
        // into their owner's shared memory (slot = the writer's rank), so
        // the owner can add the S partials of its rows in rank order.
        const int S = (int)gridDim.z, me = (int)cluster_rank();
        constexpr int R = MT * kBM;
        const int rows_max = (R + S - 1) / S;
        float* part = reinterpret_cast<float*>(smem);
        const uint32_t pbase = smem_u32(part);
        // 1. every CTA of the cluster is past its main loop (its ring is free)
        cluster_sync_all();
        if (have) {
            uint32_t rb[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) rb[q] = q < S ? dsmem_map(pbase, (uint32_t)q) : 0u;
#pragma unroll 1
            for (int mt = 0; mt < MT; ++mt) {
                const int tr = mt * kBM + warp * 32 + lane;  // tile row of this thread
                int q = 0;
                while (q + 1 < S && tr >= (q + 1) * R / S) ++q;
                const int lr = tr - q * R / S;
                const uint32_t dst = rb[q] + (uint32_t)(((me * rows_max + lr) * kPld) * 4);
                const uint32_t tbase = tmem_d + mt * kAccCols + ((uint32_t)(warp * 32) << 16);
                for (int c = 0; c < nt; c += 32) {
                    float v[32];
                    tmem_ld32(tbase + c, v);
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        if (c + 4 * j < nt) dsmem_st4(dst + (uint32_t)((c + 4 * j) * 4), v[4 * j], v[4 * j + 1],
                                                      v[4 * j + 2], v[4 * j + 3]);
                }
            }
        }
        // 2. every partial row has reached its owner (also after a failure:
        //    every CTA arrives)
        cluster_sync_all();
        // 3. this CTA's rows: the S partials added in rank order, then written
        const int r0 = me * R / S, r1 = (me + 1) * R / S;
        constexpr int kC4 = nt / 4;
        if (have) {
            for (int idx = threadIdx.x; idx < (r1 - r0) * kC4; idx += kGemmThreads) {
                const int lr = idx / kC4, c = 4 * (idx % kC4);
                const int row = m0 + r0 + lr;
                if (row >= p.M) continue;
                const float* src = part + (size_t)lr * kPld + c;
                float4 acc = *reinterpret_cast<const float4*>(src);
                for (int q = 1; q < S; ++q) {
                    const float4 t = *reinterpret_cast<const float4*>(src + (size_t)q * rows_max * kPld);
                    acc.x += t.x;
                    acc.y += t.y;
                    acc.z += t.z;
                    acc.w += t.w;
                }
                if constexpr (F8) {
                    const float sa = __ldg(p.a_scale + row);
                    acc.x = round_bf16f(acc.x * (sa * s_bsc[c]));
                    acc.y = round_bf16f(acc.y * (sa * s_bsc[c + 1]));
                    acc.z = round_bf16f(acc.z * (sa * s_bsc[c + 2]));
                    acc.w = round_bf16f(acc.w * (sa * s_bsc[c + 3]));
                }
                float* dst = p.C + (size_t)row * p.ldc + n0 + c;
                if constexpr (EPI == kGemmAdd) red_add4(dst, acc);
                else *reinterpret_cast<float4*>(dst) = acc;
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

// 2-D [rows][K] row-major operand (bf16 or E4M3), boxes of box_rows rows x
// 128 bytes with the 128-byte swizzle; rows past `rows` read as zeros.
bool make_map(CUtensorMap* m, const void* base, int rows, int K, int box_rows, bool e4m3) {
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

// The output C [rows][cols] (row stride ld elements), fp32 or bf16, as boxes
// of 32 rows x 64 bytes with the 64-byte swizzle; rows past `rows` are not written.
bool make_store_map(CUtensorMap* m, void* base, int rows, int cols, int ld, bool bf16) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const int esz = bf16 ? 2 : 4;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)ld * esz};
    const cuuint32_t box[2] = {(cuuint32_t)(64 / esz), 32};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MT, int MMA_N>
constexpr int gemm_smem_bytes() {
    return gemm_stages<MT, MMA_N>() * (int)(gemm_a_tile<MT>() + MMA_N * 128) + 1024;
}

template <int EPI, int MMA_N, bool F8, int MT, bool SPLIT>
cudaError_t launch_t(const void* A, const void* B, const GemmParams& p, int splits, cudaStream_t s) {
    constexpr int smem = gemm_smem_bytes<MT, MMA_N>();
    static bool attr = false;
    auto kern = gemm_kernel<EPI, MMA_N, F8, MT, SPLIT>;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    CUtensorMap ma, mb, mc;
    if (!make_map(&ma, A, p.M, p.K, kBM * MT, F8)) return cudaErrorInvalidValue;
    if (EPI == kGemmSwiglu) {
        // B = [gate rows; up rows] of a [2 n_half][K] matrix; 128 + 128 rows per tile
        if (!make_map(&mb, B, 2 * p.n_half, p.K, MMA_N / 2, F8)) return cudaErrorInvalidValue;
        if (!p.out_bf16 || !make_store_map(&mc, p.out_bf16, p.M, p.N, p.ldc, true)) return cudaErrorInvalidValue;
    } else {
        if (!make_map(&mb, B, p.N, p.K, MMA_N, F8)) return cudaErrorInvalidValue;
        if (!p.C || !make_store_map(&mc, p.C, p.M, p.N, p.ldc, false)) return cudaErrorInvalidValue;
    }
    const int nt = EPI == kGemmSwiglu ? MMA_N / 2 : MMA_N;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((p.M + kBM * MT - 1) / (kBM * MT), p.N / nt, splits);
    cfg.blockDim = dim3(kGemmThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    if (SPLIT) {
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = 1;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = splits;
        cfg.attrs = at;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, kern, ma, mb, mc, p);
}

// How many clusters of S CTAs of the split kernels run at once (cached; the
// SMs of a GPC hold whole clusters only).
int cluster_capacity(int S, int num_sms) {
    static int cap[9] = {0};
    if (S <= 1) return num_sms;
    if (S > 8) return 0;
    if (!cap[S]) {
        constexpr int smem = gemm_smem_bytes<2, 160>();
        auto kern = gemm_kernel<kGemmAdd, 160, false, 2, true>;
        int n = 0;
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(1, 1, S);
        cfg.blockDim = dim3(kGemmThreads);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = 1;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = S;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) == cudaSuccess &&
            cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess && n > 0)
            cap[S] = n * S;
        else
            cap[S] = (num_sms / (2 * S)) * S;  // unknown: assume half the SMs
    }
    return cap[S];
}

// Modelled time of one tile configuration, in microseconds: whole waves of
// CTAs, each taking its k-blocks at a per-k-block time plus ~2 us of
// prologue and epilogue, plus ~5 us (E4M3: ~8) for the cluster reduction
// of a split.
// The per-k-block times are fits to this kernel's timings on GB300 at
// M = 512 (the prefill's shapes): the main loop is bound neither by L2 nor
// by the MMAs alone but by the SM's shared-memory traffic (TMA writes plus
// the MMAs' operand reads), which grows with the tile width; E4M3 k-blocks
// (128 elements) take ~1.4x a bf16 k-block (64).  Two 128-row accumulators
// pay off only for the SwiGLU tile, where they turn two waves into one.
double tile_cost(int M, int N, int K, int epi, bool fp8, const GemmTile& t, int num_sms) {
    const int kbe = fp8 ? 2 * kBK : kBK;
    const long long tiles = (long long)((M + kBM * t.mt - 1) / (kBM * t.mt)) * (N / t.bn);
    const int kb = (K / kbe + t.splits - 1) / t.splits;
    const int cap = cluster_capacity(t.splits, num_sms);
    if (cap <= 0) return 1e30;
    const long long waves = (tiles * t.splits + cap - 1) / cap;
    double t_kb;
    if (epi == kGemmSwiglu) t_kb = t.mt == 2 ? 0.84 : 0.48;
    else t_kb = t.mt == 2 ? 0.30 + 0.0015 * t.bn : 0.262 + 0.00085 * t.bn;
    if (fp8) t_kb *= 1.4;
    // the reduction of an E4M3 split also scales and rounds every element
    return (double)waves * (kb * t_kb + 2.0) + (t.splits > 1 ? (fp8 ? 8.0 : 5.0) : 0.0);
}

bool tile_ok(int M, int N, int K, int epi, bool fp8, const GemmTile& t) {
    const int kbe = fp8 ? 2 * kBK : kBK;
    if (M < 1 || N < 1 || K < kbe || K % kbe) return false;
    if (t.mt != 1 && t.mt != 2) return false;
    if (t.splits < 1 || t.splits > 8 || t.splits > K / kbe) return false;
    if (epi == kGemmSwiglu) return t.bn == 128 && t.splits == 1 && N % 128 == 0;
    const bool bn_ok = t.bn == 64 || t.bn == 80 || t.bn == 128 || t.bn == 160 || t.bn == 192;
    return bn_ok && N % t.bn == 0 && t.splits <= 4;
}

template <int EPI, bool F8>
cudaError_t launch_tile(const void* A, const void* B, const GemmParams& p, const GemmTile& t, cudaStream_t s) {
    if constexpr (EPI == kGemmSwiglu) {
        return t.mt == 2 ? launch_t<EPI, 256, F8, 2, false>(A, B, p, 1, s) : launch_t<EPI, 256, F8, 1, false>(A, B, p, 1, s);
    } else {
#define TTS_GEMM_N(MT, SP)                                                             \
    switch (t.bn) {                                                                  \
        case 64: return launch_t<EPI, 64, F8, MT, SP>(A, B, p, t.splits, s);         \
        case 80: return launch_t<EPI, 80, F8, MT, SP>(A, B, p, t.splits, s);         \
        case 128: return launch_t<EPI, 128, F8, MT, SP>(A, B, p, t.splits, s);       \
        case 160: return launch_t<EPI, 160, F8, MT, SP>(A, B, p, t.splits, s);       \
        default: return launch_t<EPI, 192, F8, MT, SP>(A, B, p, t.splits, s);        \
    }
        if (t.splits > 1) {
            if (t.mt == 2) TTS_GEMM_N(2, true)
            TTS_GEMM_N(1, true)
        }
        if (t.mt == 2) TTS_GEMM_N(2, false)
        TTS_GEMM_N(1, false)
#undef TTS_GEMM_N
    }
}

}  // namespace

GemmTile gemm_pick(int M, int N, int K, int epi, bool fp8, int num_sms, int splits) {
    GemmTile best{0, 0, 0};
    double best_t = 1e300;
    // automatic choice: at most two K splits (more measured slower at these
    // shapes: the reduction costs more than the extra SMs give); 256-row
    // tiles for the SwiGLU GEMM only
    const int s_max = splits > 0 ? splits : 2;
    for (int mt : {1, 2})
        for (int bn : {64, 80, 128, 160, 192})
            for (int S = 1; S <= s_max; ++S) {
                if (splits > 0 && S != splits) continue;
                if (splits <= 0 && mt == 2 && epi != kGemmSwiglu) continue;
                const GemmTile t{mt, bn, S};
                if (!tile_ok(M, N, K, epi, fp8, t)) continue;
                const double c = tile_cost(M, N, K, epi, fp8, t, num_sms);
                if (c < best_t * (1.0 - 1e-9)) {  // ties keep the earlier (smaller) configuration
                    best_t = c;
                    best = t;
                }
            }
    return best;
}

bool gemm_shape_ok(int N, int K, int epi, bool fp8) {
    return gemm_pick(kBM, N, K, epi, fp8, 152, 1).mt != 0;
}

cudaError_t launch_gemm(const void* A, const void* B, const GemmParams& p_in, int epi, bool fp8, GemmTile t,
                        int num_sms, cudaStream_t s) {
    GemmParams p = p_in;
    if (t.mt == 0) t = gemm_pick(p.M, p.N, p.K, epi, fp8, num_sms, t.splits);
    if (!tile_ok(p.M, p.N, p.K, epi, fp8, t)) return cudaErrorInvalidValue;
    if (fp8 && (!p.a_scale || !p.b_scale)) return cudaErrorInvalidValue;
    if (epi == kGemmSwiglu && p.n_half != p.N) return cudaErrorInvalidValue;
    const int nkb = p.K / (fp8 ? 2 * kBK : kBK);
    p.kb_per_split = (nkb + t.splits - 1) / t.splits;
    if ((long long)p.kb_per_split * (t.splits - 1) >= nkb) return cudaErrorInvalidValue;  // an empty split
    if (fp8) {
        if (epi == kGemmStore) return launch_tile<kGemmStore, true>(A, B, p, t, s);
        if (epi == kGemmAdd) return launch_tile<kGemmAdd, true>(A, B, p, t, s);
        return launch_tile<kGemmSwiglu, true>(A, B, p, t, s);
    }
    if (epi == kGemmStore) return launch_tile<kGemmStore, false>(A, B, p, t, s);
    if (epi == kGemmAdd) return launch_tile<kGemmAdd, false>(A, B, p, t, s);
    return launch_tile<kGemmSwiglu, false>(A, B, p, t, s);
}

}  // namespace tts

// ---- stand-alone entry points ------------------------------------------------------
namespace {
int gemm_entry(const void* A, const void* B, const float* a_scale, const float* b_scale, void* C, int M, int N, int K,
               int epi, bool fp8, tts::GemmTile t, void* stream, const char* name) {
    using namespace tts;
    if (!A || !B || !C || epi < kGemmStore || epi > kGemmSwiglu) return TTS_ERR_ARG;
    if (fp8 && (!a_scale || !b_scale)) return TTS_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) | reinterpret_cast<uintptr_t>(C)) & 15)
        return TTS_ERR_ARG;
    if (t.mt != 0 && !tile_ok(M, N, K, epi, fp8, t)) return TTS_ERR_ARG;  // before any device call
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return TTS_ERR_CUDA;
    if (t.mt == 0) t = gemm_pick(M, N, K, epi, fp8, sms, t.splits);
    if (!tile_ok(M, N, K, epi, fp8, t)) return TTS_ERR_ARG;
    GemmParams p{};
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
    const cudaError_t e = launch_gemm(A, B, p, epi, fp8, t, sms, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        std::fprintf(stderr, "tts: %s failed: %s\n", name, cudaGetErrorString(e));
        return TTS_ERR_CUDA;
    }
    return TTS_OK;
}
}  // namespace

extern "C" int tts_gemm_bf16(const void* A, const void* B, void* C, int M, int N, int K, int epi, int splits,
                             void* stream) {
    return gemm_entry(A, B, nullptr, nullptr, C, M, N, K, epi, false, tts::GemmTile{0, 0, splits > 0 ? splits : 0},
                      stream, "tts_gemm_bf16");
}

extern "C" int tts_gemm_fp8(const void* A8, const void* B8, const float* a_scale, const float* b_scale, void* C, int M,
                            int N, int K, int epi, void* stream) {
    return gemm_entry(A8, B8, a_scale, b_scale, C, M, N, K, epi, true, tts::GemmTile{0, 0, 0}, stream, "tts_gemm_fp8");
}

extern "C" int tts_gemm_tiled(const void* A, const void* B, const float* a_scale, const float* b_scale, void* C, int M,
                              int N, int K, int epi, int fp8, int tile_rows, int tile_cols, int splits, void* stream) {
    if (tile_rows != 128 && tile_rows != 256) return TTS_ERR_ARG;
    return gemm_entry(A, B, a_scale, b_scale, C, M, N, K, epi, fp8 != 0,
                      tts::GemmTile{tile_rows / 128, tile_cols, splits}, stream, "tts_gemm_tiled");
}

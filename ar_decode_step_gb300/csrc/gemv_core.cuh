// Building blocks of the M = 1 weight-streaming projections, shared by the
// per-projection GEMV kernel (gemv.cu) and the persistent decode-step kernel
// (step.cu).  A CTA = one producer warp + kConsumerWarps consumer warps.
//
// Producer: streams the CTA's row range of a weight matrix through a ring of
// shared-memory stages.  A stage is a group of RS whole rows (RS a power of
// two, up to 40 KB) filled by one bulk copy on the TMA engine (two for
// gate/up: RS/2 gate rows and the matching RS/2 up rows); completion is
// counted on the slot's "full" mbarrier, consumers free the slot on its
// "empty" mbarrier.
//
// Consumers, bf16 weights: warp w owns column segment w % WPR of row slot
// w / WPR (WPR segments per row, stage_geom); a stage's rows are taken one row
// slot per pass: equal bytes per warp, direct activation indexing, one shuffle
// reduction per row, packed fp32 FMAs against fp32 activations.
// Consumers, E4M3 weights: the stage loop runs on the tensor cores (E4M3 x
// E4M3 mma.sync m16n8k32, fp32 accumulation), the stage's rows as A and the
// quantised activation as B.  A stage of R rows is cut into P = 16 / R
// K-subranges per row, and each subrange into one piece per warp, so a warp's
// 16 MMA rows are all (row, subrange) pairs of the stage.  Each lane feeds
// its own 16-byte chunks of its two MMA rows and the matching activation
// chunk, so the products of MMA row m meet only in output column m mod 8: the
// partial sums are the MMA's diagonal.  Lanes of odd and even MMA rows take
// the two halves of each 128-byte group in opposite order, which keeps the
// 16-byte shared-memory loads free of bank conflicts.
// Either way, per-(row, segment) partials are summed in segment order
// (deterministic) before the epilogue.
//
// Activations: staged in shared memory once per projection, fp32 planes for
// bf16 weights, E4M3 bytes (per-token scale) for FP8 weights.
#pragma once

#include <type_traits>

#include "kernels.h"

namespace tts {
namespace core {

constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;  // + one producer warp (the last)
constexpr int kMaxStages = 8;
constexpr int kBarrierBytes = 128;         // room for 8 full + 8 empty barriers

// ---- chunk dot products ------------------------------------------------------
// Two fp32 FMAs in one instruction (packed f32x2): (e, o) += (a0, a1) * (b0, b1),
// each rounded like fmaf.
__device__ __forceinline__ void ffma2(float& e, float& o, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 pa, pb, pc;\n\t"
        "mov.b64 pa, {%2, %3};\n\t"
        "mov.b64 pb, {%4, %5};\n\t"
        "mov.b64 pc, {%0, %1};\n\t"
        "fma.rn.f32x2 pc, pa, pb, pc;\n\t"
        "mov.b64 {%0, %1}, pc;\n\t}"
        : "+f"(e), "+f"(o)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// BF16: 8 weights x fp32 activations held as two float4 planes; two
// independent FMA chains (even / odd elements), issued as packed pairs.
__device__ __forceinline__ void dot_bf16(const uint4 w, const float4 a, const float4 b, float& e, float& o) {
    ffma2(e, o, bf16lo(w.x), bf16hi(w.x), a.x, a.y);
    ffma2(e, o, bf16lo(w.y), bf16hi(w.y), a.z, a.w);
    ffma2(e, o, bf16lo(w.z), bf16hi(w.z), b.x, b.y);
    ffma2(e, o, bf16lo(w.w), bf16hi(w.w), b.z, b.w);
}

// D += A . B for one m16n8k32 tile: A 16 x 32 E4M3 (row-major fragments
// a0..a3), B 32 x 8 E4M3 (column fragments b0, b1), D 16 x 8 fp32.
__device__ __forceinline__ void mma_e4m3(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// fp32 -> E4M3 byte (round to nearest even, saturating to +-448).
__device__ __forceinline__ uint32_t e4m3_byte(float x) {
    return (uint32_t)__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
}
// x / sa for the four elements of v as E4M3 bytes, v.x in the lowest byte
// (pairs converted by one instruction each, same rounding as e4m3_byte).
__device__ __forceinline__ uint32_t e4m3x4_div(const float4 v, float sa, float rsa) {
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(div_rn_by(v.x, sa, rsa), div_rn_by(v.y, sa, rsa)),
                                                 __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(div_rn_by(v.z, sa, rsa), div_rn_by(v.w, sa, rsa)),
                                                 __NV_SATFINITE, __NV_E4M3);
    return lo | (hi << 16);
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

// Barrier among the consumer warps only (the producer warp does not take part).
__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory"); }
// The same barrier, returning whether v was true in any consumer thread: a
// decision every consumer thread takes alike (to stop after a failed wait).
__device__ __forceinline__ bool consumer_sync_or(bool v) {
    unsigned r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "bar.red.or.pred po, 1, %2, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"((unsigned)v), "n"(kConsumers)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ float consumer_sum(float v, float* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = warp_sum(v);
    consumer_sync();
    if (lane == 0) red[warp] = v;
    consumer_sync();
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kConsumerWarps; ++i) s += red[i];  // fixed order: deterministic
    consumer_sync();
    return s;
}
// The sum of s and the max of m over the consumer threads, with one barrier:
// red[0..15] must not be read any more from an earlier call, which holds when
// calls are separated by at least one consumer barrier (as the stagings of
// successive phases are).
__device__ __forceinline__ void consumer_sum_max(float& s, float& m, float* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    s = warp_sum(s);
    m = warp_max(m);
    if (lane == 0) {
        red[warp] = s;
        red[kConsumerWarps + warp] = m;
    }
    consumer_sync();
    s = red[0];
    m = red[kConsumerWarps];
#pragma unroll
    for (int i = 1; i < kConsumerWarps; ++i) {  // fixed order: deterministic
        s += red[i];
        m = fmaxf(m, red[kConsumerWarps + i]);
    }
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
    consumer_sync();
    return s;
}

// ---- data exchange between the phases of the persistent step -----------------
// Each vector a phase of the persistent step hands to the next (qkv, the
// attention output, the residual stream after the attention and after the
// MLP, the MLP activation) has a buffer of its own per layer, set to kUnset
// before every launch, and an arrival counter, also kUnset at launch.
// Producers store their elements once, then each producing CTA adds 1 to the
// counter, with no fence in between.  A consumer CTA waits (one thread
// polling) until the counter shows every producer, then loads the vector and
// re-reads any element still kUnset: the data is the signal, the counter
// only says when to start reading (it keeps thousands of threads from
// polling the data lines while the producers work).  So no CTA waits for a
// fence, and there is no grid barrier.  Arithmetic never makes the bit
// pattern kUnset (a negative NaN with every payload bit set; NaNs from
// arithmetic are the canonical 0x7fffffff).
constexpr uint32_t kUnset = 0xffffffffu;

__device__ __forceinline__ bool unset4(const float4& v) {
    return __float_as_uint(v.x) == kUnset || __float_as_uint(v.y) == kUnset || __float_as_uint(v.z) == kUnset ||
           __float_as_uint(v.w) == kUnset;
}
__device__ __forceinline__ float4 ld_relaxed4(const float4* p) {
    float4 v;
    asm volatile("ld.relaxed.gpu.global.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed(float* p, float v) {
    asm volatile("st.relaxed.gpu.global.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

// What a polling wait needs: where to record a timeout, the CTA's abort flag
// (set by any of its threads that gave up) and the wait's limit in ns.
struct Poll {
    int* err;
    volatile int* abort;
    uint64_t limit_ns;
};

// Re-read the float4 at p until none of its elements is kUnset and return
// it.  If the wait ran out (the timeout is recorded) or the launch is
// aborting, *w.abort is set and the value returned is still unset.  (Values
// go in and out by value: a reference would move the caller's registers to
// local memory.)
static __device__ __noinline__ float4 poll4_wait(const float4* p, const Poll& w) {
    const uint64_t t0 = globaltimer_ns();
    for (unsigned n = 1;; ++n) {
        __nanosleep(64);
        const float4 v = ld_relaxed4(p);
        if (!unset4(v)) return v;
        if ((n & 15) == 0) {
            if (*w.abort || (w.err && (*reinterpret_cast<volatile int*>(w.err) & kErrTimeout))) {
                *w.abort = 1;
                return v;
            }
            if (globaltimer_ns() - t0 > w.limit_ns) {
                if (w.err) atomicOr(w.err, kErrTimeout);
                *w.abort = 1;
                return v;
            }
        }
    }
}
// One float4 of an exchanged vector, waiting until it is written (still
// unset only if the wait failed).
__device__ __forceinline__ float4 poll4(const float4* p, const Poll& w) {
    const float4 v = ld_relaxed4(p);
    return unset4(v) ? poll4_wait(p, w) : v;
}

// Announce this CTA's stores of an exchanged vector: after every consumer
// thread issued its stores, one relaxed add to the vector's counter.
__device__ __forceinline__ void xch_publish(unsigned* ctr) {
    consumer_sync();
    if (threadIdx.x == 0) asm volatile("red.relaxed.gpu.global.add.u32 [%0], 1;" ::"l"(ctr) : "memory");
}
// Thread 0's half of xch_wait.
static __device__ __noinline__ void xch_wait_thread(const unsigned* ctr, unsigned n, const Poll& w) {
    uint64_t t0 = 0;
    for (unsigned k = 0;; ++k) {
        unsigned v;
        asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
        if (v - kUnset >= n) return;  // the counter started at kUnset
        __nanosleep(32);
        if ((k & 15) == 15) {
            if (*w.abort || (w.err && (*reinterpret_cast<volatile int*>(w.err) & kErrTimeout))) {
                *w.abort = 1;
                return;
            }
            const uint64_t t = globaltimer_ns();
            if (!t0) t0 = t;
            else if (t - t0 > w.limit_ns) {
                if (w.err) atomicOr(w.err, kErrTimeout);
                *w.abort = 1;
                return;
            }
        }
    }
}
// Wait until n producer CTAs have announced their stores to the vector of
// counter ctr (thread 0 polls; the other consumer threads wait at the
// barrier).  False, for every consumer thread alike, if the wait ran out or
// the launch is aborting.
__device__ __forceinline__ bool xch_wait(const unsigned* ctr, unsigned n, const Poll& w) {
    if (threadIdx.x == 0) xch_wait_thread(ctr, n, w);
    return !consumer_sync_or(*w.abort);
}

// ---- one projection as seen by one CTA ---------------------------------------
struct Proj {
    const unsigned char* W;  // [rows][K] weights (gate/up: 2N rows)
    const float* wscale;     // FP8 per-row scales
    float* y;                // output (or the residual stream for kEpiResid)
    int N, K;                // outputs, inner dimension
    int rs;                  // rows per ring stage
    int wpr;                 // column segments per row
    int fp8;                 // weights are E4M3 (else bf16)
    int swiglu;              // rows [0,N) gate, [N,2N) up
    int r0, r1;              // this CTA's output rows [r0, r1) (proj_split_rows)
};

// Output rows of this CTA: an even split of N over the grid.
__device__ __forceinline__ void proj_split_rows(Proj& j) {
    j.r0 = (int)((long long)blockIdx.x * j.N / gridDim.x);
    j.r1 = (int)((long long)(blockIdx.x + 1) * j.N / gridDim.x);
}

// Hides v's value from the optimiser: what is derived from it is computed
// where it is used instead of being hoisted out of loops and kept in registers.
__device__ __forceinline__ int opaque(int v) {
    asm volatile("" : "+r"(v));
    return v;
}
__device__ __forceinline__ unsigned char* opaque_ptr(unsigned char* v) {
    asm volatile("" : "+l"(v));
    return v;
}

// log2 of a power of two.  The stage geometry's row counts (rs, and so the
// output rows per stage) and segments per row (wpr) are powers of two, so
// the per-phase set-up divides by shifting: a run-time integer division
// costs tens of instructions (64-bit ones a subroutine call), paid by every
// consumer thread at the start of every phase.
__device__ __forceinline__ int ilog2(int x) { return 31 - __clz(x); }

__device__ __forceinline__ int proj_cpr(const Proj& j) { return j.K / (j.fp8 ? 16 : 8); }
__device__ __forceinline__ int proj_opst(const Proj& j) { return j.swiglu ? j.rs / 2 : j.rs; }
__device__ __forceinline__ void proj_rows(const Proj& j, int& r0, int& r1) {
    r0 = j.r0;
    r1 = j.r1;
}
__device__ __forceinline__ int proj_stages(const Proj& j) {
    int r0, r1;
    proj_rows(j, r0, r1);
    const int opst = proj_opst(j);
    return (r1 - r0 + opst - 1) >> ilog2(opst);
}

// Ring of shared-memory stages; `it` counts stages since the ring was set up
// (producer and consumers each keep their own copy, in step).
struct Ring {
    uint64_t* full;
    uint64_t* empty;
    unsigned char* buf;
    uint32_t slot_bytes;
    int ns;
    uint32_t ns_magic;  // ring_magic(ns)
};

// floor(2^32 / ns) + 1 for a ring of ns >= 2 slots (every ring here has at
// least two): it / ns = __umulhi(it, ring_magic(ns)) exactly for every
// it < 2^32 / ns (the error term stays below 1 / ns; division by an
// invariant integer through a multiply-high, as in Granlund and Montgomery,
// "Division by invariant integers using multiplication", PLDI 1994), which
// saves the consumers a run-time division at every phase start.
__host__ __device__ inline uint32_t ring_magic(int ns) { return 0xffffffffu / (uint32_t)ns + 1u; }
// Slot and phase parity of ring stage `it`.
__device__ __forceinline__ void ring_pos(const Ring& r, int it, int& slot, uint32_t& phase) {
    const uint32_t q = __umulhi((uint32_t)it, r.ns_magic);
    slot = it - (int)q * r.ns;
    phase = q & 1u;
}

__device__ __forceinline__ void ring_init(const Ring& r) {
    for (int s = 0; s < r.ns; ++s) {
        mbar_init(&r.full[s], 1);
        mbar_init(&r.empty[s], kConsumerWarps);
    }
    fence_mbar_init();
}

// Producer (one thread): copy stage s of projection j into the next ring slot
// (advancing it).  Returns false (and sets *abort) if a wait ran out.
__device__ __forceinline__ bool produce_stage(const Proj& j, int s, const Ring& ring, int& it, uint64_t pol,
                                              volatile int* abort, int* err, unsigned long long* wait_ns = nullptr,
                                              unsigned long long* stage_tr = nullptr, int stage_tr_n = 0) {
    int r0, r1;
    proj_rows(j, r0, r1);
    const size_t rowb = (size_t)proj_cpr(j) * 16;
    const int opst = proj_opst(j);
    int slot;
    uint32_t ph;
    ring_pos(ring, it, slot, ph);
    const uint64_t tw = wait_ns ? globaltimer_ns() : 0;
    const bool got = mbar_wait_or_abort(&ring.empty[slot], ph ^ 1, abort);
    if (wait_ns) *wait_ns += globaltimer_ns() - tw;
    if (!got) {
        if (err) atomicOr(err, kErrTimeout);
        *abort = 1;
        return false;
    }
    const int o0 = r0 + s * opst;
    const int no = min(opst, r1 - o0);
    unsigned char* dst = ring.buf + (size_t)slot * ring.slot_bytes;
    if (stage_tr && it < stage_tr_n) stage_tr[4 * it] = globaltimer_ns();
    if (j.swiglu) {
        mbar_arrive_expect_tx(&ring.full[slot], (uint32_t)(2 * no * rowb));
        bulk_g2s(dst, j.W + (size_t)o0 * rowb, (uint32_t)(no * rowb), &ring.full[slot], pol);
        bulk_g2s(dst + (size_t)opst * rowb, j.W + ((size_t)j.N + o0) * rowb, (uint32_t)(no * rowb),
                 &ring.full[slot], pol);
    } else {
        mbar_arrive_expect_tx(&ring.full[slot], (uint32_t)(no * rowb));
        bulk_g2s(dst, j.W + (size_t)o0 * rowb, (uint32_t)(no * rowb), &ring.full[slot], pol);
    }
    ++it;
    return true;
}

// Producer (one thread): stream projection j's rows of this CTA into the ring.
// Returns false (and sets *abort) if a wait ran out.
__device__ __forceinline__ bool produce(const Proj& j, const Ring& ring, int& it, uint64_t pol,
                                        volatile int* abort, int* err) {
    int r0, r1;
    proj_rows(j, r0, r1);
    const size_t rowb = (size_t)proj_cpr(j) * 16;
    const int opst = proj_opst(j);
    const int nst = (r1 - r0 + opst - 1) >> ilog2(opst);
    for (int s = 0; s < nst; ++s, ++it) {
        int slot;
        uint32_t ph;
        ring_pos(ring, it, slot, ph);
        if (!mbar_wait_or_abort(&ring.empty[slot], ph ^ 1, abort)) {
            if (err) atomicOr(err, kErrTimeout);
            *abort = 1;
            return false;
        }
        const int o0 = r0 + s * opst;
        const int no = min(opst, r1 - o0);
        unsigned char* dst = ring.buf + (size_t)slot * ring.slot_bytes;
        if (j.swiglu) {
            mbar_arrive_expect_tx(&ring.full[slot], (uint32_t)(2 * no * rowb));
            bulk_g2s(dst, j.W + (size_t)o0 * rowb, (uint32_t)(no * rowb), &ring.full[slot], pol);
            bulk_g2s(dst + (size_t)opst * rowb, j.W + ((size_t)j.N + o0) * rowb, (uint32_t)(no * rowb),
                     &ring.full[slot], pol);
        } else {
            mbar_arrive_expect_tx(&ring.full[slot], (uint32_t)(no * rowb));
            bulk_g2s(dst, j.W + (size_t)o0 * rowb, (uint32_t)(no * rowb), &ring.full[slot], pol);
        }
    }
    return true;
}

// Producer after an abort: wait (bounded) for the copies still in flight.
__device__ __forceinline__ void drain(const Ring& ring, int it) {
    for (int i = it > ring.ns ? it - ring.ns : 0; i < it; ++i) {
        int slot;
        uint32_t ph;
        ring_pos(ring, i, slot, ph);
        mbar_wait(&ring.full[slot], ph);
    }
}

// Stage the activation vector for a projection with inner dimension K:
//   x (fp32, global, written by other CTAs: read through L2) -> optional
//   RMSNorm with gain gamma -> shared memory, fp32 planes (bf16 weights) or,
//   with FP8 weights, per-token E4M3 quantisation with scale amax/448 stored
//   as E4M3 bytes in order.  Returns the activation scale (1 for bf16).
//   Consumers only.
template <bool FP8, bool RMS>
__device__ __forceinline__ float stage_x(const float* x, const __nv_bfloat16* gamma, int K, float eps,
                                         unsigned char* xs, float* red) {
    const int cpr = K / (FP8 ? 16 : 8);
    const float4* x4 = reinterpret_cast<const float4*>(x);
    float scale_in = 1.0f;
    if constexpr (RMS) {
        float ss = 0.f;
        for (int i = threadIdx.x; i < K / 4; i += kConsumers) {
            const float4 v = __ldcg(x4 + i);
            ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
        }
        ss = consumer_sum(ss, red);
        scale_in = 1.0f / sqrtf(ss / (float)K + eps);
    }
    auto load = [&](int i) {
        float4 v = __ldcg(x4 + i);
        if constexpr (RMS) {
            const uint2 g = *reinterpret_cast<const uint2*>(gamma + 4 * i);
            v.x = v.x * scale_in * bf16lo(g.x);
            v.y = v.y * scale_in * bf16hi(g.x);
            v.z = v.z * scale_in * bf16lo(g.y);
            v.w = v.w * scale_in * bf16hi(g.y);
        }
        return v;
    };
    float sa = 1.0f;
    if constexpr (!FP8) {
        float4* xs4 = reinterpret_cast<float4*>(xs);
        for (int i = threadIdx.x; i < K / 4; i += kConsumers) {
            const int e = 4 * i;  // chunk e/8, plane (e%8)/4
            xs4[((e & 7) >> 2) * cpr + (e >> 3)] = load(i);
        }
    } else {
        // normalise, amax, then quantise (the normalised values are recomputed)
        float amax = 0.f;
        for (int i = threadIdx.x; i < K / 4; i += kConsumers) {
            const float4 v = load(i);
            amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
        }
        amax = consumer_max(amax, red);
        sa = __fdiv_rn(fmaxf(amax, 1e-12f), 448.0f);
        const float rsa = __frcp_rn(sa);
        uint32_t* xs4 = reinterpret_cast<uint32_t*>(xs);  // E4M3 bytes, in order
        for (int i = threadIdx.x; i < K / 4; i += kConsumers) {
            const float4 v = load(i);
            xs4[i] = e4m3x4_div(v, sa, rsa);
        }
    }
    consumer_sync();
    return sa;
}

// ---- activation segments in registers -----------------------------------------
// A consumer warp's column segment [c0, c1) of a projection is the same in
// every stage, so with bf16 weights each lane keeps the activations of its
// chunks c0 + lane + 32 i (at most kMaxLaneChunks) in registers, two fp32
// planes per chunk.  E4M3 weights (tensor cores) read their activation chunks
// from the staged bytes in shared memory instead.
template <bool FP8>
struct XSeg {
    static constexpr int kChunks = kMaxLaneChunks;
    float4 a[kChunks], b[kChunks];  // elements 0-3 and 4-7 of each 8-weight chunk
};
template <>
struct XSeg<true> {
    const unsigned char* xs;  // E4M3 activation bytes in shared memory (read per MMA pair)
};

// This warp's segment of projection j.
__device__ __forceinline__ void proj_segment(const Proj& j, int warp, int& rslot, int& sg, int& c0, int& c1) {
    const int CPR = proj_cpr(j), lw = ilog2(j.wpr);
    rslot = warp >> lw;
    sg = warp & (j.wpr - 1);
    c0 = (sg * CPR) >> lw;
    c1 = ((sg + 1) * CPR) >> lw;
}

// Segment from the shared memory written by stage_x: fp32 planes for bf16
// weights, E4M3 bytes for FP8 (in the order the lane's MMAs consume them).
template <bool FP8>
__device__ __forceinline__ void load_xseg_smem(const unsigned char* xs, int CPR, int c0, int c1, XSeg<FP8>& x) {
    const int lane = threadIdx.x & 31;
    if constexpr (!FP8) {
#pragma unroll
        for (int i = 0; i < XSeg<FP8>::kChunks; ++i) {
            const int c = c0 + lane + 32 * i;
            x.a[i] = c < c1 ? reinterpret_cast<const float4*>(xs)[c] : float4{};
            x.b[i] = c < c1 ? reinterpret_cast<const float4*>(xs)[CPR + c] : float4{};
        }
    } else {
        x.xs = xs;
    }
}

// A plain (un-normalised) fp32 activation vector for bf16 weights: the lane's
// segment straight from global memory (through L2: other CTAs wrote it) into
// registers, all loads in flight at once.  Needs no shared staging and no
// block barrier.  Same values and layout as load_xseg_smem after stage_x.
// With a Poll, x is an exchanged vector: elements still kUnset are re-read
// until written (all loads are first issued together); a failed wait sets
// *w->abort.
__device__ __forceinline__ void load_xseg_plain(const float* x, int c0, int c1, XSeg<false>& xr,
                                                const Poll* w = nullptr) {
    const int lane = threadIdx.x & 31;
    const float4* x4 = reinterpret_cast<const float4*>(x);
#pragma unroll
    for (int i = 0; i < kMaxLaneChunks; ++i) {
        const int c = c0 + lane + 32 * i;
        xr.a[i] = c < c1 ? ld_relaxed4(x4 + 2 * c) : float4{};
        xr.b[i] = c < c1 ? ld_relaxed4(x4 + 2 * c + 1) : float4{};
    }
    if (!w) return;
#pragma unroll
    for (int i = 0; i < kMaxLaneChunks; ++i) {
        const int c = c0 + lane + 32 * i;
        if (c < c1) {
            if (unset4(xr.a[i])) xr.a[i] = poll4_wait(x4 + 2 * c, *w);
            if (unset4(xr.b[i])) xr.b[i] = poll4_wait(x4 + 2 * c + 1, *w);
        }
    }
}

// Stage an exchanged activation vector (see "data exchange" above) for a
// projection with inner dimension K into the shared layout of stage_x,
// waiting for its elements:
//   RMS:   x = h * r * gamma, r = 1/sqrt(sum(h^2)/K + eps)   (K <= kMaxRmsK)
//   FP8:   sa = max(amax, 1e-12)/448, amax over the (normalised) values (for
//          RMS inputs r * max |h * gamma|, reduced with the sum), or the
//          site's static scale when one is set; x8 = e4m3(x/sa) as bytes
// (plain bf16 inputs are not staged: the stage loop reads them itself).
// Every thread waits for its own elements, then the CTA reduces the
// statistics in a fixed order.  Plain FP8 inputs go through xf, an fp32
// scratch of K floats in shared memory, filled by asynchronous copies.
// Returns sa (1 for bf16), or -1 if a wait ran out (every consumer thread
// returns, having passed the same barriers).
template <bool FP8, bool RMS>
__device__ float stage_x_xch(const float* x, const __nv_bfloat16* gamma, int K, float eps, const float* sa_static,
                             float* calib, unsigned char* xs, float* xf, float* red, const Poll& w) {
    const int cpr = K / (FP8 ? 16 : 8);
    const float4* x4 = reinterpret_cast<const float4*>(x);
    const int n4 = K / 4;
    if (FP8 && sa_static) prefetch_l1(sa_static);
    float sa = 1.0f;
    if constexpr (RMS) {
        constexpr int kB = kMaxRmsK / 4 / kConsumers;
        float4 v[kB];
        uint2 g[kB];
#pragma unroll
        for (int k = 0; k < kB; ++k) {
            const int i = threadIdx.x + k * kConsumers;
            if (i < n4) {
                v[k] = ld_relaxed4(x4 + i);
                g[k] = *reinterpret_cast<const uint2*>(gamma + 4 * i);
            }
        }
        // sum of squares and (FP8) max |h * gamma| in one reduction: the
        // normalised amax is r * max |h * gamma| (r > 0)
        float ss = 0.f, am = 0.f;
#pragma unroll
        for (int k = 0; k < kB; ++k) {
            const int i = threadIdx.x + k * kConsumers;
            if (i < n4) {
                if (unset4(v[k])) v[k] = poll4_wait(x4 + i, w);
                ss += v[k].x * v[k].x + v[k].y * v[k].y + v[k].z * v[k].z + v[k].w * v[k].w;
                if constexpr (FP8)
                    am = fmaxf(fmaxf(am, fmaxf(fabsf(v[k].x * bf16lo(g[k].x)), fabsf(v[k].y * bf16hi(g[k].x)))),
                               fmaxf(fabsf(v[k].z * bf16lo(g[k].y)), fabsf(v[k].w * bf16hi(g[k].y))));
            }
        }
        consumer_sum_max(ss, am, red);
        const float r = rsqrtf(ss * __frcp_rn((float)K) + eps);
#pragma unroll
        for (int k = 0; k < kB; ++k) {
            v[k].x *= r * bf16lo(g[k].x);
            v[k].y *= r * bf16hi(g[k].x);
            v[k].z *= r * bf16lo(g[k].y);
            v[k].w *= r * bf16hi(g[k].y);
        }
        if constexpr (FP8) {
            am *= r;
            sa = __fdiv_rn(fmaxf(am, 1e-12f), 448.0f);
            // non-negative floats order like their bit patterns
            if (calib && threadIdx.x == 0) atomicMax(reinterpret_cast<int*>(calib), __float_as_int(am));
            if (sa_static) {
                const float ss_ = *sa_static;
                if (ss_ > 0.f) sa = ss_;  // static: values beyond 448 * sa saturate
            }
        }
        const float rsa = __frcp_rn(sa);  // x / sa by div_rn_by: one division per CTA, not per element
#pragma unroll
        for (int k = 0; k < kB; ++k) {
            const int i = threadIdx.x + k * kConsumers;
            if (i < n4) {
                const int e = 4 * i;
                if constexpr (!FP8) {
                    reinterpret_cast<float4*>(xs)[((e & 7) >> 2) * cpr + (e >> 3)] = v[k];
                } else {
                    reinterpret_cast<uint32_t*>(xs)[i] =
                        e4m3x4_div(v[k], sa, rsa);
                }
            }
        }
    } else {
        static_assert(FP8, "plain bf16 inputs are read by the stage loop");
        // the whole vector into xf at once, then the elements still unset re-read
        for (int i = threadIdx.x; i < n4; i += kConsumers) cp_async16(xf + 4 * i, x4 + i);
        cp_async_wait_all();
        float am = 0.f;
        for (int i = threadIdx.x; i < n4; i += kConsumers) {
            float4 v = reinterpret_cast<const float4*>(xf)[i];
            if (unset4(v)) {
                v = poll4_wait(x4 + i, w);
                reinterpret_cast<float4*>(xf)[i] = v;
            }
            am = fmaxf(am, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
        }
        float unused = 0.f;
        consumer_sum_max(unused, am, red);
        sa = __fdiv_rn(fmaxf(am, 1e-12f), 448.0f);
        if (calib && threadIdx.x == 0) atomicMax(reinterpret_cast<int*>(calib), __float_as_int(am));
        if (sa_static) {
            const float ss_ = *sa_static;
            if (ss_ > 0.f) sa = ss_;
        }
        const float rsa = __frcp_rn(sa);
        for (int i = threadIdx.x; i < n4; i += kConsumers) {
            const float4 v = reinterpret_cast<const float4*>(xf)[i];
            reinterpret_cast<uint32_t*>(xs)[i] =
                e4m3x4_div(v, sa, rsa);
        }
    }
    return consumer_sync_or(*w.abort) ? -1.0f : sa;
}

// Where the persistent step's epilogue puts its outputs (both optional).
struct EpiOut {
    float* rows;  // kEpiResid: shared-memory copy of this CTA's rows of y (read and updated
                  //   instead of global memory), or null
    float* xout;  // the exchange buffer of y: every output stored there for the next phase
                  //   (y itself is then written only by kEpiResid, the residual stream kept
                  //   for the host)
};

// The tensor-core FP8 stage loop's per-lane constants for one projection (the
// same in every stage: worked out once, outside the stage loop).  A stage
// holds `rs` rows (a power of two, 2..16; SwiGLU: rs / 2 gate rows, then their
// rs / 2 up rows) of cpr 16-byte chunks; P = 16 / rs subranges of cpr / P
// chunks per row.  Lane (g, q) of warp w works on subrange kap = g / (8 / P)
// and on rows ra = g mod (8 / P) and rb = ra + rs / 2, which it feeds as MMA
// rows g and g + 8; subrange kap's piece of warp w is its units
// [w u / 8, (w + 1) u / 8) of u = cpr / (4 P) units of 4 chunks.
struct Fp8Lane {
    int a_off, b_off;   // byte offset, within a stage, of this lane's first chunk of rows ra and rb
    int x_off;          // byte offset of its first activation chunk
    int a_out, b_out;   // output rows of ra and rb within a stage (an up row maps to its gate row)
    int a_part, b_part; // their partial-sum slots: r * wpr + w P + kap
    int nu;             // 4-chunk units of this warp's piece
    int odd;            // g & 1
};
__device__ __forceinline__ Fp8Lane fp8_lane(int cpr, size_t rowb, int rs, int opst, int wpr) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
    const int lr = ilog2(rs);                         // rs = 2^lr, 2 <= rs <= kFp8MmaRows = 16
    const int P = kFp8MmaRows >> lr, gpr = rs >> 1;   // subranges per row, lane groups per subrange
    const int kap = g >> (lr - 1), ra = g & (gpr - 1), rb = ra + gpr;
    const int ls = cpr >> (4 - lr), units = ls / 4;   // chunks and 4-chunk units per subrange
    const int u0 = warp * units / kConsumerWarps;
    const int c0 = kap * ls + 4 * u0 + q;         // this lane's first chunk
    Fp8Lane L;
    L.a_off = (int)(ra * rowb) + 16 * c0;
    L.b_off = (int)(rb * rowb) + 16 * c0;
    L.x_off = 16 * c0;
    L.a_out = ra < opst ? ra : ra - opst;
    L.b_out = rb < opst ? rb : rb - opst;
    L.a_part = ra * wpr + warp * P + kap;
    L.b_part = rb * wpr + warp * P + kap;
    L.nu = (warp + 1) * units / kConsumerWarps - u0;
    L.odd = g & 1;
    return L;
}

// One ring stage of E4M3 rows on the tensor cores (lane constants from
// fp8_lane).  Per 128-byte group (8 chunks) of a lane's piece, lanes of even g
// take chunks q and 4 + q in that order, lanes of odd g the other way round
// (conflict-free 16-byte loads); a trailing unit of 4 chunks takes chunk q.
// Each lane's activation chunk is the one matching its row chunk, so
// D[m][m mod 8] is MMA row m's partial sum.  The four MMAs of a group go to
// four accumulators, added in a fixed order.  A row is fed as zeros unless its
// output row is below `nv`.  Writes the partial sums of the valid rows into
// part (this stage's slots).
__device__ __forceinline__ void fp8_stage(const unsigned char* sbuf, const Fp8Lane& L, int nv,
                                          const unsigned char* xs, float* part) {
    const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
    const bool va = L.a_out < nv, vb = L.b_out < nv;
    const unsigned char* pa = sbuf + L.a_off;
    const unsigned char* pb = sbuf + L.b_off;
    const unsigned char* px = xs + L.x_off;
    const int off0 = 64 * L.odd, off1 = 64 * (L.odd ^ 1);  // the two halves of a group, odd rows swapped
    const int groups = L.nu >> 1;
    float d[4][4] = {};
#pragma unroll 2
    for (int t = 0; t < groups; ++t) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int off = 128 * t + (h ? off1 : off0);
            const uint4 wa = va ? *reinterpret_cast<const uint4*>(pa + off) : uint4{};
            const uint4 wb = vb ? *reinterpret_cast<const uint4*>(pb + off) : uint4{};
            const uint4 x = *reinterpret_cast<const uint4*>(px + off);
            mma_e4m3(d[2 * h], wa.x, wb.x, wa.y, wb.y, x.x, x.y);
            mma_e4m3(d[2 * h + 1], wa.z, wb.z, wa.w, wb.w, x.z, x.w);
        }
    }
    if (L.nu & 1) {  // trailing unit: chunk q of every lane's 4
        const int off = 128 * groups;
        const uint4 wa = va ? *reinterpret_cast<const uint4*>(pa + off) : uint4{};
        const uint4 wb = vb ? *reinterpret_cast<const uint4*>(pb + off) : uint4{};
        const uint4 x = *reinterpret_cast<const uint4*>(px + off);
        mma_e4m3(d[0], wa.x, wb.x, wa.y, wb.y, x.x, x.y);
        mma_e4m3(d[1], wa.z, wb.z, wa.w, wb.w, x.z, x.w);
    }
    // D[g][g] sits in lane (g, g / 2) as element g & 1, D[g + 8][g] as element
    // 2 + (g & 1) (selects, not an index: a lane-dependent index would put d
    // in local memory)
    if (q == (g >> 1)) {
        float sa_[4], sb_[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            sa_[k] = L.odd ? d[k][1] : d[k][0];
            sb_[k] = L.odd ? d[k][3] : d[k][2];
        }
        if (va) part[L.a_part] = (sa_[0] + sa_[1]) + (sa_[2] + sa_[3]);
        if (vb) part[L.b_part] = (sb_[0] + sb_[1]) + (sb_[2] + sb_[3]);
    }
}

// Consumers: reduce projection j's stages from the ring against the lane's
// activation registers, then apply the epilogue to this CTA's outputs.
// `part` holds proj_stages(j) * rs * wpr floats.  Returns false if a wait ran
// out or the launch is aborting (every consumer thread alike).
template <bool FP8, int EPI>
__device__ __forceinline__ bool consume(const Proj& j, const Ring& ring, int& it, const XSeg<FP8>& xr, float sa,
                                        float* part, volatile int* abort, int* err,
                                        unsigned long long* wait_ns = nullptr, const EpiOut* so = nullptr,
                                        unsigned long long* stage_tr = nullptr, int stage_tr_n = 0) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int r0, r1;
    proj_rows(j, r0, r1);
    const int nrows = r1 - r0;
    const int CPR = proj_cpr(j), RS = j.rs, WPR = j.wpr, SLOTS = kConsumerWarps >> ilog2(WPR),
              NP = RS >> ilog2(SLOTS);
    const size_t rowb = (size_t)CPR * 16;
    const int opst = proj_opst(j), lo = ilog2(opst);
    const int nst = (nrows + opst - 1) >> lo;
    int rslot, sg, c0, c1;
    proj_segment(j, warp, rslot, sg, c0, c1);
    Fp8Lane fl{};
    if constexpr (FP8) fl = fp8_lane(CPR, rowb, RS, opst, WPR);
    // FP8: the epilogue's per-row weight scales are pulled into L1 now, so
    // that its loads hit L1 instead of waiting for L2 behind the weight
    // stream; a prefetch holds no register, so nothing waits for it
    if constexpr (FP8) {
        if (threadIdx.x < nrows) {
            prefetch_l1(j.wscale + r0 + threadIdx.x);
            if (EPI == kEpiSwiglu) prefetch_l1(j.wscale + j.N + r0 + threadIdx.x);
        }
    }

    bool ok = true;
    unsigned long long waited = 0;  // ns spent waiting for data (traced runs; stored once at the end)
    int slot;                       // ring slot and phase of stage `it`, advanced per stage
    uint32_t phase;
    ring_pos(ring, it, slot, phase);
    for (int s = 0; s < nst; ++s, ++it) {
        const bool timed = wait_ns && threadIdx.x == 0;  // traced runs: thread 0 times its data waits
        const uint64_t tw = timed ? globaltimer_ns() : 0;
        // the warp stops as one: a lane that gave up stops its neighbours too
        const bool got = __all_sync(0xffffffffu, mbar_wait_or_abort(&ring.full[slot], phase, abort));
        if (timed) waited += globaltimer_ns() - tw;
        if (!got) {
            if (lane == 0 && err) atomicOr(err, kErrTimeout);
            *abort = 1;
            ok = false;
            break;
        }
        const long long clk0 = stage_tr ? clock64() : 0;
        unsigned long long* str = nullptr;  // traced warps: 0 (first row of the trace), the last (second row)
        if (stage_tr && lane == 0 && it < stage_tr_n && (warp == 0 || warp == kConsumerWarps - 1))
            str = stage_tr + (warp == 0 ? 0 : stage_tr_n * 4) + 4 * it;
        if (str) str[1] = globaltimer_ns();
        const unsigned char* sbuf = ring.buf + (size_t)slot * ring.slot_bytes;
        if constexpr (FP8) {
            fp8_stage(sbuf, fl, nrows - s * opst, xr.xs, part + (size_t)s * RS * WPR);
        } else {
            for (int ps = 0; ps < NP; ++ps) {
                const int r = ps * SLOTS + rslot;          // row of the stage
                const int orow = r & (opst - 1);           // its output row within the stage (gate row for up)
                if (s * opst + orow < nrows) {
                    const uint4* wrow = reinterpret_cast<const uint4*>(sbuf + r * rowb);
                    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int i = 0; i < XSeg<FP8>::kChunks; ++i) {
                        const int c = c0 + lane + 32 * i;
                        if (c < c1) dot_bf16(wrow[c], xr.a[i], xr.b[i], acc[2 * (i & 1)], acc[2 * (i & 1) + 1]);
                    }
                    const float v = warp_sum((acc[0] + acc[1]) + (acc[2] + acc[3]));
                    if (lane == 0) part[(s * RS + r) * WPR + sg] = v;
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&ring.empty[slot]);
        if (str) {
            str[2] = globaltimer_ns();
            str[3] = (unsigned long long)(clock64() - clk0);  // SM cycles of this stage
        }
        if (++slot == ring.ns) {
            slot = 0;
            phase ^= 1;
        }
    }
    if (wait_ns && threadIdx.x == 0) *wait_ns += waited;
    if (consumer_sync_or(!ok || *abort)) return false;

    // per-row sums over segments (in segment order) and the epilogue
    for (int r = threadIdx.x; r < nrows; r += kConsumers) {
        const int n = r0 + r;
        const int s = r >> lo, jj = r & (opst - 1);
        auto row_sum = [&](int rs_) {
            const float* pr = part + (s * RS + rs_) * WPR;
            float acc = 0.f;
            for (int q = 0; q < WPR; ++q) acc += pr[q];
            return acc;
        };
        if constexpr (EPI == kEpiSwiglu) {
            float g = row_sum(jj), u = row_sum(RS / 2 + jj);
            float m;
            if constexpr (FP8) {
                g = round_bf16(g * (sa * j.wscale[n]));
                u = round_bf16(u * (sa * j.wscale[j.N + n]));
                m = round_bf16(silu(g) * u);
            } else {
                m = silu(g) * u;
            }
            if (so && so->xout) st_relaxed(so->xout + n, m);
            else j.y[n] = m;
        } else {
            float o = row_sum(jj);
            if constexpr (FP8) o = round_bf16(o * (sa * j.wscale[n]));
            if constexpr (EPI == kEpiResid) {
                if (so && so->rows) {
                    o = so->rows[r] + o;
                    so->rows[r] = o;
                } else {
                    o = __ldcg(j.y + n) + o;
                }
            }
            if (so && so->xout) {
                st_relaxed(so->xout + n, o);
                if constexpr (EPI == kEpiResid) j.y[n] = o;
            } else {
                j.y[n] = o;
            }
        }
    }
    return true;
}

// load_xseg_smem + consume.  consume_call is the separate (not inlined)
// function: its registers are allocated on their own, so the state the caller
// keeps across phases cannot push the bf16 stage loop's activation registers
// (up to 20 float4 per lane) into local memory.  The FP8 loop keeps only a
// pointer to its activation bytes; there the call's register save and restore
// cost more than they protect (FP8 1.65 -> 1.54 ms/frame inlined, while bf16
// inlined spilled and lost), so proj_phase inlines consume_body for FP8.
// Returns the advanced stage counter, or -1 if a wait ran out.
// `xplain`: bf16 weights only, a plain activation vector read from global
// memory directly (then xs is not used); else the shared planes in xs.
template <bool FP8, int EPI>
__device__ __forceinline__ int consume_body(const Proj& j, const Ring& ring, int it, const unsigned char* xs, float sa,
                                            float* part, volatile int* abort, int* err, unsigned long long* wait_ns,
                                            const EpiOut* so, unsigned long long* stage_tr, int stage_tr_n,
                                            const float* xplain, const Poll* poll) {
    int rslot, sg, c0, c1;
    proj_segment(j, threadIdx.x >> 5, rslot, sg, c0, c1);
    XSeg<FP8> xr;
    if constexpr (!FP8) {
        // a failed wait sets *abort: the stage loop then stops, all threads alike
        if (xplain) load_xseg_plain(xplain, c0, c1, xr, poll);
        else load_xseg_smem<false>(xs, proj_cpr(j), c0, c1, xr);
    } else {
        load_xseg_smem<true>(xs, proj_cpr(j), c0, c1, xr);
    }
    return consume<FP8, EPI>(j, ring, it, xr, sa, part, abort, err, wait_ns, so, stage_tr, stage_tr_n) ? it : -1;
}
template <bool FP8, int EPI>
__device__ __noinline__ int consume_call(const Proj j, const Ring ring, int it, const unsigned char* xs, float sa,
                                        float* part, volatile int* abort, int* err, unsigned long long* wait_ns,
                                        const EpiOut* so, unsigned long long* stage_tr, int stage_tr_n,
                                        const float* xplain = nullptr, const Poll* poll = nullptr) {
    return consume_body<FP8, EPI>(j, ring, it, xs, sa, part, abort, err, wait_ns, so, stage_tr, stage_tr_n, xplain,
                                  poll);
}
// The stage loop and epilogue as proj_phase runs them: inlined for FP8, a
// call for bf16 (see above).
template <bool FP8, int EPI>
__device__ __forceinline__ int consume_phase(const Proj& j, const Ring& ring, int it, const unsigned char* xs,
                                             float sa, float* part, volatile int* abort, int* err,
                                             unsigned long long* wait_ns, const EpiOut* so,
                                             unsigned long long* stage_tr, int stage_tr_n,
                                             const float* xplain = nullptr, const Poll* poll = nullptr) {
    if constexpr (FP8)
        return consume_body<FP8, EPI>(j, ring, it, xs, sa, part, abort, err, wait_ns, so, stage_tr, stage_tr_n,
                                      xplain, poll);
    else
        return consume_call<FP8, EPI>(j, ring, it, xs, sa, part, abort, err, wait_ns, so, stage_tr, stage_tr_n,
                                      xplain, poll);
}

// Philox4x32-10 counter-based generator (Salmon, Moraes, Dror and Shaw,
// "Parallel random numbers: as easy as 1, 2, 3", SC'11): ten rounds of the
// 4 x 32-bit Philox S-box, the key bumped by the Weyl increments each round.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
        const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
        c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return c;
}

// Temperature sampling for codebook k at frame t, one warp ("Higgs Audio v3
// TTS-4B on FlashRT", section 4 sampling policy: stable softmax and a
// stateless categorical draw keyed by the request seed).  u in [0, 1) is the
// top 24 bits of the first Philox word for counter (t, k, 0, 0) and key seed;
// the code is the first v whose running sum of exp((x_v - max) / T) exceeds
// u times the total.  Lane l sums the contiguous chunk [l c, (l+1) c) of the
// V logits (c = ceil(V / 32)), a warp scan orders the chunks, and the lane
// holding the crossing walks its chunk.  Returns the code in every lane.
__device__ __forceinline__ int sample_codebook(const float* row, int V, float T, unsigned long long seed, int t,
                                               int k) {
    const int lane = threadIdx.x & 31;
    const int c = (V + 31) / 32;
    const int v0 = min(V, lane * c), v1 = min(V, v0 + c);
    float mx = -INFINITY;
    for (int v = v0; v < v1; ++v) mx = fmaxf(mx, __ldcg(row + v));
    mx = warp_max(mx);
    const float invT = 1.0f / T;
    float sum = 0.f;
    for (int v = v0; v < v1; ++v) sum += expf((__ldcg(row + v) - mx) * invT);
    float incl = sum;  // inclusive scan over lanes
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    const float total = __shfl_sync(0xffffffffu, incl, 31);
    const uint4 r = philox4x32_10(make_uint4((uint32_t)t, (uint32_t)k, 0u, 0u), (uint32_t)seed,
                                  (uint32_t)(seed >> 32));
    const float u = (float)(r.x >> 8) * (1.0f / 16777216.0f);
    const float target = u * total;
    const unsigned hit = __ballot_sync(0xffffffffu, incl > target);
    int code = -1;
    if (hit) {
        const int owner = __ffs(hit) - 1;
        if (lane == owner) {
            float run = incl - sum;
            for (int v = v0; v < v1; ++v) {
                const float e = expf((__ldcg(row + v) - mx) * invT);
                run += e;
                if (run > target) { code = v; break; }
                if (e > 0.f) code = v;  // rounding: the crossing is at the chunk's last weight
            }
        }
        code = __shfl_sync(0xffffffffu, code, owner);
    } else {
        // u * total rounded up to the total: the last code with a non-zero weight
        int last = -1;
        for (int v = v0; v < v1; ++v)
            if (expf((__ldcg(row + v) - mx) * invT) > 0.f) last = v;
        const unsigned has = __ballot_sync(0xffffffffu, last >= 0);
        code = has ? __shfl_sync(0xffffffffu, last, 31 - __clz(has)) : 0;
    }
    return code < 0 ? 0 : code;
}

// Codebook head, after every CTA stored its logits: the last CTA to arrive
// takes the per-codebook greedy argmax (ties: lowest code; or, with a positive
// temperature in the state, a sampled code: sample_codebook) under the delay
// mask (codebook k is BOS-pad before frame k and EOC from frame eoc + k on;
// "Higgs Audio v3 TTS-4B on FlashRT", section 4 sampling policy and section 5),
// records the codes (next step's input and the history ring) and advances the
// position and frame.  `counter` holds `base` before the first arrival and is
// put back to it.  Consumers only.
__device__ __forceinline__ void head_tail(const float* logits, int n_cb, int V, DevState* st, unsigned* counter,
                                          unsigned base, int* hist, int hist_cap, int* s_last, int* s_codes) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    consumer_sync();  // every thread's logits stores precede thread 0's release below
    if (threadIdx.x == 0) {
        unsigned old;  // acquire-release: the last CTA then sees every CTA's logits
        asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(counter) : "memory");
        *s_last = old - base == gridDim.x - 1;
    }
    consumer_sync();
    if (!*s_last) return;
    const int t = st->t, eoc = st->eoc;
    const float T = st->temperature;
    for (int k = warp; k < n_cb; k += kConsumerWarps) {
        if (T > 0.f) {
            const int c = sample_codebook(logits + (size_t)k * V, V, T, st->seed, t, k);
            if (lane == 0) s_codes[k] = t < k ? V - 2 : (eoc >= 0 && t >= eoc + k) ? V - 1 : c;
            continue;
        }
        float best = -INFINITY;
        int bi = 0x7fffffff;
        for (int v = lane; v < V; v += 32) {
            const float x = __ldcg(logits + (size_t)k * V + v);
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
            int c = bi;
            if (t < k) c = V - 2;
            else if (eoc >= 0 && t >= eoc + k) c = V - 1;
            s_codes[k] = c;
        }
    }
    consumer_sync();
    if (threadIdx.x == 0) {
        if (eoc < 0 && s_codes[0] == V - 1) st->eoc = t;
        int* hrow = hist + (size_t)(st->hist_idx % hist_cap) * n_cb;
        for (int k = 0; k < n_cb; ++k) {
            st->codes[k] = s_codes[k];
            hrow[k] = s_codes[k];
        }
        st->hist_idx += 1;
        st->t = t + 1;
        st->pos += 1;
        *counter = base;
    }
}

}  // namespace core
}  // namespace tts

// The whole decode step (or one prefill position) as one persistent kernel.
//
// One CTA per SM, all co-resident (cooperative launch).  The producer warp of
// each CTA streams, back to back, every weight range the CTA owns over the
// whole step -- QKV, O-proj, gate/up, down-proj of layer 0, then layer 1, ...,
// then the codebook head -- through its ring of shared-memory stages, never
// waiting on anything but free ring slots.  The eight consumer warps walk
// the phases of the step ("Higgs Audio v3 TTS-4B on FlashRT", section 5):
//
//   embed:   h = sum_k E_k[c_k] (this CTA's slice)
//   per layer l:
//     QKV:   x = RMSNorm(h) (+FP8 quant); qkv rows
//     attn:  per (kv head, split) unit: q/k RMSNorm + RoPE, bf16 KV write,
//            online-softmax attention over the split, last unit merges
//     O:     x = attn (+quant); h += W_o x
//     GU:    x = RMSNorm(h) (+quant); act = silu(gate) * up
//     down:  x = act (+quant); h += W_d x
//   head:    x = RMSNorm(h); logits; last CTA: greedy argmax under the delay
//            mask, codes, position and frame advance (prefill: advance only)
//
// There is no grid barrier: every vector a phase hands on (h, qkv, the
// attention output, the MLP activation) is stored into an exchange buffer of
// its own (one per layer and kind, all 0xffffffff at launch), each producing
// CTA then bumps the vector's arrival counter without a fence, and the next
// phase starts reading once the counter is complete, re-reading any element
// still unset (the data exchange in gemv_core.cuh).  No CTA waits for a
// fence or for the CTAs that do not feed it.  The producer never waits for the
// consumers of other CTAs: it
// keeps its ring full with the next phase's weights, so HBM streams through
// norms, attention and the waits.  Every wait is bounded (kWaitLimitNs) and
// stops early once any CTA has recorded a timeout; then the kernel records
// kErrTimeout, lets its in-flight copies land and returns.
#pragma once

#include "gemv_core.cuh"

namespace tts {

namespace {

using namespace core;

constexpr int kMaxHRows = 256;     // rows of h one CTA owns, at most
constexpr int kAttnMinChunk = 64;   // positions per attention split, at least (no merge below)

// The exchange buffers of StepParams::xch (layout: step_xch_words).
enum XchKind { kXQkv = 0, kXAttn, kXHo, kXAct, kXHd };  // qkv, attention output, h after attention / MLP, act

// Vector `kind` of layer l; l = -1: h after the embedding (any kind).
__device__ __forceinline__ float* xch_vec(const StepParams& p, int l, int kind) {
    if (l < 0) return p.xch;
    const int QKVR = (p.n_q + 2 * p.n_kv) * kHeadDim, A = p.n_q * kHeadDim;
    float* b = p.xch + p.hidden + (size_t)l * step_xch_layer_words(p.hidden, QKVR, A, p.inter);
    switch (kind) {
        case kXQkv: return b;
        case kXAttn: return b + QKVR;
        case kXHo: return b + QKVR + A;
        case kXAct: return b + QKVR + A + p.hidden;
        default: return b + QKVR + A + p.hidden + p.inter;
    }
}
// The last-arriver tickets: attention of (layer l, unit slot u) at
// l * n_q + u (u: the kv head, or the q head when a unit serves one q head),
// the head at n_layers * n_q.  Each starts the launch at kUnset.
__device__ __forceinline__ unsigned* xch_tickets(const StepParams& p) {
    return reinterpret_cast<unsigned*>(xch_vec(p, p.n_layers, kXQkv));
}
// The arrival counter of vector `kind` of layer l (l = -1: the embedding).
__device__ __forceinline__ unsigned* xch_counter(const StepParams& p, int l, int kind) {
    return xch_tickets(p) + p.n_layers * p.n_q + 1 + (l < 0 ? 0 : 1 + 5 * l + kind);
}
__device__ __forceinline__ Poll step_poll(const StepParams& p, volatile int* abort) {
    return Poll{&p.st->err, abort, p.wait_limit_ns ? p.wait_limit_ns : kWaitLimitNs};
}

constexpr int kAttnStep = 8;  // positions a warp scores at once

template <int G>
struct AttnSmem {
    float qs[G][kHeadDim];  // normalised, rotated, pre-scaled queries
    float knew[kHeadDim], vnew[kHeadDim];
    float wm[kConsumerWarps][G], wl[kConsumerWarps][G];
    float wo[kConsumerWarps][G][kHeadDim];
    float pw[kConsumerWarps][kAttnStep][G];  // a warp's softmax weights of its current positions
};

// Sum each of the kAttnStep entries of v over the 32 lanes of the warp (a
// reduce-scatter: each halving step exchanges half of the entries with one
// partner lane, then the lanes holding the same entry add up).  Lane l ends
// with the total of entry l mod kAttnStep in v[0].
__device__ __forceinline__ void warp_reduce_scatter(float (&v)[kAttnStep]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = kAttnStep / 2; o >= 1; o >>= 1) {
        const bool up = lane & o;
#pragma unroll
        for (int i = 0; i < o; ++i) {
            const float keep = up ? v[i + o] : v[i];
            const float send = up ? v[i] : v[i + o];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
#pragma unroll
    for (int o = kAttnStep; o < 32; o <<= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
}

// One (kv head g, split) unit of the decode attention of one layer, run by the
// consumer warps of this CTA.  The cached K and V rows of the unit's positions
// are read from global memory, a step ahead of their use (an L2 prefetch of
// them measured slower: it competes with the weight stream).  The new
// position's row comes from the QKV output: the
// unit waits for its q/k/v rows in the exchange buffer (a failed wait sets the
// abort flag; the unit then writes no cache row).  Returns false (every
// consumer thread alike) if a wait ran out or the launch is aborting.
template <int G, bool TRACE>
__device__ __forceinline__ bool attention_unit(const StepParams& p, const StepLayer& L, int layer, int pos, int g,
                                               int q0, bool write_kv, int split, int nsplit, int chunk,
                                               unsigned char* scratch, int* s_last, const Poll& w) {
    auto mark = [&](int k) {  // traced launches: the unit's progress
        if constexpr (TRACE)
            if (threadIdx.x == 0)
                p.trace[(size_t)blockIdx.x * p.trace_stride + 8 + 27 * p.n_layers + 4 * layer + k] = globaltimer_ns();
    };
    AttnSmem<G>& sm = *reinterpret_cast<AttnSmem<G>*>(scratch);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int len = pos + 1;
    const int t0 = split * chunk, t1 = min(len, t0 + chunk);
    const bool has_new = t1 == len;
    const float2* rope = p.rope + (size_t)pos * (kHeadDim / 2);
    const float scale = 1.0f / sqrtf((float)kHeadDim);
    const size_t cache_off = ((size_t)layer * p.n_kv + g) * p.max_pos * kHeadDim;
    __nv_bfloat16* kc = p.kc + cache_off;
    __nv_bfloat16* vc = p.vc + cache_off;
    const float* qkv = xch_vec(p, layer, kXQkv);
    float* out = xch_vec(p, layer, kXAttn);

    // q/k RMSNorm over head_dim then rotate-half RoPE: lane l holds dims
    // 4l..4l+3; its rotation partner dims (+-64) sit in lane l^16.  Returns
    // whether the lane's row elements arrived.
    auto norm_rope = [&](const float* src, const __nv_bfloat16* gamma, float* dst, float post) {
        // the gains and this position's (cos, sin) pairs do not depend on the
        // exchanged row: their loads go out before the wait for it
        const uint2 gb = *reinterpret_cast<const uint2*>(gamma + 4 * lane);
        const float4 cs01 = *reinterpret_cast<const float4*>(rope + ((4 * lane) & 63));
        const float4 cs23 = *reinterpret_cast<const float4*>(rope + ((4 * lane) & 63) + 2);
        const float4 v = poll4(reinterpret_cast<const float4*>(src) + lane, w);
        const bool ok = !unset4(v);
        const float ss = warp_sum(v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w);
        const float r = rsqrtf(ss * (1.0f / kHeadDim) + p.eps);
        const float a[4] = {v.x * r * bf16lo(gb.x), v.y * r * bf16hi(gb.x), v.z * r * bf16lo(gb.y),
                            v.w * r * bf16hi(gb.y)};
        const float c[4] = {cs01.x, cs01.z, cs23.x, cs23.z}, sn[4] = {cs01.y, cs01.w, cs23.y, cs23.w};
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const float partner = __shfl_xor_sync(0xffffffffu, a[jj], 16);
            dst[4 * lane + jj] = (lane < 16 ? a[jj] * c[jj] - partner * sn[jj] : a[jj] * c[jj] + partner * sn[jj]) * post;
        }
        return ok;
    };
    // The cached rows do not depend on this step: issue the loads of the
    // warp's first positions before the q/k loads (one memory round trip).
    // Warp w scores positions in steps of kAttnStep: step i covers
    // [t0 + kAttnStep (w + 8 i), +kAttnStep); lane l holds dims 4 (l mod 32)
    // .. +3 of each key and value row (whole rows are one coalesced load per
    // position).  The new position's row (t1 - 1 when has_new) comes from
    // shared memory.
    const int tcache_end = has_new ? t1 - 1 : t1;  // cached rows; the new row comes from smem
    uint2 ka[kAttnStep];  // the key rows of the warp's next step
    uint2 va[kAttnStep];  // the value rows of its current step
    auto load_k = [&](int tb) {
#pragma unroll
        for (int b = 0; b < kAttnStep; ++b) {
            const int t = tb + b;
            ka[b] = t < tcache_end ? *reinterpret_cast<const uint2*>(kc + (size_t)t * kHeadDim + 4 * lane)
                                   : make_uint2(0u, 0u);
        }
    };
    auto load_v = [&](int tb) {
#pragma unroll
        for (int b = 0; b < kAttnStep; ++b) {
            const int t = tb + b;
            va[b] = t < tcache_end ? *reinterpret_cast<const uint2*>(vc + (size_t)t * kHeadDim + 4 * lane)
                                   : make_uint2(0u, 0u);
        }
    };
    load_k(t0 + kAttnStep * warp);
    load_v(t0 + kAttnStep * warp);
    // warp w < G takes query head q0 + w; the new key/value row goes to the
    // first warp without a query head, or to the last warp (after its query
    // head) when the group fills every consumer warp
    static_assert(G <= kConsumerWarps, "one consumer warp per query head of the group");
    constexpr int kNewRowWarp = G < kConsumerWarps ? G : kConsumerWarps - 1;
    if (warp < G) norm_rope(qkv + (size_t)(q0 + warp) * kHeadDim, L.qn, sm.qs[warp], scale);
    if (has_new && warp == kNewRowWarp) {
        const bool okk = norm_rope(qkv + (size_t)(p.n_q + g) * kHeadDim, L.kn, sm.knew, 1.0f);
        const float4 v4 = poll4(reinterpret_cast<const float4*>(qkv + (size_t)(p.n_q + p.n_kv + g) * kHeadDim) + lane, w);
        const bool okv = !unset4(v4);
        // a row that never arrived is not cached; of the units sharing a kv
        // head, one writes it (the others use their own identical copy)
        const bool store = __all_sync(0xffffffffu, okk && okv) && write_kv;
        __syncwarp();
        const float vf[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const int d = 4 * lane + jj;
            const __nv_bfloat16 kb = __float2bfloat16_rn(sm.knew[d]);
            const __nv_bfloat16 vb = __float2bfloat16_rn(vf[jj]);
            if (store) {
                kc[(size_t)pos * kHeadDim + d] = kb;
                vc[(size_t)pos * kHeadDim + d] = vb;
            }
            sm.knew[d] = __bfloat162float(kb);
            sm.vnew[d] = __bfloat162float(vb);
        }
    }
    consumer_sync();
    mark(0);

    float m[G], l[G], o[G][4], qr[G][4];
#pragma unroll
    for (int jj = 0; jj < G; ++jj) {
        m[jj] = -INFINITY;
        l[jj] = 0.f;  // this lane's share of the softmax denominator (summed over the warp at the end)
#pragma unroll
        for (int i = 0; i < 4; ++i) { o[jj][i] = 0.f; qr[jj][i] = sm.qs[jj][4 * lane + i]; }
    }
    const int new_t = has_new ? t1 - 1 : -1;
    float (*pw)[G] = sm.pw[warp];
    for (int tb = t0 + kAttnStep * warp; tb < t1; tb += kAttnStep * kConsumerWarps) {
        // the value rows of these positions (the first step's came with its
        // key rows): in flight while the scores are formed
        if (tb != t0 + kAttnStep * warp) load_v(tb);
        // partial scores of the lane's 4 dims, reduced over the warp: lane l
        // ends with the full score of position tb + l mod kAttnStep for every head
        float sc[G][kAttnStep];
#pragma unroll
        for (int b = 0; b < kAttnStep; ++b) {
            float k4[4];
            if (tb + b == new_t) {
#pragma unroll
                for (int i = 0; i < 4; ++i) k4[i] = sm.knew[4 * lane + i];
            } else {
                k4[0] = bf16lo(ka[b].x); k4[1] = bf16hi(ka[b].x); k4[2] = bf16lo(ka[b].y); k4[3] = bf16hi(ka[b].y);
            }
#pragma unroll
            for (int jj = 0; jj < G; ++jj)
                sc[jj][b] = qr[jj][0] * k4[0] + qr[jj][1] * k4[1] + qr[jj][2] * k4[2] + qr[jj][3] * k4[3];
        }
        // the next step's key rows: in flight during the reduction and P.V
        load_k(tb + kAttnStep * kConsumerWarps);
        const int tl = tb + (lane & (kAttnStep - 1));  // the position this lane's scores belong to
        const bool live = tl < t1;
#pragma unroll
        for (int jj = 0; jj < G; ++jj) {
            warp_reduce_scatter(sc[jj]);
            const float sj = live ? sc[jj][0] : -INFINITY;
            const float mn = fmaxf(m[jj], warp_max(sj));
            const float corr = __expf(m[jj] - mn);
            const float pj = live ? __expf(sj - mn) : 0.f;
            l[jj] = l[jj] * corr + (lane < kAttnStep ? pj : 0.f);
#pragma unroll
            for (int i = 0; i < 4; ++i) o[jj][i] *= corr;
            m[jj] = mn;
            if (lane < kAttnStep) pw[lane][jj] = pj;
        }
        __syncwarp();
        // o[h] += sum_b p[h][b] V[tb + b] over the lane's dims
#pragma unroll
        for (int b = 0; b < kAttnStep; ++b) {
            float v4[4];
            if (tb + b == new_t) {
#pragma unroll
                for (int i = 0; i < 4; ++i) v4[i] = sm.vnew[4 * lane + i];
            } else {
                v4[0] = bf16lo(va[b].x); v4[1] = bf16hi(va[b].x); v4[2] = bf16lo(va[b].y); v4[3] = bf16hi(va[b].y);
            }
#pragma unroll
            for (int jj = 0; jj < G; ++jj) {
                const float pj = pw[b][jj];
#pragma unroll
                for (int i = 0; i < 4; ++i) o[jj][i] += pj * v4[i];
            }
        }
        __syncwarp();
    }
#pragma unroll
    for (int jj = 0; jj < G; ++jj) l[jj] = warp_sum(l[jj]);
    mark(1);
#pragma unroll
    for (int jj = 0; jj < G; ++jj) {
        if (lane == 0) { sm.wm[warp][jj] = m[jj]; sm.wl[warp][jj] = l[jj]; }
#pragma unroll
        for (int i = 0; i < 4; ++i) sm.wo[warp][jj][4 * lane + i] = o[jj][i];
    }
    if (consumer_sync_or(*w.abort)) return false;

    // merge the warps; a single split writes the output directly
    const int u = q0 / G;  // the unit's slot: kv head g (G = the group), or q head q0 (G = 1)
    float* po = p.part_o + (((size_t)u * p.S + split) * G) * kHeadDim;
    float* pml = p.part_ml + (((size_t)u * p.S + split) * G) * 2;
    for (int idx = threadIdx.x; idx < G * kHeadDim; idx += kConsumers) {
        const int jj = idx / kHeadDim, d = idx % kHeadDim;
        float M = -INFINITY;
        for (int w2 = 0; w2 < kConsumerWarps; ++w2) M = fmaxf(M, sm.wm[w2][jj]);
        float Ls = 0.f, O = 0.f;
        for (int w2 = 0; w2 < kConsumerWarps; ++w2) {
            const float c = sm.wm[w2][jj] == -INFINITY ? 0.f : __expf(sm.wm[w2][jj] - M);
            Ls += sm.wl[w2][jj] * c;
            O += sm.wo[w2][jj][d] * c;
        }
        if (nsplit == 1) {
            st_relaxed(out + (size_t)(q0 + jj) * kHeadDim + d, O / Ls);
        } else {
            po[idx] = O;
            if (d == 0) { pml[2 * jj] = M; pml[2 * jj + 1] = Ls; }
        }
    }
    if (nsplit == 1) {
        consumer_sync();
        mark(2);
        mark(3);
        return true;
    }
    mark(2);
    // the last split of this kv head merges all splits (the ticket starts at
    // kUnset: arrival k, from 0, reads kUnset + k).  One acquire-release add
    // by thread 0 after the barrier orders every thread's partial stores
    // before it and, in the merging CTA, the other splits' stores before every
    // thread's loads after the next barrier (measured faster than a fence in
    // every thread: FP8 1.735 -> 1.711 ms/frame)
    consumer_sync();
    if (threadIdx.x == 0) {
        unsigned old;
        asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                     : "=r"(old)
                     : "l"(xch_tickets(p) + layer * p.n_q + u)
                     : "memory");
        *s_last = old + 1u == (unsigned)(nsplit - 1);
    }
    consumer_sync();
    if (*s_last) {
        // every split's (max, sum) pairs and partial outputs in one round trip:
        // the pairs into shared memory, the outputs of this thread's entries
        // (idx = threadIdx.x + 256 e) into registers, kMergeBatch splits at a time
        constexpr int kMergeBatch = 20;
        constexpr int kEntries = (G * kHeadDim + kConsumers - 1) / kConsumers;
        const float* po0 = p.part_o + ((size_t)u * p.S * G) * kHeadDim;
        const float* pml0 = p.part_ml + ((size_t)u * p.S * G) * 2;
        float* mlw = &sm.wo[0][0][0];  // reuse: [nsplit][G][2] pairs, then [nsplit][G] weights
        float pv[kEntries][kMergeBatch];
        auto load_po = [&](int s0) {
#pragma unroll
            for (int e = 0; e < kEntries; ++e) {
                const int idx = threadIdx.x + kConsumers * e;
                const int jj = idx / kHeadDim, d = idx % kHeadDim;
#pragma unroll
                for (int b = 0; b < kMergeBatch; ++b)
                    pv[e][b] = (idx < G * kHeadDim && s0 + b < nsplit)
                                   ? __ldcg(po0 + ((size_t)(s0 + b) * G + jj) * kHeadDim + d) : 0.f;
            }
        };
        load_po(0);
        for (int i = threadIdx.x; i < nsplit * G * 2; i += kConsumers) mlw[i] = __ldcg(pml0 + i);
        consumer_sync();
        float* wgt = mlw + nsplit * G * 2;
        float* lsum = wgt + nsplit * G;
        if (threadIdx.x < G) {
            const int jj = threadIdx.x;
            float M = -INFINITY;
            for (int s = 0; s < nsplit; ++s) M = fmaxf(M, mlw[(s * G + jj) * 2]);
            float Ls = 0.f;
            for (int s = 0; s < nsplit; ++s) {
                const float c = __expf(mlw[(s * G + jj) * 2] - M);
                wgt[s * G + jj] = c;
                Ls += mlw[(s * G + jj) * 2 + 1] * c;
            }
            lsum[jj] = Ls;
        }
        consumer_sync();
        float acc[kEntries] = {};
        for (int s0 = 0; s0 < nsplit; s0 += kMergeBatch) {
            if (s0 > 0) load_po(s0);
#pragma unroll
            for (int e = 0; e < kEntries; ++e) {
                const int jj = (threadIdx.x + kConsumers * e) / kHeadDim;
#pragma unroll
                for (int b = 0; b < kMergeBatch; ++b)
                    if (s0 + b < nsplit) acc[e] += pv[e][b] * wgt[(s0 + b) * G + jj];
            }
        }
#pragma unroll
        for (int e = 0; e < kEntries; ++e) {
            const int idx = threadIdx.x + kConsumers * e;
            if (idx < G * kHeadDim) {
                const int jj = idx / kHeadDim, d = idx % kHeadDim;
                st_relaxed(out + (size_t)(q0 + jj) * kHeadDim + d, acc[e] / lsum[jj]);
            }
        }
    }
    consumer_sync();
    mark(3);
    return true;
}

// Per-CTA constants of one launch, worked out once at kernel start and kept
// in shared memory: the phase functions read them there instead of holding
// them in registers across the step.
struct CtaState {
    int pos, nsplit, chunk, nunits;
    int qsub;                      // attention units per kv head and split: 1 (all G q heads) or G (one each)
    int unit_g, unit_j, unit_split;  // this CTA's attention unit (kv head, q head within it, split), if any
    int rows[5][2];                // this CTA's output rows per projection kind
    unsigned long long* cwait;     // traced runs: consumer wait per projection (thread 0), else null
    unsigned long long* cstr;      // traced runs: this CTA's per-stage trace, else null
    int cstr_n;
};

// Dynamic shared memory: barriers | per-layer pointer table | activation /
// attention scratch | partials | ring.
struct StepSmem {
    StepLayer* sl;
    unsigned char* xs;
    float* part;
    Ring ring;
};
__device__ __forceinline__ StepSmem step_smem(unsigned char* smem, const StepParams& p) {
    StepSmem m;
    const int tbl_bytes = (p.n_layers * (int)sizeof(StepLayer) + 127) & ~127;
    m.sl = reinterpret_cast<StepLayer*>(smem + kBarrierBytes);
    m.xs = smem + kBarrierBytes + tbl_bytes;
    m.part = reinterpret_cast<float*>(m.xs + p.xs_bytes);
    m.ring = Ring{reinterpret_cast<uint64_t*>(smem), reinterpret_cast<uint64_t*>(smem) + p.ns,
                  m.xs + p.xs_bytes + p.part_bytes, (uint32_t)p.slot_bytes, p.ns, p.ns_magic};
    return m;
}

// Projection `kind` (0 QKV, 1 O, 2 gate/up, 3 down, 4 head) of layer l as this CTA sees it.
__device__ __forceinline__ Proj step_proj(const StepParams& p, const StepLayer* sl, const CtaState& cs, int kind,
                                          int l, bool fp8) {
    Proj j{};
    j.fp8 = (fp8 && kind != 4) ? 1 : 0;
    j.rs = p.rs[kind];
    j.wpr = p.wpr[kind];
    j.r0 = cs.rows[kind][0];
    j.r1 = cs.rows[kind][1];
    const int A = p.n_q * kHeadDim;
    if (kind == 4) {
        j.W = reinterpret_cast<const unsigned char*>(p.head);
        j.y = p.logits;
        j.N = p.n_cb * p.cb_vocab;
        j.K = p.hidden;
        return j;
    }
    const StepLayer& L = sl[l];
    switch (kind) {
        case 0: j.W = static_cast<const unsigned char*>(L.wqkv); j.wscale = L.sqkv; j.y = p.qkv;
                j.N = A + 2 * p.n_kv * kHeadDim; j.K = p.hidden; break;
        case 1: j.W = static_cast<const unsigned char*>(L.wo); j.wscale = L.so; j.y = p.h;
                j.N = p.hidden; j.K = A; break;
        case 2: j.W = static_cast<const unsigned char*>(L.wgu); j.wscale = L.sgu; j.y = p.act;
                j.N = p.inter; j.K = p.hidden; j.swiglu = 1; break;
        default: j.W = static_cast<const unsigned char*>(L.wd); j.wscale = L.sd; j.y = p.h;
                 j.N = p.hidden; j.K = p.inter; break;
    }
    return j;
}

template <bool TRACE>
__device__ __forceinline__ void trace_mark(const StepParams& p, int ev) {
    if constexpr (TRACE)
        if (threadIdx.x == 0) p.trace[(size_t)blockIdx.x * p.trace_stride + ev] = globaltimer_ns();
}

// One projection phase of the consumers: stage the activation vector from its
// exchange buffer (waiting for it, with the norm / quantisation its kind
// needs), reduce this CTA's stages from the ring, apply the epilogue (storing
// the outputs into their exchange buffer).  For bf16 a call of its own
// (proj_phase below): its registers are allocated apart from the state the
// step keeps across phases.  Returns the advanced stage counter, or -1 if a
// wait ran out or the launch is aborting (every consumer thread alike).
template <bool FP8_, int KIND, bool TRACE>
__device__ __forceinline__ int proj_phase_body(const StepParams& p, const CtaState& cs, unsigned char* smem, int l,
                                               int it, float* red, volatile int* abort, float* s_hrows) {
    constexpr bool FP8 = FP8_ && KIND != 4;  // the head is bf16 in both precisions
    const StepSmem m = step_smem(smem, p);
    const Proj j = step_proj(p, m.sl, cs, KIND, l, FP8);
    const int ev = 1 + 14 * l + (KIND == 0 ? 0 : KIND == 1 ? 5 : KIND == 2 ? 8 : KIND == 3 ? 11 : 0);
    const int A = p.n_q * kHeadDim;
    // FP8 activation site of this projection: static scale and calibration
    const float* site_sa = FP8 && p.fp8_sa ? p.fp8_sa + 4 * l + KIND : nullptr;
    float* site_cal = FP8 && p.fp8_calib ? p.fp8_calib + 4 * l + KIND : nullptr;
    const Poll w = step_poll(p, abort);
    // this projection's input: h after the previous layer (the embedding for
    // layer 0), the attention output, h after the attention, the MLP
    // activation, h after the last layer
    const int xl = KIND == 0 ? l - 1 : KIND == 4 ? p.n_layers - 1 : l;
    const int xk = KIND == 1 ? kXAttn : KIND == 2 ? kXHo : KIND == 3 ? kXAct : kXHd;
    const float* x = xch_vec(p, xl, xk);
    float sa = 1.0f;
    // every CTA produces a slice of every exchanged vector
    if (!xch_wait(xch_counter(p, xl, xk), gridDim.x, w)) return -1;
    if constexpr (KIND == 0) {
        sa = stage_x_xch<FP8, true>(x, m.sl[l].ln_in, p.hidden, p.eps, site_sa, site_cal, m.xs, nullptr, red, w);
    } else if constexpr (KIND == 2) {
        sa = stage_x_xch<FP8, true>(x, m.sl[l].ln_post, p.hidden, p.eps, site_sa, site_cal, m.xs, nullptr, red, w);
    } else if constexpr (KIND == 4) {
        sa = stage_x_xch<false, true>(x, p.final_norm, p.hidden, p.eps, nullptr, nullptr, m.xs, nullptr, red, w);
    } else if constexpr (FP8) {
        sa = stage_x_xch<true, false>(x, nullptr, KIND == 1 ? A : p.inter, p.eps, site_sa, site_cal, m.xs,
                                      reinterpret_cast<float*>(m.xs + p.xf_off), red, w);
    }
    // (bf16 O and down inputs are not staged: the stage loop's lanes load their
    // segments of the exchanged vector straight into registers, waiting there)
    if (sa < 0.f) return -1;
    if constexpr (KIND == 4) trace_mark<TRACE>(p, 1 + 14 * p.n_layers);
    else trace_mark<TRACE>(p, ev);

    // the stage loop and epilogue (consume_phase: for bf16 a function of its
    // own, allocated apart from the staging code above, so that it keeps the
    // activation segment and the loop state in registers; inlined for FP8).
    // Traced launches also record the consumers' data waits and CTA 0's
    // per-stage times.
    unsigned long long* cw = TRACE && cs.cwait && KIND < 4 ? cs.cwait + 4 * l + KIND : nullptr;
    unsigned long long* str = TRACE ? cs.cstr : nullptr;
    const int str_n = TRACE ? cs.cstr_n : 0;
    if constexpr (KIND == 1 || KIND == 3) {
        // residual add on this CTA's rows of h (kept in shared memory)
        const EpiOut so{s_hrows, xch_vec(p, l, KIND == 1 ? kXHo : kXHd)};
        it = consume_phase<FP8, kEpiResid>(j, m.ring, it, m.xs, sa, m.part, abort, &p.st->err, cw, &so, str, str_n,
                                          FP8 ? nullptr : x, &w);
        if constexpr (TRACE && KIND == 3) {
            // layer-level checks: this CTA's rows of the residual stream after the layer
            if (p.hsnap && it >= 0)
                for (int r = threadIdx.x; r < j.r1 - j.r0; r += kConsumers)
                    p.hsnap[(size_t)(l + 1) * p.hidden + j.r0 + r] = s_hrows[r];
        }
    } else if constexpr (KIND == 2) {
        const EpiOut so{nullptr, xch_vec(p, l, kXAct)};
        it = consume_phase<FP8, kEpiSwiglu>(j, m.ring, it, m.xs, sa, m.part, abort, &p.st->err, cw, &so, str, str_n);
    } else if constexpr (KIND == 0) {
        const EpiOut so{nullptr, xch_vec(p, l, kXQkv)};
        it = consume_phase<FP8, kEpiStore>(j, m.ring, it, m.xs, sa, m.part, abort, &p.st->err, cw, &so, str, str_n);
    } else {
        it = consume_phase<FP8, kEpiStore>(j, m.ring, it, m.xs, sa, m.part, abort, &p.st->err, cw, nullptr, str,
                                          str_n);
    }
    const bool ok = it >= 0;
    if constexpr (KIND < 4)
        if (ok) xch_publish(xch_counter(p, l, KIND == 0 ? kXQkv : KIND == 1 ? kXHo : KIND == 2 ? kXAct : kXHd));
    if constexpr (KIND == 4) trace_mark<TRACE>(p, 1 + 14 * p.n_layers + 1);
    else trace_mark<TRACE>(p, ev + 1);
    return ok ? it : -1;
}

template <bool FP8_, int KIND, bool TRACE>
__device__ __noinline__ int proj_phase_call(const StepParams& p, const CtaState& cs, unsigned char* smem, int l,
                                            int it, float* red, volatile int* abort, float* s_hrows) {
    return proj_phase_body<FP8_, KIND, TRACE>(p, cs, smem, l, it, red, abort, s_hrows);
}
// A projection phase as the step kernel runs it: a call of its own for bf16
// (and the bf16 head), inlined for FP8, whose phases hold few registers
// (FP8 1.557 -> 1.528 ms/frame; bf16 inlined measured no better).
template <bool FP8_, int KIND, bool TRACE>
__device__ __forceinline__ int proj_phase(const StepParams& p, const CtaState& cs, unsigned char* smem, int l, int it,
                                          float* red, volatile int* abort, float* s_hrows) {
    if constexpr (FP8_ && KIND != 4)
        return proj_phase_body<FP8_, KIND, TRACE>(p, cs, smem, l, it, red, abort, s_hrows);
    else
        return proj_phase_call<FP8_, KIND, TRACE>(p, cs, smem, l, it, red, abort, s_hrows);
}

// This CTA's attention unit of layer l (CTAs without one only announce that
// they are done).  Returns the advanced stage counter, or -1 if a wait ran
// out or the launch is aborting (every consumer thread alike).
template <int G, bool TRACE>
__device__ __forceinline__ int attn_phase_body(const StepParams& p, const CtaState& cs, unsigned char* smem, int l,
                                               int it, int* s_last, volatile int* abort) {
    if ((int)blockIdx.x < cs.nunits) {
        const Poll w = step_poll(p, abort);
        if (!xch_wait(xch_counter(p, l, kXQkv), gridDim.x, w)) return -1;
        const StepSmem m = step_smem(smem, p);
        bool ok;
        if (G > 1 && cs.qsub > 1)
            ok = attention_unit<1, TRACE>(p, m.sl[l], l, cs.pos, cs.unit_g, cs.unit_g * G + cs.unit_j,
                                          cs.unit_j == 0, cs.unit_split, cs.nsplit, cs.chunk, m.xs, s_last, w);
        else
            ok = attention_unit<G, TRACE>(p, m.sl[l], l, cs.pos, cs.unit_g, cs.unit_g * G, true, cs.unit_split,
                                          cs.nsplit, cs.chunk, m.xs, s_last, w);
        if (!ok) return -1;
    }
    // after its merge, if this unit merged: every CTA counts, so the count is
    // complete only once every kv head's output is stored
    xch_publish(xch_counter(p, l, kXAttn));
    return it;
}

template <int G, bool TRACE>
__device__ __noinline__ int attn_phase_call(const StepParams& p, const CtaState& cs, unsigned char* smem, int l,
                                            int it, int* s_last, volatile int* abort) {
    return attn_phase_body<G, TRACE>(p, cs, smem, l, it, s_last, abort);
}
// The attention phase as the step kernel runs it: inlined in the FP8 kernel
// (FP8 1.530 -> 1.503 ms/frame), a call of its own in the bf16 one (inlined,
// the bf16 step measured no better at its headline workload).
template <bool FP8, int G, bool TRACE>
__device__ __forceinline__ int attn_phase(const StepParams& p, const CtaState& cs, unsigned char* smem, int l, int it,
                                          int* s_last, volatile int* abort) {
    if constexpr (FP8)
        return attn_phase_body<G, TRACE>(p, cs, smem, l, it, s_last, abort);
    else
        return attn_phase_call<G, TRACE>(p, cs, smem, l, it, s_last, abort);
}

template <int PREC, int G, bool TRACE>
__global__ void __launch_bounds__(kThreads, 1) step_kernel(const __grid_constant__ StepParams p_in) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(16) StepParams s_p;  // the launch parameters, for the phase functions
    __shared__ CtaState s_cs;
    __shared__ float red[32];
    __shared__ int s_last;
    __shared__ int s_codes[kMaxCodebooks];
    __shared__ volatile int s_abort;
    __shared__ float s_hrows[kMaxHRows];  // this CTA's rows of the residual stream h

    constexpr bool FP8 = PREC == kFP8;
    const StepParams& p = p_in;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const StepSmem m = step_smem(smem, p);
    {
        // parameters and the layer pointer table (read on every stage) into shared memory
        static_assert(sizeof(StepParams) % 8 == 0, "StepParams is copied in 8-byte words");
        const unsigned long long* ps = reinterpret_cast<const unsigned long long*>(&p_in);
        unsigned long long* pd = reinterpret_cast<unsigned long long*>(&s_p);
        for (int i = threadIdx.x; i < (int)(sizeof(StepParams) / 8); i += blockDim.x) pd[i] = ps[i];
        const unsigned long long* src = reinterpret_cast<const unsigned long long*>(p.layers);
        unsigned long long* dst = reinterpret_cast<unsigned long long*>(m.sl);
        for (int i = threadIdx.x; i < p.n_layers * (int)(sizeof(StepLayer) / 8); i += blockDim.x) dst[i] = src[i];
    }
    const int A = p.n_q * kHeadDim;
    if (threadIdx.x < 5) {
        const int N = threadIdx.x == 0 ? A + 2 * p.n_kv * kHeadDim
                    : threadIdx.x == 2 ? p.inter
                    : threadIdx.x == 4 ? p.n_cb * p.cb_vocab
                                       : p.hidden;
        s_cs.rows[threadIdx.x][0] = (int)((long long)blockIdx.x * N / gridDim.x);
        s_cs.rows[threadIdx.x][1] = (int)((long long)(blockIdx.x + 1) * N / gridDim.x);
    }
    if (threadIdx.x == 0) {
        ring_init(m.ring);
        s_abort = 0;
        const int pos = p.st->pos;
        s_cs.pos = pos;
        // attention work split for this position
        const int len = pos + 1;
        int S = gridDim.x / p.n_kv;
        if (S > p.S) S = p.S;
        if (S < 1) S = 1;
        int chunk = (len + S - 1) / S;
        if (chunk < kAttnMinChunk) chunk = kAttnMinChunk;
        s_cs.chunk = chunk;
        s_cs.nsplit = (len + chunk - 1) / chunk;
        // short contexts leave most CTAs without a unit: then each q head of
        // a kv head gets a unit of its own (the units of one kv head read the
        // same cached rows; one of them writes the new row)
        s_cs.qsub = (G > 1 && p.n_kv * G * s_cs.nsplit <= (int)gridDim.x) ? G : 1;
        s_cs.nunits = p.n_kv * s_cs.qsub * s_cs.nsplit;
        const int uq = blockIdx.x / s_cs.nsplit;  // (kv head, q head within it)
        s_cs.unit_split = blockIdx.x % s_cs.nsplit;
        s_cs.unit_g = uq / s_cs.qsub;
        s_cs.unit_j = uq % s_cs.qsub;
        s_cs.cwait = TRACE ? p.trace + (size_t)blockIdx.x * p.trace_stride + 8 + 19 * p.n_layers : nullptr;
        s_cs.cstr = (TRACE && p.stage_trace && blockIdx.x == 0) ? p.stage_trace : nullptr;
        s_cs.cstr_n = p.stage_trace_stride / 4;
    }
    __syncthreads();
    const int pos = s_cs.pos;

    // ---- warm L2 with every layer's small parameters ---------------------------
    // Norm gains, FP8 scales and this position's RoPE row are read on the
    // consumers' critical path right after a wait; a first touch would queue
    // behind the saturated weight stream.  The idle lanes of the producer warp
    // spread L2 prefetches of all of them over the CTAs at kernel start.
    if (warp == kConsumerWarps && lane > 0) {
        const int n_items = 8 * p.n_layers + 2;
        const int A2 = A + 2 * p.n_kv * kHeadDim;
        for (int item = blockIdx.x * 31 + (lane - 1); item < n_items; item += gridDim.x * 31) {
            const void* ptr = nullptr;
            uint32_t bytes = 0;
            if (item < 8 * p.n_layers) {
                const StepLayer& L = m.sl[item / 8];
                switch (item % 8) {
                    case 0: ptr = L.ln_in; bytes = p.hidden * 2; break;
                    case 1: ptr = L.ln_post; bytes = p.hidden * 2; break;
                    case 2: ptr = L.qn; bytes = kHeadDim * 2; break;
                    case 3: ptr = L.kn; bytes = kHeadDim * 2; break;
                    case 4: ptr = L.sqkv; bytes = A2 * 4; break;
                    case 5: ptr = L.so; bytes = p.hidden * 4; break;
                    case 6: ptr = L.sgu; bytes = 2 * p.inter * 4; break;
                    default: ptr = L.sd; bytes = p.hidden * 4; break;
                }
            } else if (item == 8 * p.n_layers) {
                ptr = p.final_norm;
                bytes = p.hidden * 2;
            } else if (pos >= 0 && pos < p.max_pos) {
                ptr = p.rope + (size_t)pos * (kHeadDim / 2);
                bytes = kHeadDim / 2 * sizeof(float2);
            }
            if (ptr)
                for (uint32_t off = 0; off < bytes; off += 32768)
                    prefetch_l2_bulk(static_cast<const unsigned char*>(ptr) + off, min(32768u, bytes - off));
        }
    }

    // ---- producer warp: every weight range of the step, in phase order --------
    // Two cursors walk the same stage sequence: the copy cursor fills ring
    // slots as they free up; the prefetch cursor runs up to p.pf_stages stages
    // ahead asking L2 for the data.  A projection's byte ranges are worked out
    // once when a cursor enters it; per stage the producer only adds offsets
    // (it is a single thread: integer divisions per stage would throttle it).
    if (warp == kConsumerWarps) {
        if (lane == 0) {
            struct Seg {  // this CTA's part of one projection
                const unsigned char* a;  // first row of its range (gate rows for gate/up)
                const unsigned char* b;  // matching up rows, or null
                uint32_t stage_bytes;    // bytes of a full stage, per range
                uint32_t last_bytes;     // bytes of the last stage, per range
                uint32_t b_off;          // offset of the up rows inside a slot
                int nst;
            };
            const Ring& ring = m.ring;
            const int nkinds = p.decode ? 4 * p.n_layers + 1 : 4 * p.n_layers;
            auto seg_of = [&](int q) {
                const int kind = q == 4 * p.n_layers ? 4 : q % 4;
                const Proj j = step_proj(p, m.sl, s_cs, kind, q == 4 * p.n_layers ? 0 : q / 4, FP8);
                const uint32_t rowb = (uint32_t)proj_cpr(j) * 16u;
                const int opst = proj_opst(j), nrows = j.r1 - j.r0;
                Seg sg;
                sg.a = j.W + (size_t)j.r0 * rowb;
                sg.b = j.swiglu ? j.W + ((size_t)j.N + j.r0) * rowb : nullptr;
                sg.nst = (nrows + opst - 1) >> ilog2(opst);
                sg.stage_bytes = (uint32_t)opst * rowb;
                sg.last_bytes = (uint32_t)(nrows - (sg.nst - 1) * opst) * rowb;
                sg.b_off = (uint32_t)opst * rowb;
                return sg;
            };
            const uint64_t pol = l2_evict_first_policy();
            unsigned long long* tr = TRACE ? p.trace + (size_t)blockIdx.x * p.trace_stride + 4 + 14 * p.n_layers
                                           : nullptr;
            unsigned long long* str = TRACE ? s_cs.cstr : nullptr;
            const int str_n = s_cs.cstr_n;

            // prefetch cursor
            int pq = 0, ps = 0, pidx = 0;
            Seg psg = seg_of(0);
            auto prefetch_upto = [&](int limit) {
                // pidx counts real stages only (it is compared with the copy
                // cursor): segments without stages are stepped over
                while (pq < nkinds && pidx < limit) {
                    if (ps < psg.nst) {
                        const uint32_t bytes = ps + 1 < psg.nst ? psg.stage_bytes : psg.last_bytes;
                        const size_t off = (size_t)ps * psg.stage_bytes;
                        prefetch_l2_bulk(psg.a + off, bytes);
                        if (psg.b) prefetch_l2_bulk(psg.b + off, bytes);
                        ++pidx;
                        ++ps;
                    }
                    if (ps >= psg.nst) {
                        ps = 0;
                        if (++pq < nkinds) psg = seg_of(pq);
                    }
                }
            };

            int it = 0, slot = 0;
            uint32_t parity = 1;  // first pass over the ring: slots start free
            bool ok = true;
            for (int q = 0; q < nkinds && ok; ++q) {
                const Seg sg = seg_of(q);
                unsigned long long* pw = TRACE && q < 4 * p.n_layers
                                             ? p.trace + (size_t)blockIdx.x * p.trace_stride + 8 + 23 * p.n_layers + q
                                             : nullptr;
                unsigned long long waited = 0;  // stored once per projection (traced runs)
                for (int s2 = 0; s2 < sg.nst; ++s2) {
                    prefetch_upto(it + p.pf_stages);
                    const uint64_t tw = pw ? globaltimer_ns() : 0;
                    // While the slot is still busy (the consumers are in a norm, a
                    // wait or attention) keep HBM streaming: run the L2 prefetch
                    // further ahead, up to p.pf_max stages past the copy cursor.
                    bool got = mbar_try_wait(&ring.empty[slot], parity);
                    while (!got && pq < nkinds && pidx < it + p.pf_max) {
                        prefetch_upto(pidx + 1);
                        got = mbar_try_wait(&ring.empty[slot], parity);
                    }
                    if (!got && !mbar_wait_or_abort(&ring.empty[slot], parity, &s_abort)) {
                        atomicOr(&p.st->err, kErrTimeout);
                        s_abort = 1;
                        ok = false;
                        break;
                    }
                    if (pw) waited += globaltimer_ns() - tw;
                    if (str && it < str_n) str[4 * it] = globaltimer_ns();
                    const uint32_t bytes = s2 + 1 < sg.nst ? sg.stage_bytes : sg.last_bytes;
                    const size_t off = (size_t)s2 * sg.stage_bytes;
                    unsigned char* dst = ring.buf + (size_t)slot * ring.slot_bytes;
                    mbar_arrive_expect_tx(&ring.full[slot], sg.b ? 2 * bytes : bytes);
                    bulk_g2s(dst, sg.a + off, bytes, &ring.full[slot], pol);
                    if (sg.b) bulk_g2s(dst + sg.b_off, sg.b + off, bytes, &ring.full[slot], pol);
                    ++it;
                    if (++slot == ring.ns) {
                        slot = 0;
                        parity ^= 1;
                    }
                }
                if (pw) *pw = waited;
                if (tr) tr[q == 4 * p.n_layers ? 5 * (p.n_layers - 1) + 4 : 5 * (q / 4) + q % 4] = globaltimer_ns();
            }
            if (tr) tr[5 * p.n_layers + 1] = globaltimer_ns();
            if (!ok) drain(ring, it);
        }
        return;
    }

    // ---- consumer warps ------------------------------------------------------------
    trace_mark<TRACE>(p, 0);
    if (pos < 0 || pos >= p.max_pos) {
        if (threadIdx.x == 0) {
            atomicOr(&p.st->err, kErrPos | kErrTimeout);  // kErrTimeout stops the others' waits early
            s_abort = 1;
        }
        return;
    }

    // embed: this CTA's slice of h = sum_k E_k[c_k]
    {
        if (threadIdx.x < p.n_cb) {
            int c = p.decode ? p.st->codes[threadIdx.x] : p.prompt[(size_t)p.st->prefill_row * p.n_cb + threadIdx.x];
            if (c < 0 || c >= p.cb_vocab) {
                atomicOr(&p.st->err, kErrCode);
                c = 0;
            }
            s_codes[threadIdx.x] = c;
        }
        consumer_sync();
        const int i0 = (int)((long long)blockIdx.x * p.hidden / gridDim.x);
        const int i1 = (int)((long long)(blockIdx.x + 1) * p.hidden / gridDim.x);
        float* h0 = xch_vec(p, -1, kXHd);
        for (int i = i0 + threadIdx.x; i < i1; i += kConsumers) {
            float acc = 0.f;
            for (int k = 0; k < p.n_cb; ++k)
                acc += __bfloat162float(p.embed[((size_t)k * p.cb_vocab + s_codes[k]) * p.hidden + i]);
            p.h[i] = acc;
            s_hrows[i - i0] = acc;
            if (!p.fault_skip_embed) st_relaxed(h0 + i, acc);
            if constexpr (TRACE)
                if (p.hsnap) p.hsnap[i] = acc;
        }
        if (!p.fault_skip_embed) xch_publish(xch_counter(p, -1, 0));
    }

    // per layer: QKV | attention | O-proj | gate/up | down, each phase waiting
    // only for the exchanged elements it reads (no barrier between phases:
    // trace events 2, 4, 7, 10 and 13 repeat the event before them)
    int it = 0;
    for (int l = 0; l < p.n_layers; ++l) {
        const int ev = 1 + 14 * l;
        if ((it = proj_phase<FP8, 0, TRACE>(s_p, s_cs, smem, l, it, red, &s_abort, s_hrows)) < 0) return;
        trace_mark<TRACE>(p, ev + 2);
        if ((it = attn_phase<FP8, G, TRACE>(s_p, s_cs, smem, l, it, &s_last, &s_abort)) < 0) return;
        trace_mark<TRACE>(p, ev + 3);
        trace_mark<TRACE>(p, ev + 4);
        if ((it = proj_phase<FP8, 1, TRACE>(s_p, s_cs, smem, l, it, red, &s_abort, s_hrows)) < 0) return;
        trace_mark<TRACE>(p, ev + 7);
        if ((it = proj_phase<FP8, 2, TRACE>(s_p, s_cs, smem, l, it, red, &s_abort, s_hrows)) < 0) return;
        trace_mark<TRACE>(p, ev + 10);
        if ((it = proj_phase<FP8, 3, TRACE>(s_p, s_cs, smem, l, it, red, &s_abort, s_hrows)) < 0) return;
        trace_mark<TRACE>(p, ev + 13);
    }
    if (p.decode) {
        if ((it = proj_phase<FP8, 4, TRACE>(s_p, s_cs, smem, 0, it, red, &s_abort, s_hrows)) < 0) return;
        head_tail(p.logits, p.n_cb, p.cb_vocab, p.st, xch_tickets(p) + p.n_layers * p.n_q, kUnset, p.hist,
                  p.hist_cap, &s_last, s_codes);
        trace_mark<TRACE>(p, 1 + 14 * p.n_layers + 2);
    }
    if (!p.decode && blockIdx.x == 0 && threadIdx.x == 0) {
        p.st->pos = pos + 1;
        p.st->prefill_row += 1;
    }
}

template <int PREC, int G>
cudaError_t launch_step_t(const StepParams& p, int grid, int smem, cudaStream_t s) {
    auto kern = p.trace ? step_kernel<PREC, G, true> : step_kernel<PREC, G, false>;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

// Per-precision entry points (one translation unit each, compiled in parallel).
template <int PREC>
cudaError_t step_prepare_prec(int G, int smem) {
#define TTS_STEP_PREP(GG)                                                                                  \
    if (G == GG) {                                                                                         \
        cudaError_t e = cudaFuncSetAttribute(step_kernel<PREC, GG, false>,                                 \
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);           \
        if (e == cudaSuccess)                                                                              \
            e = cudaFuncSetAttribute(step_kernel<PREC, GG, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                     smem);                                                                \
        return e;                                                                                          \
    }
    TTS_STEP_PREP(1) TTS_STEP_PREP(2) TTS_STEP_PREP(4) TTS_STEP_PREP(8)
#undef TTS_STEP_PREP
    return cudaErrorInvalidValue;
}

template <int PREC>
cudaError_t launch_step_prec(const StepParams& p, int G, int grid, int smem, cudaStream_t s) {
    if (G == 1) return launch_step_t<PREC, 1>(p, grid, smem, s);
    if (G == 2) return launch_step_t<PREC, 2>(p, grid, smem, s);
    if (G == 4) return launch_step_t<PREC, 4>(p, grid, smem, s);
    if (G == 8) return launch_step_t<PREC, 8>(p, grid, smem, s);
    return cudaErrorInvalidValue;
}

}  // namespace
}  // namespace tts

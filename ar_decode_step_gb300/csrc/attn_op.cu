// Standalone entry point for one layer's decode attention: the step's kernel
// (q/k RMSNorm + RoPE + bf16 KV write + split-K GQA attention) driven from
// plain pointers, outside a context.
#include <cmath>
#include <cstdio>
#include <mutex>

#include "kernels.h"
#include "tts_decode.h"

using namespace tts;

namespace {

// Scratch layout for one call: [DevState][tickets n_kv][RoPE row 64 x float2]
// [partial max/sum n_kv*S*G*2][partial outputs n_kv*S*G*128], 256-byte aligned.
struct AttnScratch {
    size_t st, counters, rope, part_ml, part_o, total;
};

size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }

AttnScratch scratch_layout(int n_q, int n_kv, int S) {
    AttnScratch L{};
    const int G = n_q / n_kv;
    size_t off = 0;
    L.st = off;       off = up256(off + sizeof(DevState));
    L.counters = off; off = up256(off + sizeof(unsigned) * n_kv);
    L.rope = off;     off = up256(off + sizeof(float2) * (kHeadDim / 2));
    L.part_ml = off;  off = up256(off + sizeof(float) * (size_t)n_kv * S * G * 2);
    L.part_o = off;   off = up256(off + sizeof(float) * (size_t)n_kv * S * G * kHeadDim);
    L.total = off;
    return L;
}

int check_args(const float* qkv, const void* qn, const void* kn, const void* kc, const void* vc,
               const float* out, int n_q, int n_kv, int max_pos, int pos) {
    if (!qkv || !qn || !kn || !kc || !vc || !out) return TTS_ERR_ARG;
    if (n_kv < 1 || n_q < 1 || n_q % n_kv) return TTS_ERR_ARG;
    const int G = n_q / n_kv;
    if (G != 1 && G != 2 && G != 4 && G != 8) return TTS_ERR_ARG;
    if (max_pos < 1 || max_pos > 65536) return TTS_ERR_ARG;
    if (pos < 0) return TTS_ERR_ARG;
    if (pos >= max_pos) return TTS_ERR_FULL;
    return TTS_OK;
}

// The RoPE row of one position: cos/sin of pos * theta^(-2i/128) (fp64 angle).
void rope_row(int pos, float theta, float2* row) {
    for (int i = 0; i < kHeadDim / 2; ++i) {
        const double inv_f = std::pow((double)theta, -2.0 * i / (double)kHeadDim);
        const double ang = (double)pos * inv_f;
        row[i] = make_float2((float)std::cos(ang), (float)std::sin(ang));
    }
}

// Fill the call's scratch (zeroed tickets and state, the RoPE row) and launch.
cudaError_t run_attention(char* scratch, const AttnScratch& L, const float* qkv, const void* qn,
                          const void* kn, void* kc, void* vc, float* out, int n_q, int n_kv, int max_pos,
                          int pos, float eps, float theta, int S, cudaStream_t s) {
    float2 row[kHeadDim / 2];
    rope_row(pos, theta, row);
    cudaError_t e = cudaMemsetAsync(scratch, 0, L.rope, s);  // state + tickets start at zero
    if (e != cudaSuccess) return e;
    e = cudaMemcpyAsync(scratch + L.rope, row, sizeof(row), cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return e;
    AttnParams a{};
    a.qkv = qkv;
    a.q_norm = static_cast<const __nv_bfloat16*>(qn);
    a.k_norm = static_cast<const __nv_bfloat16*>(kn);
    a.rope = nullptr;
    a.rope_row = reinterpret_cast<const float2*>(scratch + L.rope);  // the one row of this position
    a.kc = static_cast<__nv_bfloat16*>(kc);
    a.vc = static_cast<__nv_bfloat16*>(vc);
    a.out = out;
    a.part_o = reinterpret_cast<float*>(scratch + L.part_o);
    a.part_ml = reinterpret_cast<float*>(scratch + L.part_ml);
    a.counter = reinterpret_cast<unsigned*>(scratch + L.counters);
    a.st = reinterpret_cast<DevState*>(scratch + L.st);
    a.pos_override = pos;
    a.n_q = n_q;
    a.n_kv = n_kv;
    a.max_pos = max_pos;
    a.S = S;
    a.eps = eps;
    e = launch_attention(a, LaunchCfg{0, 0, false}, s);
    if (e != cudaSuccess) return e;
    return cudaSuccess;
}

int read_err(const char* scratch, const AttnScratch& L, cudaStream_t s) {
    DevState st{};
    if (cudaMemcpyAsync(&st, scratch + L.st, sizeof(st), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return TTS_ERR_CUDA;
    return st.err ? TTS_ERR_DEVICE : TTS_OK;
}

}  // namespace

extern "C" int tts_attention_decode(const float* qkv, const void* q_norm, const void* k_norm, void* k_cache,
                                    void* v_cache, float* out, int n_q, int n_kv, int max_pos, int pos,
                                    float eps, float rope_theta, void* stream) {
    int rc = check_args(qkv, q_norm, k_norm, k_cache, v_cache, out, n_q, n_kv, max_pos, pos);
    if (rc != TTS_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int S = attn_splits_for(max_pos);
    const AttnScratch L = scratch_layout(n_q, n_kv, S);
    void* scratch = nullptr;
    cudaError_t e = cudaMallocAsync(&scratch, L.total, s);
    if (e != cudaSuccess) return TTS_ERR_CUDA;
    e = run_attention(static_cast<char*>(scratch), L, qkv, q_norm, k_norm, k_cache, v_cache, out, n_q, n_kv,
                      max_pos, pos, eps, rope_theta, S, s);
    rc = (e == cudaSuccess) ? read_err(static_cast<char*>(scratch), L, s) : TTS_ERR_CUDA;
    cudaFreeAsync(scratch, s);
    if (cudaStreamSynchronize(s) != cudaSuccess) return TTS_ERR_CUDA;
    if (e != cudaSuccess) std::fprintf(stderr, "tts: attention launch failed: %s\n", cudaGetErrorString(e));
    return rc;
}

// ---------------------------------------------------------------------------
// Allocation-free variant.  Some callers cannot allocate device memory at the
// point of the call: code running inside another runtime's memory budget, a
// caller holding no allocator of its own (an embedded or real-time host loop
// that must never hit cudaMalloc's implicit synchronisation or failure), or a
// process whose allocations are frozen after start-up.  This entry point takes
// its scratch from one fixed array in device global memory instead.
//
// The array belongs to this file's device module.  Under lazy module loading
// (the CUDA default) a module is loaded on a device -- and its global arrays
// created there -- the first time the process touches it on that device: here
// that is the address lookup below, and the attention kernel's module loads on
// its first launch.  Both can allocate, so the first call on each device
// belongs to the caller's set-up, while allocation is still allowed (tts_init
// also performs the lookup for its device).  After that the array stays until
// the process exits or the device is reset.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kStaticScratchBytes = size_t(2) << 20;  // 2 MiB
__device__ __align__(256) char g_attn_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
void* g_static_addr[kMaxDevices] = {};

}  // namespace

namespace tts {

// Device address of the array on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device (with that device current) and cached.  A device reset
// (cudaDeviceReset) unloads the module, which makes the cached address stale:
// a process that resets a device must not call the allocation-free entry
// point on that device afterwards.
int static_scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TTS_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return TTS_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (!g_static_addr[dev]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_attn_static_scratch);
        if (e != cudaSuccess) {
            std::fprintf(stderr, "tts: cudaGetSymbolAddress of the static scratch failed: %s\n",
                         cudaGetErrorString(e));
            return TTS_ERR_CUDA;
        }
        g_static_addr[dev] = p;
    }
    *out = g_static_addr[dev];
    return TTS_OK;
}

}  // namespace tts

extern "C" int tts_attention_decode_noalloc(const float* qkv, const void* q_norm, const void* k_norm,
                                            void* k_cache, void* v_cache, float* out, int n_q, int n_kv,
                                            int max_pos, int pos, float eps, float rope_theta, void* stream) {
    int rc = check_args(qkv, q_norm, k_norm, k_cache, v_cache, out, n_q, n_kv, max_pos, pos);
    if (rc != TTS_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int S = attn_splits_for(max_pos);
    const AttnScratch L = scratch_layout(n_q, n_kv, S);
    if (L.total > kStaticScratchBytes) {
        std::fprintf(stderr,
                     "tts_attention_decode_noalloc: n_q=%d, max_pos=%d needs %zu bytes of scratch; "
                     "the static array holds %zu\n",
                     n_q, max_pos, L.total, kStaticScratchBytes);
        return TTS_ERR_ARG;
    }
    void* base = nullptr;
    rc = static_scratch_address(&base);
    if (rc != TTS_OK) return rc;
    char* scratch = static_cast<char*>(base);
    // run_attention zeroes the tickets and the state word before the launch;
    // the partial buffers are fully written before they are read.
    const cudaError_t e = run_attention(scratch, L, qkv, q_norm, k_norm, k_cache, v_cache, out, n_q, n_kv,
                                        max_pos, pos, eps, rope_theta, S, s);
    if (e != cudaSuccess) {
        std::fprintf(stderr, "tts: attention launch failed: %s\n", cudaGetErrorString(e));
        return TTS_ERR_CUDA;
    }
    return read_err(scratch, L, s);
}

// Host side of the persistent decode-step kernel: launch geometry and the
// per-precision dispatch (kernels in step_bf16.cu / step_fp8.cu).
#include "kernels.h"

namespace tts {

cudaError_t step_prepare_bf16(int G, int smem);
cudaError_t step_prepare_fp8(int G, int smem);
cudaError_t launch_step_bf16(const StepParams& p, int G, int grid, int smem, cudaStream_t s);
cudaError_t launch_step_fp8(const StepParams& p, int G, int grid, int smem, cudaStream_t s);

cudaError_t step_prepare(int prec, int G, int smem) {
    return prec == kFP8 ? step_prepare_fp8(G, smem) : step_prepare_bf16(G, smem);
}

int step_attn_scratch_bytes(int G) {
    // AttnSmem<G> (step_kernel.cuh): queries, the new key and value rows, per
    // warp softmax state, partial outputs and the weights of 8 positions
    return (int)(sizeof(float) * (G * kHeadDim + 2 * kHeadDim + 2 * kConsumerWarps * G +
                                  kConsumerWarps * G * kHeadDim + kConsumerWarps * 8 * G));
}

int step_threads() { return (kConsumerWarps + 1) * 32; }

cudaError_t launch_step(const StepParams& p, int prec, int G, int grid, int smem, cudaStream_t s) {
    return prec == kFP8 ? launch_step_fp8(p, G, grid, smem, s) : launch_step_bf16(p, G, grid, smem, s);
}

}  // namespace tts

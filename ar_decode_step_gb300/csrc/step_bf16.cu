// The persistent decode-step kernel, BF16 weights (kernel code in step_kernel.cuh).
#include "step_kernel.cuh"

namespace tts {
cudaError_t step_prepare_bf16(int G, int smem) { return step_prepare_prec<kBF16>(G, smem); }
cudaError_t launch_step_bf16(const StepParams& p, int G, int grid, int smem, cudaStream_t s) {
    return launch_step_prec<kBF16>(p, G, grid, smem, s);
}
}  // namespace tts

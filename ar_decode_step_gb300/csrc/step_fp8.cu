// The persistent decode-step kernel, FP8 (E4M3) weights (kernel code in step_kernel.cuh).
#include "step_kernel.cuh"

namespace tts {
cudaError_t step_prepare_fp8(int G, int smem) { return step_prepare_prec<kFP8>(G, smem); }
cudaError_t launch_step_fp8(const StepParams& p, int G, int grid, int smem, cudaStream_t s) {
    return launch_step_prec<kFP8>(p, G, grid, smem, s);
}
}  // namespace tts

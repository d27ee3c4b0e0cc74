// tail.cu -- the Gemma sandwich tail that follows the routed phase 2, as a launch of its own (the
// streaming GEMV's phase 2 runs the same row function inside its fused combine).
//
// Source page (docs.rs, turbospark-runtime 0.3.0): Gemma-4 batched routed prefill
// (src/families/gemma4/moe_batch.rs), the per-token tail encoded on the same command buffer after
// the fused phase 2 (the steps and their rounding: tail_common.cuh).
#include "tail_common.cuh"

namespace tsmoe {

namespace {

constexpr int kTailThreads = 1024;

// One CTA per token row.
__global__ void __launch_bounds__(kTailThreads) gemma_tail_kernel(TailArgs a) {
    __shared__ float v[kTailMaxH];
    __shared__ float rs;
    pdl_wait();                 // y comes from the previous kernel
    pdl_launch_dependents();
    const int t = blockIdx.x;
    if (t >= a.T) return;
    gemma_tail_rows(a, t, 1, v, &rs, static_cast<int>(threadIdx.x), kTailThreads, [] { __syncthreads(); });
}

}  // namespace

cudaError_t launch_gemma_tail(const TailArgs& a, cudaStream_t s) {
    if (a.T <= 0) return cudaSuccess;
    return launch_pdl(gemma_tail_kernel, dim3(a.T), dim3(kTailThreads), 0, s, a);
}

}  // namespace tsmoe

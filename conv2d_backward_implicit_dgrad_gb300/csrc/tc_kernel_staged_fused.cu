// tcgen05 implicit-GEMM dgrad, staged mode with the fused epilogue
// (ReLU-backward mask and/or accumulation into grad_input).
#include "tc_kernel.cuh"

namespace dgrad {

cudaError_t launch_tc_staged_fused(const MainParams &p, const Tiling &t, cudaStream_t stream, bool pdl) {
    if (t.kc != 32 || !p.a_tma || !p.a_staged) return cudaErrorInvalidValue;
    return launch_mode<true, 1, true>(p, t, stream, pdl);
}

}  // namespace dgrad

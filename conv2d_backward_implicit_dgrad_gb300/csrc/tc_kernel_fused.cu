// tcgen05 implicit-GEMM dgrad, tensor-copy mode with the fused epilogue
// (ReLU-backward mask and/or accumulation into grad_input).
#include "tc_kernel.cuh"

namespace dgrad {

cudaError_t launch_tc_fused(const MainParams &p, const Tiling &t, cudaStream_t stream, bool pdl) {
    if (t.kc != 32 || !p.a_tma) return cudaErrorInvalidValue;
    return launch_mode<true, 1>(p, t, stream, pdl);
}

}  // namespace dgrad

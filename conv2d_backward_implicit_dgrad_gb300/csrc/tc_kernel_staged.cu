// tcgen05 implicit-GEMM dgrad, staged mode (each A stage one tensor copy of
// the caller's grad_out, transposed in shared memory), plain stores; the
// fused-epilogue instances are in tc_kernel_staged_fused.cu.
#include "tc_kernel.cuh"

namespace dgrad {

#ifdef DGRAD_TRACE
// Tracing builds only: this unit's per-CTA cycle counters (every unit that
// includes tc_kernel.cuh holds its own copy).
extern "C" int dgrad_trace_read_staged(unsigned long long *host, int n) {
    if (n > kTraceCtas * kTraceSlots) n = kTraceCtas * kTraceSlots;
    if (cudaMemcpyFromSymbol(host, g_trace, sizeof(unsigned long long) * n) != cudaSuccess) return -1;
    static unsigned long long zeros[kTraceCtas * kTraceSlots];
    return cudaMemcpyToSymbol(g_trace, zeros, sizeof(zeros)) == cudaSuccess ? 0 : -1;
}
#endif

cudaError_t launch_tc_staged(const MainParams &p, const Tiling &t, cudaStream_t stream, bool pdl) {
    if (t.kc != 32 || !p.a_tma || !p.a_staged) return cudaErrorInvalidValue;
    if (p.relu_in != nullptr || p.accumulate != 0) return launch_tc_staged_fused(p, t, stream, pdl);
    return launch_mode<true, 0, true>(p, t, stream, pdl);
}

}  // namespace dgrad

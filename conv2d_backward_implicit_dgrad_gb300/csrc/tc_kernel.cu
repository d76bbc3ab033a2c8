// tcgen05 implicit-GEMM dgrad, plain-store instantiations: tensor-copy mode
// (packed frame) without the fused epilogue, and producer-warp mode with the
// fused epilogue chosen at run time.  The fused tensor-copy instantiations
// live in tc_kernel_fused.cu and the staged-mode ones in tc_kernel_staged.cu,
// so the sets compile in parallel.
#include "tc_kernel.cuh"

namespace dgrad {

#ifdef DGRAD_TRACE
// Tracing builds only: copy (and clear) the per-CTA cycle counters.
extern "C" int dgrad_trace_read(unsigned long long *host, int n) {
    if (n > kTraceCtas * kTraceSlots) n = kTraceCtas * kTraceSlots;
    if (cudaMemcpyFromSymbol(host, g_trace, sizeof(unsigned long long) * n) != cudaSuccess) return -1;
    static unsigned long long zeros[kTraceCtas * kTraceSlots];
    return cudaMemcpyToSymbol(g_trace, zeros, sizeof(zeros)) == cudaSuccess ? 0 : -1;
}
#endif

cudaError_t launch_tc(const MainParams &p, const Tiling &t, cudaStream_t stream, bool pdl) {
    if (t.kc != 32) return cudaErrorInvalidValue;
    if (!p.a_tma) return launch_mode<false, 2>(p, t, stream, pdl);
    if (p.a_tmem) return launch_tc_tmem(p, t, stream, pdl);
    if (p.a_staged) return launch_tc_staged(p, t, stream, pdl);
    if (p.relu_in != nullptr || p.accumulate != 0) return launch_tc_fused(p, t, stream, pdl);
    return launch_mode<true, 0>(p, t, stream, pdl);
}

}  // namespace dgrad

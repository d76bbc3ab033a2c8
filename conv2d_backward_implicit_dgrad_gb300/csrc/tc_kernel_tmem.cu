// tcgen05 implicit-GEMM dgrad, tensor-memory A mode (1x1 kernel, stride 1,
// no padding): tensor copies of the caller's NCHW grad_out, moved by the
// epilogue warps into tensor memory, where the MMA reads its A operand.
// One phase and one tap per chunk, so the epilogue is the plain one-phase
// form; plain and fused-store instances.
#include "tc_kernel.cuh"

namespace dgrad {

#ifdef DGRAD_TRACE
// Tracing builds only: this unit's per-CTA cycle counters.
extern "C" int dgrad_trace_read_tmem(unsigned long long *host, int n) {
    if (n > kTraceCtas * kTraceSlots) n = kTraceCtas * kTraceSlots;
    if (cudaMemcpyFromSymbol(host, g_trace, sizeof(unsigned long long) * n) != cudaSuccess) return -1;
    static unsigned long long zeros[kTraceCtas * kTraceSlots];
    return cudaMemcpyToSymbol(g_trace, zeros, sizeof(zeros)) == cudaSuccess ? 0 : -1;
}
#endif

cudaError_t launch_tc_tmem(const MainParams &p, const Tiling &t, cudaStream_t stream, bool pdl) {
    if (t.kc != 32 || !p.a_tma || !p.a_tmem || epi_form(p.vec_w, p.s, p.max_sub) != 0) return cudaErrorInvalidValue;
    if (p.relu_in != nullptr || p.accumulate != 0) return launch_kc<32, true, 0, 1, 1, false, true>(p, t, stream, pdl);
    return launch_kc<32, true, 0, 0, 1, false, true>(p, t, stream, pdl);
}

}  // namespace dgrad

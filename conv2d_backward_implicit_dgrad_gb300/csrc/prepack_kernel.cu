// Weight pre-pack: OIHW fp32 weights -> the K-major packed layout the main
// kernels stream (see PrepackParams).  Replaces meganeura's per-element
// implicit W^T reads (its A-tile load decomposes k into (co, kh, kw) with
// divisions and reads weight with a strided index) by one pass that writes
// each (slice, chunk) block contiguously, keeps only the taps each phase
// uses, zero-pads channels, and (TF32 precision) rounds to TF32 once.
#include <cuda_runtime.h>

#include "dgrad_internal.h"
#include "ptx.cuh"

namespace dgrad {

namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) prepack_kernel(const __grid_constant__ PrepackParams p) {
    // Let the main kernel start its prologue while this grid runs; it reads
    // the packed weights only after griddepcontrol.wait.
    dev::grid_launch_dependents();
    const long long stride = static_cast<long long>(gridDim.x) * kThreads;
    const int G = p.kc / 4;
    for (long long i = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; i < p.total; i += stride) {
        long long rest = i;
        const int e = static_cast<int>(rest % 4);
        rest /= 4;
        int j, gq;
        if (p.layout == 1) {   // [tap][j][swizzled 16-byte chunk][4]
            const int pos = static_cast<int>(rest % G);
            rest /= G;
            j = static_cast<int>(rest % p.bn);
            rest /= p.bn;
            gq = pos ^ (j & 7);
        } else {               // [tap][gq][j][4]
            j = static_cast<int>(rest % p.bn);
            rest /= p.bn;
            gq = static_cast<int>(rest % G);
            rest /= G;
        }
        const int t = static_cast<int>(rest % p.n_taps);
        rest /= p.n_taps;
        const int c = static_cast<int>(rest % p.n_chunks);
        const int sl = static_cast<int>(rest / p.n_chunks);
        const int co = c * p.kc + 4 * gq + e;
        const int ci = sl * p.bn + j;
        float v = 0.f;
        if (co < p.Co && ci < p.Ci)
            v = __ldg(p.w + ((static_cast<size_t>(co) * p.Ci + ci) * p.kH + p.tap_kh[t]) * p.kW + p.tap_kw[t]);
        if (p.round_tf32) v = dev::round_tf32(v);
        p.wp[i] = v;
    }
}

}  // namespace

cudaError_t launch_prepack(const PrepackParams &p, cudaStream_t stream) {
    long long blocks = (p.total + kThreads - 1) / kThreads;
    if (blocks > 4096) blocks = 4096;
    if (blocks < 1) blocks = 1;
    prepack_kernel<<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace dgrad

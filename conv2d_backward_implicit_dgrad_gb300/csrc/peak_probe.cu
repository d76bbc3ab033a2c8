// FP32 FFMA throughput probe (include/dgrad_probe.h): eight independent
// dependent-FMA chains per thread keep every FFMA pipe of an SM busy once a
// few warps per scheduler are resident, so blocks * 256 * 8 * iters FMAs over
// the event-timed launch is the pipe's rate.
#include <cuda_runtime.h>

#include "dgrad.h"
#include "dgrad_internal.h"
#include "dgrad_probe.h"

namespace {

constexpr int kProbeThreads = 256;
constexpr int kChains = 8;

__global__ void __launch_bounds__(kProbeThreads) ffma_probe_kernel(int iters, float m, float c, float *out) {
    float x[kChains];
#pragma unroll
    for (int i = 0; i < kChains; ++i) x[i] = static_cast<float>(threadIdx.x + i);
#pragma unroll 1
    for (int it = 0; it < iters; it += 4) {
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int i = 0; i < kChains; ++i) x[i] = fmaf(x[i], m, c);
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kChains; ++i) s += x[i];
    out[static_cast<size_t>(blockIdx.x) * kProbeThreads + threadIdx.x] = s;
}

}  // namespace

extern "C" int dgrad_probe_ffma(int blocks, int iters, float *out, void *stream) {
    if (blocks < 1 || iters < 4 || iters % 4 != 0 || out == nullptr) return DGRAD_ERR_INVALID_ARG;
    ffma_probe_kernel<<<blocks, kProbeThreads, 0, static_cast<cudaStream_t>(stream)>>>(iters, 0.999999f, 1e-6f,
                                                                                       out);
    return dgrad::cuda_status(cudaGetLastError());
}

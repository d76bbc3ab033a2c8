// Exact-fp32 implicit-GEMM dgrad on the CUDA cores (FFMA), over the same
// phase split, zero-padded grad_out frame and packed weights as the tcgen05
// path.
//
// One CTA computes 128 output positions x BN input channels of one phase.
// For each chunk of KC output channels it stages the frame band
// [P0, P0 + a_rows) and the phase's packed weights in shared memory, then
// every thread accumulates PPT positions x 4 channels in registers: for each
// tap and 4-channel group, PPT 16-byte A reads and 4 16-byte B reads feed
// PPT*16 FFMAs (meganeura's 4x4 register micro-tile, widened along K).
#include <cuda_runtime.h>

#include "dgrad_internal.h"
#include "gather.cuh"
#include "ptx.cuh"

namespace dgrad {

namespace {

constexpr int kThreads = 256;

template <int BN, int KC>
__global__ void __launch_bounds__(kThreads) simt_dgrad_kernel(const __grid_constant__ MainParams p) {
    extern __shared__ __align__(16) float sm[];
    constexpr int G = KC / 4;           // 4-channel groups per chunk
    constexpr int CG = BN / 4;          // threads along input channels
    constexpr int PG = kThreads / CG;   // threads along positions
    constexpr int PPT = kBlockM / PG;   // positions per thread
    float *As = sm;                                            // [G][a_rows][4]
    float *Bs = sm + static_cast<size_t>(G) * p.a_rows * 4;    // [taps][G][BN][4]

    const int tile = blockIdx.x, slice = blockIdx.y;
    const PhaseDesc pd = p.phase[blockIdx.z];
    const int P0 = tile * kBlockM;
    const int tid = threadIdx.x;
    const int cg = tid / PG, pg = tid % PG;

    float acc[PPT][4];
#pragma unroll
    for (int i = 0; i < PPT; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

    const float4 *A4 = reinterpret_cast<const float4 *>(As);
    const float4 *B4 = reinterpret_cast<const float4 *>(Bs);
    for (int c = 0; c < p.n_chunks && pd.tap_count > 0; ++c) {
        __syncthreads();
        dev::fill_a_stage<KC>(As, p, P0, c * KC, tid, kThreads);
        const size_t woff = ((static_cast<size_t>(slice) * p.n_chunks + c) * p.n_taps + pd.tap_begin) * KC * BN;
        const float4 *src = reinterpret_cast<const float4 *>(p.wp + woff);
        const int n4 = pd.tap_count * KC * BN / 4;
        for (int i = tid; i < n4; i += kThreads) reinterpret_cast<float4 *>(Bs)[i] = __ldg(src + i);
        __syncthreads();
        for (int t = 0; t < pd.tap_count; ++t) {
            const int shift = p.tap[pd.tap_begin + t].shift;
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float4 b[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) b[j] = B4[(t * G + g) * BN + cg * 4 + j];
#pragma unroll
                for (int i = 0; i < PPT; ++i) {
                    const float4 a = A4[g * p.a_rows + pg + i * PG + shift];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        acc[i][j] = fmaf(a.x, b[j].x, acc[i][j]);
                        acc[i][j] = fmaf(a.y, b[j].y, acc[i][j]);
                        acc[i][j] = fmaf(a.z, b[j].z, acc[i][j]);
                        acc[i][j] = fmaf(a.w, b[j].w, acc[i][j]);
                    }
                }
            }
        }
    }

    // Overwrite grad_input (phase outputs with no taps are written as 0), or
    // apply the fused epilogue.
    const size_t plane = static_cast<size_t>(p.H) * p.W;
#pragma unroll
    for (int i = 0; i < PPT; ++i) {
        const int P = P0 + pg + i * PG;
        int n, q, u;
        dev::decode_position(p, P, n, q, u);
        if (P >= p.positions || q >= pd.Hq || u >= pd.Wq) continue;
        const int ih = p.s * q + pd.a, iw = p.s * u + pd.b;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int ci = slice * BN + cg * 4 + j;
            if (ci < p.Ci) {
                const size_t idx = (static_cast<size_t>(n) * p.Ci + ci) * plane + static_cast<size_t>(ih) * p.W + iw;
                float v = acc[i][j];
                if (p.relu_in && !(__ldg(p.relu_in + idx) > 0.f)) v = 0.f;   // fused ReLU backward
                if (p.accumulate) v = p.gi[idx] + v;                         // fused accumulate-into
                p.gi[idx] = v;
            }
        }
    }
}

template <int BN, int KC>
cudaError_t launch_bn_kc(const MainParams &p, const Tiling &t, cudaStream_t stream) {
    auto kern = simt_dgrad_kernel<BN, KC>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, t.smem_bytes);
    if (e != cudaSuccess) return e;
    dim3 grid(t.n_tiles, t.n_slices, p.n_phases);
    kern<<<grid, kThreads, t.smem_bytes, stream>>>(p);
    return cudaGetLastError();
}

template <int BN>
cudaError_t launch_bn(const MainParams &p, const Tiling &t, cudaStream_t stream) {
    switch (t.kc) {
        case 8: return launch_bn_kc<BN, 8>(p, t, stream);
        case 16: return launch_bn_kc<BN, 16>(p, t, stream);
        case 32: return launch_bn_kc<BN, 32>(p, t, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_simt(const MainParams &p, const Tiling &t, cudaStream_t stream) {
    switch (t.bn) {
        case 16: return launch_bn<16>(p, t, stream);
        case 32: return launch_bn<32>(p, t, stream);
        case 64: return launch_bn<64>(p, t, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace dgrad

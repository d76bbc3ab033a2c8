// dgrad for few input channels (stems) as a GEMM followed by col2im.
//
//   P[position][(ci,kh,kw)] = sum over co of V[position][co] * weight[co][ci][kh][kw]
//
// (V the packed grad_out frame) is a dense GEMM with N = Ci*kH*kW columns:
// one tcgen05 MMA of 128 positions x N per K step, where the phase-split
// kernel would issue a 16-wide slice per tap.  Every P element belongs to
// grad_input[n][ci][oh*s - ph + kh][ow*s - pw + kw] (the forward mapping of
// doppler's conv2d_backward_input.wgsl), so col2im adds it there.  A CTA
// owns bands of R input rows: it runs the GEMM tiles of every position that
// reaches its band, adds their P values into the band in shared memory and
// writes the band out whole, so each grad_input element is written once.
// Each epilogue warp adds into its own copy of the band: for one tap the 32
// positions of a warp land on 32 different elements, and a warp's taps run
// in program order, so there are no concurrent updates of one element and
// no atomics; the four copies are summed in a fixed order when the band is
// written (results are the same bit for bit from run to run).  GEMM columns
// are tap-major, r = (kh*kW + kw)*Ci + ci: the CI channels of one tap are
// independent updates issued together.
//
// Roles (192 threads): warps 0-3 col2im epilogue (tensor memory -> shared-
// memory band -> grad_input), warp 4 TMEM allocation + MMA issue (converged
// warp, one elected lane), warp 5 one thread of copies (packed weights once,
// then per tile and 32-channel chunk one 2-D tensor copy of the frame).
// All waits are bounded.
#include <cuda_runtime.h>

#include "dgrad_internal.h"
#include "ptx.cuh"

namespace dgrad {

namespace {

constexpr int kCThreads = 192;
constexpr int kCEpiThreads = 128;
constexpr int kCMmaWarp = 4;
constexpr int kCLoadWarp = 5;
constexpr int kCMaxAStages = 4;
constexpr int kCMaxChunks = 32;
constexpr uint32_t kCStageBytes = kBlockM * 128;

struct CBars {
    uint64_t a_full[kCMaxAStages];
    uint64_t a_empty[kCMaxAStages];
    uint64_t b_full[kCMaxChunks];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    volatile int abort_flag;
};
static_assert(sizeof(CBars) <= 1024, "barrier block");

__device__ __forceinline__ void cfail(CBars *b, const C2iParams &p) {
    b->abort_flag = 1;
    atomicOr(p.err, kErrTimeout);
}

__device__ __forceinline__ int floor_div(int a, int b) { return a >= 0 ? a / b : -((-a + b - 1) / b); }

// Band b: image n, input rows [r0, r0 + R); the frame positions of the
// grad_out rows that reach it, [pa, pb), in tiles of 128.
struct Band {
    int n, r0, pa, pb, tiles;
};

__device__ __forceinline__ Band band_of(const C2iParams &p, int b) {
    Band d;
    d.n = b / p.bands_per_img;
    d.r0 = (b - d.n * p.bands_per_img) * p.R;
    const int lo = max(0, -floor_div(-(d.r0 + p.ph - p.kH + 1), p.s));   // ceil((r0 + ph - kH + 1) / s)
    const int hi = min(p.oH - 1, floor_div(d.r0 + p.R - 1 + p.ph, p.s));
    d.pa = (d.n * p.Hv + lo + p.Ph) * p.Wp;
    d.pb = (d.n * p.Hv + hi + 1 + p.Ph) * p.Wp;
    d.tiles = hi >= lo ? (d.pb - d.pa + kBlockM - 1) / kBlockM : 0;
    return d;
}

template <int CI>
__global__ void __launch_bounds__(kCThreads, 1) c2i_dgrad_kernel(const __grid_constant__ C2iParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    CBars *bars = reinterpret_cast<CBars *>(smem);
    const uint32_t b_base = (dev::smem_u32(smem) + 1024u + 1023u) & ~1023u;
    const uint32_t a_base = b_base + static_cast<uint32_t>(p.n_chunks * p.chunk_bytes);
    float *band = reinterpret_cast<float *>(smem + (a_base + static_cast<uint32_t>(p.a_stages) * kCStageBytes -
                                                    dev::smem_u32(smem)));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < p.a_stages; ++i) {
            dev::mbar_init(dev::smem_u32(&bars->a_full[i]), 1);
            dev::mbar_init(dev::smem_u32(&bars->a_empty[i]), 1);
        }
        for (int i = 0; i < p.n_chunks; ++i) dev::mbar_init(dev::smem_u32(&bars->b_full[i]), 1);
        for (int i = 0; i < 2; ++i) {
            dev::mbar_init(dev::smem_u32(&bars->acc_full[i]), 1);
            dev::mbar_init(dev::smem_u32(&bars->acc_empty[i]), kCEpiThreads);
        }
        dev::mbar_init(dev::smem_u32(&bars->drain), 1);
        bars->abort_flag = 0;
        dev::fence_mbar_init();
    }
    if (warp == kCMmaWarp) {
        dev::tmem_alloc(dev::smem_u32(&bars->tmem_base), p.tmem_cols);
        dev::tmem_relinquish();
    }
    dev::tc_fence_before();
    __syncthreads();
    dev::tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    const long long tmo = p.timeout_ns;

    if (warp == kCLoadWarp) {
        // ---------------------------------------------------- copies
        if (lane == 0) {
            dev::prefetch_tensormap(&p.a_map);
            dev::grid_dependency_wait();   // packed weights and frame come from the preceding kernel
            for (int c = 0; c < p.n_chunks; ++c) {
                const uint32_t bar = dev::smem_u32(&bars->b_full[c]);
                dev::mbar_arrive_expect_tx(bar, static_cast<uint32_t>(p.chunk_bytes));
                dev::bulk_g2s(b_base + static_cast<uint32_t>(c * p.chunk_bytes),
                              reinterpret_cast<const uint8_t *>(p.wp) + static_cast<size_t>(c) * p.chunk_bytes,
                              static_cast<uint32_t>(p.chunk_bytes), bar);
            }
            int last[kCMaxAStages];
            for (int i = 0; i < kCMaxAStages; ++i) last[i] = -1;
            int stage = 0;
            uint32_t parity = 0;
            bool ok = true;
            for (int b = blockIdx.x; ok && b < p.n_bands && !bars->abort_flag; b += gridDim.x) {
                const Band d = band_of(p, b);
                for (int t = 0; ok && t < d.tiles; ++t) {
                    for (int c = 0; c < p.n_chunks; ++c) {
                        if (!dev::mbar_wait(dev::smem_u32(&bars->a_empty[stage]), parity ^ 1, tmo)) {
                            cfail(bars, p);
                            ok = false;
                            break;
                        }
                        const uint32_t bar = dev::smem_u32(&bars->a_full[stage]);
                        dev::mbar_arrive_expect_tx(bar, kCStageBytes);
                        dev::tma_load_2d(a_base + static_cast<uint32_t>(stage) * kCStageBytes, &p.a_map, 32 * c,
                                         d.pa + t * kBlockM, bar);
                        last[stage] = static_cast<int>(parity);
                        if (++stage == p.a_stages) stage = 0, parity ^= 1;
                    }
                }
            }
            // Never leave with a copy in flight into this CTA's shared memory.
            for (int c = 0; c < p.n_chunks; ++c) dev::mbar_wait(dev::smem_u32(&bars->b_full[c]), 0, tmo);
            for (int i = 0; i < p.a_stages; ++i)
                if (last[i] >= 0) dev::mbar_wait(dev::smem_u32(&bars->a_full[i]), last[i], tmo);
        }
        __syncwarp();
    } else if (warp == kCMmaWarp) {
        // ---------------------------------------------------- MMA issuer
        int stage = 0, acc = 0;
        uint32_t parity = 0, acc_parity = 0;
        bool ok = true, b_ready = false;
        for (int b = blockIdx.x; ok && b < p.n_bands && !bars->abort_flag; b += gridDim.x) {
            const Band d = band_of(p, b);
            for (int t = 0; ok && t < d.tiles; ++t) {
                if (!__all_sync(0xffffffffu,
                                dev::mbar_wait(dev::smem_u32(&bars->acc_empty[acc]), acc_parity ^ 1, tmo))) {
                    ok = false;
                    break;
                }
                if (!b_ready) {
                    for (int c = 0; ok && c < p.n_chunks; ++c)
                        if (!__all_sync(0xffffffffu, dev::mbar_wait(dev::smem_u32(&bars->b_full[c]), 0, tmo)))
                            ok = false;
                    if (!ok) break;
                    b_ready = true;
                }
                dev::tc_fence_after();
                const uint32_t dcol = tmem + static_cast<uint32_t>(acc * p.bn);
                for (int c = 0; c < p.n_chunks; ++c) {
                    if (!__all_sync(0xffffffffu,
                                    dev::mbar_wait(dev::smem_u32(&bars->a_full[stage]), parity, tmo))) {
                        ok = false;
                        break;
                    }
                    dev::tc_fence_after();
                    const uint64_t ad = dev::smem_desc_sw128(a_base + static_cast<uint32_t>(stage) * kCStageBytes, 0);
                    const uint64_t bd = dev::smem_desc_sw128(b_base + static_cast<uint32_t>(c * p.chunk_bytes), 0);
#pragma unroll
                    for (int k8 = 0; k8 < 4; ++k8)
                        dev::mma_tf32_elect(dcol, dev::desc_add(ad, 32 * k8), dev::desc_add(bd, 32 * k8), p.idesc,
                                            (c > 0 || k8 > 0) ? 1u : 0u);
                    dev::mma_commit_elect(dev::smem_u32(&bars->a_empty[stage]));
                    if (++stage == p.a_stages) stage = 0, parity ^= 1;
                }
                if (!ok) break;
                dev::mma_commit_elect(dev::smem_u32(&bars->acc_full[acc]));
                if (++acc == 2) acc = 0, acc_parity ^= 1;
            }
        }
        if (!ok && lane == 0) cfail(bars, p);
        // Every MMA this warp issued has finished before tensor memory is freed.
        dev::mma_commit_elect(dev::smem_u32(&bars->drain));
        dev::mbar_wait(dev::smem_u32(&bars->drain), 0, tmo);
    } else {
        // ---------------------------------------------------- col2im epilogue
        const int et = threadIdx.x;   // 0..127: tensor-memory lane = tile row
        const int band_floats = CI * p.R * p.pitch;
        float *mine = band + warp * band_floats;   // this warp's copy of the band
        const int taps = p.kH * p.kW;
        int acc = 0;
        uint32_t acc_parity = 0;
        bool ok = true;
        for (int b = blockIdx.x; ok && b < p.n_bands; b += gridDim.x) {
            const Band d = band_of(p, b);
            for (int i = et; i < 4 * band_floats; i += kCEpiThreads) band[i] = 0.f;
            dev::named_bar(1, kCEpiThreads);
            for (int t = 0; t < d.tiles; ++t) {
                const bool got = dev::mbar_wait(dev::smem_u32(&bars->acc_full[acc]), acc_parity, tmo);
                if (!dev::named_bar_and(1, kCEpiThreads, got)) {
                    if (!got) cfail(bars, p);
                    ok = false;
                    break;
                }
                dev::tc_fence_after();
                // this thread's position and the part of the band its row can reach
                const int P = d.pa + t * kBlockM + et;
                const int rem = P - d.n * p.Hv * p.Wp;
                const int y = rem / p.Wp, x = rem - y * p.Wp;
                const int oh = y - p.Ph, ow = x - p.Pw;
                const bool valid = P < d.pb && oh >= 0 && oh < p.oH && ow >= 0 && ow < p.oW;
                const int kh_lo = d.r0 + p.ph - oh * p.s;   // kernel rows landing in the band: [kh_lo, kh_lo + R)
                const int base = (oh * p.s - p.ph - d.r0) * p.pitch + ow * p.s;   // band offset of tap (0, 0), ci 0
                const uint32_t taddr = tmem + (static_cast<uint32_t>(warp * 32) << 16) +
                                       static_cast<uint32_t>(acc * p.bn);
                // 16 taps (16 * CI columns) per batch of tensor-memory loads
                for (int t0 = 0; t0 < taps; t0 += 16) {
                    uint32_t r[CI][16];
#pragma unroll
                    for (int k = 0; k < CI; ++k)
                        if ((t0 * CI + 16 * k) < p.bn)
                            dev::tmem_ld16(taddr + static_cast<uint32_t>(t0 * CI + 16 * k), r[k]);
                    dev::tmem_wait_ld();
                    if (!valid) continue;
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int tap = t0 + j;
                        if (tap >= taps) break;
                        const int c0 = tap * CI;
                        if (static_cast<unsigned>(p.col_kh[c0] - kh_lo) >= static_cast<unsigned>(p.R)) continue;
                        float *dst = mine + base + p.col_off[c0];   // ci 0; channel ci sits ci * R * pitch further
                        float old[CI];
#pragma unroll
                        for (int ci = 0; ci < CI; ++ci) old[ci] = dst[ci * p.R * p.pitch];
#pragma unroll
                        for (int ci = 0; ci < CI; ++ci) {
                            const int col = j * CI + ci;   // column of this batch
                            dst[ci * p.R * p.pitch] = old[ci] + __uint_as_float(r[col >> 4][col & 15]);
                        }
                    }
                }
                dev::tc_fence_before();
                dev::mbar_arrive(dev::smem_u32(&bars->acc_empty[acc]));
                if (++acc == 2) acc = 0, acc_parity ^= 1;
            }
            if (!ok) break;
            dev::named_bar(1, kCEpiThreads);   // every addition of the band is done
            // write the band: rows [r0, min(r0 + R, H)) of every input channel, the four
            // warp copies summed in a fixed order, fused epilogue applied
            const int rows = min(p.R, p.H - d.r0);
            const int per_ci = rows * p.W;
            for (int i = et; i < CI * per_ci; i += kCEpiThreads) {
                const int ci = i / per_ci;
                const int rr = (i - ci * per_ci) / p.W;
                const int iw = i - ci * per_ci - rr * p.W;
                const int o_band = (ci * p.R + rr) * p.pitch + iw + p.pw;
                float v = ((band[o_band] + band[band_floats + o_band]) + band[2 * band_floats + o_band]) +
                          band[3 * band_floats + o_band];
                const size_t o = ((static_cast<size_t>(d.n) * p.Ci + ci) * p.H + d.r0 + rr) * p.W + iw;
                if (p.relu_in && !(__ldg(p.relu_in + o) > 0.f)) v = 0.f;
                if (p.accumulate) v = p.gi[o] + v;
                p.gi[o] = v;
            }
            dev::named_bar(1, kCEpiThreads);   // before the band is cleared for the next one
        }
    }

    dev::tc_fence_before();
    __syncthreads();
    dev::tc_fence_after();
    if (warp == kCMmaWarp) dev::tmem_dealloc(tmem, p.tmem_cols);
}

}  // namespace

cudaError_t launch_c2i(const C2iParams &p, const Tiling &t, cudaStream_t stream, bool pdl) {
    if (p.n_chunks > kCMaxChunks || p.a_stages > kCMaxAStages) return cudaErrorInvalidValue;
    void (*kern)(C2iParams) = nullptr;
    switch (p.Ci) {
        case 1: kern = c2i_dgrad_kernel<1>; break;
        case 2: kern = c2i_dgrad_kernel<2>; break;
        case 3: kern = c2i_dgrad_kernel<3>; break;
        case 4: kern = c2i_dgrad_kernel<4>; break;
        default: return cudaErrorInvalidValue;
    }
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, t.smem_bytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(t.grid);
    cfg.blockDim = dim3(kCThreads);
    cfg.dynamicSmemBytes = t.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace dgrad

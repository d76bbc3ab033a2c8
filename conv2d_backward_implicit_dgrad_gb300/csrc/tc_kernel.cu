// Warp-specialised tcgen05 implicit-GEMM dgrad (TF32 operands, fp32
// accumulation in tensor memory), one persistent CTA per SM.
//
// GEMM view (meganeura conv2d_grad_input_gemm.wgsl, header comment), turned
// so that output positions are the MMA's M:
//   D[P, ci] = sum over (tap t, co) of V[P + shift_t][co] * Wp[t][co][ci]
// for every sub-pixel phase (each with its own accumulator), where V is the
// zero-padded, flattened grad_out frame and Wp the pre-packed weights.
//
// Roles (448 threads):
//   warps 0-3   epilogue: tensor memory -> registers -> grad_input (NCHW)
//   warp  4     tensor-memory allocation and the single MMA-issuing thread
//   warp  5     one thread streaming packed weights with bulk copies (TMA)
//   warps 6-13  producers: grad_out band -> shared memory (A operand)
// Pipelines (all mbarriers, all waits bounded):
//   A ring   a_stages  producers -> MMA        (A_full / A_empty)
//   B ring   b_stages  weight loader -> MMA    (B_full / B_empty); when the
//            whole packed weight of the launch fits, it is loaded once
//   acc      acc_bufs  MMA -> epilogue         (acc_full / acc_empty)
#include <cuda_runtime.h>

#include "dgrad_internal.h"
#include "gather.cuh"
#include "ptx.cuh"

namespace dgrad {

namespace {

constexpr int kEpiWarps = 4;
constexpr int kMmaWarp = 4;
constexpr int kLoadWarp = 5;
constexpr int kProdWarp0 = 6;
constexpr int kProdWarps = 8;
constexpr int kThreads = (kProdWarp0 + kProdWarps) * 32;
constexpr int kMaxAStages = 4;
constexpr int kMaxBStages = 32;

struct Barriers {
    uint64_t a_full[kMaxAStages];
    uint64_t a_empty[kMaxAStages];
    uint64_t b_full[kMaxBStages];
    uint64_t b_empty[kMaxBStages];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    volatile int abort_flag;
};
static_assert(sizeof(Barriers) <= 1024, "barrier block exceeds its reserved bytes");

__device__ __forceinline__ void fail(Barriers *bars, const MainParams &p) {
    bars->abort_flag = 1;
    atomicOr(p.err, kErrTimeout);
}

template <int KC>
__global__ void __launch_bounds__(kThreads, 1) tc_dgrad_kernel(const __grid_constant__ MainParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    Barriers *bars = reinterpret_cast<Barriers *>(smem);
    float *a_base = reinterpret_cast<float *>(smem + 1024);
    const int a_stage_floats = p.a_rows * KC;
    uint8_t *b_base = smem + 1024 + static_cast<size_t>(p.a_stages) * a_stage_floats * 4;

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        for (int i = 0; i < p.a_stages; ++i) {
            dev::mbar_init(dev::smem_u32(&bars->a_full[i]), kProdWarps * 32);
            dev::mbar_init(dev::smem_u32(&bars->a_empty[i]), 1);
        }
        for (int i = 0; i < p.b_stages; ++i) {
            dev::mbar_init(dev::smem_u32(&bars->b_full[i]), 1);
            dev::mbar_init(dev::smem_u32(&bars->b_empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            dev::mbar_init(dev::smem_u32(&bars->acc_full[i]), 1);
            dev::mbar_init(dev::smem_u32(&bars->acc_empty[i]), kEpiWarps * 32);
        }
        dev::mbar_init(dev::smem_u32(&bars->drain), 1);
        bars->abort_flag = 0;
        dev::fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        dev::tmem_alloc(dev::smem_u32(&bars->tmem_base), p.tmem_cols);
        dev::tmem_relinquish();
    }
    dev::tc_fence_before();
    __syncthreads();
    dev::tc_fence_after();
    const uint32_t tmem_base = bars->tmem_base;
    const long long tmo = p.timeout_ns;
    const int tile_rows = p.tm * kBlockM;

    if (warp >= kProdWarp0) {
        // ------------------------------------------------------ producers
        const int ptid = threadIdx.x - kProdWarp0 * 32;
        uint32_t it = 0;
        for (int w = blockIdx.x; w < p.n_work && !bars->abort_flag; w += gridDim.x) {
            const int P0 = (w / p.n_slices) * tile_rows;
            for (int c = 0; c < p.n_chunks; ++c, ++it) {
                const int stage = it % p.a_stages;
                const uint32_t round = it / p.a_stages;
                if (!dev::mbar_wait(dev::smem_u32(&bars->a_empty[stage]), (round & 1) ^ 1, tmo)) {
                    fail(bars, p);
                    break;
                }
                float *As = a_base + static_cast<size_t>(stage) * a_stage_floats;
                dev::fill_a_stage<KC>(As, p, P0, c * KC, ptid, kProdWarps * 32);
                dev::fence_proxy_async_smem();
                dev::mbar_arrive(dev::smem_u32(&bars->a_full[stage]));
            }
        }
    } else if (warp == kLoadWarp) {
        // ------------------------------------------------- weight loader
        if (lane == 0) {
            dev::grid_dependency_wait();   // packed weights come from the preceding kernel
            int last_round[kMaxBStages];
            for (int i = 0; i < kMaxBStages; ++i) last_round[i] = -1;
            if (p.b_resident) {
                for (int c = 0; c < p.n_chunks; ++c) {
                    const uint32_t bar = dev::smem_u32(&bars->b_full[c]);
                    dev::mbar_arrive_expect_tx(bar, p.chunk_bytes);
                    dev::bulk_g2s(dev::smem_u32(b_base + static_cast<size_t>(c) * p.chunk_bytes),
                                  reinterpret_cast<const uint8_t *>(p.wp) + static_cast<size_t>(c) * p.chunk_bytes,
                                  p.chunk_bytes, bar);
                    last_round[c] = 0;
                }
            } else {
                uint32_t it = 0;
                for (int w = blockIdx.x; w < p.n_work && !bars->abort_flag; w += gridDim.x) {
                    const int slice = w % p.n_slices;
                    bool ok = true;
                    for (int c = 0; c < p.n_chunks; ++c, ++it) {
                        const int stage = it % p.b_stages;
                        const uint32_t round = it / p.b_stages;
                        if (!dev::mbar_wait(dev::smem_u32(&bars->b_empty[stage]), (round & 1) ^ 1, tmo)) {
                            fail(bars, p);
                            ok = false;
                            break;
                        }
                        const uint32_t bar = dev::smem_u32(&bars->b_full[stage]);
                        dev::mbar_arrive_expect_tx(bar, p.chunk_bytes);
                        const size_t off = (static_cast<size_t>(slice) * p.n_chunks + c) * p.chunk_bytes;
                        dev::bulk_g2s(dev::smem_u32(b_base + static_cast<size_t>(stage) * p.chunk_bytes),
                                      reinterpret_cast<const uint8_t *>(p.wp) + off, p.chunk_bytes, bar);
                        last_round[stage] = static_cast<int>(round);
                    }
                    if (!ok) break;
                }
            }
            // Never leave with a copy in flight into this CTA's shared memory.
            for (int i = 0; i < p.b_stages && i < kMaxBStages; ++i)
                if (last_round[i] >= 0)
                    dev::mbar_wait(dev::smem_u32(&bars->b_full[i]), last_round[i] & 1, tmo);
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ---------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t a_lbo = static_cast<uint32_t>(p.a_rows) * 16;
            const uint32_t b_lbo = static_cast<uint32_t>(p.bn) * 16;
            const uint32_t a0 = dev::smem_u32(a_base);
            const uint32_t b0 = dev::smem_u32(b_base);
            uint32_t a_it = 0, b_it = 0, local = 0;
            bool ok = true;
            for (int w = blockIdx.x; ok && w < p.n_work && !bars->abort_flag; w += gridDim.x, ++local) {
                const int buf = local % p.acc_bufs;
                const uint32_t around = local / p.acc_bufs;
                if (!dev::mbar_wait(dev::smem_u32(&bars->acc_empty[buf]), (around & 1) ^ 1, tmo)) {
                    fail(bars, p);
                    break;
                }
                dev::tc_fence_after();
                const uint32_t d_base = tmem_base + buf * p.acc_cols;
                for (int c = 0; c < p.n_chunks; ++c, ++a_it, ++b_it) {
                    const int sa = a_it % p.a_stages;
                    const int sb = p.b_resident ? c : static_cast<int>(b_it % p.b_stages);
                    const uint32_t rb = p.b_resident ? 0u : b_it / p.b_stages;
                    if (!dev::mbar_wait(dev::smem_u32(&bars->a_full[sa]), (a_it / p.a_stages) & 1, tmo) ||
                        !dev::mbar_wait(dev::smem_u32(&bars->b_full[sb]), rb & 1, tmo)) {
                        fail(bars, p);
                        ok = false;
                        break;
                    }
                    dev::tc_fence_after();
                    const uint32_t a_stage = a0 + static_cast<uint32_t>(sa) * a_stage_floats * 4;
                    const uint32_t b_stage = b0 + static_cast<uint32_t>(sb) * p.chunk_bytes;
                    for (int m = 0; m < p.tm; ++m) {
                        for (int ph = 0; ph < p.n_phases; ++ph) {
                            const PhaseDesc &pd = p.phase[ph];
                            const uint32_t d = d_base + (m * p.n_phases + ph) * p.bn;
                            for (int t = pd.tap_begin; t < pd.tap_begin + pd.tap_count; ++t) {
                                const uint32_t a_row = static_cast<uint32_t>(m * kBlockM + p.tap[t].shift) * 16;
#pragma unroll
                                for (int k8 = 0; k8 < KC / 8; ++k8) {
                                    const uint64_t ad = dev::smem_desc(a_stage + 2 * k8 * a_lbo + a_row, a_lbo, 128);
                                    const uint64_t bd = dev::smem_desc(
                                        b_stage + static_cast<uint32_t>((t * (KC / 4) + 2 * k8) * p.bn) * 16, b_lbo,
                                        128);
                                    const uint32_t acc = (c > 0 || t > pd.tap_begin || k8 > 0) ? 1u : 0u;
                                    dev::mma_tf32(d, ad, bd, p.idesc, acc);
                                }
                            }
                        }
                    }
                    dev::mma_commit(dev::smem_u32(&bars->a_empty[sa]));
                    if (!p.b_resident) dev::mma_commit(dev::smem_u32(&bars->b_empty[sb]));
                }
                if (!ok) break;
                dev::mma_commit(dev::smem_u32(&bars->acc_full[buf]));
            }
            // Drain: every MMA issued above has finished before TMEM is freed.
            dev::mma_commit(dev::smem_u32(&bars->drain));
            if (!dev::mbar_wait(dev::smem_u32(&bars->drain), 0, tmo)) fail(bars, p);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------- epilogue
        const int ew = warp;   // 0..3: tensor-memory lanes 32*ew .. 32*ew+31
        const size_t plane = static_cast<size_t>(p.H) * p.W;
        uint32_t local = 0;
        for (int w = blockIdx.x; w < p.n_work && !bars->abort_flag; w += gridDim.x, ++local) {
            const int tile = w / p.n_slices, slice = w % p.n_slices;
            const int buf = local % p.acc_bufs;
            const uint32_t around = local / p.acc_bufs;
            if (!dev::mbar_wait(dev::smem_u32(&bars->acc_full[buf]), around & 1, tmo)) {
                fail(bars, p);
                break;
            }
            dev::tc_fence_after();
            const int ci0 = slice * p.bn;
            const int nci = min(p.bn, p.Ci - ci0);
            for (int m = 0; m < p.tm; ++m) {
                const int P = tile * tile_rows + m * kBlockM + ew * 32 + lane;
                int n, q, u;
                dev::decode_position(p, P, n, q, u);
                const bool pos_ok = P < p.positions;
                for (int ph = 0; ph < p.n_phases; ++ph) {
                    const PhaseDesc &pd = p.phase[ph];
                    const bool valid = pos_ok && q < pd.Hq && u < pd.Wq;
                    const int ih = p.s * q + pd.a, iw = p.s * u + pd.b;
                    float *dst = p.gi + (static_cast<size_t>(n) * p.Ci + ci0) * plane +
                                 static_cast<size_t>(ih) * p.W + iw;
                    if (pd.tap_count == 0) {
                        if (valid)
                            for (int j = 0; j < nci; ++j) dst[j * plane] = 0.f;
                        continue;
                    }
                    const uint32_t col0 = tmem_base + (static_cast<uint32_t>(ew * 32) << 16) + buf * p.acc_cols +
                                          (m * p.n_phases + ph) * p.bn;
                    for (int c0 = 0; c0 < p.bn; c0 += 16) {
                        uint32_t r[16];
                        dev::tmem_ld16(col0 + c0, r);
                        dev::tmem_wait_ld();
                        if (valid) {
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                if (c0 + j < nci) dst[(c0 + j) * plane] = __uint_as_float(r[j]);
                        }
                    }
                }
            }
            dev::tc_fence_before();
            dev::mbar_arrive(dev::smem_u32(&bars->acc_empty[buf]));
        }
    }

    dev::tc_fence_before();
    __syncthreads();
    dev::tc_fence_after();
    if (warp == kMmaWarp) dev::tmem_dealloc(tmem_base, p.tmem_cols);
}

template <int KC>
cudaError_t launch_kc(const MainParams &p, const Tiling &t, cudaStream_t stream, bool pdl) {
    auto kern = tc_dgrad_kernel<KC>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, t.smem_bytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(t.grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = t.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace

cudaError_t launch_tc(const MainParams &p, const Tiling &t, cudaStream_t stream, bool pdl) {
    switch (t.kc) {
        case 8: return launch_kc<8>(p, t, stream, pdl);
        case 16: return launch_kc<16>(p, t, stream, pdl);
        case 32: return launch_kc<32>(p, t, stream, pdl);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace dgrad

// Exact-fp32 implicit-GEMM dgrad on the CUDA cores (FFMA), over the same
// phase split, zero-padded frame geometry and packed weights as the tcgen05
// path.
//
// One work unit is 128 output positions x BN input channels of one phase
// (1024 positions for 4-channel slices, inputs with at most 4 channels).
// For each chunk of KC output channels the frame band [P0, P0 + a_rows) and
// the phase's packed weights sit in shared memory, and every thread
// accumulates PPT positions x 4 channels in registers: for each tap and
// 4-channel group, PPT 16-byte A reads and 4 16-byte B reads feed PPT*16
// FFMAs (meganeura's 4x4 register micro-tile, widened along K).  Two ways to
// fill the shared memory:
//  - frame plans (simt_pipe_kernel): the pipeline of the tensor-core path.  A
//    loader warp copies each chunk's band from the packed channels-last
//    frame (tensor copies of 4 channels x up to 256 rows, landing as the
//    [KC/4][a_rows][4] layout the FFMA loop reads) and the phase's weights
//    (one bulk copy) into a ring of stages under mbarriers; eight compute
//    warps wait for a stage, run the register tiles and release it.  CTAs are
//    persistent over work units, so copies for the next chunks and units run
//    under the FFMAs and the stores.
//  - no frame (simt_dgrad_kernel: plans without a frame buffer, such as
//    dgrad_run_noalloc's, and the few-channel, many-tap shapes where the
//    frame does not pay): every thread of the CTA gathers the band from NCHW
//    grad_out, then all compute, one stage per chunk.
#include <cuda_runtime.h>

#include "dgrad_internal.h"
#include "gather.cuh"
#include "ptx.cuh"

namespace dgrad {

namespace {

constexpr int kThreads = 256;

// Ring position: stage index and the parity of its current round.
struct Ring {
    int stage = 0;
    uint32_t parity = 0;
    __device__ __forceinline__ void next(int n) {
        if (++stage == n) {
            stage = 0;
            parity ^= 1;
        }
    }
};

__device__ __forceinline__ void decode_unit(const MainParams &p, int u, int &tile, int &slice, int &phase) {
    // the units of one tile (its slices and phases) are consecutive: they
    // read the same frame band, so later copies of it hit L2
    const int per_tile = p.n_slices * p.n_phases;
    tile = u / per_tile;
    const int rem = u - tile * per_tile;
    slice = rem / p.n_phases;
    phase = rem - slice * p.n_phases;
}

template <int BN, int KC>
__global__ void __launch_bounds__(kThreads) simt_dgrad_kernel(const __grid_constant__ MainParams p) {
    extern __shared__ __align__(16) float sm[];
    constexpr int G = KC / 4;           // 4-channel groups per chunk
    constexpr int CG = BN / 4;          // threads along input channels
    constexpr int PG = kThreads / CG;   // threads along positions
    constexpr int UM = simt_unit_rows(BN);   // positions per unit
    constexpr int PPT = UM / PG;        // positions per thread
    float *As = sm;                                            // [G][a_rows][4]
    float *Bs = sm + static_cast<size_t>(G) * p.a_rows * 4;    // [taps][G][BN][4]

    int tile, slice, phase;
    decode_unit(p, blockIdx.x, tile, slice, phase);
    const PhaseDesc pd = p.phase[phase];
    const int P0 = tile * UM;
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
    if (t.n_work > 0x7fffffffLL) return cudaErrorInvalidValue;
    dim3 grid(static_cast<unsigned>(t.n_work));   // one CTA per unit; a tile's slices and phases are consecutive
    kern<<<grid, kThreads, t.smem_bytes, stream>>>(p);
    return cudaGetLastError();
}

// ------------------------------------------------------------ frame plans
struct PipeBars {
    uint64_t full[kSimtMaxStages];    // the stage's copies have landed
    uint64_t empty[kSimtMaxStages];   // the eight compute warps are done with the stage
    uint64_t never;                   // failure-detection test: a barrier that nothing completes
    volatile int abort_flag;
};
static_assert(sizeof(PipeBars) <= kSimtPipeHeader, "barrier block exceeds its reserved bytes");

__device__ __forceinline__ void pipe_fail(PipeBars *bars, const MainParams &p) {
    bars->abort_flag = 1;
    atomicOr(p.err, kErrTimeout);
}


// kWide (BN = 64): 128 compute threads, each an 8 x 8 register tile --
// positions w*32 + tp + 4i (i < 8) of compute warp w and channels tc + 8j
// (j < 8), lane = (tc << 2) | tp -- and two CTAs per SM.  A 16-byte warp load
// takes four shared-memory passes (one per quarter warp): the 8 x 4 tiles'
// 12 loads per 128 FFMAs ask 0.375 passes per FFMA instruction of a port that
// serves 0.25 (four FFMA pipes, one pass per clock); the 8 x 8 tiles' 16 loads
// per 256 FFMAs ask 0.25.
// Unit schedules of the frame pipeline.  Round-robin (kSnake = false): CTA b
// of G takes units b, b + G, ..., the units of a tile consecutive.  For plans
// whose phases differ in tap count (kSnake = true): CTA b takes the units at
// positions b, 2G-1-b, 2G+b, 4G-1-b, ... of the units sorted by their phase's
// tap count, most first (a tile's slices consecutive within a phase), so that
// every CTA gets a similar share of taps -- round-robin with the phase fastest
// gave each CTA one phase (with 4 phases and 152 CTAs the 4-tap phase's CTAs
// did four times the 1-tap phase's work).  The plain form is its own instance:
// the schedule code in the same kernel slowed the one-phase plans by 1-5 %.
__device__ __forceinline__ int phase_rank(const MainParams &p, int ph) {
    const int t = p.phase[ph].tap_count;
    int rank = 0;
    for (int q = 0; q < p.n_phases; ++q) {
        const int tq = p.phase[q].tap_count;
        rank += (tq > t || (tq == t && q < ph)) ? 1 : 0;
    }
    return rank;
}

// Unit at schedule position k of the sorted schedule.
__device__ __forceinline__ void sorted_unit(const MainParams &p, long long k, int &tile, int &slice, int &phase) {
    const int per_phase = p.n_tiles * p.n_slices;
    const int r = static_cast<int>(k / per_phase), rem = static_cast<int>(k - static_cast<long long>(r) * per_phase);
    phase = 0;
    for (int ph = 0; ph < p.n_phases; ++ph)
        if (phase_rank(p, ph) == r) phase = ph;
    tile = rem / p.n_slices;
    slice = rem - tile * p.n_slices;
}

template <bool kSnake>
struct UnitIter;
template <>
struct UnitIter<false> {
    int u = static_cast<int>(blockIdx.x);
    // The next unit of this CTA; false past its last one.
    __device__ __forceinline__ bool next(const MainParams &p, int &tile, int &slice, int &phase) {
        if (u >= p.n_work) return false;
        decode_unit(p, u, tile, slice, phase);
        u += static_cast<int>(gridDim.x);
        return true;
    }
};
template <>
struct UnitIter<true> {
    long long j = 0;   // round
    __device__ __forceinline__ bool next(const MainParams &p, int &tile, int &slice, int &phase) {
        const long long G = gridDim.x, b = blockIdx.x;
        while (j * G < p.n_work) {
            const long long k = (j & 1) ? (j + 1) * G - 1 - b : j * G + b;
            ++j;
            if (k >= p.n_work) continue;   // a partial last round
            sorted_unit(p, k, tile, slice, phase);
            return true;
        }
        return false;
    }
};

template <int BN, int KC, bool kWide, bool kSnake = false>
__global__ void __launch_bounds__(simt_pipe_threads(kWide), kWide ? 2 : 1)
    simt_pipe_kernel(const __grid_constant__ MainParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    static_assert(!kWide || BN == 64, "8 x 8 tiles: 64-channel slices");
    constexpr int NC = simt_pipe_threads(kWide) - 32;   // compute threads
    constexpr int G = KC / 4;           // 4-channel groups per chunk
    constexpr int CG = BN / 4;          // threads along input channels (8 x 4 tiles)
    constexpr int PG = kWide ? 1 : NC / CG;   // threads along positions (8 x 4 tiles)
    constexpr int PPT = kWide ? 8 : kBlockM / PG;   // positions per thread
    PipeBars *bars = reinterpret_cast<PipeBars *>(smem);
    uint8_t *stages = smem + kSimtPipeHeader;
    const int a_bytes = G * p.a_rows * 16;
    const int stage_bytes = simt_stage_bytes(p.a_rows, KC, BN, p.tap_group);
    const int tid = threadIdx.x;
    const int warp = tid / 32, lane = tid % 32;
    const long long tmo = p.timeout_ns;

    if (tid == 0) {
        for (int i = 0; i < p.a_stages; ++i) {
            dev::mbar_init(dev::smem_u32(&bars->full[i]), 1);
            dev::mbar_init(dev::smem_u32(&bars->empty[i]), NC / 32);
        }
        dev::mbar_init(dev::smem_u32(&bars->never), 1);
        bars->abort_flag = 0;
        dev::fence_mbar_init();
    }
    __syncthreads();

    if (warp == NC / 32) {
        // ------------------------------------------------------------ loader
        if (lane == 0) {
            dev::prefetch_tensormap(&p.a_map);
            dev::grid_dependency_wait();   // the frame and the packed weights come from the pack kernel
            int last_parity[kSimtMaxStages];   // parity of each stage's last fill, -1 if never filled
            for (int i = 0; i < kSimtMaxStages; ++i) last_parity[i] = -1;
            Ring ring;
            bool ok = true;
            int tile, slice, phase;
            UnitIter<kSnake> it;
            while (ok && !bars->abort_flag && it.next(p, tile, slice, phase)) {
                const PhaseDesc &pd = p.phase[phase];
                if (pd.tap_count == 0) continue;
                const int P0 = tile * kBlockM;
                const uint32_t b_bytes = static_cast<uint32_t>(pd.tap_count) * KC * BN * 4;
                for (int c = 0; c < p.n_chunks; ++c) {
                    if (!dev::mbar_wait(dev::smem_u32(&bars->empty[ring.stage]), ring.parity ^ 1, tmo)) {
                        pipe_fail(bars, p);
                        ok = false;
                        break;
                    }
                    const uint32_t bar = dev::smem_u32(&bars->full[ring.stage]);
                    const uint32_t dst = dev::smem_u32(stages + static_cast<size_t>(ring.stage) * stage_bytes);
                    dev::mbar_arrive_expect_tx(bar, static_cast<uint32_t>(a_bytes) + b_bytes);
                    // A: group g of the chunk (channels c*KC + 4g ..) into [g][a_rows][4],
                    // a_nbox copies of a_box_rows rows; rows past the frame read as zeros
                    for (int g = 0; g < G; ++g)
                        for (int b = 0; b < p.a_nbox; ++b)
                            dev::tma_load_2d(dst + static_cast<uint32_t>(g * p.a_rows + b * p.a_box_rows) * 16,
                                             &p.a_map, c * KC + 4 * g, P0 + b * p.a_box_rows, bar);
                    // B: the phase's taps of (slice, chunk), one contiguous block
                    const size_t woff = ((static_cast<size_t>(slice) * p.n_chunks + c) * p.n_taps + pd.tap_begin) *
                                        static_cast<size_t>(KC * BN);
                    dev::bulk_g2s(dst + static_cast<uint32_t>(a_bytes), p.wp + woff, b_bytes, bar);
                    last_parity[ring.stage] = static_cast<int>(ring.parity);
                    ring.next(p.a_stages);
                }
            }
            // Never leave with a copy in flight into this CTA's shared memory.
            for (int i = 0; i < p.a_stages; ++i)
                if (last_parity[i] >= 0) dev::mbar_wait(dev::smem_u32(&bars->full[i]), last_parity[i], tmo);
        }
        __syncwarp();
        return;
    }

    // --------------------------------------------------------- compute warps
    // 8 x 4 tiles: positions pg + i*PG, channels cg*4 + j; 8 x 8 tiles:
    // positions prow + 4i, channels tc + 8j
    const int cg = tid / PG, pg = tid % PG;
    const int tp = lane & 3, tc = lane >> 2, prow = warp * 32 + tp;
    Ring ring;
    bool ok = true;
    // Failure-detection test: a bounded wait on a barrier that nothing
    // completes runs out; the CTA then stops (the loader's waits run out too).
    if (p.wait_test && !__all_sync(0xffffffffu, dev::mbar_wait(dev::smem_u32(&bars->never), 0, tmo))) {
        if (lane == 0) pipe_fail(bars, p);
        ok = false;
    }
    const size_t plane = static_cast<size_t>(p.H) * p.W;
    UnitIter<kSnake> it;
    int tile, slice, phase;
    while (ok && !bars->abort_flag && it.next(p, tile, slice, phase)) {
        const PhaseDesc &pd = p.phase[phase];
        const int P0 = tile * kBlockM;
        constexpr int CPT = kWide ? 8 : 4;   // channels per thread
        float acc[PPT][CPT];
#pragma unroll
        for (int i = 0; i < PPT; ++i)
#pragma unroll
            for (int j = 0; j < CPT; ++j) acc[i][j] = 0.f;
        for (int c = 0; pd.tap_count > 0 && c < p.n_chunks; ++c) {
            if (!__all_sync(0xffffffffu, dev::mbar_wait(dev::smem_u32(&bars->full[ring.stage]), ring.parity, tmo))) {
                if (lane == 0) pipe_fail(bars, p);
                ok = false;
                break;
            }
            const uint8_t *st = stages + static_cast<size_t>(ring.stage) * stage_bytes;
            const float4 *A4 = reinterpret_cast<const float4 *>(st);
            const float4 *B4 = reinterpret_cast<const float4 *>(st + a_bytes);
            for (int t = 0; t < pd.tap_count; ++t) {
                const int shift = p.tap[pd.tap_begin + t].shift;
                if constexpr (kWide) {
                    const float4 *Ab = A4 + prow + shift;
                    const float4 *Bb = B4 + t * G * BN + tc;
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        float4 a[8], b[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) a[i] = Ab[g * p.a_rows + 4 * i];
#pragma unroll
                        for (int j = 0; j < 8; ++j) b[j] = Bb[g * BN + 8 * j];
#pragma unroll
                        for (int i = 0; i < 8; ++i)
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                acc[i][j] = fmaf(a[i].x, b[j].x, acc[i][j]);
                                acc[i][j] = fmaf(a[i].y, b[j].y, acc[i][j]);
                                acc[i][j] = fmaf(a[i].z, b[j].z, acc[i][j]);
                                acc[i][j] = fmaf(a[i].w, b[j].w, acc[i][j]);
                            }
                    }
                } else {
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
            // this warp's reads of the stage are done
            __syncwarp();
            if (lane == 0) dev::mbar_arrive(dev::smem_u32(&bars->empty[ring.stage]));
            ring.next(p.a_stages);
        }
        if (!ok) break;
        // Overwrite grad_input (phase outputs with no taps are written as 0),
        // or apply the fused epilogue.
#pragma unroll
        for (int i = 0; i < PPT; ++i) {
            const int P = P0 + (kWide ? prow + 4 * i : pg + i * PG);
            int n, q, uu;
            dev::decode_position(p, P, n, q, uu);
            if (P >= p.positions || q >= pd.Hq || uu >= pd.Wq) continue;
            const int ih = p.s * q + pd.a, iw = p.s * uu + pd.b;
#pragma unroll
            for (int j = 0; j < CPT; ++j) {
                const int ci = slice * BN + (kWide ? tc + 8 * j : cg * 4 + j);
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
}

template <int BN, int KC, bool kWide, bool kSnake = false>
cudaError_t launch_pipe_kc(const MainParams &p, const Tiling &t, cudaStream_t stream) {
    auto kern = simt_pipe_kernel<BN, KC, kWide, kSnake>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, t.smem_bytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(t.grid);
    cfg.blockDim = dim3(simt_pipe_threads(kWide));
    cfg.dynamicSmemBytes = t.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    // 8 x 8 tiles on few taps: no dependent launch (two of these CTAs fit
    // beside the pack's blocks on an SM and, resident early, slow the pack)
    cfg.numAttrs = kWide && t.tap_group <= 4 ? 0 : 1;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int BN>
cudaError_t launch_pipe_bn(const MainParams &p, const Tiling &t, cudaStream_t stream) {
    bool differ = false;   // phases of different tap counts: the sorted schedule
    for (int q = 1; q < p.n_phases; ++q) differ = differ || p.phase[q].tap_count != p.phase[0].tap_count;
    if constexpr (BN == 64) {
        if (t.simt_wide) {
            switch (t.kc + (differ ? 1 : 0)) {
                case 8: return launch_pipe_kc<BN, 8, true>(p, t, stream);
                case 16: return launch_pipe_kc<BN, 16, true>(p, t, stream);
                case 32: return launch_pipe_kc<BN, 32, true>(p, t, stream);
                case 9: return launch_pipe_kc<BN, 8, true, true>(p, t, stream);
                case 17: return launch_pipe_kc<BN, 16, true, true>(p, t, stream);
                case 33: return launch_pipe_kc<BN, 32, true, true>(p, t, stream);
                default: return cudaErrorInvalidValue;
            }
        }
    }
    if (differ) {
        switch (t.kc) {
            case 8: return launch_pipe_kc<BN, 8, false, true>(p, t, stream);
            case 16: return launch_pipe_kc<BN, 16, false, true>(p, t, stream);
            case 32: return launch_pipe_kc<BN, 32, false, true>(p, t, stream);
            default: return cudaErrorInvalidValue;
        }
    }
    switch (t.kc) {
        case 8: return launch_pipe_kc<BN, 8, false>(p, t, stream);
        case 16: return launch_pipe_kc<BN, 16, false>(p, t, stream);
        case 32: return launch_pipe_kc<BN, 32, false>(p, t, stream);
        default: return cudaErrorInvalidValue;
    }
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
    if (t.bn == 4) return t.a_tma ? cudaErrorInvalidValue : launch_bn<4>(p, t, stream);
    if (t.a_tma) {
        switch (t.bn) {
            case 16: return launch_pipe_bn<16>(p, t, stream);
            case 32: return launch_pipe_bn<32>(p, t, stream);
            case 64: return launch_pipe_bn<64>(p, t, stream);
            default: return cudaErrorInvalidValue;
        }
    }
    switch (t.bn) {
        case 16: return launch_bn<16>(p, t, stream);
        case 32: return launch_bn<32>(p, t, stream);
        case 64: return launch_bn<64>(p, t, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace dgrad

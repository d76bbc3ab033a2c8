// Weight gradient (wgrad) kernels: position frames, the tcgen05 split-K
// GEMM and the deterministic reduction of its partial tiles.
//
// Main kernel (one persistent CTA per SM, 192 threads):
//   warps 0-3  epilogue: tensor memory -> registers -> partial tile in global
//              memory (a warp stores 32 consecutive rows of one column: 128
//              contiguous bytes per store instruction)
//   warp  4    tensor-memory allocation and the MMA loop (whole warp
//              converged, one elected lane issues)
//   warp  5    one thread issuing the tensor copies: per 32-position chunk,
//              one box of each (tap, input-channel block) segment of the row
//              tile from the input copies (A) and one box of grad_out's
//              frame (B); with split precision the same boxes again from the
//              lo halves, and the MMA warp issues A_hi*B_lo, A_lo*B_hi and
//              A_hi*B_hi per chunk
// A work unit is (row tile, column tile, K split); its 128 x bn fp32
// accumulator lives in tensor memory (two sets, so that one unit's
// epilogue overlaps the next unit's MMAs).  Every wait is bounded.
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "wgrad_internal.h"

namespace dgrad {

namespace {

constexpr int kWThreads = 192;
constexpr int kWEpiWarps = 4;
constexpr int kWMmaWarp = 4;
constexpr int kWLoadWarp = 5;
constexpr int kWBarrierBytes = 1024;
constexpr uint32_t kWStageA = 128 * 128;   // 128 rows x 32 fp32

struct WRing {
    int stage = 0;
    uint32_t parity = 0;
    __device__ __forceinline__ void next(int n) {
        if (++stage == n) {
            stage = 0;
            parity ^= 1;
        }
    }
};

struct WBars {
    uint64_t full[kWgMaxStages];
    uint64_t empty[kWgMaxStages];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    volatile int abort_flag;
};
static_assert(sizeof(WBars) <= kWBarrierBytes, "barrier block");

__device__ __forceinline__ void wfail(WBars *b, const WgradMainParams &p) {
    b->abort_flag = 1;
    atomicOr(p.err, kErrTimeout);
}

struct WUnit {
    int mt, nt, c0, c1, s0, s1;
};

// Unit w = (ks * n_mt + mt) * n_nt + nt: the K split varies slowest, so the
// units running at the same time cover every row and column tile of a few
// K ranges and share their frame data in L2 (an input-copy chunk is read by
// the kH taps of its column, a grad_out chunk by every row tile).
__device__ __forceinline__ WUnit decode_unit(const WgradMainParams &p, int w) {
    WUnit u;
    const int tiles = p.n_mt * p.n_nt;
    const int ks = w / tiles;
    const int rest = w - ks * tiles;
    u.nt = rest % p.n_nt;
    u.mt = rest / p.n_nt;
    u.c0 = ks * p.cps;
    u.c1 = min(u.c0 + p.cps, p.total_chunks);
    u.s0 = u.mt * p.spt;
    u.s1 = min(u.s0 + p.spt, p.n_segs);
    return u;
}

__global__ void __launch_bounds__(kWThreads, 1) wgrad_main_kernel(const __grid_constant__ WgradMainParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    WBars *bars = reinterpret_cast<WBars *>(smem);
    const uint32_t stage0 = (dev::smem_u32(smem) + kWBarrierBytes + 1023u) & ~1023u;
    const uint32_t half_bytes = kWStageA + static_cast<uint32_t>(p.bn) * 128u;   // A | B of one half
    const uint32_t stage_bytes = half_bytes * (p.split ? 2u : 1u);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < p.stages; ++i) {
            dev::mbar_init(dev::smem_u32(&bars->full[i]), 1);
            dev::mbar_init(dev::smem_u32(&bars->empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            dev::mbar_init(dev::smem_u32(&bars->acc_full[i]), 1);
            dev::mbar_init(dev::smem_u32(&bars->acc_empty[i]), kWEpiWarps * 32);
        }
        dev::mbar_init(dev::smem_u32(&bars->drain), 1);
        bars->abort_flag = 0;
        dev::fence_mbar_init();
    }
    if (warp == kWMmaWarp) {
        dev::tmem_alloc(dev::smem_u32(&bars->tmem_base), p.tmem_cols);
        dev::tmem_relinquish();
    }
    dev::tc_fence_before();
    __syncthreads();
    dev::tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    const long long tmo = p.timeout_ns;

    if (warp == kWLoadWarp) {
        // ---------------------------------------------------- tensor copies
        if (lane == 0) {
            dev::prefetch_tensormap(&p.x_map);
            dev::prefetch_tensormap(&p.g_map);
            int last_parity[kWgMaxStages];
            for (int i = 0; i < kWgMaxStages; ++i) last_parity[i] = -1;
            WRing ring;
            bool ok = true;
            for (int w = blockIdx.x; ok && w < p.n_units && !bars->abort_flag; w += gridDim.x) {
                const WUnit u = decode_unit(p, w);
                const uint32_t bytes = (static_cast<uint32_t>((u.s1 - u.s0) * p.seg_rows) * 128u +
                                        static_cast<uint32_t>(p.bn) * 128u) *
                                       (p.split ? 2u : 1u);
                for (int c = u.c0; c < u.c1; ++c) {
                    if (!dev::mbar_wait(dev::smem_u32(&bars->empty[ring.stage]), ring.parity ^ 1, tmo)) {
                        wfail(bars, p);
                        ok = false;
                        break;
                    }
                    const uint32_t bar = dev::smem_u32(&bars->full[ring.stage]);
                    dev::mbar_arrive_expect_tx(bar, bytes);
                    const int n = c / p.cpi;
                    const int k0 = (c - n * p.cpi) * 32;
                    const uint32_t dst = stage0 + static_cast<uint32_t>(ring.stage) * stage_bytes;
                    for (int h = 0; h <= p.split; ++h) {   // half h at dst + h * half_bytes
                        const uint32_t hd = dst + static_cast<uint32_t>(h) * half_bytes;
                        for (int s = u.s0; s < u.s1; ++s) {
                            const int4 sg = p.seg[s];
                            dev::tma_load_4d(hd + static_cast<uint32_t>((s - u.s0) * p.seg_rows) * 128u, &p.x_map,
                                             k0 + sg.z, sg.y, n, sg.x + h * p.n_copies, bar);
                        }
                        dev::tma_load_3d(hd + kWStageA, &p.g_map, k0, u.nt * p.bn, n + h * p.N, bar);
                    }
                    last_parity[ring.stage] = static_cast<int>(ring.parity);
                    ring.next(p.stages);
                }
            }
            // Never leave with a copy in flight into this CTA's shared memory.
            for (int i = 0; i < p.stages; ++i)
                if (last_parity[i] >= 0) dev::mbar_wait(dev::smem_u32(&bars->full[i]), last_parity[i], tmo);
        }
        __syncwarp();
    } else if (warp == kWMmaWarp) {
        // ---------------------------------------------------- MMA issuer
        WRing ring, racc;
        bool ok = true;
        for (int w = blockIdx.x; ok && w < p.n_units && !bars->abort_flag; w += gridDim.x, racc.next(2)) {
            const WUnit u = decode_unit(p, w);
            if (!__all_sync(0xffffffffu,
                            dev::mbar_wait(dev::smem_u32(&bars->acc_empty[racc.stage]), racc.parity ^ 1, tmo))) {
                if (lane == 0) wfail(bars, p);
                break;
            }
            dev::tc_fence_after();
            const uint32_t d = tmem + static_cast<uint32_t>(racc.stage * p.bn);
            for (int c = u.c0; c < u.c1; ++c, ring.next(p.stages)) {
                if (!__all_sync(0xffffffffu,
                                dev::mbar_wait(dev::smem_u32(&bars->full[ring.stage]), ring.parity, tmo))) {
                    if (lane == 0) wfail(bars, p);
                    ok = false;
                    break;
                }
                dev::tc_fence_after();
                const uint32_t a = stage0 + static_cast<uint32_t>(ring.stage) * stage_bytes;
                const uint64_t ad = dev::smem_desc_sw128(a, 0);
                const uint64_t bd = dev::smem_desc_sw128(a + kWStageA, 0);
                if (p.split) {
                    // lo halves one half further on; the small cross terms first
                    const uint64_t adl = dev::smem_desc_sw128(a + half_bytes, 0);
                    const uint64_t bdl = dev::smem_desc_sw128(a + half_bytes + kWStageA, 0);
                    const uint64_t pa[3] = {ad, adl, ad}, pb[3] = {bdl, bd, bd};
#pragma unroll
                    for (int q = 0; q < 3; ++q)
#pragma unroll
                        for (int k8 = 0; k8 < 4; ++k8)
                            dev::mma_tf32_elect(d, dev::desc_add(pa[q], 32 * k8), dev::desc_add(pb[q], 32 * k8),
                                                p.idesc, (c > u.c0 || q > 0 || k8 > 0) ? 1u : 0u);
                } else {
#pragma unroll
                    for (int k8 = 0; k8 < 4; ++k8)
                        dev::mma_tf32_elect(d, dev::desc_add(ad, 32 * k8), dev::desc_add(bd, 32 * k8), p.idesc,
                                            (c > u.c0 || k8 > 0) ? 1u : 0u);
                }
                dev::mma_commit_elect(dev::smem_u32(&bars->empty[ring.stage]));
            }
            if (!ok) break;
            dev::mma_commit_elect(dev::smem_u32(&bars->acc_full[racc.stage]));
        }
        // Every MMA this warp issued has finished before tensor memory is freed.
        dev::mma_commit_elect(dev::smem_u32(&bars->drain));
        dev::mbar_wait(dev::smem_u32(&bars->drain), 0, tmo);
    } else {
        // ---------------------------------------------------- epilogue
        const int ew = warp;   // warps 0-3 read tensor-memory lanes 32*ew .. 32*ew + 31
        WRing racc;
        for (int w = blockIdx.x; w < p.n_units; w += gridDim.x, racc.next(2)) {
            const bool got = dev::mbar_wait(dev::smem_u32(&bars->acc_full[racc.stage]), racc.parity, tmo);
            if (!dev::named_bar_and(1, kWEpiWarps * 32, got)) {
                if (!got) wfail(bars, p);
                break;
            }
            dev::tc_fence_after();
            const uint32_t taddr = tmem + (static_cast<uint32_t>(ew * 32) << 16) + static_cast<uint32_t>(racc.stage * p.bn);
            float *dst = p.part + static_cast<size_t>(w) * p.bn * 128 + ew * 32 + lane;
            for (int j0 = 0; j0 < p.bn; j0 += 64) {
                uint32_t r[4][16];
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    if (j0 + 16 * k < p.bn) dev::tmem_ld16(taddr + static_cast<uint32_t>(j0 + 16 * k), r[k]);
                dev::tmem_wait_ld();
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    if (j0 + 16 * k >= p.bn) break;
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        dst[static_cast<size_t>(j0 + 16 * k + j) * 128] = __uint_as_float(r[k][j]);
                }
            }
            dev::tc_fence_before();
            dev::mbar_arrive(dev::smem_u32(&bars->acc_empty[racc.stage]));
        }
    }

    dev::tc_fence_before();
    __syncthreads();
    dev::tc_fence_after();
    if (warp == kWMmaWarp) dev::tmem_dealloc(tmem, p.tmem_cols);
}

// Position frames: gf (grad_out rows padded to Wf, planes to Kimg) and the
// input copies xc, TF32-rounded.  Thread item i writes the 4 consecutive
// positions 4i .. 4i+3 of the concatenated buffers (32-bit indices: the host
// keeps both below 2^31 groups); a thread takes kUnroll items a grid-stride
// apart per pass and issues all their loads before any store.  With split
// precision the item also writes lo = tf32(v - hi) one half further on.
__device__ __forceinline__ float4 wgrad_pack_item(const WgradPackParams &p, int i, int g4, int gper, int xper,
                                                  int nci, bool g_vec) {
    float v[4];
    if (i < g4) {
        const int plane = i / gper;   // n * Co + co
        const int k = (i - plane * gper) * 4;
        const float *src = p.go + static_cast<size_t>(plane) * p.oH * p.oW;
        int oh = k / p.Wf, ow = k - oh * p.Wf;
        if (g_vec && oh < p.oH) {
            const float4 t = __ldg(reinterpret_cast<const float4 *>(src + k));
            v[0] = t.x, v[1] = t.y, v[2] = t.z, v[3] = t.w;
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                v[e] = (oh < p.oH && ow < p.oW) ? __ldg(src + oh * p.oW + ow) : 0.f;
                if (++ow == p.Wf) ow = 0, ++oh;
            }
        }
    } else {
        const int j = i - g4;
        const int plane = j / xper;   // (copy * N + n) * Ci + ci
        const int k = (j - plane * xper) * 4;
        const int c = plane / nci;
        const int kw = c / p.n_rh, rh = p.rh_list[c - kw * p.n_rh];
        const float *src = p.x + static_cast<size_t>(plane - c * nci) * p.H * p.W;
        int y = k / p.Wf, u = k - y * p.Wf;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int ih = p.s * (y - p.Ty) + rh, iw = p.s * u + kw - p.pw;
            v[e] = (u < p.oW && ih >= 0 && ih < p.H && iw >= 0 && iw < p.W) ? __ldg(src + ih * p.W + iw) : 0.f;
            if (++u == p.Wf) u = 0, ++y;
        }
    }
    return make_float4(v[0], v[1], v[2], v[3]);
}

__global__ void __launch_bounds__(256) wgrad_pack_kernel(const __grid_constant__ WgradPackParams p) {
    constexpr int kUnroll = 4;
    const int total = static_cast<int>(p.g4 + p.x4);
    const int step = gridDim.x * blockDim.x;
    const int g4 = static_cast<int>(p.g4);
    const int gper = p.Kimg / 4, xper = p.Lx / 4;
    const int nci = p.N * p.Ci;
    const bool g_vec = p.Wf == p.oW;   // frame rows are grad_out rows: 16-byte loads
    for (int i0 = blockIdx.x * blockDim.x + threadIdx.x; i0 < total; i0 += kUnroll * step) {
        float4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int i = i0 + u * step;
            if (i < total) v[u] = wgrad_pack_item(p, i, g4, gper, xper, nci, g_vec);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int i = i0 + u * step;
            if (i < total) {
                float *dst = i < g4 ? p.gf + static_cast<size_t>(i) * 4 : p.xc + static_cast<size_t>(i - g4) * 4;
                const float4 x = v[u];
                const float4 hi = make_float4(dev::round_tf32(x.x), dev::round_tf32(x.y), dev::round_tf32(x.z),
                                              dev::round_tf32(x.w));
                *reinterpret_cast<float4 *>(dst) = hi;
                if (p.split) {
                    const size_t half = static_cast<size_t>(i < g4 ? p.g4 : p.x4) * 4;
                    *reinterpret_cast<float4 *>(dst + half) =
                        make_float4(dev::round_tf32(x.x - hi.x), dev::round_tf32(x.y - hi.y),
                                    dev::round_tf32(x.z - hi.z), dev::round_tf32(x.w - hi.w));
                }
            }
        }
    }
}

// grad_weight from the partial tiles: thread i takes partial element (row
// tile, column tile, column, row), row fastest (coalesced reads), sums its
// K splits (eight independent running sums, combined in a fixed order) and
// writes the OIHW element the row stands for.
__global__ void __launch_bounds__(256) wgrad_reduce_kernel(const __grid_constant__ WgradReduceParams p) {
    const long long step = static_cast<long long>(gridDim.x) * blockDim.x;
    const size_t split_stride = static_cast<size_t>(p.n_mt) * p.n_nt * p.bn * 128;   // one K split of every tile
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < p.total; i += step) {
        const int row = static_cast<int>(i & 127);
        long long rest = i >> 7;
        const int col = static_cast<int>(rest % p.bn);
        rest /= p.bn;
        const int nt = static_cast<int>(rest % p.n_nt);
        const int mt = static_cast<int>(rest / p.n_nt);
        const int sl = row / p.seg_rows;
        const int seg = mt * p.spt + sl;
        if (sl >= p.spt || seg >= p.n_segs) continue;
        const int t = seg / p.cpt;
        const int ci = (seg - t * p.cpt) * p.seg_rows + (row - sl * p.seg_rows);
        const int co = nt * p.bn + col;
        if (ci >= p.Ci || co >= p.Co) continue;
        const float *src = p.part + ((static_cast<size_t>(mt) * p.n_nt + nt) * p.bn + col) * 128 + row;
        float acc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = 0.f;
        int ks = 0;
        for (; ks + 8 <= p.n_ks; ks += 8) {
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] += __ldg(src + static_cast<size_t>(ks + j) * split_stride);
        }
        for (int j = 0; ks < p.n_ks; ++ks, ++j) acc[j] += __ldg(src + static_cast<size_t>(ks) * split_stride);
        const float sum = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
        p.dw[(static_cast<size_t>(co) * p.Ci + ci) * p.taps + t] = sum;
    }
}

}  // namespace

cudaError_t launch_wgrad_pack(const WgradPackParams &p, cudaStream_t stream) {
    const long long total = p.g4 + p.x4;
    long long blocks = (total + 4 * 256 - 1) / (4 * 256);   // four items per thread
    if (blocks > 152LL * 64) blocks = 152LL * 64;
    if (blocks < 1) blocks = 1;
    wgrad_pack_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_wgrad_main(const WgradMainParams &p, int grid, int smem_bytes, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(wgrad_main_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess) return e;
    wgrad_main_kernel<<<grid, kWThreads, smem_bytes, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_wgrad_reduce(const WgradReduceParams &p, cudaStream_t stream) {
    long long blocks = (p.total + 255) / 256;
    if (blocks > 152LL * 8) blocks = 152LL * 8;
    if (blocks < 1) blocks = 1;
    wgrad_reduce_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace dgrad

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

#include <type_traits>

#include "ptx.cuh"
#include "wgrad_internal.h"

// Cycle accounting per CTA, compiled in only with -DDGRAD_TRACE (a tracing
// build used to see where a launch spends its time).  Slots: loader waits on
// empty stages, MMA waits on full stages, MMA waits on a free accumulator,
// MMA issue, epilogue waits, epilogue work, chunks, units, cycle of the first
// full stage, of the MMA loop's end, of the epilogue's end.
#ifdef DGRAD_TRACE
namespace dgrad {
constexpr int kWTraceSlots = 16;
constexpr int kWTraceCtas = 1024;
__device__ unsigned long long g_wtrace[kWTraceCtas * kWTraceSlots];
}  // namespace dgrad
#define WG_TRACE_ADD(slot, v) \
    atomicAdd(&g_wtrace[(blockIdx.x % kWTraceCtas) * kWTraceSlots + (slot)], (unsigned long long)(v))
#define WG_TRACE_CLOCK(x) const long long x = clock64()
extern "C" int wgrad_trace_read(unsigned long long *host, int n) {
    if (n > dgrad::kWTraceCtas * dgrad::kWTraceSlots) n = dgrad::kWTraceCtas * dgrad::kWTraceSlots;
    if (cudaMemcpyFromSymbol(host, dgrad::g_wtrace, sizeof(unsigned long long) * n) != cudaSuccess) return -1;
    static unsigned long long zeros[dgrad::kWTraceCtas * dgrad::kWTraceSlots];
    return cudaMemcpyToSymbol(dgrad::g_wtrace, zeros, sizeof(zeros)) == cudaSuccess ? 0 : -1;
}
#else
#define WG_TRACE_ADD(slot, v) ((void)0)
#define WG_TRACE_CLOCK(x) ((void)0)
#endif

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
    uint64_t never;   // failure-detection test: a barrier nothing completes
    uint32_t tmem_base;
    volatile int abort_flag;
};
static_assert(sizeof(WBars) <= kWBarrierBytes, "barrier block");

__device__ __forceinline__ void wfail(WBars *b, uint32_t *err, WBars *) {
    b->abort_flag = 1;
    atomicOr(err, kErrTimeout);
}
__device__ __forceinline__ void wfail(WBars *b, const WgradMainParams &p) { wfail(b, p.err, b); }

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
        dev::mbar_init(dev::smem_u32(&bars->never), 1);
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
    dev::grid_launch_dependents();   // the reduction reads the partial tiles only after griddepcontrol.wait

    if (warp == kWLoadWarp) {
        // ---------------------------------------------------- tensor copies
        if (lane == 0) {
            dev::prefetch_tensormap(&p.x_map);
            dev::prefetch_tensormap(&p.g_map);
            dev::grid_dependency_wait();   // the frames come from the pack kernel
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
                    WG_TRACE_CLOCK(tl0);
                    if (!dev::mbar_wait(dev::smem_u32(&bars->empty[ring.stage]), ring.parity ^ 1, tmo)) {
                        wfail(bars, p);
                        ok = false;
                        break;
                    }
                    WG_TRACE_CLOCK(tl1);
                    WG_TRACE_ADD(0, tl1 - tl0);
                    const uint32_t bar = dev::smem_u32(&bars->full[ring.stage]);
                    dev::mbar_arrive_expect_tx(bar, bytes);
                    const int n = c / p.cpi;   // image group
                    const int r = c - n * p.cpi;   // chunk within the group
                    const uint32_t dst = stage0 + static_cast<uint32_t>(ring.stage) * stage_bytes;
                    for (int h = 0; h <= p.split; ++h) {   // half h at dst + h * half_bytes
                        const uint32_t hd = dst + static_cast<uint32_t>(h) * half_bytes;
                        for (int s = u.s0; s < u.s1; ++s) {
                            const int4 sg = p.seg[s];
                            const uint32_t sd = hd + static_cast<uint32_t>((s - u.s0) * p.seg_rows) * 128u;
                            if (p.blocked)   // chunk = position r of group n; the tap offset in positions
                                dev::tma_load_4d(sd, &p.x_map, 0, sg.y, n * p.Px + r + (sg.z >> 5),
                                                 sg.x + h * p.n_copies, bar);
                            else
                                dev::tma_load_4d(sd, &p.x_map, r * 32 + sg.z, sg.y, n, sg.x + h * p.n_copies, bar);
                        }
                        if (p.blocked)
                            dev::tma_load_3d(hd + kWStageA, &p.g_map, 0, u.nt * p.bn, (n + h * p.Q) * p.cpi + r, bar);
                        else
                            dev::tma_load_3d(hd + kWStageA, &p.g_map, r * 32, u.nt * p.bn, n + h * p.Q, bar);
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
        if (p.wait_test && !__all_sync(0xffffffffu, dev::mbar_wait(dev::smem_u32(&bars->never), 0, tmo))) {
            if (lane == 0) wfail(bars, p);   // the test's wait ran out: no MMA is issued
            ok = false;
        }
        WG_TRACE_CLOCK(t_start);
        bool first = true;
        for (int w = blockIdx.x; ok && w < p.n_units && !bars->abort_flag; w += gridDim.x, racc.next(2)) {
            const WUnit u = decode_unit(p, w);
            WG_TRACE_CLOCK(ta0);
            if (!__all_sync(0xffffffffu,
                            dev::mbar_wait(dev::smem_u32(&bars->acc_empty[racc.stage]), racc.parity ^ 1, tmo))) {
                if (lane == 0) wfail(bars, p);
                break;
            }
            WG_TRACE_CLOCK(ta1);
            if (lane == 0) {
                WG_TRACE_ADD(2, ta1 - ta0);
                WG_TRACE_ADD(7, 1);
            }
            dev::tc_fence_after();
            const uint32_t d = tmem + static_cast<uint32_t>(racc.stage * p.bn);
            for (int c = u.c0; c < u.c1; ++c, ring.next(p.stages)) {
                WG_TRACE_CLOCK(tf0);
                if (!__all_sync(0xffffffffu,
                                dev::mbar_wait(dev::smem_u32(&bars->full[ring.stage]), ring.parity, tmo))) {
                    if (lane == 0) wfail(bars, p);
                    ok = false;
                    break;
                }
                WG_TRACE_CLOCK(tf1);
                if (lane == 0) {
                    WG_TRACE_ADD(1, tf1 - tf0);
                    WG_TRACE_ADD(6, 1);
                    if (first) WG_TRACE_ADD(8, tf1 - t_start);
                }
                first = false;
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
                WG_TRACE_CLOCK(tf2);
                if (lane == 0) WG_TRACE_ADD(3, tf2 - tf1);
            }
            if (!ok) break;
            dev::mma_commit_elect(dev::smem_u32(&bars->acc_full[racc.stage]));
        }
        WG_TRACE_CLOCK(t_mend);
        if (lane == 0) WG_TRACE_ADD(9, t_mend - t_start);
        // Every MMA this warp issued has finished before tensor memory is freed.
        dev::mma_commit_elect(dev::smem_u32(&bars->drain));
        dev::mbar_wait(dev::smem_u32(&bars->drain), 0, tmo);
    } else {
        // ---------------------------------------------------- epilogue
        const int ew = warp;   // warps 0-3 read tensor-memory lanes 32*ew .. 32*ew + 31
        WRing racc;
        WG_TRACE_CLOCK(t_estart);
        for (int w = blockIdx.x; w < p.n_units; w += gridDim.x, racc.next(2)) {
            WG_TRACE_CLOCK(te0);
            const bool got = dev::mbar_wait(dev::smem_u32(&bars->acc_full[racc.stage]), racc.parity, tmo);
            if (!dev::named_bar_and(1, kWEpiWarps * 32, got)) {
                if (!got) wfail(bars, p);
                break;
            }
            WG_TRACE_CLOCK(te1);
            if (threadIdx.x == 0) WG_TRACE_ADD(4, te1 - te0);
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
            WG_TRACE_CLOCK(te2);
            if (threadIdx.x == 0) WG_TRACE_ADD(5, te2 - te1);
        }
        WG_TRACE_CLOCK(t_eend);
        if (threadIdx.x == 0) WG_TRACE_ADD(10, t_eend - t_estart);
    }

    dev::tc_fence_before();
    __syncthreads();
    dev::tc_fence_after();
    if (warp == kWMmaWarp) dev::tmem_dealloc(tmem, p.tmem_cols);
}

// ------------------------------------------------------------ run mode
// One persistent CTA per SM, 192 threads, the same warp roles as the segment
// kernel.  Unit w = (((q * nksq + ks) * cpt + cb) * n_nt + nt) * n_sets + set:
// chunks (frame positions) [c0, c1) of image group q, input channel block
// cb, output channel tile nt, tiles [set * tpu, ...).  Stage k of a unit is
// chunks c0 + k*L .. + L - 1: per tile one tensor copy of L + spt - 1
// position blocks, and one copy of the L grad_out blocks; chunk i of the
// stage reads tile rows from block i on and grad_out block i.  Accumulators:
// acc_sets sets of tpu * bn columns (two when they fit, so that one unit's
// epilogue overlaps the next unit's MMAs).
__device__ __forceinline__ void run_decode(const WgradRunParams &p, int w, int &q, int &cb, int &nt, int &t0,
                                           int &t1, int &c0, int &c1, int &slot) {
    const int set = w % p.n_sets;
    slot = w / p.n_sets;   // (q, ks, cb, nt): the unit's row of partial tiles
    int rest = slot;
    nt = rest % p.n_nt;
    rest /= p.n_nt;
    cb = rest % p.cpt;
    rest /= p.cpt;
    const int ks = rest % p.nksq;
    q = rest / p.nksq;
    c0 = ks * p.cps;
    c1 = min(c0 + p.cps, p.Pg);
    t0 = set * p.tpu;
    t1 = min(t0 + p.tpu, p.n_tiles);
}

template <bool kSplit>   // split precision: a template parameter, so the plain kernel carries none of it
__global__ void __launch_bounds__(kWThreads, 1) wgrad_run_kernel(const __grid_constant__ WgradRunParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    WBars *bars = reinterpret_cast<WBars *>(smem);
    const uint32_t base0 = (dev::smem_u32(smem) + kWBarrierBytes + 1023u) & ~1023u;
    const uint32_t xb = static_cast<uint32_t>(p.xbox_bytes);
    const uint32_t half_bytes = static_cast<uint32_t>(p.tpu) * xb + static_cast<uint32_t>(p.bbox_bytes);
    const uint32_t stage_bytes = half_bytes * (kSplit ? 2u : 1u);   // split precision: hi half, then lo half
    const uint32_t blk = static_cast<uint32_t>(p.seg_rows) * 128u;   // one position block of a tile copy
    const uint32_t gblk = static_cast<uint32_t>(p.bn) * 128u;        // one grad_out block
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
        dev::mbar_init(dev::smem_u32(&bars->never), 1);
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
    dev::grid_launch_dependents();   // the reduction reads the partial tiles only after griddepcontrol.wait
    const uint32_t acc_cols = static_cast<uint32_t>(p.tpu * p.bn);

    if (warp == kWLoadWarp) {
        // ---------------------------------------------------- tensor copies
        if (lane == 0) {
            dev::prefetch_tensormap(&p.x_map);
            dev::prefetch_tensormap(&p.g_map);
            dev::grid_dependency_wait();   // the frames come from the pack kernel
            int last_parity[kWgMaxStages];
            for (int i = 0; i < kWgMaxStages; ++i) last_parity[i] = -1;
            WRing ring;
            bool ok = true;
            for (int w = blockIdx.x; ok && w < p.n_units && !bars->abort_flag; w += gridDim.x) {
                int q, cb, nt, t0, t1, c0, c1, slot;
                run_decode(p, w, q, cb, nt, t0, t1, c0, c1, slot);
                const uint32_t bytes =
                    (static_cast<uint32_t>(t1 - t0) * xb + static_cast<uint32_t>(p.bbox_bytes)) * (kSplit ? 2u : 1u);
                for (int c = c0; c < c1; c += p.L) {
                    WG_TRACE_CLOCK(tl0);
                    if (!dev::mbar_wait(dev::smem_u32(&bars->empty[ring.stage]), ring.parity ^ 1, tmo)) {
                        wfail(bars, p.err, bars);
                        ok = false;
                        break;
                    }
                    WG_TRACE_CLOCK(tl1);
                    WG_TRACE_ADD(0, tl1 - tl0);
                    const uint32_t bar = dev::smem_u32(&bars->full[ring.stage]);
                    dev::mbar_arrive_expect_tx(bar, bytes);
                    for (int h = 0; h <= (kSplit ? 1 : 0); ++h) {
                        const uint32_t dst =
                            base0 + static_cast<uint32_t>(ring.stage) * stage_bytes + static_cast<uint32_t>(h) * half_bytes;
                        for (int t = t0; t < t1; ++t) {
                            const int2 tl = p.tile[t];   // copy, position offset
                            dev::tma_load_4d(dst + static_cast<uint32_t>(t - t0) * xb, &p.x_map, 0, cb * p.seg_rows,
                                             q * p.Px + c + tl.y, tl.x + h * p.n_copies, bar);
                        }
                        dev::tma_load_3d(dst + static_cast<uint32_t>(p.tpu) * xb, &p.g_map, 0, nt * p.bn,
                                         (q + h * p.Q) * p.Pg + c, bar);
                    }
                    last_parity[ring.stage] = static_cast<int>(ring.parity);
                    ring.next(p.stages);
                }
            }
            // Never leave with a copy in flight into this CTA's shared memory.
            for (int i = 0; i < p.stages; ++i)
                if (last_parity[i] >= 0)
                    dev::mbar_wait(dev::smem_u32(&bars->full[i]), static_cast<uint32_t>(last_parity[i]), tmo);
        }
        __syncwarp();
    } else if (warp == kWMmaWarp) {
        // ---------------------------------------------------- MMA issuer
        WRing ring, racc;
        bool ok = true;
        if (p.wait_test && !__all_sync(0xffffffffu, dev::mbar_wait(dev::smem_u32(&bars->never), 0, tmo))) {
            if (lane == 0) wfail(bars, p.err, bars);   // the test's wait ran out: no MMA is issued
            ok = false;
        }
        WG_TRACE_CLOCK(t_start);
        bool firstc = true;
        for (int w = blockIdx.x; ok && w < p.n_units && !bars->abort_flag; w += gridDim.x, racc.next(p.acc_sets)) {
            int q, cb, nt, t0, t1, c0, c1, slot;
            run_decode(p, w, q, cb, nt, t0, t1, c0, c1, slot);
            if (!__all_sync(0xffffffffu,
                            dev::mbar_wait(dev::smem_u32(&bars->acc_empty[racc.stage]), racc.parity ^ 1, tmo))) {
                if (lane == 0) wfail(bars, p.err, bars);
                break;
            }
            dev::tc_fence_after();
            const uint32_t d0 = tmem + static_cast<uint32_t>(racc.stage) * acc_cols;
            for (int c = c0; c < c1; c += p.L, ring.next(p.stages)) {
                WG_TRACE_CLOCK(tf0);
                if (!__all_sync(0xffffffffu,
                                dev::mbar_wait(dev::smem_u32(&bars->full[ring.stage]), ring.parity, tmo))) {
                    if (lane == 0) wfail(bars, p.err, bars);
                    ok = false;
                    break;
                }
                WG_TRACE_CLOCK(tf1);
                if (lane == 0) {
                    WG_TRACE_ADD(1, tf1 - tf0);
                    WG_TRACE_ADD(6, 1);
                    if (firstc) WG_TRACE_ADD(8, tf1 - t_start);
                }
                firstc = false;
                dev::tc_fence_after();
                const uint32_t sbase = base0 + static_cast<uint32_t>(ring.stage) * stage_bytes;
                const uint64_t xd = dev::smem_desc_sw128(sbase, 0);
                const uint64_t gd = dev::smem_desc_sw128(sbase + static_cast<uint32_t>(p.tpu) * xb, 0);
                const uint32_t lo = kSplit ? half_bytes : 0u;   // byte offset of the lo half
                const int n = min(p.L, c1 - c);
                for (int i = 0; i < n; ++i) {
                    const uint64_t bd = dev::desc_add(gd, static_cast<uint32_t>(i) * gblk);
                    const uint32_t acc = (c > c0 || i > 0) ? 1u : 0u;
                    for (int t = 0; t < t1 - t0; ++t) {
                        const uint64_t ad = dev::desc_add(xd, static_cast<uint32_t>(t) * xb + static_cast<uint32_t>(i) * blk);
                        const uint32_t d = d0 + static_cast<uint32_t>(t * p.bn);
                        if constexpr (kSplit) {   // hi*lo, lo*hi, hi*hi: the small cross terms first
#pragma unroll
                            for (int k8 = 0; k8 < 4; ++k8)
                                dev::mma_tf32_elect(d, dev::desc_add(ad, 32 * k8), dev::desc_add(bd, lo + 32 * k8),
                                                    p.idesc, k8 > 0 ? 1u : acc);
#pragma unroll
                            for (int k8 = 0; k8 < 4; ++k8)
                                dev::mma_tf32_elect(d, dev::desc_add(ad, lo + 32 * k8), dev::desc_add(bd, 32 * k8),
                                                    p.idesc, 1u);
                        }
#pragma unroll
                        for (int k8 = 0; k8 < 4; ++k8)
                            dev::mma_tf32_elect(d, dev::desc_add(ad, 32 * k8), dev::desc_add(bd, 32 * k8), p.idesc,
                                                (k8 > 0 || kSplit) ? 1u : acc);
                    }
                }
                dev::mma_commit_elect(dev::smem_u32(&bars->empty[ring.stage]));
                WG_TRACE_CLOCK(tf2);
                if (lane == 0) WG_TRACE_ADD(3, tf2 - tf1);
            }
            if (!ok) break;
            dev::mma_commit_elect(dev::smem_u32(&bars->acc_full[racc.stage]));
        }
        WG_TRACE_CLOCK(t_mend);
        if (lane == 0) WG_TRACE_ADD(9, t_mend - t_start);
        // Every MMA this warp issued has finished before tensor memory is freed.
        dev::mma_commit_elect(dev::smem_u32(&bars->drain));
        dev::mbar_wait(dev::smem_u32(&bars->drain), 0, tmo);
    } else {
        // ---------------------------------------------------- epilogue
        const int ew = warp;   // warps 0-3 read tensor-memory lanes 32*ew .. 32*ew + 31
        WRing racc;
        WG_TRACE_CLOCK(t_estart);
        for (int w = blockIdx.x; w < p.n_units; w += gridDim.x, racc.next(p.acc_sets)) {
            int q, cb, nt, t0, t1, c0, c1, slot;
            run_decode(p, w, q, cb, nt, t0, t1, c0, c1, slot);
            WG_TRACE_CLOCK(te0);
            const bool got = dev::mbar_wait(dev::smem_u32(&bars->acc_full[racc.stage]), racc.parity, tmo);
            if (!dev::named_bar_and(1, kWEpiWarps * 32, got)) {
                if (!got) wfail(bars, p.err, bars);
                break;
            }
            WG_TRACE_CLOCK(te1);
            if (threadIdx.x == 0) WG_TRACE_ADD(4, te1 - te0);
            dev::tc_fence_after();
            for (int t = t0; t < t1; ++t) {
                const uint32_t taddr = tmem + (static_cast<uint32_t>(ew * 32) << 16) + racc.stage * acc_cols +
                                       static_cast<uint32_t>((t - t0) * p.bn);
                float *dst = p.part + (static_cast<size_t>(slot) * p.n_tiles + t) * p.bn * 128 + ew * 32 + lane;
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
            }
            dev::tc_fence_before();
            dev::mbar_arrive(dev::smem_u32(&bars->acc_empty[racc.stage]));
            WG_TRACE_CLOCK(te2);
            if (threadIdx.x == 0) WG_TRACE_ADD(5, te2 - te1);
        }
        WG_TRACE_CLOCK(t_eend);
        if (threadIdx.x == 0) WG_TRACE_ADD(10, t_eend - t_estart);
    }

    dev::tc_fence_before();
    __syncthreads();
    dev::tc_fence_after();
    if (warp == kWMmaWarp) dev::tmem_dealloc(tmem, p.tmem_cols);
}

// Position frames: gf (grad_out) and the input copies xc, f images
// interleaved along K, TF32-rounded.  Thread item i writes the 4 consecutive
// K elements 4i .. 4i+3 of the concatenated buffers (32-bit indices: the
// host keeps both below 2^31 groups); a thread takes kUnroll items a
// grid-stride apart per pass and issues all their loads before any store.
// With split precision the item also writes lo = tf32(v - hi) one half
// further on.
__device__ __forceinline__ float4 wgrad_pack_item(const WgradPackParams &p, int i, int g4, int gper, int xper,
                                                  int qci, bool g_vec) {
    float v[4];
    const int fm = (1 << p.lf) - 1;
    if (i < g4) {
        const int plane = i / gper;   // q * Co + co
        const int k = (i - plane * gper) * 4;
        const int q = plane / p.Co, co = plane - q * p.Co;
        if (g_vec) {   // f = 1 and frame rows are grad_out rows: one 16-byte load
            const int oh = k / p.Wf;
            const float *src = p.go + static_cast<size_t>(plane) * p.oH * p.oW;
            if (oh < p.oH) {
                const float4 t = __ldg(reinterpret_cast<const float4 *>(src + k));
                v[0] = t.x, v[1] = t.y, v[2] = t.z, v[3] = t.w;
            } else {
                v[0] = v[1] = v[2] = v[3] = 0.f;
            }
        } else {
            int j = k & fm, pos = k >> p.lf;
            int oh = pos / p.Wf, ow = pos - oh * p.Wf;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int n = (q << p.lf) + j;
                v[e] = (n < p.N && oh < p.oH && ow < p.oW)
                           ? __ldg(p.go + ((static_cast<size_t>(n) * p.Co + co) * p.oH + oh) * p.oW + ow)
                           : 0.f;
                if (++j > fm) {   // next position
                    j = 0;
                    if (++ow == p.Wf) ow = 0, ++oh;
                }
            }
        }
    } else {
        const int jx = i - g4;
        const int plane = jx / xper;   // (copy * Q + q) * Ci + ci
        const int k = (jx - plane * xper) * 4;
        const int c = plane / qci;
        const int rest = plane - c * qci;
        const int q = rest / p.Ci, ci = rest - q * p.Ci;
        const int4 cp = p.copy[c];   // rh, rw, r
        int j = k & fm, pos = k >> p.lf;
        int y = pos / p.Wf, u = pos - y * p.Wf;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int n = (q << p.lf) + j;
            const int ih = p.s * (y - p.Ty) + cp.x, iw = p.s * (u - p.Tu + cp.z) + cp.y;
            v[e] = (n < p.N && ih >= 0 && ih < p.H && iw >= 0 && iw < p.W)
                       ? __ldg(p.x + ((static_cast<size_t>(n) * p.Ci + ci) * p.H + ih) * p.W + iw)
                       : 0.f;
            if (++j > fm) {   // next position
                j = 0;
                if (++u == p.Wf) u = 0, ++y;
            }
        }
    }
    return make_float4(v[0], v[1], v[2], v[3]);
}

__global__ void __launch_bounds__(256) wgrad_pack_kernel(const __grid_constant__ WgradPackParams p) {
    // Let the main kernel start its prologue while this grid runs; it reads
    // what this grid writes only after griddepcontrol.wait.
    dev::grid_launch_dependents();
    constexpr int kUnroll = 4;
    const int total = static_cast<int>(p.g4 + p.x4);
    const int step = gridDim.x * blockDim.x;
    const int g4 = static_cast<int>(p.g4);
    const int gper = p.Kimg / 4, xper = p.Lx / 4;
    const int qci = p.Q * p.Ci;
    const bool g_vec = p.lf == 0 && p.Wf == p.oW;
    for (int i0 = blockIdx.x * blockDim.x + threadIdx.x; i0 < total; i0 += kUnroll * step) {
        float4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int i = i0 + u * step;
            if (i < total) v[u] = wgrad_pack_item(p, i, g4, gper, xper, qci, g_vec);
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

// Batch-blocked frames: block b transposes kWgPackTile frame positions of
// kWgPackCh consecutive channels for the 32 images of one group, gathered
// image by image (a warp reads 32 consecutive positions of one image plane)
// into shared memory and written position by position (a warp writes the 32
// images of one position and channel: one 128-byte row; the block's channels
// are adjacent rows).  Blocks [0, g_tiles) fill gf, the rest xc; channel
// blocks vary fastest, so neighbouring blocks write neighbouring rows.  The
// block's decode and each thread's position arithmetic are shared by its
// channels, and all of a thread's loads are issued before the first store.
__global__ void __launch_bounds__(256) wgrad_pack_blocked_kernel(const __grid_constant__ WgradPackParams p) {
    dev::grid_launch_dependents();   // as wgrad_pack_kernel
    __shared__ float tile[kWgPackCh][kWgPackTile][33];
    const int b = static_cast<int>(blockIdx.x);   // the host keeps the block count below 2^31
    const bool is_g = b < p.g_tiles;
    const int bl = is_g ? b : b - static_cast<int>(p.g_tiles);
    const int C = is_g ? p.Co : p.Ci;
    const int P = is_g ? p.Pg : p.Px;
    const int ntile = (P + kWgPackTile - 1) / kWgPackTile;
    const int ncb = (C + kWgPackCh - 1) / kWgPackCh;
    const int cb = bl % ncb;
    int rest = bl / ncb;
    const int pt = rest % ntile;
    rest /= ntile;
    const int q = rest % p.Q;
    const int c = rest / p.Q;   // input copy (xc only)
    const int p0 = pt * kWgPackTile;
    const int ch0 = cb * kWgPackCh;
    const int nch = min(kWgPackCh, C - ch0);
    // gather: thread t reads position p0 + (t & 63) of images (t >> 6) + 4e, for each channel
    {
        const int pp = threadIdx.x & (kWgPackTile - 1);
        const int pos = p0 + pp;
        const int y = pos / p.Wf, u = pos - y * p.Wf;
        int ih, iw, hh, ww;
        const float *base;
        size_t img_stride;
        if (is_g) {
            ih = y, iw = u, hh = p.oH, ww = p.oW;
            base = p.go + static_cast<size_t>(ch0) * p.oH * p.oW;
            img_stride = static_cast<size_t>(p.Co) * p.oH * p.oW;
        } else {
            const int4 cp = p.copy[c];
            ih = p.s * (y - p.Ty) + cp.x, iw = p.s * (u - p.Tu) + cp.y, hh = p.H, ww = p.W;
            base = p.x + static_cast<size_t>(ch0) * p.H * p.W;
            img_stride = static_cast<size_t>(p.Ci) * p.H * p.W;
        }
        const size_t plane = static_cast<size_t>(hh) * ww;
        const bool ok = pos < P && ih >= 0 && ih < hh && iw >= 0 && iw < ww;
        const int jt = threadIdx.x >> 6;
        const int n_ok = p.N - q * 32;   // images of this group that exist
        const float *src = base + (ok ? static_cast<size_t>(ih) * ww + iw : 0) + static_cast<size_t>(q * 32 + jt) * img_stride;
        const size_t step = 4 * img_stride;
        float v[kWgPackCh][8];
#pragma unroll
        for (int k = 0; k < kWgPackCh; ++k)
#pragma unroll
            for (int e = 0; e < 8; ++e)
                v[k][e] = (ok && k < nch && jt + 4 * e < n_ok) ? __ldg(src + k * plane + e * step) : 0.f;
#pragma unroll
        for (int k = 0; k < kWgPackCh; ++k)
#pragma unroll
            for (int e = 0; e < 8; ++e) tile[k][pp][jt + 4 * e] = v[k][e];
    }
    __syncthreads();
    // write: thread t writes images 4*(t & 7) .. +3 of positions p0 + (t >> 3) + 32e, each channel (one 16-byte
    // store each; eight threads write one 128-byte row)
    const int j4 = (threadIdx.x & 7) * 4;
    float *dst;
    size_t half;
    if (is_g) {
        dst = p.gf + (static_cast<size_t>(q) * p.Pg * C + ch0) * 32 + j4;
        half = static_cast<size_t>(p.g4) * 4;
    } else {
        dst = p.xc + ((static_cast<size_t>(c) * p.Q + q) * p.Px * C + ch0) * 32 + j4;
        half = static_cast<size_t>(p.x4) * 4;
    }
    const size_t row = static_cast<size_t>(C) * 32;   // floats between consecutive positions
#pragma unroll
    for (int e = 0; e < kWgPackTile / 32; ++e) {
        const int pp = (threadIdx.x >> 3) + 32 * e;
        if (p0 + pp >= P) break;
        float *d = dst + static_cast<size_t>(p0 + pp) * row;
#pragma unroll
        for (int k = 0; k < kWgPackCh; ++k) {
            if (k >= nch) break;
            const float4 v = make_float4(tile[k][pp][j4], tile[k][pp][j4 + 1], tile[k][pp][j4 + 2], tile[k][pp][j4 + 3]);
            const float4 hi = make_float4(dev::round_tf32(v.x), dev::round_tf32(v.y), dev::round_tf32(v.z),
                                          dev::round_tf32(v.w));
            *reinterpret_cast<float4 *>(d + k * 32) = hi;
            if (p.split)
                *reinterpret_cast<float4 *>(d + k * 32 + half) =
                    make_float4(dev::round_tf32(v.x - hi.x), dev::round_tf32(v.y - hi.y),
                                dev::round_tf32(v.z - hi.z), dev::round_tf32(v.w - hi.w));
        }
    }
}

// grad_weight from the partial tiles.  A thread takes four consecutive
// partial elements (rows of one column: one 16-byte load per split); the
// eight warps of a block form 8 / W groups of W warps, warp w of a group
// summing K splits w, w + W, ... of the group's 128 elements (W = the power of
// two that leaves each warp at most about eight splits), and the group's
// first warp adds the W sums in a fixed order and writes each element's OIHW
// position.  Deterministic for a given plan.
__device__ __forceinline__ void wgrad_reduce_store(const WgradReduceParams &p, long long i, float sum) {
    if (p.plane) {   // split = [row tile][column][rows of the tile]; rows (kw, ci), columns (kh, co)
        const long long tile = 128LL * p.bn;
        const int mt = static_cast<int>(i / tile);
        const long long w = i - mt * tile;
        const int rows = min(128, p.a_rows - mt * 128);
        const int col = static_cast<int>(w / rows), r = mt * 128 + static_cast<int>(w - static_cast<long long>(col) * rows);
        const int kw = r / p.ci_rows, ci = r - kw * p.ci_rows;
        const int kh = col / p.co_rows, co = col - kh * p.co_rows;
        if (ci >= p.Ci || co >= p.Co || kh >= p.kH) return;
        p.dw[(static_cast<size_t>(co) * p.Ci + ci) * p.taps + kh * p.kW + kw] = sum;
        return;
    }
    const int row = static_cast<int>(i & 127);
    long long rest = i >> 7;
    const int col = static_cast<int>(rest % p.bn);
    rest /= p.bn;
    const int sl = row / p.seg_rows;
    int t, ci, nt;
    if (p.run_mode) {   // element (cb, nt, tile, col, row); tile = taps of one group at adjacent positions
        const int tile = static_cast<int>(rest % p.n_tiles);
        rest /= p.n_tiles;
        nt = static_cast<int>(rest % p.n_nt);
        const int cb = static_cast<int>(rest / p.n_nt);
        const int2 tl = p.tile[tile];
        const int j = tl.y + sl;   // tap within the group
        const int2 gr = p.grp[tl.x];
        if (sl >= p.spt || j >= gr.y) return;
        t = p.taps_of[gr.x + j];
        ci = cb * p.seg_rows + (row - sl * p.seg_rows);
    } else {       // element (mt, nt, col, row); row tile of (tap, ci block) segments
        nt = static_cast<int>(rest % p.n_nt);
        const int mt = static_cast<int>(rest / p.n_nt);
        const int seg = mt * p.spt + sl;
        if (sl >= p.spt || seg >= p.n_segs) return;
        t = seg / p.cpt;
        ci = (seg - t * p.cpt) * p.seg_rows + (row - sl * p.seg_rows);
    }
    const int co = nt * p.bn + col;
    if (ci >= p.Ci || co >= p.Co) return;
    p.dw[(static_cast<size_t>(co) * p.Ci + ci) * p.taps + t] = sum;
}

template <int kV>   // partial elements per thread: 4 (16-byte loads) or 1 (more threads for deep split counts)
__global__ void __launch_bounds__(256) wgrad_reduce_kernel(const __grid_constant__ WgradReduceParams p) {
    using Vec = typename std::conditional<kV == 4, float4, float>::type;
    __shared__ Vec wsum[8][32];
    dev::grid_dependency_wait();   // the partial tiles come from the main kernel
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int W = p.red_warps;                 // warps per element group (1, 2, 4 or 8)
    const int grp = warp / W, wi = warp - grp * W;
    const long long e0 = (static_cast<long long>(blockIdx.x) * (8 / W) + grp) * (32 * kV) + lane * kV;
    const size_t st = static_cast<size_t>(p.total) / kV;   // one K split of every tile, in Vec units
    float a[4][kV];   // four independent chains: splits wi + W*(4i + c) go to chain c
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int k = 0; k < kV; ++k) a[c][k] = 0.f;
    if (e0 < p.total) {
        const Vec *src = reinterpret_cast<const Vec *>(p.part + static_cast<size_t>(e0));
        for (int ks = wi; ks < p.n_ks; ks += 4 * W) {
            Vec u[4];
#pragma unroll
            for (int c = 0; c < 4; ++c)
                if (ks + c * W < p.n_ks) u[c] = __ldg(src + static_cast<size_t>(ks + c * W) * st);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                if (ks + c * W >= p.n_ks) break;
                const float *uf = reinterpret_cast<const float *>(&u[c]);
#pragma unroll
                for (int k = 0; k < kV; ++k) a[c][k] += uf[k];
            }
        }
    }
    Vec mine;
    float *mf = reinterpret_cast<float *>(&mine);
#pragma unroll
    for (int k = 0; k < kV; ++k) mf[k] = (a[0][k] + a[1][k]) + (a[2][k] + a[3][k]);
    wsum[warp][lane] = mine;
    __syncthreads();
    if (wi != 0 || e0 >= p.total) return;
    float sum[kV];
#pragma unroll
    for (int k = 0; k < kV; ++k) sum[k] = mf[k];
    for (int j = 1; j < W; ++j) {   // fixed order
        const Vec v = wsum[warp + j][lane];
        const float *vf = reinterpret_cast<const float *>(&v);
#pragma unroll
        for (int k = 0; k < kV; ++k) sum[k] += vf[k];
    }
#pragma unroll
    for (int k = 0; k < kV; ++k) wgrad_reduce_store(p, e0 + k, sum[k]);
}

}  // namespace

cudaError_t launch_wgrad_pack(const WgradPackParams &p, cudaStream_t stream) {
    if (p.blocked) {
        const long long blocks = p.g_tiles + p.x_tiles;
        if (blocks < 1 || blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
        wgrad_pack_blocked_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p);
        return cudaGetLastError();
    }
    const long long total = p.g4 + p.x4;
    long long blocks = (total + 4 * 256 - 1) / (4 * 256);   // four items per thread
    if (blocks > 152LL * 64) blocks = 152LL * 64;
    if (blocks < 1) blocks = 1;
    wgrad_pack_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(p);
    return cudaGetLastError();
}

// Launch with programmatic dependent launch: the kernel may start while the
// previous kernel on the stream finishes, and waits for its results with
// griddepcontrol.wait.
template <typename Params>
cudaError_t launch_pdl(void (*kern)(Params), const Params &p, int grid, int threads, int smem_bytes,
                       cudaStream_t stream) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

cudaError_t launch_wgrad_main(const WgradMainParams &p, int grid, int smem_bytes, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(wgrad_main_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess) return e;
    return launch_pdl(wgrad_main_kernel, p, grid, kWThreads, smem_bytes, stream);
}

cudaError_t launch_wgrad_run(const WgradRunParams &p, int grid, int smem_bytes, cudaStream_t stream) {
    auto kern = p.split ? wgrad_run_kernel<true> : wgrad_run_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, p, grid, kWThreads, smem_bytes, stream);
}

cudaError_t launch_wgrad_reduce(const WgradReduceParams &p, cudaStream_t stream) {
    // 16-byte loads (four in flight per thread: 64 bytes) unless that leaves
    // fewer threads than one block per SM
    const int v = (p.total / 4) * p.red_warps >= 152LL * 256 ? 4 : 1;
    const long long per_block = 32LL * v * (8 / p.red_warps);   // partial elements per block
    const long long blocks = (p.total + per_block - 1) / per_block;
    if (blocks < 1 || blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    return v == 4 ? launch_pdl(wgrad_reduce_kernel<4>, p, static_cast<int>(blocks), 256, 0, stream)
                  : launch_pdl(wgrad_reduce_kernel<1>, p, static_cast<int>(blocks), 256, 0, stream);
}

}  // namespace dgrad

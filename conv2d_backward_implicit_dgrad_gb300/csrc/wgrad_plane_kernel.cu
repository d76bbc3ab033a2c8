// Weight gradient, plane mode: the tcgen05 split-K GEMM reading the
// caller's NCHW tensors directly (no frames, no pack pass).  The operand
// definitions are in wgrad_internal.h (WgradPlaneParams).
//
// One CTA per SM, 192 threads, over the chunks [c0, c1) of its K range
// (chunk c: image c / cpi, positions 32*(c % cpi) .. + 31):
//   warps 0-3  build the shifted kernel columns of A from the unshifted
//              one in shared memory: a thread takes one row (kw, ci) of a
//              chunk, reads its source row's eight 16-byte pieces, shifts
//              them by kw - pw positions (the piece past the chunk's edge
//              comes from one 16-byte load of the input), zeroes the
//              positions whose column leaves the row, and writes the
//              destination row (both rows have the same swizzle phase);
//              after the last chunk, the epilogue: tensor memory ->
//              registers -> this CTA's partial split (a warp stores 32
//              consecutive rows of one column per instruction)
//   warp  4    tensor-memory allocation and the MMA loop (n_mt tiles of
//              128 x nb x 8 per K step, four K steps per chunk)
//   warp  5    one thread issuing the tensor copies: per chunk the
//              unshifted column of A and the kH row-shifted copies of B
// A stage is [A: n_mt x 128 rows][B: nb rows], every row 128 bytes (32 fp32
// positions) in the 128-byte swizzle; the MMA takes the TF32 part of each
// value.  Rows no copy writes (A past kW * ci_rows, B past kH * co_rows) are
// zeroed once at the start and feed only accumulator rows and columns the
// reduction ignores.  Every wait is bounded.
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "wgrad_internal.h"

// Cycle accounting per CTA, compiled in only with -DDGRAD_TRACE (a tracing
// build).  Slots: loader waits on empty stages, MMA waits on full stages,
// gather waits on empty stages, gather issue, MMA issue, epilogue wait,
// epilogue work, chunks, cycle of the first full stage, of the MMA loop's
// end, of the gather's last copy landing, of the loader's first copy.
#ifdef DGRAD_TRACE
namespace dgrad {
constexpr int kPTraceSlots = 12;
constexpr int kPTraceCtas = 1024;
__device__ unsigned long long g_ptrace[kPTraceCtas * kPTraceSlots];
}  // namespace dgrad
#define WP_TRACE_ADD(slot, v) \
    atomicAdd(&g_ptrace[(blockIdx.x % kPTraceCtas) * kPTraceSlots + (slot)], (unsigned long long)(v))
#define WP_TRACE_CLOCK(x) const long long x = clock64()
extern "C" int wgrad_plane_trace_read(unsigned long long *host, int n) {
    if (n > dgrad::kPTraceCtas * dgrad::kPTraceSlots) n = dgrad::kPTraceCtas * dgrad::kPTraceSlots;
    if (cudaMemcpyFromSymbol(host, dgrad::g_ptrace, sizeof(unsigned long long) * n) != cudaSuccess) return -1;
    static unsigned long long zeros[dgrad::kPTraceCtas * dgrad::kPTraceSlots];
    return cudaMemcpyToSymbol(dgrad::g_ptrace, zeros, sizeof(zeros)) == cudaSuccess ? 0 : -1;
}
#else
#define WP_TRACE_ADD(slot, v) ((void)0)
#define WP_TRACE_CLOCK(x) ((void)0)
#endif

namespace dgrad {

namespace {

constexpr int kPThreads = 192;
constexpr int kPGatherWarps = 4;
constexpr int kPMmaWarp = 4;
constexpr int kPLoadWarp = 5;
constexpr int kPBarrierBytes = 1024;
constexpr uint32_t kPTile = 128 * 128;   // one 128-row tile of A
constexpr int kPMaxShifts = 6;           // kernel columns other than pw (kW <= 7)
constexpr int kPMaxRowsPerThread = 4;    // shifted rows per thread: (kW - 1) * ci_rows <= 512

__device__ __forceinline__ float4 lds128(uint32_t a) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ void sts128(uint32_t a, float4 v) {
    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
                 : "memory");
}

// Elements E .. E + 3 of the eight values (a, b), E in 1 .. 3.
template <int E>
__device__ __forceinline__ float4 window4(float4 a, float4 b) {
    if constexpr (E == 1) return make_float4(a.y, a.z, a.w, b.x);
    if constexpr (E == 2) return make_float4(a.z, a.w, b.x, b.y);
    return make_float4(a.w, b.x, b.y, b.z);
}

__device__ __forceinline__ float4 keep4(float4 v, uint32_t bits) {
    return make_float4((bits & 1u) ? v.x : 0.f, (bits & 2u) ? v.y : 0.f, (bits & 4u) ? v.z : 0.f,
                       (bits & 8u) ? v.w : 0.f);
}

// Destination row (kw, ci) from source row (pw, ci) of the same stage:
// position k takes source position k + D (0 < |D| < 4), from the edge piece
// past either end; positions whose bit in `keep` is clear are zero.  Both
// rows have swizzle phase ph: 16-byte piece j sits at (j ^ ph) * 16.  The
// eight loads are issued before the first store.
template <int D>
__device__ __forceinline__ void shift_row(uint32_t src, uint32_t dst, int ph, float4 edge, uint32_t keep) {
    float4 v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = lds128(src + (static_cast<uint32_t>(j ^ ph) << 4));
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        float4 w;
        if constexpr (D < 0)
            w = window4<4 + D>(j == 0 ? edge : v[j - 1], v[j]);
        else
            w = window4<D>(v[j], j == 7 ? edge : v[j + 1]);
        sts128(dst + (static_cast<uint32_t>(j ^ ph) << 4), keep4(w, keep >> (4 * j)));
    }
}

__device__ __forceinline__ void shift_row_any(int d, uint32_t src, uint32_t dst, int ph, float4 edge, uint32_t keep) {
    switch (d) {
        case -3: shift_row<-3>(src, dst, ph, edge, keep); break;
        case -2: shift_row<-2>(src, dst, ph, edge, keep); break;
        case -1: shift_row<-1>(src, dst, ph, edge, keep); break;
        case 1: shift_row<1>(src, dst, ph, edge, keep); break;
        case 2: shift_row<2>(src, dst, ph, edge, keep); break;
        default: shift_row<3>(src, dst, ph, edge, keep); break;
    }
}

struct PBars {
    uint64_t xfull[kWgMaxStages];   // the stage's input copy has landed (expect_tx)
    uint64_t bfull[kWgMaxStages];   // its grad_out copies have landed (expect_tx)
    uint64_t sfull[kWgMaxStages];   // its shifted rows are written (one arrival per shifting thread)
    uint64_t empty[kWgMaxStages];   // the stage's MMAs have read it
    uint64_t acc_full;
    uint64_t drain;
    uint64_t never;        // failure-detection test: a barrier nothing completes
    uint64_t tmem_ready;   // the MMA warp has allocated tensor memory (tmem_base is written)
    uint32_t tmem_base;
    volatile int abort_flag;
};
static_assert(sizeof(PBars) <= kPBarrierBytes, "barrier block");

struct PRing {
    int stage = 0;
    uint32_t parity = 0;
    __device__ __forceinline__ void next(int n) {
        if (++stage == n) {
            stage = 0;
            parity ^= 1;
        }
    }
};

__device__ __forceinline__ void pfail(PBars *b, uint32_t *err) {
    b->abort_flag = 1;
    atomicOr(err, kErrTimeout);
}

__global__ void __launch_bounds__(kPThreads, 1) wgrad_plane_kernel(const __grid_constant__ WgradPlaneParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    PBars *bars = reinterpret_cast<PBars *>(smem);
    const uint32_t base0 = (dev::smem_u32(smem) + kPBarrierBytes + 1023u) & ~1023u;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    WP_TRACE_CLOCK(t_start);
    const int c0 = static_cast<int>(static_cast<long long>(blockIdx.x) * p.total_chunks / gridDim.x);
    const int c1 = static_cast<int>(static_cast<long long>(blockIdx.x + 1) * p.total_chunks / gridDim.x);
    const int a_rows = p.kW * p.ci_rows, b_rows = p.kH * p.co_rows;
    if (threadIdx.x == 0) {
        for (int i = 0; i < p.stages; ++i) {
            dev::mbar_init(dev::smem_u32(&bars->xfull[i]), 1);
            dev::mbar_init(dev::smem_u32(&bars->bfull[i]), 1);
            dev::mbar_init(dev::smem_u32(&bars->sfull[i]), kPGatherWarps * 32);
            dev::mbar_init(dev::smem_u32(&bars->empty[i]), 1);
        }
        dev::mbar_init(dev::smem_u32(&bars->acc_full), 1);
        dev::mbar_init(dev::smem_u32(&bars->drain), 1);
        dev::mbar_init(dev::smem_u32(&bars->never), 1);
        dev::mbar_init(dev::smem_u32(&bars->tmem_ready), 1);
        bars->abort_flag = 0;
        dev::fence_mbar_init();
    }
    // Rows that no copy writes: zero, once (16 bytes per thread and step).
    {
        const uint32_t a_pad = static_cast<uint32_t>(p.n_mt * 128 - a_rows) * 128u;
        const uint32_t b_pad = static_cast<uint32_t>(p.nb - b_rows) * 128u;
        for (int s = 0; s < p.stages; ++s) {
            const uint32_t st = base0 + static_cast<uint32_t>(s) * p.stage_bytes;
            const uint32_t az = st + static_cast<uint32_t>(a_rows) * 128u;
            const uint32_t bz = st + p.a_bytes + static_cast<uint32_t>(b_rows) * 128u;
            for (uint32_t o = threadIdx.x * 16u; o < a_pad; o += kPThreads * 16u)
                asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(az + o), "r"(0u) : "memory");
            for (uint32_t o = threadIdx.x * 16u; o < b_pad; o += kPThreads * 16u)
                asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(bz + o), "r"(0u) : "memory");
        }
        dev::fence_proxy_async_smem();
    }
    // The loader starts at once; the MMA warp allocates tensor memory after
    // this barrier (the allocation's latency overlaps the first copies).
    __syncthreads();
    const long long tmo = p.timeout_ns;
    dev::grid_launch_dependents();   // the reduction reads the partial splits only after griddepcontrol.wait

    if (warp == kPLoadWarp) {
        // ---------------------------------------------------- tensor copies
        if (lane == 0) {
            dev::prefetch_tensormap(&p.x_map);
            dev::prefetch_tensormap(&p.g_map);
            dev::grid_dependency_wait();   // the inputs may come from the previous kernel
            const uint32_t xbytes = static_cast<uint32_t>(p.ci_rows) * 128u;
            const uint32_t bbytes = static_cast<uint32_t>(b_rows) * 128u;
            int last_parity[kWgMaxStages];
            for (int i = 0; i < kWgMaxStages; ++i) last_parity[i] = -1;
            PRing ring;
            for (int c = c0; c < c1 && !bars->abort_flag; ++c) {
                WP_TRACE_CLOCK(tl0);
                if (!dev::mbar_wait(dev::smem_u32(&bars->empty[ring.stage]), ring.parity ^ 1, tmo)) {
                    pfail(bars, p.err);
                    break;
                }
                WP_TRACE_CLOCK(tl1);
                WP_TRACE_ADD(0, tl1 - tl0);
                if (c == c0) WP_TRACE_ADD(11, tl1 - t_start);
                const int n = c / p.cpi;
                const int q0 = (c - n * p.cpi) * 32;
                const uint32_t dst = base0 + static_cast<uint32_t>(ring.stage) * p.stage_bytes;
                // the input first: the shifting threads wait for it alone
                const uint32_t xbar = dev::smem_u32(&bars->xfull[ring.stage]);
                dev::mbar_arrive_expect_tx(xbar, xbytes);
                dev::tma_load_3d(dst + static_cast<uint32_t>(p.pw * p.ci_rows) * 128u, &p.x_map, q0, 0, n, xbar);
                const uint32_t bbar = dev::smem_u32(&bars->bfull[ring.stage]);
                dev::mbar_arrive_expect_tx(bbar, bbytes);
                for (int kh = 0; kh < p.kH; ++kh)   // row shift: a multiple of 4 positions (W is)
                    dev::tma_load_3d(dst + p.a_bytes + static_cast<uint32_t>(kh * p.co_rows) * 128u, &p.g_map,
                                     q0 - (kh - p.ph) * p.W, 0, n, bbar);
                last_parity[ring.stage] = static_cast<int>(ring.parity);
                ring.next(p.stages);
            }
            // Never leave with a copy in flight into this CTA's shared memory.
            for (int i = 0; i < p.stages; ++i)
                if (last_parity[i] >= 0) {
                    dev::mbar_wait(dev::smem_u32(&bars->xfull[i]), static_cast<uint32_t>(last_parity[i]), tmo);
                    dev::mbar_wait(dev::smem_u32(&bars->bfull[i]), static_cast<uint32_t>(last_parity[i]), tmo);
                }
        }
        __syncwarp();
    } else if (warp == kPMmaWarp) {
        // ---------------------------------------------------- MMA issuer
        dev::tmem_alloc(dev::smem_u32(&bars->tmem_base), p.tmem_cols);
        dev::tmem_relinquish();
        dev::tc_fence_before();
        __syncwarp();
        dev::tc_fence_after();
        const uint32_t tmem = bars->tmem_base;
        if (lane == 0) dev::mbar_arrive(dev::smem_u32(&bars->tmem_ready));   // for the epilogue warps
        PRing ring;
        bool ok = true;
        if (p.wait_test && !__all_sync(0xffffffffu, dev::mbar_wait(dev::smem_u32(&bars->never), 0, tmo))) {
            if (lane == 0) pfail(bars, p.err);   // the test's wait ran out: no MMA is issued
            ok = false;
        }
        for (int c = c0; ok && c < c1 && !bars->abort_flag; ++c, ring.next(p.stages)) {
            WP_TRACE_CLOCK(tf0);
            const bool landed = dev::mbar_wait(dev::smem_u32(&bars->xfull[ring.stage]), ring.parity, tmo) &&
                                dev::mbar_wait(dev::smem_u32(&bars->bfull[ring.stage]), ring.parity, tmo) &&
                                dev::mbar_wait(dev::smem_u32(&bars->sfull[ring.stage]), ring.parity, tmo);
            if (!__all_sync(0xffffffffu, landed)) {
                if (lane == 0) pfail(bars, p.err);
                ok = false;
                break;
            }
            WP_TRACE_CLOCK(tf1);
            if (lane == 0) {
                WP_TRACE_ADD(1, tf1 - tf0);
                WP_TRACE_ADD(7, 1);
                if (c == c0) WP_TRACE_ADD(8, tf1 - t_start);
            }
            dev::tc_fence_after();
            const uint32_t a = base0 + static_cast<uint32_t>(ring.stage) * p.stage_bytes;
            const uint64_t bd = dev::smem_desc_sw128(a + p.a_bytes, 0);
            for (int mt = 0; mt < p.n_mt; ++mt) {
                const uint64_t ad = dev::smem_desc_sw128(a + static_cast<uint32_t>(mt) * kPTile, 0);
                const uint32_t d = tmem + static_cast<uint32_t>(mt * p.nb);
#pragma unroll
                for (int k8 = 0; k8 < 4; ++k8)
                    dev::mma_tf32_elect(d, dev::desc_add(ad, 32 * k8), dev::desc_add(bd, 32 * k8), p.idesc,
                                        (c > c0 || k8 > 0) ? 1u : 0u);
            }
            dev::mma_commit_elect(dev::smem_u32(&bars->empty[ring.stage]));
            WP_TRACE_CLOCK(tf2);
            if (lane == 0) WP_TRACE_ADD(4, tf2 - tf1);
        }
        WP_TRACE_CLOCK(t_mend);
        if (lane == 0) WP_TRACE_ADD(9, t_mend - t_start);
        if (ok && !bars->abort_flag) dev::mma_commit_elect(dev::smem_u32(&bars->acc_full));
        // Every MMA this warp issued has finished before tensor memory is freed.
        dev::mma_commit_elect(dev::smem_u32(&bars->drain));
        dev::mbar_wait(dev::smem_u32(&bars->drain), 0, tmo);
    } else {
        // ---------------------------------------------------- shifted columns, then epilogue
        dev::grid_dependency_wait();   // the input may come from the previous kernel
        const int t = threadIdx.x;     // 0 .. 127
        const int n_rows = (p.kW - 1) * p.ci_rows;   // rows (kw != pw, ci)
        // This thread's rows r = t, t + 128, ... (the same in every chunk):
        // source and destination offsets in a stage, swizzle phase, column
        // shift, shift index, whether the row is a real input channel, and the
        // element offset of its edge piece from the chunk's first position
        // in the image.
        uint32_t r_src[kPMaxRowsPerThread], r_dst[kPMaxRowsPerThread];
        int r_ph[kPMaxRowsPerThread], r_d[kPMaxRowsPerThread], r_j[kPMaxRowsPerThread];
        bool r_real[kPMaxRowsPerThread];
        long long r_edge[kPMaxRowsPerThread];
#pragma unroll
        for (int i = 0; i < kPMaxRowsPerThread; ++i) {
            const int r = t + i * kPGatherWarps * 32;
            const int j = r < n_rows ? r / p.ci_rows : 0, ci = r < n_rows ? r - j * p.ci_rows : 0;
            const int kw = j < p.pw ? j : j + 1;
            r_src[i] = static_cast<uint32_t>(p.pw * p.ci_rows + ci) * 128u;
            r_dst[i] = static_cast<uint32_t>(kw * p.ci_rows + ci) * 128u;
            r_ph[i] = ci & 7;
            r_d[i] = kw - p.pw;
            r_j[i] = j;
            r_real[i] = r < n_rows && ci < p.Ci;
            r_edge[i] = static_cast<long long>(ci) * p.HW + (kw < p.pw ? -4 : 32);
        }
        const int w32 = 32 % p.W;
        int n = c0 / p.cpi;
        int q0 = (c0 - n * p.cpi) * 32;
        int col = (q0 + lane) % p.W;   // column of position q0 + lane
        PRing ring;
        bool ok = true;
        // Every exit from this loop is agreed by the whole warp (the loop
        // body holds warp-wide ballots).
        for (int c = c0; c < c1 && !__any_sync(0xffffffffu, bars->abort_flag != 0); ++c, ring.next(p.stages)) {
            WP_TRACE_CLOCK(tg0);
            const float *plane = p.x + static_cast<size_t>(n) * p.Ci * p.HW + q0;
            // The 16-byte piece past the chunk's edge, for each row of this
            // thread: positions q0 - 4 .. q0 - 1 (left shifts) or q0 + 32 ..
            // q0 + 35 (right shifts), zero off the plane.  Loaded before the
            // stage is waited for.
            float4 edge[kPMaxRowsPerThread];
#pragma unroll
            for (int i = 0; i < kPMaxRowsPerThread; ++i) {
                edge[i] = make_float4(0.f, 0.f, 0.f, 0.f);
                const int e0 = q0 + (r_d[i] < 0 ? -4 : 32);
                if (r_real[i] && e0 >= 0 && e0 < p.HW)
                    edge[i] = __ldg(reinterpret_cast<const float4 *>(plane + r_edge[i]));
            }
            // Per row: bit k set where position q0 + k keeps its column + d
            // inside the row (and is on the plane).  The ballots run in every
            // lane (uniform loops); each lane keeps its own row's.
            const bool on = q0 + lane < p.HW;
            uint32_t kp[kPMaxRowsPerThread];
#pragma unroll
            for (int i = 0; i < kPMaxRowsPerThread; ++i) {
                kp[i] = 0;
                if (i * kPGatherWarps * 32 >= n_rows) break;   // no row of this pass in any thread
#pragma unroll
                for (int jj = 0; jj < kPMaxShifts; ++jj) {
                    if (jj >= p.kW - 1) break;
                    const int d = (jj < p.pw ? jj : jj + 1) - p.pw;
                    const uint32_t b = __ballot_sync(0xffffffffu, on && col + d >= 0 && col + d < p.W);
                    kp[i] = r_j[i] == jj ? b : kp[i];
                }
            }
            if (!__all_sync(0xffffffffu, dev::mbar_wait(dev::smem_u32(&bars->xfull[ring.stage]), ring.parity, tmo))) {
                if (lane == 0) pfail(bars, p.err);
                ok = false;
                break;
            }
            WP_TRACE_CLOCK(tg1);
            if (threadIdx.x == 0) WP_TRACE_ADD(2, tg1 - tg0);
            const uint32_t st = base0 + static_cast<uint32_t>(ring.stage) * p.stage_bytes;
#pragma unroll
            for (int i = 0; i < kPMaxRowsPerThread; ++i)
                if (t + i * kPGatherWarps * 32 < n_rows)
                    shift_row_any(r_d[i], st + r_src[i], st + r_dst[i], r_ph[i], edge[i], kp[i]);
            // The rows reach the tensor core's operand reads (async proxy).
            dev::fence_proxy_async_smem();
            dev::mbar_arrive(dev::smem_u32(&bars->sfull[ring.stage]));
            WP_TRACE_CLOCK(tg2);
            if (threadIdx.x == 0) WP_TRACE_ADD(3, tg2 - tg1);
            // next chunk: 32 positions on, or the next image
            q0 += 32;
            col += w32;
            if (col >= p.W) col -= p.W;
            if (q0 >= p.cpi * 32) {
                q0 = 0;
                ++n;
                col = lane % p.W;
            }
        }
        WP_TRACE_CLOCK(t_gend);
        if (threadIdx.x == 0) WP_TRACE_ADD(10, t_gend - t_start);
        // Epilogue: warps 0-3 read tensor-memory lanes 32*warp .. 32*warp + 31.
        const bool got = ok && dev::mbar_wait(dev::smem_u32(&bars->tmem_ready), 0, tmo) &&
                         dev::mbar_wait(dev::smem_u32(&bars->acc_full), 0, tmo);
        if (dev::named_bar_and(1, kPGatherWarps * 32, got)) {
            const uint32_t tmem = bars->tmem_base;
            WP_TRACE_CLOCK(te1);
            if (threadIdx.x == 0) WP_TRACE_ADD(5, te1 - t_gend);
            dev::tc_fence_after();
            float *split = p.part + static_cast<size_t>(blockIdx.x) * a_rows * p.nb;
            // Each warp stores 32 consecutive rows of one column per
            // instruction.  (Assembling the split in the free stage ring and
            // writing it with one bulk copy measured slower: 12k cycles vs 6k.)
            for (int mt = 0; mt < p.n_mt; ++mt) {
                const int rows = min(128, a_rows - mt * 128);
                if (warp * 32 >= rows) continue;   // warp-uniform: rows is a multiple of 8
                const int row = warp * 32 + lane;
                const uint32_t taddr = tmem + (static_cast<uint32_t>(warp * 32) << 16) + static_cast<uint32_t>(mt * p.nb);
                float *dst = split + static_cast<size_t>(mt) * 128 * p.nb + row;
                for (int j0 = 0; j0 < p.nb; j0 += 64) {
                    uint32_t r[4][16];
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        if (j0 + 16 * k < p.nb) dev::tmem_ld16(taddr + static_cast<uint32_t>(j0 + 16 * k), r[k]);
                    dev::tmem_wait_ld();
                    if (row < rows) {
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            if (j0 + 16 * k >= p.nb) break;
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                dst[static_cast<size_t>(j0 + 16 * k + j) * rows] = __uint_as_float(r[k][j]);
                        }
                    }
                }
            }
            WP_TRACE_CLOCK(te2);
            if (threadIdx.x == 0) WP_TRACE_ADD(6, te2 - te1);
        } else if (ok && !got) {
            pfail(bars, p.err);
        }
    }

    dev::tc_fence_before();
    __syncthreads();
    dev::tc_fence_after();
    if (warp == kPMmaWarp) dev::tmem_dealloc(bars->tmem_base, p.tmem_cols);
}

// Launch with programmatic dependent launch: the kernel may start while the
// previous kernel on the stream finishes; every thread that reads the
// inputs waits for it with griddepcontrol.wait first.
cudaError_t launch_plane_pdl(const WgradPlaneParams &p, int grid, int smem_bytes, cudaStream_t stream) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kPThreads);
    cfg.dynamicSmemBytes = smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, wgrad_plane_kernel, p);
}

}  // namespace

cudaError_t launch_wgrad_plane(const WgradPlaneParams &p, int grid, int smem_bytes, cudaStream_t stream) {
    if (grid < 1 || grid > p.total_chunks) return cudaErrorInvalidValue;
    cudaError_t e =
        cudaFuncSetAttribute(wgrad_plane_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess) return e;
    return launch_plane_pdl(p, grid, smem_bytes, stream);
}

}  // namespace dgrad

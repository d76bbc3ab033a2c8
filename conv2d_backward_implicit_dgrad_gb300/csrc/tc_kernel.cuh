// Warp-specialised tcgen05 implicit-GEMM dgrad (TF32 operands, fp32
// accumulation in tensor memory), one persistent CTA per SM.
//
// GEMM view (meganeura conv2d_grad_input_gemm.wgsl, header comment), turned
// so that output positions are the MMA's M:
//   D[P, ci] = sum over (tap t, co) of V[P + shift_t][co] * Wp[t][co][ci]
// for every sub-pixel phase (each with its own accumulator), where V is the
// zero-padded, flattened grad_out frame and Wp the pre-packed weights.
// Grouped plans issue the taps of one kernel row as one MMA with N = taps x
// slice: the A window is shared, each tap lands in its own sub-accumulator
// one output row further down per column step, and the epilogue adds the
// sub-accumulators back with the matching row shifts.
//
// Roles (448 threads with producer warps, 192 in tensor-copy mode):
//   warps 0-3   epilogue: tensor memory -> registers -> grad_input
//   warp  4     tensor-memory allocation; the MMA loop (whole warp, one
//               elected lane issues)
//   warp  5     one thread streaming packed weights with bulk copies (TMA);
//               in tensor-copy mode (packed channels-last frame) it also
//               copies each A stage with 2-D tensor copies
//   warps 6-13  producer mode: a band of grad_out -> shared memory (A
//               operand), 32 channels per stage, rows in the 128-byte
//               swizzled K-major layout of the tensor core
//   staged mode (tensor copies of the caller's grad_out itself): two
//               transposer warps after the epilogue warps turn each copied
//               stage, in place, into that layout
//   tensor-memory A mode (1x1, stride 1, no padding): the epilogue warps
//               also move each copied 32-channel chunk of a tile from shared
//               into tensor memory, where the MMA reads its A operand
// Pipelines (all mbarriers, all waits bounded):
//   A ring   a_stages  loader/producers -> MMA (A_full / A_empty)
//   B ring   b_stages  weight loader -> MMA    (B_full / B_empty); when the
//            whole packed weight of the launch fits, it is loaded once
//   acc      acc_bufs  MMA -> epilogue         (acc_full / acc_empty)
#pragma once

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
constexpr int kThreadsTmaA = kProdWarp0 * 32;
constexpr int kMaxAStages = 8;
constexpr int kMaxBStages = 32;
constexpr int kRowSlots = kProdWarps * 32 / 4;   // 4-byte producer: threads per channel lane
constexpr int kMaxRowsPerThread = 16;            // a_rows <= kRowSlots * kMaxRowsPerThread
constexpr int kGroupThreads = 128;               // quad producer: threads per producer group
constexpr int kQuadBatch = 4;                    // quad producer: warp items with loads in flight
constexpr int kGroupTableOffset = 1024;          // bytes into shared memory: MMA group table
constexpr int kXchgOffset = 3072;                // epilogue row exchange; operand stages follow at the next
                                                 // 1024-byte boundary

constexpr int kTransWarps = 2;                   // staged mode: transposer warps
constexpr int kTransThreads = kTransWarps * 32;
constexpr int kTransRows = 4;                    // rows per transposer thread (A stages of <= 256 rows)
constexpr int kTransBar = 3;                     // named barrier of the transposers (1, 2: epilogue groups)

struct Barriers {
    uint64_t a_full[kMaxAStages];
    uint64_t a_empty[kMaxAStages];
    uint64_t stg_full[kMaxAStages];   // staged / tensor-memory A modes: the stage's tensor copies have landed
    uint64_t stg_empty[kMaxAStages];  // tensor-memory A mode: the stage's copies have been read
    uint64_t ta_full[4];              // tensor-memory A mode: an A slot in tensor memory is written
    uint64_t ta_empty[4];             // tensor-memory A mode: the MMAs reading an A slot are done
    uint64_t b_full[kMaxBStages];
    uint64_t b_empty[kMaxBStages];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t drain;
    uint64_t never;   // failure-detection test: a barrier that nothing completes
    uint32_t tmem_base;
    volatile int abort_flag;
};
static_assert(sizeof(Barriers) <= kGroupTableOffset, "barrier block exceeds its reserved bytes");
static_assert(kGroupTableOffset + kMaxTaps * 16 <= kXchgOffset, "MMA group table exceeds its reserved bytes");

// Cycle accounting per CTA, compiled in only with -DDGRAD_TRACE (a tracing
// build used to see where a launch spends its time).  Slots: MMA waits on
// acc_empty / A_full / B_full, MMA issue, producer waits on A_empty,
// producer issue, epilogue waits on acc_full, epilogue work, units, chunks,
// launch-relative cycle of the first MMA, of the MMA loop's end, of the
// producers' end, of the epilogue's end; global-timer ns at the CTA's start
// and end, and its span in cycles.  In the grouped one-phase epilogue, slots
// 4, 5, 14 and 15 hold its publish pass, barrier, combine-and-store loop and
// last stores instead.
#ifdef DGRAD_TRACE
constexpr int kTraceSlots = 20;
constexpr int kTraceCtas = 1024;
__device__ unsigned long long g_trace[kTraceCtas * kTraceSlots];
#define DGRAD_TRACE_ADD(slot, v) \
    atomicAdd(&g_trace[(blockIdx.x % kTraceCtas) * kTraceSlots + (slot)], (unsigned long long)(v))
#define DGRAD_TRACE_CLOCK(x) const long long x = clock64()
#define DGRAD_TRACE_SET(slot, v) (g_trace[(blockIdx.x % kTraceCtas) * kTraceSlots + (slot)] = (unsigned long long)(v))
#else
#define DGRAD_TRACE_SET(slot, v) ((void)0)
#define DGRAD_TRACE_ADD(slot, v) ((void)0)
#define DGRAD_TRACE_CLOCK(x) ((void)0)
#endif

__device__ __forceinline__ void fail(Barriers *bars, const MainParams &p) {
    bars->abort_flag = 1;
    atomicOr(p.err, kErrTimeout);
}

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

// ------------------------------------------------------------------ producers
// Number of grad_out elements of image n (plane order j = oh*oW + ow) whose
// frame position is below P.
__device__ __forceinline__ int plane_elems_below(const MainParams &p, int n, int P) {
    const int rel = P - (n * p.Hv + p.Ph) * p.Wp - p.Pw;
    if (rel <= 0) return 0;
    const int oh = rel / p.Wp;
    if (oh >= p.oH) return p.oH * p.oW;
    return oh * p.oW + min(rel - oh * p.Wp, p.oW);
}

// First frame position of a tile and the end of the positions its outputs
// may lie in.  Tiles run across images, or (img_tiles > 0, staged mode)
// each image has img_tiles tiles of its own, so that a band never holds two
// images; positions past the tile's image are then never outputs of it.
__device__ __forceinline__ int tile_origin(const MainParams &p, int tile, int &lim) {
    if (p.img_tiles) {
        const int n = tile / p.img_tiles;
        lim = (n + 1) * p.HvWp;
        return n * p.HvWp + (tile - n * p.img_tiles) * p.tile_step;
    }
    lim = p.positions;
    return tile * p.tile_step;
}

// Staged mode.  The loader's tensor copy writes the band's grad_out elements
// channel by channel at the start of the A stage: element x0 + e of channel
// 32c + k of the image's plane at float k*stg_box + e (x0 = the band's first
// element rounded down to a multiple of 4, channels past Co and elements past
// the plane read as zeros).  The transposer warps read every value they will
// write into registers, meet at a named barrier (after which nothing of the
// copy is read again), and write the band in the MMA's layout: row r (frame
// position P0 + r) holds its element's 32 channels, TF32-rounded (split
// precision: the hi or lo part), in the 128-byte swizzle; rows with no
// element (frame padding, other images) are zeros.  Thread t takes rows
// t, t + 64, ...: a warp's loads of one channel read consecutive words, and
// its 16-byte stores of one chunk land in eight different bank groups.
template <int KC, int kEG>
__device__ __forceinline__ void transpose_stages(const MainParams &p, Barriers *bars, float *a_base,
                                                 int a_stage_floats, long long tmo) {
    constexpr int kW0 = kProdWarp0 + (kEG - 1) * kEpiWarps;
    const int tt = static_cast<int>(threadIdx.x) - kW0 * 32;
    const uint32_t a0 = dev::smem_u32(a_base);
    Ring ring;
    // The two warps leave together: whether to go on is agreed at the named
    // barrier of every stage (a wait that ran out, or an abort, in either).
    for (int w = blockIdx.x; w < p.n_work; w += gridDim.x) {
        int lim;
        const int P0 = tile_origin(p, w / p.n_slices, lim);
        const int n = P0 / p.HvWp;
        const int x0 = plane_elems_below(p, n, P0) & ~3;
        int loc[kTransRows];   // element of row tt + 64*i in the copy, or -1
#pragma unroll
        for (int i = 0; i < kTransRows; ++i) {
            const int r = tt + kTransThreads * i;
            const int P = P0 + r;
            loc[i] = -1;
            if (r < p.band_rows && P < lim) {
                const int rel = P - n * p.HvWp;
                const int y = rel / p.Wp;
                const int oh = y - p.Ph, ow = rel - y * p.Wp - p.Pw;
                if (static_cast<unsigned>(oh) < static_cast<unsigned>(p.oH) &&
                    static_cast<unsigned>(ow) < static_cast<unsigned>(p.oW))
                    loc[i] = oh * p.oW + ow - x0;
            }
        }
        for (int c = 0; c < p.n_chunks; ++c, ring.next(p.a_stages)) {
            DGRAD_TRACE_CLOCK(tw0);
            const bool got = !bars->abort_flag &&
                             dev::mbar_wait(dev::smem_u32(&bars->stg_full[ring.stage]), ring.parity, tmo);
            DGRAD_TRACE_CLOCK(tw1);
            if (tt == 0) DGRAD_TRACE_ADD(4, tw1 - tw0);
            const float *stg = a_base + static_cast<size_t>(ring.stage) * a_stage_floats;
            float v[kTransRows][KC];
#pragma unroll
            for (int i = 0; i < kTransRows; ++i) {
#pragma unroll
                for (int k = 0; k < KC; ++k)
                    v[i][k] = (got && loc[i] >= 0) ? stg[k * p.stg_box + loc[i]] : 0.f;
            }
            // Every read of the copy is done (nothing of it is read again),
            // and every transposer thread has its data.
            if (!dev::named_bar_and(kTransBar, kTransThreads, got)) {
                if (!got) fail(bars, p);
                return;
            }
            DGRAD_TRACE_CLOCK(tw15);
            if (tt == 0) DGRAD_TRACE_ADD(15, tw15 - tw1);
            const int pass = p.split_chunks ? c / p.split_chunks : 0;
            const uint32_t as = a0 + static_cast<uint32_t>(ring.stage) * a_stage_floats * 4;
#pragma unroll
            for (int i = 0; i < kTransRows; ++i) {
                const int r = tt + kTransThreads * i;
                if (r < p.a_rows) {
#pragma unroll
                    for (int k = 0; k < KC; ++k) {
                        float x = v[i][k];
                        if (p.split_chunks) {
                            const float hi = dev::round_tf32_int(x);
                            x = pass == 1 ? dev::round_tf32_int(x - hi) : hi;
                        } else if (p.round_tf32) {
                            x = dev::round_tf32_int(x);
                        }
                        v[i][k] = x;
                    }
                    const uint32_t row = as + static_cast<uint32_t>(r) * 128;
#pragma unroll
                    for (int g = 0; g < KC / 4; ++g)
                        asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(
                                         row + (static_cast<uint32_t>(g ^ (r & 7)) << 4)),
                                     "f"(v[i][4 * g]), "f"(v[i][4 * g + 1]), "f"(v[i][4 * g + 2]),
                                     "f"(v[i][4 * g + 3])
                                     : "memory");
                }
            }
            // The stores reach the tensor core's (async-proxy) operand reads.
            dev::fence_proxy_async_smem();
            dev::mbar_arrive(dev::smem_u32(&bars->a_full[ring.stage]));
            DGRAD_TRACE_CLOCK(tw2);
            if (tt == 0) DGRAD_TRACE_ADD(5, tw2 - tw15);
        }
    }
}

// Tensor-memory A mode (1x1 kernel, stride 1, no padding: a tile's A rows
// are 128 consecutive grad_out positions with no shifted windows).  For each
// 32-channel chunk the loader copies the tile's plane elements from NCHW
// grad_out into a shared-memory stage: a copy of 128 elements x 32 channels
// of the tile's first image, and when the tile runs into the next image a
// second one from that image's first element (channel k, element e of copy
// b at float (b*32 + k)*128 + e).  Epilogue thread t (tensor-memory lane t =
// tile row t) reads its position's 32 channels (a warp's loads of one
// channel are consecutive words), TF32-rounds them (split precision: the
// hi or lo part) and writes them as 32 columns of an A slot in tensor
// memory; the MMA then reads A from there.  Waits are agreed by the warp
// (the tensor-memory store is a warp-wide instruction).  Returns false if a
// wait ran out (recorded; the caller's unit ends).
template <int KC>
__device__ __forceinline__ bool write_tmem_a(const MainParams &p, Barriers *bars, const float *a_base,
                                             int a_stage_floats, uint32_t tmem_base, int tile, int ew, int lane,
                                             Ring &rs, Ring &rt, long long tmo) {
    const int t = ew * 32 + lane;
    const int plane = p.oH * p.oW;
    int lim;
    const int P0 = tile_origin(p, tile, lim);   // image-aligned tiles: every valid row is in box 0
    const int n0 = P0 / plane, x0 = P0 - n0 * plane;
    const int P = P0 + t;
    const bool valid = P < lim;
    int off = 0;
    if (valid) {
        const int n = P / plane, j = P - n * plane;
        off = n == n0 ? j - x0 : KC * kBlockM + j;
    }
    const uint32_t tl = tmem_base + (static_cast<uint32_t>(ew * 32) << 16) + static_cast<uint32_t>(p.a_tcol);
    // (Issuing chunk c's store before fetching chunk c + 1 measured slower:
    // it holds chunk c's slot back while chunk c + 1's copy is awaited.)
    for (int c = 0; c < p.n_chunks; ++c, rs.next(p.a_stages), rt.next(p.a_tslots)) {
        DGRAD_TRACE_CLOCK(tw0);
        if (!__all_sync(0xffffffffu, dev::mbar_wait(dev::smem_u32(&bars->stg_full[rs.stage]), rs.parity, tmo))) {
            if (lane == 0) fail(bars, p);
            return false;
        }
        DGRAD_TRACE_CLOCK(tw1);
        if (t == 0) DGRAD_TRACE_ADD(4, tw1 - tw0);
        const float *stg = a_base + static_cast<size_t>(rs.stage) * a_stage_floats;
        float v[KC];
#pragma unroll
        for (int k = 0; k < KC; ++k) v[k] = valid ? stg[k * kBlockM + off] : 0.f;
        dev::mbar_arrive(dev::smem_u32(&bars->stg_empty[rs.stage]));   // the stage may be refilled
        const int pass = p.split_chunks ? c / p.split_chunks : 0;
#pragma unroll
        for (int k = 0; k < KC; ++k) {
            if (p.split_chunks) {
                const float hi = dev::round_tf32_int(v[k]);
                v[k] = pass == 1 ? dev::round_tf32_int(v[k] - hi) : hi;
            } else if (p.round_tf32) {
                v[k] = dev::round_tf32_int(v[k]);
            }
        }
        DGRAD_TRACE_CLOCK(tw2);
        if (t == 0) DGRAD_TRACE_ADD(15, tw2 - tw1);
        if (!__all_sync(0xffffffffu, dev::mbar_wait(dev::smem_u32(&bars->ta_empty[rt.stage]), rt.parity ^ 1, tmo))) {
            if (lane == 0) fail(bars, p);
            return false;
        }
        dev::tmem_st32(tl + static_cast<uint32_t>(rt.stage * KC), v);
        dev::tmem_wait_st();
        dev::tc_fence_before();
        dev::mbar_arrive(dev::smem_u32(&bars->ta_full[rt.stage]));
        DGRAD_TRACE_CLOCK(tw3);
        if (t == 0) DGRAD_TRACE_ADD(5, tw3 - tw2);
    }
    return true;
}

// Quad producer.  The 256 producer threads form two groups of 128 that fill
// alternate A stages, so two stages' loads are in flight.  Inside a stage, a
// warp item is 8 consecutive aligned quads (4 plane elements) x 16 channels:
// lane (qsub, cg) loads channels cg*4..cg*4+3 of its quad with 16-byte loads
// (each load instruction reads four full 128-byte lines), transposes the
// 4x4 block in registers, rounds to TF32 and writes four 16-byte row chunks.
// Lanes 8p..8p+7 hold quads 2p, 2p+1 x cg 0..3: their rows sit 4 apart, so
// the swizzled chunk positions of one store phase are all distinct.  Frame
// rows with no grad_out element are written as zeros.
template <int KC>
__device__ __forceinline__ void produce_quads(const MainParams &p, Barriers *bars, float *a_base, int a_stage_floats,
                                              int tile_step, long long tmo) {
    const int gtid = threadIdx.x - kProdWarp0 * 32;
    const int group = gtid / kGroupThreads;
    const int tid = gtid % kGroupThreads;
    const int gw = tid / 32, lane = tid % 32;
    const int qsub = ((lane >> 3) << 1) | ((lane >> 2) & 1);
    const int cg = lane & 3;
    const int plane = p.oH * p.oW;
    const int img = p.Hv * p.Wp;
    const uint32_t a0 = dev::smem_u32(a_base);
    constexpr int kZeroRowsPerThread = (kRowSlots * kMaxRowsPerThread + kGroupThreads - 1) / kGroupThreads;
    Ring ring;
    uint32_t it = 0;
    for (int w = blockIdx.x; w < p.n_work && !bars->abort_flag; w += gridDim.x) {
        const int P0 = (w / p.n_slices) * tile_step;
        const int P1 = P0 + p.a_rows;
        // Rows of this thread that hold no grad_out element (zeros), as a mask.
        uint32_t zero_mask = 0;
#pragma unroll
        for (int i = 0; i < kZeroRowsPerThread; ++i) {
            const int r = tid + kGroupThreads * i;
            if (r < p.a_rows && dev::frame_row_offset(p, P0 + r) < 0) zero_mask |= 1u << i;
        }
        // Images overlapping the band and their quad ranges.
        const int n_lo = min(P0 / img, p.N - 1);
        const int n_hi = min((P1 - 1) / img, p.N - 1);
        int seg_n[kMaxBandImages], seg_jlo[kMaxBandImages], seg_jhi[kMaxBandImages], seg_q0[kMaxBandImages];
        int seg_start[kMaxBandImages + 1];
        int items = 0;
#pragma unroll
        for (int s = 0; s < kMaxBandImages; ++s) {
            const int n = n_lo + s;
            seg_n[s] = n;
            seg_jlo[s] = seg_jhi[s] = seg_q0[s] = 0;
            seg_start[s] = items;
            if (n <= n_hi) {
                const int jlo = plane_elems_below(p, n, P0), jhi = plane_elems_below(p, n, P1);
                seg_jlo[s] = jlo;
                seg_jhi[s] = jhi;
                seg_q0[s] = jlo >> 2;
                if (jhi > jlo) items += (((jhi + 3) >> 2) - seg_q0[s] + 7) / 8 * 2;   // octets x 2 halves
            }
        }
        seg_start[kMaxBandImages] = items;

        for (int c = 0; c < p.n_chunks; ++c, ++it, ring.next(p.a_stages)) {
            if (static_cast<int>(it & 1) != group) continue;
            DGRAD_TRACE_CLOCK(tw0);
            if (!dev::mbar_wait(dev::smem_u32(&bars->a_empty[ring.stage]), ring.parity ^ 1, tmo)) {
                fail(bars, p);
                return;
            }
            DGRAD_TRACE_CLOCK(tw1);
            if (gtid == 0) DGRAD_TRACE_ADD(4, tw1 - tw0);
            const uint32_t as = a0 + static_cast<uint32_t>(ring.stage) * a_stage_floats * 4;
            // zero rows
#pragma unroll
            for (int i = 0; i < kZeroRowsPerThread; ++i) {
                if (zero_mask & (1u << i)) {
                    const uint32_t row = as + static_cast<uint32_t>(tid + kGroupThreads * i) * 128;
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        asm volatile("st.shared.v4.f32 [%0], {%1, %1, %1, %1};" ::"r"(row + 16 * k), "f"(0.f)
                                     : "memory");
                }
            }
            // data quads, kQuadBatch warp items with their loads in flight
            for (int base = gw; base < items; base += 4 * kQuadBatch) {
                float4 v[kQuadBatch][4];
                int jq[kQuadBatch], nq[kQuadBatch], jloq[kQuadBatch], jhiq[kQuadBatch], hq[kQuadBatch];
#pragma unroll
                for (int b = 0; b < kQuadBatch; ++b) {
                    const int item = base + 4 * b;
                    jq[b] = -1;
                    nq[b] = jloq[b] = jhiq[b] = hq[b] = 0;
                    if (item < items) {
                        // segment of the item (selects over static indices: no local memory)
                        int sn = seg_n[0], sjlo = seg_jlo[0], sjhi = seg_jhi[0], sq0 = seg_q0[0], sst = seg_start[0];
#pragma unroll
                        for (int k = 1; k < kMaxBandImages; ++k) {
                            if (item >= seg_start[k]) {
                                sn = seg_n[k];
                                sjlo = seg_jlo[k];
                                sjhi = seg_jhi[k];
                                sq0 = seg_q0[k];
                                sst = seg_start[k];
                            }
                        }
                        const int local = item - sst;
                        const int half = local & 1;
                        const int j = (sq0 + (local >> 1) * 8 + qsub) * 4;
                        if (j < sjhi) {
                            jq[b] = j;
                            nq[b] = sn;
                            jloq[b] = sjlo;
                            jhiq[b] = sjhi;
                            hq[b] = half;
                            const int ch = c * KC + half * 16 + cg * 4;
                            const float4 *src = reinterpret_cast<const float4 *>(
                                p.go + (static_cast<size_t>(sn) * p.Co + ch) * plane + j);
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                v[b][k] = (ch + k < p.Co) ? __ldg(src + static_cast<size_t>(k) * (plane / 4))
                                                          : make_float4(0.f, 0.f, 0.f, 0.f);
                        }
                    }
                }
                DGRAD_TRACE_CLOCK(tq1);
                if (gtid == 0) DGRAD_TRACE_ADD(14, tq1 - tw1);
#pragma unroll
                for (int b = 0; b < kQuadBatch; ++b) {
                    if (jq[b] < 0) continue;
                    const int j = jq[b];
                    const int n = nq[b];
                    int oh = j / p.oW, ow = j - oh * p.oW;
                    const float ev[4][4] = {{v[b][0].x, v[b][1].x, v[b][2].x, v[b][3].x},
                                            {v[b][0].y, v[b][1].y, v[b][2].y, v[b][3].y},
                                            {v[b][0].z, v[b][1].z, v[b][2].z, v[b][3].z},
                                            {v[b][0].w, v[b][1].w, v[b][2].w, v[b][3].w}};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int je = j + e;
                        if (je >= jloq[b] && je < jhiq[b]) {
                            const int r = (n * p.Hv + oh + p.Ph) * p.Wp + ow + p.Pw - P0;
                            float x0 = ev[e][0], x1 = ev[e][1], x2 = ev[e][2], x3 = ev[e][3];
                            if (p.round_tf32) {
                                x0 = dev::round_tf32(x0);
                                x1 = dev::round_tf32(x1);
                                x2 = dev::round_tf32(x2);
                                x3 = dev::round_tf32(x3);
                            }
                            const uint32_t dst = as + static_cast<uint32_t>(r) * 128 +
                                                 (static_cast<uint32_t>((hq[b] * 4 + cg) ^ (r & 7)) << 4);
                            asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "f"(x0), "f"(x1),
                                         "f"(x2), "f"(x3)
                                         : "memory");
                        }
                        if (++ow == p.oW) {
                            ow = 0;
                            ++oh;
                        }
                    }
                }
            }
            DGRAD_TRACE_CLOCK(tw2);
            if (gtid == 0) DGRAD_TRACE_ADD(5, tw2 - tw1);
            if (gtid == 0) DGRAD_TRACE_ADD(15, 1);
            // The writer makes its stores visible to the tensor core's
            // (async-proxy) operand reads, then releases the stage.
            dev::fence_proxy_async_smem();
            dev::mbar_arrive(dev::smem_u32(&bars->a_full[ring.stage]));
        }
    }
}

// 4-byte producer (any shape).  Thread (pr, e) copies frame rows
// r = pr + kRowSlots*i, channel e of every 4-channel group with
// asynchronous copies (zero-fill for padding).  One warp instruction moves 8
// consecutive rows x 4 channels into eight distinct 16-byte chunks of the
// swizzled rows.  The tensor core reads the TF32 part of these fp32 values.
template <int KC>
__device__ __forceinline__ void produce_async4(const MainParams &p, Barriers *bars, float *a_base, int a_stage_floats,
                                               int tile_step, long long tmo) {
    const int ptid = threadIdx.x - kProdWarp0 * 32;
    const int e = ptid & 3, pr = ptid >> 2;
    const int sw = pr & 7;
    const size_t plane = static_cast<size_t>(p.oH) * p.oW;
    const uint32_t a0 = dev::smem_u32(a_base) + e * 4;
    Ring ring;
    for (int w = blockIdx.x; w < p.n_work && !bars->abort_flag; w += gridDim.x) {
        const int P0 = (w / p.n_slices) * tile_step;
        int off[kMaxRowsPerThread];
#pragma unroll
        for (int i = 0; i < kMaxRowsPerThread; ++i) {
            const int r = pr + kRowSlots * i;
            off[i] = r < p.a_rows ? dev::frame_row_offset(p, P0 + r) : -1;
        }
        for (int c = 0; c < p.n_chunks; ++c, ring.next(p.a_stages)) {
            if (!dev::mbar_wait(dev::smem_u32(&bars->a_empty[ring.stage]), ring.parity ^ 1, tmo)) {
                fail(bars, p);
                dev::cp_async_wait_all();
                return;
            }
            const uint32_t as = a0 + static_cast<uint32_t>(ring.stage) * a_stage_floats * 4;
            const int co0 = c * KC + e;
#pragma unroll
            for (int i = 0; i < kMaxRowsPerThread; ++i) {
                const int r = pr + kRowSlots * i;
                if (r < p.a_rows) {
                    const uint32_t dst = as + static_cast<uint32_t>(r) * 128;
#pragma unroll
                    for (int g = 0; g < KC / 4; ++g) {
                        const int co = co0 + 4 * g;
                        const bool v = off[i] >= 0 && co < p.Co;
                        const float *src = v ? p.go + static_cast<size_t>(off[i]) + co * plane : p.go;
                        dev::cp_async_4(dst + ((g ^ sw) << 4), src, v ? 4u : 0u);
                    }
                }
            }
            dev::cp_async_arrive(dev::smem_u32(&bars->a_full[ring.stage]));
        }
    }
    dev::cp_async_wait_all();
}

// ------------------------------------------------------------------ epilogue
// Result of one 16-column batch of one phase for this warp's 32 rows (lane =
// output position, out[j] = input channel c0 + j), from registers already
// loaded from tensor memory: r[g] = sub-accumulator g.
//
// Ungrouped (S = 1) the accumulator is the result.  Grouped, sub-accumulator
// g holds, at row o, the tap whose output is row o - (S-1-g); the result of
// row o is the sum over g of sub-accumulator g at row o + (S-1-g).  Rows of
// the next warp come through shared memory (each warp publishes the first
// rows the warp above it needs); rows past the 128-row block are never
// valid outputs (the tile step leaves them out).
template <int S, int SMAX>
__device__ __forceinline__ void combine(const uint32_t (&r)[SMAX][16], float (&out)[16], float *xw, const float *xn,
                                        int lane, int bar_id) {
    if constexpr (S == 1) {
#pragma unroll
        for (int j = 0; j < 16; ++j) out[j] = __uint_as_float(r[0][j]);
    } else {
        int slot = 0;
#pragma unroll
        for (int g = 0; g < S - 1; ++g) {
            const int sh = S - 1 - g;
            if (lane < sh) {
#pragma unroll
                for (int j = 0; j < 16; ++j) xw[(slot + lane) * 16 + j] = __uint_as_float(r[g][j]);
            }
            slot += sh;
        }
        DGRAD_TRACE_CLOCK(tb0);
        dev::named_bar(bar_id, 128);
        DGRAD_TRACE_CLOCK(tb1);
        if (threadIdx.x == 0) DGRAD_TRACE_ADD(5, tb1 - tb0);
#pragma unroll
        for (int j = 0; j < 16; ++j) out[j] = __uint_as_float(r[S - 1][j]);
        slot = 0;
#pragma unroll
        for (int g = 0; g < S - 1; ++g) {
            const int sh = S - 1 - g;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                float v = __shfl_down_sync(0xffffffffu, __uint_as_float(r[g][j]), sh);
                if (lane + sh >= 32) v = xn ? xn[(slot + lane + sh - 32) * 16 + j] : 0.f;
                out[j] += v;
            }
            slot += sh;
        }
    }
}

// Stores of one finished batch: NV = 1 writes one phase (4-byte stores, a
// warp writes 32 consecutive positions of one channel row); NV = s (2 or 4)
// writes the s column phases of one row phase together: positions (q, u) of
// phases (a, 0..s-1) are the s consecutive elements s*u .. s*u+s-1 of input
// row s*q + a, one 8- or 16-byte store.
// Fused epilogue on NV consecutive elements at d: keep the new values where
// the ReLU input is > 0 (else 0), then add the values already in grad_input.
template <int NV>
__device__ __forceinline__ void fuse_values(const MainParams &p, const float *d, float (&v)[NV]) {
    if (p.relu_in) {
        const float *m = p.relu_in + (d - p.gi);
        float mv[NV];
        if constexpr (NV == 1) {
            mv[0] = __ldg(m);
        } else if constexpr (NV == 2) {
            const float2 t = __ldg(reinterpret_cast<const float2 *>(m));
            mv[0] = t.x, mv[1] = t.y;
        } else {
            const float4 t = __ldg(reinterpret_cast<const float4 *>(m));
            mv[0] = t.x, mv[1] = t.y, mv[2] = t.z, mv[3] = t.w;
        }
#pragma unroll
        for (int e = 0; e < NV; ++e) v[e] = mv[e] > 0.f ? v[e] : 0.f;
    }
    if (p.accumulate) {
        float ov[NV];
        if constexpr (NV == 1) {
            ov[0] = *d;
        } else if constexpr (NV == 2) {
            const float2 t = *reinterpret_cast<const float2 *>(d);
            ov[0] = t.x, ov[1] = t.y;
        } else {
            const float4 t = *reinterpret_cast<const float4 *>(d);
            ov[0] = t.x, ov[1] = t.y, ov[2] = t.z, ov[3] = t.w;
        }
#pragma unroll
        for (int e = 0; e < NV; ++e) v[e] = ov[e] + v[e];
    }
}

template <int NV, int CB, bool kFuse>
__device__ __forceinline__ void store_batch_as(const MainParams &p, float *dst, size_t plane, int ncols,
                                               const float (&res)[NV][CB / 16][16]) {
    float *d = dst;   // advanced by one channel plane per store
#pragma unroll
    for (int k = 0; k < CB / 16; ++k) {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            if (k * 16 + j < ncols) {
                float v[NV];
#pragma unroll
                for (int e = 0; e < NV; ++e) v[e] = res[e][k][j];
                if constexpr (kFuse) fuse_values<NV>(p, d, v);
                if constexpr (NV == 1) {
                    *d = v[0];
                } else if constexpr (NV == 2) {
                    *reinterpret_cast<float2 *>(d) = make_float2(v[0], v[1]);
                } else {
                    *reinterpret_cast<float4 *>(d) = make_float4(v[0], v[1], v[2], v[3]);
                }
            }
            d += plane;
        }
    }
}

// FUSE: 0 plain stores, 1 fused epilogue, 2 chosen per batch from the
// parameters.  Kernels built for plain stores carry none of the fused code
// (measured: even untaken, it slowed the epilogue by up to 2 us per call).
template <int NV, int CB, int FUSE>
__device__ __forceinline__ void store_batch(const MainParams &p, float *dst, size_t plane, int ncols,
                                            const float (&res)[NV][CB / 16][16]) {
    if constexpr (FUSE == 2) {
        if (p.relu_in != nullptr || p.accumulate != 0)
            store_batch_as<NV, CB, true>(p, dst, plane, ncols, res);
        else
            store_batch_as<NV, CB, false>(p, dst, plane, ncols, res);
    } else {
        store_batch_as<NV, CB, FUSE == 1>(p, dst, plane, ncols, res);
    }
}

// Epilogue state of one warp across the batches of a work unit.
struct EpiCtx {
    const MainParams *p;
    uint32_t tbase;       // tensor-memory address of this warp's lanes in the unit's accumulator set
    bool row_ok;
    int n, q, u, ci0, nci;
    float *xbase;         // this group's row-exchange area
    int slots, ew, lane, bar_id;
    uint32_t xcount;      // row exchanges done (alternates the exchange buffers)
};

// One work unit's output rows for this warp: every phase, every input
// channel of the slice, in batches of CB columns (CB / 16 slices of 16): a
// batch's tensor-memory loads (for NV phases, up to SMAX sub-accumulators
// each) are issued together and waited for once.  The previous batch's
// stores go out before a batch's loads; the last batch's values are returned
// in `pend` (stored by the caller after it has released the accumulator set).
template <int NV, int SMAX, int CB, int FUSE>
__device__ __forceinline__ void epilogue_unit(EpiCtx &e, float (&pend)[NV][CB / 16][16], float *&pend_dst,
                                              int &pend_cols) {
    constexpr int K = CB / 16;
    const MainParams &p = *e.p;
    const size_t plane = static_cast<size_t>(p.H) * p.W;
    for (int ph0 = 0; ph0 < p.n_phases; ph0 += NV) {
        const PhaseDesc &pd0 = p.phase[ph0];
        const bool valid = e.row_ok && e.q < pd0.Hq && e.u < pd0.Wq;
        const int ih = p.s * e.q + pd0.a, iw = p.s * e.u + pd0.b;
        float *dst = p.gi + (static_cast<size_t>(e.n) * p.Ci + e.ci0) * plane + static_cast<size_t>(ih) * p.W + iw;
        for (int c0 = 0; c0 < p.bn; c0 += CB) {
            if (pend_dst) store_batch<NV, CB, FUSE>(p, pend_dst, plane, pend_cols, pend);
            uint32_t r[NV][K][SMAX][16];
            DGRAD_TRACE_CLOCK(tl0);
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                const int sub = p.phase[ph0 + v].tap_count ? p.phase[ph0 + v].sub : 0;
                const int col = p.phase[ph0 + v].col;
#pragma unroll
                for (int k = 0; k < K; ++k) {
                    if (c0 + 16 * k >= p.bn) break;
#pragma unroll
                    for (int g = 0; g < SMAX; ++g)
                        if (g < sub)
                            dev::tmem_ld16(e.tbase + static_cast<uint32_t>(col + g * p.bn + c0 + 16 * k), r[v][k][g]);
                }
            }
            dev::tmem_wait_ld();
            DGRAD_TRACE_CLOCK(tl1);
            if (threadIdx.x == 0) DGRAD_TRACE_ADD(4, tl1 - tl0);
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                const int sub = p.phase[ph0 + v].tap_count ? p.phase[ph0 + v].sub : 0;
#pragma unroll
                for (int k = 0; k < K; ++k) {
                    if (c0 + 16 * k >= p.bn) break;
                    float *xb = e.xbase + static_cast<size_t>((e.xcount & 1) * 4) * e.slots * 16;
                    float *xw = xb + e.ew * e.slots * 16;
                    const float *xn = e.ew < 3 ? xw + e.slots * 16 : nullptr;
                    if (sub == 0) {
#pragma unroll
                        for (int j = 0; j < 16; ++j) pend[v][k][j] = 0.f;
                    } else if (sub == 1) {
                        combine<1, SMAX>(r[v][k], pend[v][k], xw, xn, e.lane, e.bar_id);
                    } else {
                        if constexpr (SMAX >= 2) {
                            if (sub == 2) combine<2, SMAX>(r[v][k], pend[v][k], xw, xn, e.lane, e.bar_id);
                        }
                        if constexpr (SMAX >= 3) {
                            if (sub == 3) combine<3, SMAX>(r[v][k], pend[v][k], xw, xn, e.lane, e.bar_id);
                        }
                        if constexpr (SMAX >= 4) {
                            if (sub == 4) combine<4, SMAX>(r[v][k], pend[v][k], xw, xn, e.lane, e.bar_id);
                        }
                        ++e.xcount;
                    }
                }
            }
            pend_dst = valid ? dst + static_cast<size_t>(c0) * plane : nullptr;
            pend_cols = min(CB, e.nci - c0);
        }
    }
}

// A whole work unit for this warp: its tm blocks of 128 rows (one when
// grouped), then the release of the accumulator set and the last stores.
template <int NV, int SMAX, int CB, int FUSE>
__device__ __forceinline__ void epilogue_run(EpiCtx &e, int tile, uint32_t tbase0, int m_cols, uint64_t *acc_empty) {
    const MainParams &p = *e.p;
    float pend[NV][CB / 16][16];
    float *pend_dst = nullptr;
    int pend_cols = 0;
    int lim;
    const int T0 = tile_origin(p, tile, lim);
    for (int m = 0; m < p.tm; ++m) {
        const int o = m * kBlockM + e.ew * 32 + e.lane;   // row of the unit
        const int P = T0 + o;
        dev::decode_position(p, P, e.n, e.q, e.u);
        e.row_ok = o < p.tile_step && P < lim;
        e.tbase = tbase0 + static_cast<uint32_t>(m * m_cols);
        epilogue_unit<NV, SMAX, CB, FUSE>(e, pend, pend_dst, pend_cols);
    }
    // Every value of the unit is in registers: release the accumulator set
    // to the MMA, then store the last batch.
    dev::tc_fence_before();
    dev::mbar_arrive(dev::smem_u32(acc_empty));
    DGRAD_TRACE_CLOCK(ts0);
    if (pend_dst) store_batch<NV, CB, FUSE>(p, pend_dst, static_cast<size_t>(p.H) * p.W, pend_cols, pend);
    DGRAD_TRACE_CLOCK(ts1);
    if (threadIdx.x == 0) DGRAD_TRACE_ADD(14, ts1 - ts0);
}

// A whole grouped work unit of a one-phase convolution (stride 1) with S
// sub-accumulators: first every warp publishes, for all the slice's columns,
// the first rows the warp above it needs (one named barrier per unit instead
// of one per 16 columns), then each warp combines and stores its rows batch by
// batch without waiting for the others.  `ubuf` alternates the exchange
// buffer between consecutive units: a warp can start the next unit's
// publishing only after all four warps have passed this unit's barrier, i.e.
// after the reads of the buffer it would overwrite.
template <int S, int FUSE>
__device__ __forceinline__ void epilogue_run_g1(EpiCtx &e, int tile, uint32_t tbase0, uint64_t *acc_empty,
                                                uint32_t ubuf) {
    constexpr int kSlots = S * (S - 1) / 2;
    const MainParams &p = *e.p;
    const PhaseDesc &pd = p.phase[0];
    const int bnp = p.bn;
    const int o = e.ew * 32 + e.lane;   // row of the unit
    int lim;
    const int P = tile_origin(p, tile, lim) + o;
    dev::decode_position(p, P, e.n, e.q, e.u);
    e.row_ok = o < p.tile_step && P < lim;
    const uint32_t tb = tbase0 + static_cast<uint32_t>(pd.col);
    float *xb = e.xbase + static_cast<size_t>(ubuf) * 4 * kSlots * bnp;
    float *xw = xb + static_cast<size_t>(e.ew) * kSlots * bnp;
    const float *xn = e.ew < 3 ? xw + kSlots * bnp : nullptr;
    DGRAD_TRACE_CLOCK(tg0);
    for (int c0 = 0; c0 < bnp; c0 += 16) {   // publish
        uint32_t r[S - 1][16];
#pragma unroll
        for (int g = 0; g < S - 1; ++g) dev::tmem_ld16(tb + static_cast<uint32_t>(g * bnp + c0), r[g]);
        dev::tmem_wait_ld();
        int slot = 0;
#pragma unroll
        for (int g = 0; g < S - 1; ++g) {
            const int sh = S - 1 - g;
            if (e.lane < sh) {
#pragma unroll
                for (int j = 0; j < 16; ++j) xw[(slot + e.lane) * bnp + c0 + j] = __uint_as_float(r[g][j]);
            }
            slot += sh;
        }
    }
    DGRAD_TRACE_CLOCK(tg1);
    dev::named_bar(e.bar_id, 128);
    DGRAD_TRACE_CLOCK(tg2);
    if (threadIdx.x == 0) {
        DGRAD_TRACE_ADD(4, tg1 - tg0);
        DGRAD_TRACE_ADD(5, tg2 - tg1);
    }
    const size_t plane = static_cast<size_t>(p.H) * p.W;
    const bool valid = e.row_ok && e.q < pd.Hq && e.u < pd.Wq;
    const int ih = p.s * e.q + pd.a, iw = p.s * e.u + pd.b;
    float *dst = p.gi + (static_cast<size_t>(e.n) * p.Ci + e.ci0) * plane + static_cast<size_t>(ih) * p.W + iw;
    float pend[1][1][16];
    float *pend_dst = nullptr;
    int pend_cols = 0;
    for (int c0 = 0; c0 < bnp; c0 += 16) {   // combine and store
        if (pend_dst) store_batch<1, 16, FUSE>(p, pend_dst, plane, pend_cols, pend);
        uint32_t r[S][16];
#pragma unroll
        for (int g = 0; g < S; ++g) dev::tmem_ld16(tb + static_cast<uint32_t>(g * bnp + c0), r[g]);
        dev::tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) pend[0][0][j] = __uint_as_float(r[S - 1][j]);
        int slot = 0;
#pragma unroll
        for (int g = 0; g < S - 1; ++g) {
            const int sh = S - 1 - g;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                float v = __shfl_down_sync(0xffffffffu, __uint_as_float(r[g][j]), sh);
                if (e.lane + sh >= 32) v = xn ? xn[(slot + e.lane + sh - 32) * bnp + c0 + j] : 0.f;
                pend[0][0][j] += v;
            }
            slot += sh;
        }
        pend_dst = valid ? dst + static_cast<size_t>(c0) * plane : nullptr;
        pend_cols = min(16, e.nci - c0);
    }
    // Every value of the unit is in registers: release the accumulator set,
    // then store the last batch.
    dev::tc_fence_before();
    dev::mbar_arrive(dev::smem_u32(acc_empty));
    DGRAD_TRACE_CLOCK(tg3);
    if (pend_dst) store_batch<1, 16, FUSE>(p, pend_dst, plane, pend_cols, pend);
    DGRAD_TRACE_CLOCK(tg4);
    if (threadIdx.x == 0) {
        DGRAD_TRACE_ADD(14, tg3 - tg2);
        DGRAD_TRACE_ADD(15, tg4 - tg3);
    }
}

// Epilogue forms, one kernel instantiation each (so that each form's
// registers are allocated on their own): phases stored together (NV),
// sub-accumulators per phase (SMAX) and columns per tensor-memory wait (CB),
// at most 64 loaded registers per batch.
template <int kEpi> struct EpiForm;
template <> struct EpiForm<0> { static constexpr int NV = 1, SMAX = 1, CB = 64; };
template <> struct EpiForm<1> { static constexpr int NV = 1, SMAX = 2, CB = 32; };
template <> struct EpiForm<2> { static constexpr int NV = 1, SMAX = 3, CB = 16; };
template <> struct EpiForm<3> { static constexpr int NV = 1, SMAX = 4, CB = 16; };
template <> struct EpiForm<4> { static constexpr int NV = 2, SMAX = 1, CB = 32; };
template <> struct EpiForm<5> { static constexpr int NV = 2, SMAX = 2, CB = 16; };
template <> struct EpiForm<6> { static constexpr int NV = 4, SMAX = 1, CB = 16; };

__host__ __device__ constexpr int epi_form(int vec_w, int s, int max_sub) {
    return (vec_w && s == 4) ? 6
         : (vec_w && s == 2) ? (max_sub <= 1 ? 4 : 5)
         : (max_sub <= 1 ? 0 : max_sub == 2 ? 1 : max_sub == 3 ? 2 : 3);
}

// kEpi selects the epilogue form (EpiForm).  Registers: each SM sub-
// partition holds a quarter of the register file and a quarter of the
// block's warps (rounded up), so 6 warps leave 255 per thread and 14 warps
// (producer mode) 128.
// kEG: epilogue warp groups (2: warps 6-9 form a second group that takes
// every other work unit and the second accumulator set; tensor-copy mode).
// kStg: staged mode (tensor copies of the caller's grad_out, transposed by
// kTransWarps warps placed after the epilogue warps).
template <bool kTmaA, int kEG, bool kStg>
constexpr int kernel_threads() {
    return kTmaA ? (kProdWarp0 + (kEG - 1) * kEpiWarps + (kStg ? kTransWarps : 0)) * 32 : kThreads;
}

// kTA: tensor-memory A mode (the epilogue warps write A into tensor memory).
template <int KC, bool kTmaA, int kEpi, int kFuse, int kEG, bool kStg, bool kTA = false>
__global__ void __launch_bounds__(kernel_threads<kTmaA, kEG, kStg>(), 1)
    tc_dgrad_kernel(const __grid_constant__ MainParams p) {
    static_assert(kEG == 1 || (kEG == 2 && kTmaA), "a second epilogue group needs the tensor-copy mode");
    static_assert(!kStg || kTmaA, "staged copies are tensor copies");
    static_assert(!kTA || (kTmaA && !kStg && kEG == 1), "tensor-memory A: tensor copies, one epilogue group");
    static_assert(KC == 32, "operand rows are one 128-byte swizzle row of 32 TF32 values");
    extern __shared__ __align__(1024) uint8_t smem[];
    Barriers *bars = reinterpret_cast<Barriers *>(smem);
    uint4 *group_table = reinterpret_cast<uint4 *>(smem + kGroupTableOffset);
    float *xchg = reinterpret_cast<float *>(smem + kXchgOffset);
    // Operand stages start on a 1024-byte boundary of the shared window: the
    // 128-byte swizzle is a function of the address bits inside that pattern.
    const uint32_t smem0 = dev::smem_u32(smem);
    const uint32_t stage0 = (smem0 + kXchgOffset + static_cast<uint32_t>(p.xchg_bytes) + 1023) & ~1023u;
    float *a_base = reinterpret_cast<float *>(smem + (stage0 - smem0));
    const int a_stage_floats = p.a_rows * KC;
    uint8_t *b_base = reinterpret_cast<uint8_t *>(a_base) + static_cast<size_t>(p.a_stages) * a_stage_floats * 4;

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        const uint32_t a_arrivals =
            kStg ? kTransThreads : kTmaA ? 1 : (p.vec_producer ? kGroupThreads : kProdWarps * 32);
        for (int i = 0; i < p.a_stages; ++i) {
            dev::mbar_init(dev::smem_u32(&bars->a_full[i]), a_arrivals);
            dev::mbar_init(dev::smem_u32(&bars->a_empty[i]), 1);
            dev::mbar_init(dev::smem_u32(&bars->stg_full[i]), 1);
            dev::mbar_init(dev::smem_u32(&bars->stg_empty[i]), kEpiWarps * 32);
        }
        for (int i = 0; i < 4; ++i) {
            dev::mbar_init(dev::smem_u32(&bars->ta_full[i]), kEpiWarps * 32);
            dev::mbar_init(dev::smem_u32(&bars->ta_empty[i]), 1);
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
        dev::mbar_init(dev::smem_u32(&bars->never), 1);
        bars->abort_flag = 0;
        dev::fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        dev::tmem_alloc(dev::smem_u32(&bars->tmem_base), p.tmem_cols);
        dev::tmem_relinquish();
        for (int i = lane; i < p.n_mgroups; i += 32) group_table[i] = p.mgroup[i];
    }
    dev::tc_fence_before();
    __syncthreads();
    dev::tc_fence_after();
    const uint32_t tmem_base = bars->tmem_base;
    const long long tmo = p.timeout_ns;
    DGRAD_TRACE_CLOCK(t_start);
    if (threadIdx.x == 0) DGRAD_TRACE_SET(16, dev::globaltimer_ns());
    const int tile_step = p.tile_step;
    const uint32_t tap_b_bytes = static_cast<uint32_t>(p.bn) * 128;   // one tap of one chunk of B
    const int m_cols = p.acc_cols / p.tm;                              // accumulator columns of one M block

    if (!kTmaA && warp >= kProdWarp0) {
        // ------------------------------------------------------ producers
        if (p.vec_producer)
            produce_quads<KC>(p, bars, a_base, a_stage_floats, tile_step, tmo);
        else
            produce_async4<KC>(p, bars, a_base, a_stage_floats, tile_step, tmo);
        DGRAD_TRACE_CLOCK(t_pend);
        if (threadIdx.x == kProdWarp0 * 32) DGRAD_TRACE_ADD(12, t_pend - t_start);
    } else if (kStg && warp >= kProdWarp0 + (kEG - 1) * kEpiWarps) {
        // ---------------------------------------------------- transposers
        transpose_stages<KC, kEG>(p, bars, a_base, a_stage_floats, tmo);
        DGRAD_TRACE_CLOCK(t_pend);
        if (threadIdx.x == (kProdWarp0 + (kEG - 1) * kEpiWarps) * 32) DGRAD_TRACE_ADD(12, t_pend - t_start);
    } else if (warp == kLoadWarp) {
        // ------------------------------------------------- weight loader
        // B stage (c, tg) = taps [bg_tap0[tg], bg_tap0[tg+1]) of channel
        // chunk c of the work unit's slice: one contiguous block of the
        // packed weights.
        // Staged mode: grad_out comes from HBM, so the boxes of the stages
        // kPrefetchAhead ahead of the one being loaded are prefetched into
        // L2 (a CTA's stages are its units' chunks in order); the stage
        // copies then hit L2.  grad_out is the caller's input, not an output
        // of the preceding kernel, so the first ones go out before the wait.
        // Tensor-memory A mode likewise, with the boxes of the one or two
        // images of each tile.
        const int n_seq = (kStg || kTA) ? ((p.n_work - static_cast<int>(blockIdx.x) +
                                            static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x)) * p.n_chunks
                                        : 0;
        const int ahead = (kStg || kTA) ? p.prefetch_ahead : 0;
        auto prefetch_stage = [&](int s) {
            if (ahead == 0 || s >= n_seq) return;
            const int c = s % p.n_chunks;
            if (p.split_chunks && c >= p.split_chunks) return;   // passes 1 and 2 re-read pass 0's boxes
            const int w = static_cast<int>(blockIdx.x) + (s / p.n_chunks) * static_cast<int>(gridDim.x);
            int lim;
            const int P0 = tile_origin(p, w / p.n_slices, lim);
            if constexpr (kTA) {
                const int plane = p.oH * p.oW;
                const int n0 = P0 / plane, x0 = P0 - n0 * plane;
                dev::tma_prefetch_3d(&p.a_map, x0, c * KC, n0);
                if (x0 + kBlockM > plane && n0 + 1 < p.N) dev::tma_prefetch_3d(&p.a_map, 0, c * KC, n0 + 1);
            } else {
                const int n = P0 / p.HvWp;
                dev::tma_prefetch_3d(&p.a_map, plane_elems_below(p, n, P0) & ~3, c * KC, n);
            }
        };
        if (lane == 0) {
            if (kTmaA) dev::prefetch_tensormap(&p.a_map);
            if (kStg || kTA)
                for (int s = 0; s < ahead; ++s) prefetch_stage(s);
            dev::grid_dependency_wait();   // packed weights (and frame) come from the preceding kernel
            int last_parity[kMaxBStages];   // parity of each stage's last fill, -1 if never filled
            for (int i = 0; i < kMaxBStages; ++i) last_parity[i] = -1;
            int a_last_parity[kMaxAStages];
            for (int i = 0; i < kMaxAStages; ++i) a_last_parity[i] = -1;
            if (p.b_resident) {   // one slice, one stage per chunk: load everything once
                for (int c = 0; c < p.n_chunks; ++c) {
                    const uint32_t bar = dev::smem_u32(&bars->b_full[c]);
                    dev::mbar_arrive_expect_tx(bar, p.chunk_bytes);
                    dev::bulk_g2s(dev::smem_u32(b_base + static_cast<size_t>(c) * p.chunk_bytes),
                                  reinterpret_cast<const uint8_t *>(p.wp) + static_cast<size_t>(c) * p.chunk_bytes,
                                  p.chunk_bytes, bar);
                    last_parity[c] = 0;
                }
            }
            if (kTmaA || !p.b_resident) {
                Ring ring, aring;
                bool ok = true;
                int seq = 0;   // staged: this CTA's stages loaded so far
                const uint32_t a_stage_bytes = static_cast<uint32_t>(a_stage_floats) * 4;
                for (int w = blockIdx.x; ok && w < p.n_work && !bars->abort_flag; w += gridDim.x) {
                    const int slice = w % p.n_slices;
                    int lim;
                    const int P0 = tile_origin(p, w / p.n_slices, lim);
                    // staged: the band's image and its first plane element, rounded down to a
                    // 16-byte boundary (the tensor copy's innermost coordinate must be one)
                    const int sn = kStg ? P0 / p.HvWp : 0;
                    const int sx0 = kStg ? plane_elems_below(p, sn, P0) & ~3 : 0;
                    // tensor-memory A: the tile's first image and element, and whether it runs into the next image
                    const int tplane = p.oH * p.oW;
                    const int tn0 = kTA ? P0 / tplane : 0;
                    const int tx0 = kTA ? P0 - tn0 * tplane : 0;
                    const bool tcross = kTA && !p.img_tiles && tx0 + kBlockM > tplane && tn0 + 1 < p.N;
                    for (int c = 0; ok && c < p.n_chunks; ++c) {
                        if (kTmaA) {
                            // A stage: frame rows [P0, P0 + a_rows) x channels [32c, 32c + 32)
                            const uint32_t empty = dev::smem_u32(kTA ? &bars->stg_empty[aring.stage]
                                                                     : &bars->a_empty[aring.stage]);
                            if (!dev::mbar_wait(empty, aring.parity ^ 1, tmo)) {
                                fail(bars, p);
                                ok = false;
                                break;
                            }
                            const uint32_t dst = dev::smem_u32(a_base) + aring.stage * a_stage_bytes;
                            if constexpr (kTA) {
                                // channels [32cc, 32cc + 32) of the tile's positions (one or two images)
                                prefetch_stage(seq + ahead);
                                ++seq;
                                const uint32_t bar = dev::smem_u32(&bars->stg_full[aring.stage]);
                                const uint32_t box = kBlockM * KC * 4;
                                dev::mbar_arrive_expect_tx(bar, tcross ? 2 * box : box);
                                const int cc = p.split_chunks ? c % p.split_chunks : c;
                                dev::tma_load_3d(dst, &p.a_map, tx0, cc * KC, tn0, bar);
                                if (tcross) dev::tma_load_3d(dst + box, &p.a_map, 0, cc * KC, tn0 + 1, bar);
                            } else if constexpr (kStg) {
                                // grad_out elements [sx0, sx0 + stg_box) of 32 channels of image sn; split
                                // precision reads channel chunk c mod split_chunks in every K pass
                                prefetch_stage(seq + ahead);
                                ++seq;
                                const uint32_t bar = dev::smem_u32(&bars->stg_full[aring.stage]);
                                dev::mbar_arrive_expect_tx(bar, static_cast<uint32_t>(p.stg_box) * KC * 4);
                                const int cc = p.split_chunks ? c % p.split_chunks : c;
                                dev::tma_load_3d(dst, &p.a_map, sx0, cc * KC, sn, bar);
                            } else {
                                const uint32_t bar = dev::smem_u32(&bars->a_full[aring.stage]);
                                dev::mbar_arrive_expect_tx(bar, a_stage_bytes);
                                // Split precision: K pass c / split_chunks = 0, 1, 2 reads the
                                // hi, lo, hi half of the frame rows (B holds lo, hi, hi).
                                int x = c * KC;
                                if (p.split_chunks) {
                                    const int pass = c / p.split_chunks;
                                    x = (c - pass * p.split_chunks) * KC + (pass == 1 ? p.co_h : 0);
                                }
                                for (int b = 0; b < p.a_nbox; ++b)
                                    dev::tma_load_2d(dst + static_cast<uint32_t>(b * p.a_box_rows) * 128, &p.a_map,
                                                     x, P0 + b * p.a_box_rows, bar);
                            }
                            a_last_parity[aring.stage] = static_cast<int>(aring.parity);
                            aring.next(p.a_stages);
                        }
                        for (int tg = 0; !p.b_resident && tg < p.n_tgroups; ++tg) {
                            if (!dev::mbar_wait(dev::smem_u32(&bars->b_empty[ring.stage]), ring.parity ^ 1, tmo)) {
                                fail(bars, p);
                                ok = false;
                                break;
                            }
                            const int t0 = p.bg_tap0[tg];
                            const uint32_t bytes = static_cast<uint32_t>(p.bg_tap0[tg + 1] - t0) * tap_b_bytes;
                            const uint32_t bar = dev::smem_u32(&bars->b_full[ring.stage]);
                            dev::mbar_arrive_expect_tx(bar, bytes);
                            const size_t off =
                                ((static_cast<size_t>(slice) * p.n_chunks + c) * p.n_taps + t0) * tap_b_bytes;
                            dev::bulk_g2s(dev::smem_u32(b_base + static_cast<size_t>(ring.stage) * p.chunk_bytes),
                                          reinterpret_cast<const uint8_t *>(p.wp) + off, bytes, bar);
                            last_parity[ring.stage] = static_cast<int>(ring.parity);
                            ring.next(p.b_stages);
                        }
                    }
                }
            }
            // Never leave with a copy in flight into this CTA's shared memory.
            for (int i = 0; i < p.b_stages && i < kMaxBStages; ++i)
                if (last_parity[i] >= 0) dev::mbar_wait(dev::smem_u32(&bars->b_full[i]), last_parity[i], tmo);
            for (int i = 0; i < p.a_stages && i < kMaxAStages; ++i)
                if (a_last_parity[i] >= 0)
                    dev::mbar_wait(dev::smem_u32((kStg || kTA) ? &bars->stg_full[i] : &bars->a_full[i]),
                                   a_last_parity[i], tmo);
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ---------------------------------------------------- MMA issuer
        // The whole warp runs this loop converged; every wait is taken by all
        // lanes and agreed with a vote, and one elected lane issues the MMAs
        // and commits (warp-uniform descriptors stay in uniform registers).
        const uint32_t a_addr0 = dev::smem_u32(a_base);
        const uint32_t b_addr0 = dev::smem_u32(b_base);
        Ring ra, rb, racc;
        bool ok = true;
        bool first_chunk = true;
        // Failure-detection test: a bounded wait on a barrier that nothing
        // completes runs out; the whole CTA then takes its abort path.
        if (p.wait_test && !__all_sync(0xffffffffu, dev::mbar_wait(dev::smem_u32(&bars->never), 0, tmo))) {
            if (lane == 0) fail(bars, p);
            ok = false;
        }
        for (int w = blockIdx.x; ok && w < p.n_work && !bars->abort_flag; w += gridDim.x, racc.next(p.acc_bufs)) {
            DGRAD_TRACE_CLOCK(tm0);
            if (!__all_sync(0xffffffffu,
                            dev::mbar_wait(dev::smem_u32(&bars->acc_empty[racc.stage]), racc.parity ^ 1, tmo))) {
                if (lane == 0) fail(bars, p);
                break;
            }
            DGRAD_TRACE_CLOCK(tm1);
            if (lane == 0) {
                DGRAD_TRACE_ADD(0, tm1 - tm0);
                DGRAD_TRACE_ADD(8, 1);
            }
            dev::tc_fence_after();
            const uint32_t d_base = tmem_base + racc.stage * p.acc_cols;
            for (int c = 0; ok && c < p.n_chunks; ++c, ra.next(kTA ? p.a_tslots : p.a_stages)) {
                DGRAD_TRACE_CLOCK(tc0);
                const uint32_t a_ready = dev::smem_u32(kTA ? &bars->ta_full[ra.stage] : &bars->a_full[ra.stage]);
                if (!__all_sync(0xffffffffu, dev::mbar_wait(a_ready, ra.parity, tmo))) {
                    if (lane == 0) fail(bars, p);
                    ok = false;
                    break;
                }
                DGRAD_TRACE_CLOCK(tc1);
                if (lane == 0) {
                    DGRAD_TRACE_ADD(1, tc1 - tc0);
                    DGRAD_TRACE_ADD(9, 1);
                    if (first_chunk) DGRAD_TRACE_ADD(10, tc1 - t_start);
                }
                first_chunk = false;
                // Stages written with cp.async (4-byte producer) reach the
                // consumer through the barrier only; make them visible to the
                // tensor core's operand reads here.  The quad producer fences
                // its own stores instead, so this fence (which would also wait
                // for this thread's MMAs in flight) is not taken on that path.
                if (!kTmaA && !p.vec_producer) dev::fence_proxy_async_smem();
                const uint32_t a_stage = a_addr0 + static_cast<uint32_t>(ra.stage) * a_stage_floats * 4;
                for (int tg = 0; tg < p.n_tgroups; ++tg) {
                    const int sb = p.b_resident ? c : rb.stage;
                    const uint32_t pb = p.b_resident ? 0u : rb.parity;
                    DGRAD_TRACE_CLOCK(tb0);
                    if (!__all_sync(0xffffffffu, dev::mbar_wait(dev::smem_u32(&bars->b_full[sb]), pb, tmo))) {
                        if (lane == 0) fail(bars, p);
                        ok = false;
                        break;
                    }
                    DGRAD_TRACE_CLOCK(tb1);
                    if (lane == 0) DGRAD_TRACE_ADD(2, tb1 - tb0);
                    dev::tc_fence_after();
                    // B stage base, rebased so that a group's tap offset indexes it directly
                    const uint32_t b_stage = b_addr0 + static_cast<uint32_t>(sb) * p.chunk_bytes -
                                             static_cast<uint32_t>(p.bg_tap0[tg]) * tap_b_bytes;
                    const int g0 = p.bg_first[tg], g1 = p.bg_first[tg + 1];
                    for (int m = 0; m < p.tm; ++m) {
                        const uint32_t a_m = a_stage + static_cast<uint32_t>(m * kBlockM) * 128;
                        const uint32_t d_m = d_base + static_cast<uint32_t>(m * m_cols);
                        uint4 nxt = group_table[g0];
                        for (int gi = g0; gi < g1; ++gi) {
                            const uint4 cur = nxt;
                            if (gi + 1 < g1) nxt = group_table[gi + 1];   // prefetch the next group's entry
                            // A window of the group: frame rows [m*128 + shift, +128) of the
                            // stage.  The swizzle follows the absolute address bits, so the
                            // window may start on any 128-byte row with base offset 0.
                            const uint64_t ad = dev::smem_desc_sw128(a_m + cur.x, 0);
                            const uint64_t bd = dev::smem_desc_sw128(b_stage + cur.z, 0);
                            const uint32_t d = d_m + (cur.y & 0x7fffffffu);
                            const uint32_t acc0 = (c > 0 || (cur.y >> 31) == 0) ? 1u : 0u;
                            if constexpr (kTA) {
                                // A from tensor memory: slot ra.stage, K columns 8*k8 ..
                                const uint32_t at = tmem_base + static_cast<uint32_t>(p.a_tcol + ra.stage * KC);
#pragma unroll
                                for (int k8 = 0; k8 < KC / 8; ++k8)
                                    dev::mma_tf32_ts_elect(d, at + 8 * k8, dev::desc_add(bd, 32 * k8), cur.w,
                                                           k8 > 0 ? 1u : acc0);
                            } else {
#pragma unroll
                                for (int k8 = 0; k8 < KC / 8; ++k8)
                                    dev::mma_tf32_elect(d, dev::desc_add(ad, 32 * k8), dev::desc_add(bd, 32 * k8),
                                                        cur.w, k8 > 0 ? 1u : acc0);
                            }
                        }
                    }
                    if (!p.b_resident) {
                        dev::mma_commit_elect(dev::smem_u32(&bars->b_empty[sb]));
                        rb.next(p.b_stages);
                    }
                    DGRAD_TRACE_CLOCK(tb2);
                    if (lane == 0) DGRAD_TRACE_ADD(3, tb2 - tb1);
                }
                if (!ok) break;
                dev::mma_commit_elect(dev::smem_u32(kTA ? &bars->ta_empty[ra.stage] : &bars->a_empty[ra.stage]));
            }
            if (!ok) break;
            dev::mma_commit_elect(dev::smem_u32(&bars->acc_full[racc.stage]));
        }
        // Drain: every MMA issued above has finished before TMEM is freed.
        dev::mma_commit_elect(dev::smem_u32(&bars->drain));
        if (!__all_sync(0xffffffffu, dev::mbar_wait(dev::smem_u32(&bars->drain), 0, tmo)) && lane == 0)
            fail(bars, p);
        DGRAD_TRACE_CLOCK(t_mend);
        if (lane == 0) DGRAD_TRACE_ADD(11, t_mend - t_start);
    } else {
        // ------------------------------------------------------- epilogue
        // Warp ew = warp % 4 reads tensor-memory lanes 32*ew .. 32*ew+31.  (A
        // second group of four epilogue warps taking alternate units measured
        // slower: ten warps leave 168 registers per thread, six leave 255.)
        const int ew = warp & 3;
        const int slots = p.max_sub * (p.max_sub - 1) / 2;
        const int gi = (kEG == 2 && warp >= kProdWarp0) ? 1 : 0;   // epilogue group
        EpiCtx e;
        e.p = &p;
        e.xbase = xchg + static_cast<size_t>(gi) * (p.xchg_bytes / 4 / kEG);
        e.slots = slots;
        e.ew = ew;
        e.lane = lane;
        e.bar_id = 1 + gi;
        e.xcount = 0;
        Ring racc;
        Ring ta_rs, ta_rt;   // tensor-memory A mode: shared-memory stages and tensor-memory slots
        uint32_t it = 0;
        // One group: every unit, accumulator sets in turn.  Two groups: group gi
        // takes the CTA's units gi, gi + 2, ... and always accumulator set gi.
        for (int w = blockIdx.x + gi * static_cast<int>(gridDim.x); w < p.n_work;
             w += kEG * static_cast<int>(gridDim.x), ++it) {
            int stage;
            uint32_t parity;
            if constexpr (kEG == 2) {
                stage = gi;
                parity = it & 1u;
            } else {
                stage = racc.stage;
                parity = racc.parity;
                racc.next(p.acc_bufs);
            }
            const int tile = w / p.n_slices, slice = w % p.n_slices;
            // Tensor-memory A mode: first this unit's A, chunk by chunk, into tensor memory.
            bool wrote = true;
            if constexpr (kTA)
                wrote = write_tmem_a<KC>(p, bars, a_base, a_stage_floats, tmem_base, tile, ew, lane, ta_rs, ta_rt, tmo);
            DGRAD_TRACE_CLOCK(te0);
            // All four warps of the group leave together or go on together.
            const bool got = wrote && dev::mbar_wait(dev::smem_u32(&bars->acc_full[stage]), parity, tmo);
            if (!dev::named_bar_and(e.bar_id, 128, got)) {
                if (!got && wrote) fail(bars, p);
                break;
            }
            DGRAD_TRACE_CLOCK(te1);
            if (threadIdx.x == 0) DGRAD_TRACE_ADD(6, te1 - te0);
            dev::tc_fence_after();
            e.ci0 = slice * p.bn;
            e.nci = min(p.bn, p.Ci - e.ci0);
            using F = EpiForm<kEpi>;
            const uint32_t tbase0 =
                tmem_base + (static_cast<uint32_t>(ew * 32) << 16) + static_cast<uint32_t>(stage * p.acc_cols);
            if constexpr (F::NV == 1 && F::SMAX > 1) {
                if (p.xchg_unit && p.phase[0].tap_count > 0 && p.phase[0].sub == F::SMAX)
                    epilogue_run_g1<F::SMAX, kFuse>(e, tile, tbase0, &bars->acc_empty[stage], e.xcount++ & 1u);
                else
                    epilogue_run<F::NV, F::SMAX, F::CB, kFuse>(e, tile, tbase0, m_cols, &bars->acc_empty[stage]);
            } else {
                epilogue_run<F::NV, F::SMAX, F::CB, kFuse>(e, tile, tbase0, m_cols, &bars->acc_empty[stage]);
            }
            DGRAD_TRACE_CLOCK(te2);
            if (threadIdx.x == 0) DGRAD_TRACE_ADD(7, te2 - te1);
        }
        DGRAD_TRACE_CLOCK(t_eend);
        if (threadIdx.x == 0) DGRAD_TRACE_ADD(13, t_eend - t_start);
    }

    dev::tc_fence_before();
    __syncthreads();
    dev::tc_fence_after();
    if (warp == kMmaWarp) dev::tmem_dealloc(tmem_base, p.tmem_cols);
    DGRAD_TRACE_CLOCK(t_cta_end);
    if (threadIdx.x == 0) {
        DGRAD_TRACE_SET(17, dev::globaltimer_ns());
        DGRAD_TRACE_SET(18, t_cta_end - t_start);
    }
}

template <int KC, bool kTmaA, int kEpi, int kFuse, int kEG = 1, bool kStg = false, bool kTA = false>
cudaError_t launch_kc(const MainParams &p, const Tiling &t, cudaStream_t stream, bool pdl) {
    auto kern = tc_dgrad_kernel<KC, kTmaA, kEpi, kFuse, kEG, kStg, kTA>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, t.smem_bytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(t.grid);
    cfg.blockDim = dim3(kernel_threads<kTmaA, kEG, kStg>());
    cfg.dynamicSmemBytes = t.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

template <bool kTmaA, int kFuse, bool kStg = false>
cudaError_t launch_mode(const MainParams &p, const Tiling &t, cudaStream_t stream, bool pdl) {
    // Two epilogue groups for the grouped forms of plain-store tensor-copy
    // launches (the fused-epilogue instances keep one group).
    constexpr bool kTwo = kTmaA && kFuse == 0;
    constexpr int kEG2 = kTwo ? 2 : 1;
    const bool two = kTwo && p.epi_groups == 2 && p.acc_bufs == 2;
    switch (epi_form(p.vec_w, p.s, p.max_sub)) {
        case 0: return launch_kc<32, kTmaA, 0, kFuse, 1, kStg>(p, t, stream, pdl);
        case 1:
            return two ? launch_kc<32, kTmaA, 1, kFuse, kEG2, kStg>(p, t, stream, pdl)
                       : launch_kc<32, kTmaA, 1, kFuse, 1, kStg>(p, t, stream, pdl);
        case 2:
            return two ? launch_kc<32, kTmaA, 2, kFuse, kEG2, kStg>(p, t, stream, pdl)
                       : launch_kc<32, kTmaA, 2, kFuse, 1, kStg>(p, t, stream, pdl);
        case 3:
            return two ? launch_kc<32, kTmaA, 3, kFuse, kEG2, kStg>(p, t, stream, pdl)
                       : launch_kc<32, kTmaA, 3, kFuse, 1, kStg>(p, t, stream, pdl);
        case 4: return launch_kc<32, kTmaA, 4, kFuse, 1, kStg>(p, t, stream, pdl);
        case 5: return launch_kc<32, kTmaA, 5, kFuse, 1, kStg>(p, t, stream, pdl);
        default: return launch_kc<32, kTmaA, 6, kFuse, 1, kStg>(p, t, stream, pdl);
    }
}

}  // namespace

}  // namespace dgrad

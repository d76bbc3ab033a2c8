// Pack kernel: one launch that (a) packs the weights and (b) optionally packs
// grad_out into the channels-last, zero-padded frame the tcgen05 kernel
// copies with the tensor engine.
//
// (a) OIHW fp32 weights -> the packed layout of PrepackParams.  Replaces
//     meganeura's per-element implicit W^T reads (its A-tile load decomposes
//     k into (co, kh, kw) with divisions and reads weight with a strided
//     index) by one pass that writes each (slice, chunk) block contiguously,
//     keeps only the taps each phase uses, zero-pads channels, and (TF32
//     precision) rounds to TF32 once.
// (b) grad_out NCHW -> V[P][k] (FramePackParams): one block transposes a
//     tile of kFrameTileElems (consecutive frame positions x 32, 64 or 128
//     channels) through shared memory, so both the grad_out reads (along
//     positions) and the V writes (along channels) are coalesced.  Frame positions
//     outside grad_out, and channels >= Co, are written as zeros; the
//     meganeura shader's transposed padding becomes these zero rows.
#include <cuda_runtime.h>

#include "dgrad_internal.h"
#include "ptx.cuh"

namespace dgrad {

namespace {

constexpr int kThreads = 256;
static_assert(kFrameTileElems % kThreads == 0 && kFrameTileElems / 128 <= kThreads, "frame tile split");
constexpr int kMaxPrepackBlocks = 1024;

struct PackArgs {
    PrepackParams w;        // valid when w_blocks > 0
    FramePackParams f;      // valid when f_blocks > 0
    int w_blocks;
    int f_blocks;
};

__device__ void pack_weights(const PrepackParams &p, int block, int nblocks) {
    const long long stride = static_cast<long long>(nblocks) * kThreads;
    const int G = p.kc / 4;
    for (long long i = static_cast<long long>(block) * kThreads + threadIdx.x; i < p.total; i += stride) {
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
        // Split precision: chunk c is K pass c / split_chunks of channel chunk c mod split_chunks.
        const int cc = p.split_chunks ? c % p.split_chunks : c;
        const int co = cc * p.kc + 4 * gq + e;
        const int ci = sl * p.bn + j;
        float v = 0.f;
        if (co < p.Co && ci < p.Ci)
            v = __ldg(p.w + ((static_cast<size_t>(co) * p.Ci + ci) * p.kH + p.tap_kh[t]) * p.kW + p.tap_kw[t]);
        if (p.split_chunks) {
            const float hi = dev::round_tf32(v);
            v = c < p.split_chunks ? dev::round_tf32(v - hi) : hi;   // pass 0 takes the low part
        } else if (p.round_tf32) {
            v = dev::round_tf32(v);
        }
        p.wp[i] = v;
    }
}

// One frame tile of TP = kFrameTileElems / TC consecutive positions x TC
// channels.  block -> (position tile, channel group); position tiles vary
// fastest so neighbouring blocks read neighbouring grad_out runs.  Wide
// frames (many channels per position) take wide channel groups, so each
// position's row segment written is TC * 4 bytes long.
template <int TC>
__device__ void pack_frame(const FramePackParams &p, int block, float *tile, int *off) {
    constexpr int TP = kFrameTileElems / TC;
    constexpr int kStride = TP + 1;
    const int pt = block % p.pos_tiles;
    const int co0 = (block / p.pos_tiles) * TC;
    const int P0 = pt * TP;
    const int plane = p.oH * p.oW;
    if (threadIdx.x < TP) {   // grad_out offset of channel 0 at each position, or -1
        const int P = P0 + threadIdx.x;
        int o = -1;
        if (P < p.positions) {
            const int img = p.Hv * p.Wp;
            const int n = P / img, rem = P - n * img;
            const int y = rem / p.Wp, x = rem - y * p.Wp;
            const int oh = y - p.Ph, ow = x - p.Pw;
            if (oh >= 0 && oh < p.oH && ow >= 0 && ow < p.oW) o = n * p.Co * plane + oh * p.oW + ow;
        }
        off[threadIdx.x] = o;
    }
    __syncthreads();
    // read: TC channels x TP positions, coalesced along positions.  Each
    // thread keeps one position and issues all of its channel loads before
    // the first shared-memory store, so they are in flight together.
    {
        constexpr int kRowsPerPass = kThreads / TP;
        constexpr int kLoads = TC / kRowsPerPass;
        const int xi = threadIdx.x % TP;
        const int c0 = threadIdx.x / TP;
        const int o = off[xi];
        float v[kLoads];
#pragma unroll
        for (int k = 0; k < kLoads; ++k) {
            const int co = co0 + c0 + kRowsPerPass * k;
            v[k] = (o >= 0 && co < p.Co) ? __ldg(p.go + static_cast<size_t>(o) + static_cast<size_t>(co) * plane) : 0.f;
        }
#pragma unroll
        for (int k = 0; k < kLoads; ++k)
            tile[(c0 + kRowsPerPass * k) * kStride + xi] = p.round_tf32 ? dev::round_tf32(v[k]) : v[k];
    }
    __syncthreads();
    // write: each position's TC channels (TC * 4 contiguous bytes), coalesced along channels
    const int ncols = min(TP, p.positions - P0);
    const int cmax = min(TC, (p.split ? p.co_h : p.co_v) - co0);
    float *dst = p.v + static_cast<size_t>(P0) * p.co_v + co0;
    for (int i = threadIdx.x; i < TC * ncols; i += kThreads) {
        const int xi = i / TC, c = i % TC;
        if (c < cmax) {
            const float x = tile[c * kStride + xi];
            float *row = dst + static_cast<size_t>(xi) * p.co_v;
            if (p.split) {   // hi in the first half of the row, lo in the second
                const float hi = dev::round_tf32(x);
                row[c] = hi;
                row[p.co_h + c] = dev::round_tf32(x - hi);
            } else {
                row[c] = x;
            }
        }
    }
}

__global__ void __launch_bounds__(kThreads) pack_kernel(const __grid_constant__ PackArgs a) {
    // Let the main kernel start its prologue while this grid runs; it reads
    // what this grid writes only after griddepcontrol.wait.
    dev::grid_launch_dependents();
    __shared__ float tile[kFrameTileElems + 128];   // TC x (TP + 1) = kFrameTileElems + TC floats, TC <= 128
    __shared__ int off[kFrameTileElems / 32];
    if (static_cast<int>(blockIdx.x) < a.w_blocks) {
        pack_weights(a.w, blockIdx.x, a.w_blocks);
    } else {
        const int b = blockIdx.x - a.w_blocks;
        if (a.f.tile_c == 128)
            pack_frame<128>(a.f, b, tile, off);
        else if (a.f.tile_c == 64)
            pack_frame<64>(a.f, b, tile, off);
        else
            pack_frame<32>(a.f, b, tile, off);
    }
}

}  // namespace

cudaError_t launch_pack(const PrepackParams *pp, const FramePackParams *fp, cudaStream_t stream) {
    PackArgs a{};
    if (pp) {
        a.w = *pp;
        long long blocks = (pp->total + kThreads - 1) / kThreads;
        a.w_blocks = static_cast<int>(blocks < 1 ? 1 : (blocks > kMaxPrepackBlocks ? kMaxPrepackBlocks : blocks));
    }
    if (fp) {
        a.f = *fp;
        a.f_blocks = fp->pos_tiles * fp->c_groups;   // c_groups = ceil(co_v / tile_c)
    }
    const int blocks = a.w_blocks + a.f_blocks;
    if (blocks == 0) return cudaSuccess;
    pack_kernel<<<blocks, kThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace dgrad

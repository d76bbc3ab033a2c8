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
// (b) grad_out NCHW -> V[P][k] (FramePackParams): one block transposes 32
//     channels x up to 256 consecutive plane elements through a swizzled
//     shared tile, with 16-byte accesses on both sides (grad_out runs along
//     positions, frame rows along channels).  Only the rows of grad_out's
//     positions are written: the frame's zero rows and zero channels (the
//     meganeura shader's transposed padding) are set once when the plan is
//     made.
#include <cuda_runtime.h>

#include "dgrad_internal.h"
#include "ptx.cuh"

namespace dgrad {

namespace {

constexpr int kThreads = 256;
static_assert(kPackChannels == 32 && kThreads == 8 * kPackChannels && kPackSegMax % 32 == 0,
              "frame block: 8 threads per channel row, 32 positions per write step");
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
        if (p.layout == 2) {   // col2im: [chunk][r = (kh*kW + kw)*Ci + ci][swizzled 16-byte group][4]
            const int pos = static_cast<int>(rest % 8);
            rest /= 8;
            const int r = static_cast<int>(rest % p.bn);
            const int c = static_cast<int>(rest / p.bn);
            const int co = c * p.kc + 4 * (pos ^ (r & 7)) + e;
            const int taps = p.kH * p.kW;
            float v = 0.f;
            if (co < p.Co && r < p.Ci * taps) {
                const int tap = r / p.Ci, ci = r - tap * p.Ci;
                v = __ldg(p.w + (static_cast<size_t>(co) * p.Ci + ci) * taps + tap);
            }
            p.wp[i] = p.round_tf32 ? dev::round_tf32(v) : v;
            continue;
        }
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

// Shared tile of one frame block: 32 channel rows of `pitch` (= seg_len) floats.
// The 16-byte group g of row j sits at group (g & ~7) | ((g ^ (j >> 2)) & 7):
// the 16-byte stores of the read phase (8 threads along one row) and the
// 4-channel column reads of the write phase (a warp: 4 positions x 8 channel
// quads) both hit 32 distinct banks.
__device__ __forceinline__ int tile_index(int j, int e, int pitch) {
    const int g = e >> 2;
    return j * pitch + (((g & ~7) | ((g ^ (j >> 2)) & 7)) << 2) + (e & 3);
}

// One frame block: image n, channels [c0, c0 + 32) and plane elements
// [e0, e0 + len) of grad_out.
//  read:  thread t takes channel t / 8 and the 16-byte groups t % 8 + 8k of
//         its run (8 threads cover one 128-byte line), every load in flight
//         before the shared-memory stores;
//  write: thread t takes channel quad t % 8 and positions t / 8 + 32k; the
//         frame row of a position gets 4 channels per 16-byte store (a warp
//         writes 4 whole 128-byte row segments).
template <bool kVec>
__device__ void pack_frame(const FramePackParams &p, int block, float *tile) {
    constexpr int kSteps = kPackSegMax / 32;   // 16-byte groups per thread (read) and positions per thread (write)
    const int plane = p.oH * p.oW;
    const int seg = block % p.segs;
    const int rest = block / p.segs;
    const int cg = rest % p.c_groups;
    const int n = rest / p.c_groups;
    const int c0 = cg * kPackChannels;
    const int e0 = seg * p.seg_len;
    const int len = min(p.seg_len, plane - e0);
    const int t = threadIdx.x;
    {
        const int j = t >> 3, c = c0 + j;
        const int eb = (t & 7) << 2;   // first element of this thread's first group
        const float *src = p.go + (static_cast<size_t>(n) * p.Co + c) * plane + e0 + eb;
        float4 v[kSteps];
#pragma unroll
        for (int k = 0; k < kSteps; ++k) {
            const int e = eb + 32 * k;
            v[k] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (c < p.Co && e < len) {
                if (kVec && e + 4 <= len) {
                    v[k] = __ldg(reinterpret_cast<const float4 *>(src + 32 * k));
                } else {
                    v[k].x = __ldg(src + 32 * k);
                    if (e + 1 < len) v[k].y = __ldg(src + 32 * k + 1);
                    if (e + 2 < len) v[k].z = __ldg(src + 32 * k + 2);
                    if (e + 3 < len) v[k].w = __ldg(src + 32 * k + 3);
                }
            }
        }
        float *dst = tile + tile_index(j, eb, p.seg_len);   // group t%8 + 8k sits 32k floats further on
#pragma unroll
        for (int k = 0; k < kSteps; ++k)
            if (eb + 32 * k < p.seg_len) *reinterpret_cast<float4 *>(dst + 32 * k) = v[k];
    }
    __syncthreads();
    const int q = t & 7;
    const int c = c0 + 4 * q;
    if (c >= (p.split ? p.co_h : p.co_v)) return;
    int e = t >> 3;
    if (e >= len) return;
    const int pitch = p.seg_len;
    const float *s0 = tile + tile_index(4 * q, e, pitch);   // rows 4q..4q+3 at position e; +32 floats per step
    int oh = (e0 + e) / p.oW, ow = (e0 + e) - oh * p.oW;
    float *vbase = p.v + static_cast<size_t>(c);
#pragma unroll
    for (int k = 0; k < kSteps; ++k, e += 32) {
        if (e >= len) break;
        float4 x;
        x.x = s0[32 * k];
        x.y = s0[32 * k + pitch];
        x.z = s0[32 * k + 2 * pitch];
        x.w = s0[32 * k + 3 * pitch];
        const size_t P = (static_cast<size_t>(n) * p.Hv + oh + p.Ph) * p.Wp + ow + p.Pw;
        float *row = vbase + P * p.co_v;
        if (p.split) {   // hi in the first half of the row, lo in the second
            float4 hi, lo;
            hi.x = dev::round_tf32(x.x), lo.x = dev::round_tf32(x.x - hi.x);
            hi.y = dev::round_tf32(x.y), lo.y = dev::round_tf32(x.y - hi.y);
            hi.z = dev::round_tf32(x.z), lo.z = dev::round_tf32(x.z - hi.z);
            hi.w = dev::round_tf32(x.w), lo.w = dev::round_tf32(x.w - hi.w);
            *reinterpret_cast<float4 *>(row) = hi;
            *reinterpret_cast<float4 *>(row + p.co_h) = lo;
        } else {
            if (p.round_tf32) {
                x.x = dev::round_tf32(x.x), x.y = dev::round_tf32(x.y);
                x.z = dev::round_tf32(x.z), x.w = dev::round_tf32(x.w);
            }
            *reinterpret_cast<float4 *>(row) = x;
        }
        ow += 32;   // next position of this thread: 32 elements further on in the plane
        while (ow >= p.oW) {
            ow -= p.oW;
            ++oh;
        }
    }
}

__global__ void __launch_bounds__(kThreads) pack_kernel(const __grid_constant__ PackArgs a) {
    // Let the main kernel start its prologue while this grid runs; it reads
    // what this grid writes only after griddepcontrol.wait.
    dev::grid_launch_dependents();
    extern __shared__ __align__(16) float tile[];   // kPackChannels x seg_len floats
    if (static_cast<int>(blockIdx.x) < a.w_blocks) {
        pack_weights(a.w, blockIdx.x, a.w_blocks);
    } else {
        const int b = blockIdx.x - a.w_blocks;
        if (a.f.vec)
            pack_frame<true>(a.f, b, tile);
        else
            pack_frame<false>(a.f, b, tile);
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
        a.f_blocks = fp->N * fp->c_groups * fp->segs;
    }
    const int blocks = a.w_blocks + a.f_blocks;
    if (blocks == 0) return cudaSuccess;
    const size_t smem = fp ? static_cast<size_t>(kPackChannels) * fp->seg_len * sizeof(float) : 0;
    pack_kernel<<<blocks, kThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace dgrad

// Producer side of the implicit GEMM: copy a band of the zero-padded,
// flattened grad_out frame V into shared memory as the GEMM's A operand.
//
// meganeura's shader rebuilds every im2col element from (co, kh, kw, ih, iw)
// with integer divisions and a bounds test per element and per tap (its
// B-tile load).  Here each output position P of a tile reads the frame at
// P + shift[tap], so one band [P0, P0 + a_rows) of V, loaded once per
// channel chunk, serves every tap of every phase: the taps become different
// start rows of the same shared-memory matrix.  Padding (the transposed
// padding of the stride-1 case and the phase offsets of the strided case) is
// produced here as zeros.
#pragma once

#include "dgrad_internal.h"
#include "ptx.cuh"

namespace dgrad {
namespace dev {

// Address of V[v][co0] in grad_out, or nullptr where the frame is zero.
__device__ __forceinline__ const float *frame_row_src(const MainParams &p, int v, int co0) {
    if (v >= p.positions) return nullptr;
    const int n = v / p.HvWp;
    const int rem = v - n * p.HvWp;
    const int y = rem / p.Wp;
    const int x = rem - y * p.Wp;
    const int oh = y - p.Ph, ow = x - p.Pw;
    if (static_cast<unsigned>(oh) >= static_cast<unsigned>(p.oH) ||
        static_cast<unsigned>(ow) >= static_cast<unsigned>(p.oW))
        return nullptr;
    const size_t plane = static_cast<size_t>(p.oH) * p.oW;
    return p.go + (static_cast<size_t>(n) * p.Co + co0) * plane + static_cast<size_t>(oh) * p.oW + ow;
}

template <int KC>
__device__ __forceinline__ void load_frame_row(const MainParams &p, const float *src, int co0, float (&v)[KC]) {
    const size_t plane = static_cast<size_t>(p.oH) * p.oW;
    const int valid = src ? min(KC, p.Co - co0) : 0;
#pragma unroll
    for (int k = 0; k < KC; ++k) v[k] = (k < valid) ? __ldg(src + k * plane) : 0.f;
}

// Layout written: As[(g * a_rows + r) * 4 + e] = V[P0 + r][co0 + 4g + e]
// (K-major 16-byte groups; row r of group g is one core-matrix row).
template <int KC>
__device__ __forceinline__ void store_frame_row(const MainParams &p, float *As, int r, float (&v)[KC]) {
    if (p.round_tf32) {
#pragma unroll
        for (int k = 0; k < KC; ++k) v[k] = round_tf32(v[k]);
    }
#pragma unroll
    for (int g = 0; g < KC / 4; ++g)
        *reinterpret_cast<float4 *>(As + (static_cast<size_t>(g) * p.a_rows + r) * 4) =
            make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
}

// Rows are split over `nthreads` threads; consecutive threads take
// consecutive positions, so each global load instruction of a warp reads a
// contiguous run of one grad_out plane and each 16-byte shared store of a
// warp is conflict-free.  Two rows per thread are in flight at once.
template <int KC>
__device__ __forceinline__ void fill_a_stage(float *As, const MainParams &p, int P0, int co0, int tid,
                                             int nthreads) {
    int r = tid;
    for (; r + nthreads < p.a_rows; r += 2 * nthreads) {
        float v0[KC], v1[KC];
        const float *s0 = frame_row_src(p, P0 + r, co0);
        const float *s1 = frame_row_src(p, P0 + r + nthreads, co0);
        load_frame_row<KC>(p, s0, co0, v0);
        load_frame_row<KC>(p, s1, co0, v1);
        store_frame_row<KC>(p, As, r, v0);
        store_frame_row<KC>(p, As, r + nthreads, v1);
    }
    if (r < p.a_rows) {
        float v0[KC];
        load_frame_row<KC>(p, frame_row_src(p, P0 + r, co0), co0, v0);
        store_frame_row<KC>(p, As, r, v0);
    }
}

// Element offset of V[v][channel 0] in grad_out (add co * oH * oW for
// channel co), or -1 where the frame is zero.
__device__ __forceinline__ int frame_row_offset(const MainParams &p, int v) {
    if (v >= p.positions) return -1;
    const int n = v / p.HvWp;
    const int rem = v - n * p.HvWp;
    const int y = rem / p.Wp;
    const int x = rem - y * p.Wp;
    const int oh = y - p.Ph, ow = x - p.Pw;
    if (static_cast<unsigned>(oh) >= static_cast<unsigned>(p.oH) ||
        static_cast<unsigned>(ow) >= static_cast<unsigned>(p.oW))
        return -1;
    return (n * p.Co * p.oH + oh) * p.oW + ow;
}

// Decode a flattened output position into (n, q, u).
__device__ __forceinline__ void decode_position(const MainParams &p, int P, int &n, int &q, int &u) {
    n = P / p.HvWp;
    const int rem = P - n * p.HvWp;
    q = rem / p.Wp;
    u = rem - q * p.Wp;
}

}  // namespace dev
}  // namespace dgrad

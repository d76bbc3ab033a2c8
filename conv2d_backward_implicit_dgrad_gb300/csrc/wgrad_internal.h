// Internal declarations of the weight gradient (wgrad): plan geometry and
// kernel parameter blocks.
//
// GEMM view.  For tap t = (kh, kw) and input channel ci, row r = (t, ci) of
//   D[r][co] = sum over K of X[r][k] * G[co][k]
// is grad_weight[co][ci][kh][kw], with K running over the batch and the
// grad_out positions.  Both operands are K-major, i.e. positions contiguous
// per channel, which is the NCHW layout itself:
//  - G frame (gf): grad_out per (n, co) plane, rows padded to Wf (a multiple
//    of 4) and the plane to Kimg (a multiple of 32): G[co][k] with
//    k = oh*Wf + ow, 0 where ow >= oW or oh >= oH;
//  - input copies (xc): the forward input read at k by tap t is
//    x[n][ci][s*oh - ph + kh][s*ow - pw + kw].  Writing kh - ph = s*dh + rh
//    (0 <= rh < s), that is row oh + dh of the row phase rh, so copy
//    c = (kw, rh) holds xc[c][n][ci][y*Wf + u] = x[n][ci][s*(y - Ty) + rh]
//    [s*u + kw - pw] (0 outside the input and for u >= oW), and tap t reads
//    copy c at k + (dh + Ty)*Wf: a whole number of frame rows, so every
//    tensor copy starts on a 16-byte boundary.
// Split precision (TF32X3): both frames twice, hi = tf32(v) then
// lo = tf32(v - hi) (gf planes [half][n][co], xc planes [half][copy][n][ci]),
// and per chunk three K passes hi*lo, lo*hi, hi*hi.
#pragma once

#include "dgrad_internal.h"
#include "wgrad.h"

namespace dgrad {

constexpr int kWgMaxSegs = 256;     // (tap, ci block) segments of all row tiles
constexpr int kWgMaxRowPhases = 4;  // row phases rh (<= stride)
constexpr int kWgMaxStages = 8;

struct WgradGeometry {
    int N, Ci, H, W, Co, kH, kW, s, ph, pw, oH, oW;
    int Wf, Kimg, Lx, cpi;            // frame row pitch, K per image, input-copy plane, 32-position chunks per image
    int Ty;                           // leading zero rows of the input copies
    int n_rh, rh_list[kWgMaxRowPhases];
    int n_copies;                     // kW * n_rh; copy c = kw * n_rh + (index of rh)
    int taps;
    int tap_copy[kMaxTaps], tap_off[kMaxTaps];
    int seg_rows, cpt, n_segs, spt;   // rows per segment, segments per tap, all segments, segments per row tile
    int n_mt, bn, n_nt, n_ks, cps;    // tiles of rows / columns, K splits, chunks per split
    int total_chunks, n_units, grid, stages, smem_bytes, tmem_cols;
    int split;                        // 1: split precision (hi and lo halves of both frames, three K passes)
    size_t g_elems, x_elems, part_elems;   // frames: both halves when split
};

dgrad_status_t make_wgrad_geometry(int N, int Ci, int H, int W, int Co, int kH, int kW, int stride, int pad_h,
                                   int pad_w, int precision, int sm_count, WgradGeometry *g);

struct WgradPackParams {
    const float *go, *x;
    float *gf, *xc;
    int N, Ci, H, W, Co, oH, oW, s, pw, Wf, Kimg, Lx, Ty, n_rh;
    int rh_list[kWgMaxRowPhases];
    long long g4, x4;   // float4 groups of one half of gf and of xc
    int split;          // 1: write hi = tf32(v) in half 0 and lo = tf32(v - hi) in half 1
};

struct WgradMainParams {
    CUtensorMap x_map;   // xc as {Lx, Ci, N, n_copies}, box {32, seg_rows, 1, 1}, 128-byte swizzle
    CUtensorMap g_map;   // gf as {Kimg, Co, N}, box {32, bn, 1}, 128-byte swizzle
    float *part;         // partial tiles [unit][bn][128], unit = (ks * n_mt + mt) * n_nt + nt
    uint32_t *err;
    int n_mt, n_nt, n_ks, n_units, bn, seg_rows, spt, n_segs, cpi, total_chunks, cps, stages, tmem_cols;
    int split, N, n_copies;   // split precision: lo halves at image N + n (gf) and copy n_copies + c (xc)
    uint32_t idesc;
    long long timeout_ns;
    int4 seg[kWgMaxSegs];   // x: input copy, y: first input channel, z: K offset (elements)
};

struct WgradReduceParams {
    const float *part;
    float *dw;
    int Co, Ci, taps, bn, n_mt, n_nt, n_ks, seg_rows, cpt, spt, n_segs;
    long long total;   // n_mt * n_nt * bn * 128 partial elements per split
};

cudaError_t launch_wgrad_pack(const WgradPackParams &p, cudaStream_t stream);
cudaError_t launch_wgrad_main(const WgradMainParams &p, int grid, int smem_bytes, cudaStream_t stream);
cudaError_t launch_wgrad_reduce(const WgradReduceParams &p, cudaStream_t stream);

}  // namespace dgrad

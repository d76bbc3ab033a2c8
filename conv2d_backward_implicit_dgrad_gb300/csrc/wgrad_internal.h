// Internal declarations of the weight gradient (wgrad): plan geometry and
// kernel parameter blocks.
//
// GEMM view.  For tap t = (kh, kw) and input channel ci, row r = (t, ci) of
//   D[r][co] = sum over K of X[r][k] * G[co][k]
// is grad_weight[co][ci][kh][kw], with K running over the batch and the
// grad_out positions.  Both operands are K-major (positions contiguous per
// channel), held in position frames with f images interleaved along K
// (f = 4; 2 or 1 for batches below 4), image group q = n / f, j = n % f:
//  - G frame (gf): gf[q][co][(oh*Wf + ow)*f + j] = grad_out[n][co][oh][ow],
//    0 where ow >= oW, n >= N or past the last row; a plane holds Kimg
//    (a multiple of 32) positions;
//  - input copies (xc): with kh - ph = s*dh + rh and kw - pw = s*dw + rw
//    (0 <= rh, rw < s), the input read at grad_out position (oh, ow) by tap
//    t is x[n][ci][s*(oh + dh) + rh][s*(ow + dw) + rw].  Copy c = (rh, rw, r)
//    holds xc[c][q][ci][(y*Wf + u)*f + j] = x[n][ci][s*(y - Ty) + rh]
//    [s*(u - Tu + r) + rw] (0 outside the input), and tap t reads the copy
//    with r = (dw + Tu) mod (4/f) at K offset ((dh + Ty)*Wf + dw + Tu - r)*f:
//    a multiple of 4 positions, so every tensor copy starts on a 16-byte
//    boundary.  For f = 4 that is one copy per (rh, rw): the input once.
// Batch-blocked frames (f = 32): the same K index, stored position-major,
// gf[q*Pg + p][co][j] and xc[c][q*Px + p][ci][j] (p = y*Wf + u, Pg = Kimg/32,
// Px = Lx/32), so a tensor copy of one chunk for a channel block is one
// contiguous run, and every tap offset is a whole number of positions.
// Split precision (TF32X3): both frames twice, hi = tf32(v) then
// lo = tf32(v - hi) (gf planes [half][q][co], xc planes [half][copy][q][ci]),
// and per chunk three K passes hi*lo, lo*hi, hi*hi.
#pragma once

#include "dgrad_internal.h"
#include "wgrad.h"

namespace dgrad {

constexpr int kWgMaxSegs = 256;     // (tap, ci block) segments of all row tiles
constexpr int kWgMaxRowPhases = 4;  // largest stride
constexpr int kWgMaxCopies = 32;    // input copies (rh, rw, r)
constexpr int kWgPackTile = 64;     // frame positions per block of the batch-blocked pack
constexpr int kWgPackCh = 4;        // channels per block of the batch-blocked pack
constexpr int kWgMaxGroups = 16;    // run mode: tap groups (kernel row, input copy)
constexpr int kWgMaxTiles = 32;     // run mode: 128-row accumulator tiles (spt adjacent taps each)
constexpr int kWgMaxStages = 8;

struct WgradGeometry {
    int N, Ci, H, W, Co, kH, kW, s, ph, pw, oH, oW;
    int f, lf, m, Q;                  // images interleaved along K (f = 1 << lf), m = max(1, 4 / f), image groups
    int blocked;                      // f = 32, frames [position][channel][32 images]
    int direct;                       // 1x1, stride 1, no padding: no frames, copies from the caller's tensors
    int Wf, Kimg, Lx, cpi;            // frame row pitch, K per image group, input-copy plane, chunks per group
    int Ty, Tu;                       // leading zero rows and columns of the input copies
    int n_copies;
    int copy_rh[kWgMaxCopies], copy_rw[kWgMaxCopies], copy_r[kWgMaxCopies];
    int taps;
    int tap_copy[kMaxTaps], tap_off[kMaxTaps];
    int seg_rows, cpt, n_segs, spt;   // rows per segment, segments per tap, all segments, segments per row tile
    int n_mt, bn, n_nt, n_ks, cps;    // tiles of rows / columns, K splits, chunks per split
    int total_chunks, n_units, grid, stages, smem_bytes, tmem_cols;
    int split;                        // 1: split precision (hi and lo halves of both frames, three K passes)
    // Run mode (batch-blocked frames, TF32): tiles of spt taps at adjacent
    // positions; a tensor copy brings a run of L + spt - 1 positions of one
    // tile, which feeds L chunks (see WgradRunParams).
    int run_mode, n_groups, n_tiles, nksq, run_len, tpu, n_sets, acc_sets, xbox_bytes, bbox_bytes;
    int grp_copy[kWgMaxGroups], grp_base[kWgMaxGroups], grp_nt[kWgMaxGroups], grp_nmt[kWgMaxGroups];
    int grp_tap0[kWgMaxGroups];
    int grp_taps[kMaxTaps];
    int tile_grp[kWgMaxTiles], tile_m0[kWgMaxTiles];
    // Plane mode (see WgradPlaneParams): rows of one kernel column's input
    // channels and of one kernel row's output channels, each a multiple of 8.
    int plane, ci_rows, co_rows;
    size_t g_elems, x_elems, part_elems;   // frames: both halves when split
};

// allow_plane = false plans as if plane mode did not exist (the frame
// modes' tables, for the host-only descriptions).
dgrad_status_t make_wgrad_geometry(int N, int Ci, int H, int W, int Co, int kH, int kW, int stride, int pad_h,
                                   int pad_w, int precision, int sm_count, WgradGeometry *g, bool allow_plane = true);

struct WgradPackParams {
    const float *go, *x;
    float *gf, *xc;
    int N, Ci, H, W, Co, oH, oW, s, Wf, Kimg, Lx, Ty, Tu, Q, lf;
    long long g4, x4;   // float4 groups of one half of gf and of xc
    int split;          // 1: write hi = tf32(v) in half 0 and lo = tf32(v - hi) in half 1
    int4 copy[kWgMaxCopies];   // per input copy: rh, rw, r
    int blocked, Px, Pg;       // batch-blocked frames: positions per image group of xc and of gf
    long long g_tiles, x_tiles;   // blocks of the batch-blocked pack (kWgPackTile positions of kWgPackCh channels)
};

struct WgradMainParams {
    CUtensorMap x_map;   // xc as {Lx, Ci, Q, n_copies}, box {32, seg_rows, 1, 1}, 128-byte swizzle
    CUtensorMap g_map;   // gf as {Kimg, Co, Q}, box {32, bn, 1}, 128-byte swizzle
    float *part;         // partial tiles [unit][bn][128], unit = (ks * n_mt + mt) * n_nt + nt
    uint32_t *err;
    int n_mt, n_nt, n_ks, n_units, bn, seg_rows, spt, n_segs, cpi, total_chunks, cps, stages, tmem_cols;
    int split, Q, n_copies;   // split precision: lo halves at group Q + q (gf) and copy n_copies + c (xc)
    int blocked, Px;          // batch-blocked frames (chunk = one position; Px positions per xc group)
    uint32_t idesc;
    long long timeout_ns;
    int wait_test;   // failure-detection test: the MMA warp first waits on a barrier nothing completes
    int4 seg[kWgMaxSegs];   // x: input copy, y: first input channel, z: K offset (elements)
};

struct WgradReduceParams {
    const float *part;
    float *dw;
    int Co, Ci, taps, bn, n_mt, n_nt, n_ks, seg_rows, cpt, spt, n_segs;
    long long total;   // partial elements per split (segment mode n_mt * n_nt * bn * 128)
    // run mode: partial tile t holds the taps tile[t].y .. of group tile[t].x
    int run_mode, n_tiles;
    int red_warps;   // warps summing the K splits of one group of 128 elements: 1, 2, 4 or 8
    int2 tile[kWgMaxTiles];
    int2 grp[kWgMaxGroups];   // x: first entry in taps, y: taps in the group
    int taps_of[kMaxTaps];
    // plane mode: a split is [row tile][column][rows of the tile] (rows (kw, ci), columns (kh, co))
    int plane, ci_rows, co_rows, kH, kW, a_rows;
};

// Run-mode main kernel.  Chunk = one frame position of 32 images.  Tile t
// (group g, taps m0 .. m0 + spt - 1 of the group, consecutive positions, the
// taps past the group's end padding rows) is, for chunk c, the spt position
// blocks starting at c + base + m0: 128 contiguous rows of a tensor copy
// that holds positions [c, c + L + spt - 1) of the tile (one copy feeds the
// L chunks of a stage).  A unit is (tile set, ci block, co tile, image group,
// K range); its grad_out copy holds the stage's L chunks.
struct WgradRunParams {
    CUtensorMap x_map;   // batch-blocked xc, box {32, seg_rows, L + spt - 1, 1}
    CUtensorMap g_map;   // batch-blocked gf, box {32, bn, L}
    float *part;         // partial tiles [((q * nksq + ks) * cpt + cb) * n_nt + nt][tile][bn][128]
    uint32_t *err;
    int n_units, n_sets, tpu, n_tiles, cpt, n_nt, nksq, cps, Pg, Px, seg_rows, L, bn, stages, acc_sets, tmem_cols;
    int xbox_bytes, bbox_bytes;
    int split, n_copies, Q;   // split precision: lo copies at copy + n_copies and group + Q (stage: hi half, lo half)
    uint32_t idesc;
    long long timeout_ns;
    int wait_test;   // failure-detection test: the MMA warp first waits on a barrier nothing completes
    int2 tile[kWgMaxTiles];   // x: input copy, y: position offset of the tile's first tap (base + m0)
};

// Plane mode (stride 1, oH = H, oW = W, W a multiple of 4, TF32): no
// frames.  K runs over the positions q = ih*W + ow of each image's input
// plane, so that the kernel row kh moves grad_out by whole rows and the
// kernel column kw moves the input by kw - pw columns:
//   A[(kw, ci)][q] = input[n][ci][q + kw - pw]   (0 where the column leaves
//                    the row, and for q >= H*W)
//   B[(kh, co)][q] = grad_out[n][co][q - (kh - ph)*W]   (0 off the plane)
//   grad_weight[co][ci][kh][kw] = sum over n, q of A[(kw, ci)][q] * B[(kh, co)][q].
// Per 32-position chunk: each kernel row of B is one tensor copy of grad_out
// at a shifted position (a multiple of 4 positions, so 16-byte aligned); A's
// unshifted column (kw = pw) is one tensor copy of the input; the other
// columns are gathered by SIMT threads (4-byte asynchronous copies, zero
// fill) into the same 128-byte-swizzled rows.  A's rows (kw, ci) fill n_mt
// tiles of 128, B's rows (kh, co) one MMA N (nb <= 256); every CTA keeps
// all n_mt x nb accumulators in tensor memory over a contiguous range of
// chunks (images in order) and writes one partial split.
struct WgradPlaneParams {
    CUtensorMap x_map;   // input as {H*W, Ci, N}, box {32, ci_rows, 1}, 128-byte swizzle
    CUtensorMap g_map;   // grad_out as {H*W, Co, N}, box {32, co_rows, 1}, 128-byte swizzle
    const float *x;      // the input (the gathered columns read it directly)
    float *part;         // split b: [row tile][nb columns][rows of the tile], rows (kw, ci), columns (kh, co)
    uint32_t *err;
    int N, Ci, HW, W, kH, kW, ph, pw;
    int ci_rows, co_rows, nb, n_mt, cpi, total_chunks, stages, tmem_cols;
    uint32_t a_bytes, stage_bytes;   // A region (n_mt x 16 KB), A + B
    uint32_t idesc;
    long long timeout_ns;
    int wait_test;   // failure-detection test: the MMA warp first waits on a barrier nothing completes
};

cudaError_t launch_wgrad_plane(const WgradPlaneParams &p, int grid, int smem_bytes, cudaStream_t stream);
cudaError_t launch_wgrad_pack(const WgradPackParams &p, cudaStream_t stream);
cudaError_t launch_wgrad_main(const WgradMainParams &p, int grid, int smem_bytes, cudaStream_t stream);
cudaError_t launch_wgrad_run(const WgradRunParams &p, int grid, int smem_bytes, cudaStream_t stream);
cudaError_t launch_wgrad_reduce(const WgradReduceParams &p, cudaStream_t stream);

}  // namespace dgrad

// Internal declarations of libdgrad_gb300: geometry of the phase-split
// implicit GEMM, kernel parameter blocks and launchers.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "dgrad.h"

namespace dgrad {

constexpr int kMaxTaps = 128;
constexpr int kMaxPhases = 16;
constexpr int kMaxStride = 4;
constexpr int kBlockM = 128;          // GEMM rows (output positions) per MMA block
constexpr int kMaxSmem = 232448;      // opt-in dynamic shared memory per CTA on sm_103
constexpr int kSmemPerSm = 233472;    // shared memory of one SM (each resident CTA also reserves 1 KB)
constexpr int kTmemCols = 512;        // tensor-memory columns per SM
constexpr int kMaxSub = 4;            // taps of one kernel row grouped into one MMA (sub-accumulators)

// Instruction descriptor of tcgen05.mma .kind::tf32 (PTX ISA, "instruction
// descriptor" table for .kind::f16 / .kind::tf32): fp32 accumulator, TF32 A
// and B, both K-major, no negation, dense.
constexpr uint32_t tf32_idesc(int M, int N) {
    return (1u << 4)                                  // D format: F32
           | (2u << 7)                                // A format: TF32
           | (2u << 10)                               // B format: TF32
           | (static_cast<uint32_t>(N >> 3) << 17)    // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);   // M / 16
}

// Device error word values (a bit set; the host maps it to dgrad_status_t).
constexpr uint32_t kErrTimeout = 1u;

// One kernel tap that feeds a phase.  In the zero-padded grad_out frame V
// (see Geometry) the tap reads V at (output position + shift).
struct TapDesc {
    int kh, kw;   // position inside the kernel
    int shift;    // dr * Wp + dc, >= 0
    int phase;    // index of the phase the tap feeds
    int dr, dc;   // row and column offset in the frame
};

// One sub-pixel phase (a, b): input rows ih = s*q + a, columns iw = s*u + b.
// Its taps are listed row by row of the kernel (dr descending), row_len taps
// per row with dc descending by one from tap to tap.
struct PhaseDesc {
    int a, b;
    int Hq, Wq;             // output rows/cols of the phase: ceil((H-a)/s), ceil((W-b)/s)
    int tap_begin, tap_count;
    int row_len;            // taps per kernel row of the phase
    int sub;                // main kernel: sub-accumulators (row_len when taps are grouped, else 1)
    int col;                // main kernel: tensor-memory column of the phase's accumulator
};

// Phase split of the strided dgrad plus the flattened, zero-padded grad_out
// frame V that turns every phase into shifted copies of one matrix:
//   V[n][y][x] = grad_out[n][.][y - Ph][x - Pw]  (0 outside), y < Hv, x < Wp,
//   flattened position  P = (n*Hv + y)*Wp + x.
// Output (n, q, u) of any phase sits at P = (n*Hv + q)*Wp + u and its tap t
// reads V at P + shift[t].  Hv and Wp are large enough that every read made
// for a valid output either lands on the intended element or on a zero.
struct Geometry {
    int N, Ci, H, W, Co, kH, kW, s, ph, pw, oH, oW;
    int n_phases;
    PhaseDesc phase[kMaxPhases];
    int n_taps;
    TapDesc tap[kMaxTaps];
    int Ph, Pw, Hv, Wp;
    long long positions;   // N * Hv * Wp
    int max_shift;
};

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime
// (no link-time dependency on the driver library); NULL if unavailable.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// DGRAD_OK for cudaSuccess; otherwise records the error for
// dgrad_cuda_error_string, clears it and returns DGRAD_ERR_CUDA.
dgrad_status_t cuda_status(cudaError_t e);

dgrad_status_t make_geometry(int N, int Ci, int H, int W, int Co, int kH, int kW,
                             int stride, int pad_h, int pad_w, Geometry *g);

// One tcgen05 MMA group: `ntaps` taps issued as one MMA of N = ntaps * bn
// over one A window (start row a_shift), writing accumulator columns from
// col * bn on.  Taps are counted in the packing order of the weights (tap0 is
// a position in that order; the group's taps are consecutive there).  Forms:
//  - one tap per group (col = its phase);
//  - kernel-row groups (`grouped`): the taps of one kernel row of one phase;
//    sub-accumulator j holds the tap with shift a_shift + (ntaps - 1 - j),
//    i.e. the output position that many rows further down, and the epilogue
//    shifts it back;
//  - shared-shift groups (`pgroup`, stride > 1): the taps of different phases
//    with the same frame shift; each phase keeps its own accumulator, the
//    phases sit in tensor memory in an order that makes every group's phases
//    adjacent, and the first group holds a tap of every phase (it starts
//    every accumulator).
// `first`: the group starts its accumulator columns (accumulate = 0 on the
// first K step of the first chunk).
struct MGroup {
    int col, tap0, ntaps, a_shift, first;
};
struct Tiling;
// Groups of a plan, the packing order of the taps (perm[i] = geometry tap at
// packing position i) and each phase's accumulator column in units of bn
// (phase_units).  Returns the group count, or -1 when the plan's grouping
// form cannot be built for this geometry.
int build_mgroups(const Geometry &g, const Tiling &t, MGroup *out, int *perm, int *phase_units);

// Tiling of the main kernel.
struct Tiling {
    int path;          // dgrad_path_t (SIMT or TCGEN05)
    int tm;            // M blocks (kBlockM positions) per work unit
    int bn;            // input channels per slice
    int n_slices;
    int kc;            // output channels per chunk (multiple of 8)
    int n_chunks;
    int n_tiles;
    long long n_work;
    int grid;
    int a_rows;        // rows of one A stage
    int a_stages, b_stages;
    int b_resident;
    int tap_group;     // largest number of taps in one B stage (tcgen05 path)
    int n_tgroups;     // B stages per channel chunk
    int chunk_bytes;   // bytes of one B stage (tap_group taps)
    int grouped;       // 1: taps of a kernel row share one MMA (MGroup)
    int pgroup;        // 1: taps of different phases with the same shift share one MMA (MGroup)
    int tile_step;     // output positions per tile (tm*128, less the rows a grouped MMA cannot finish)
    int want_b_stages; // requested weight pipeline depth (0: automatic)
    int n_mgroups;
    int bg_first[kMaxTaps + 1];   // B stage i holds MMA groups [bg_first[i], bg_first[i+1])
    int xchg_bytes;    // shared memory for the epilogue's cross-warp row exchange
    int xchg_unit;     // 1: one exchange per unit (a single phase: every column published before one barrier)
    int epi_groups;    // epilogue warp groups taking alternate units (2 for grouped tensor-copy launches)
    int a_tma;         // 1: A stages are tensor copies (of the packed frame, or staged); 0: producer warps gather
    int a_staged;      // 1: each A stage is one tensor copy of the caller's NCHW grad_out, transposed in place
                       //    by two transposer warps (no frame, no grad_out pack)
    int stg_box;       // staged: plane elements per copy (box width, a multiple of 4, <= 256)
    int band_rows;     // frame rows an A stage must hold for the MMAs (tm*128 + the largest tap shift)
    int img_tiles;     // tiles per image when tiles never cross an image (staged); 0: tiles run across images
    int a_tmem;        // 1 (1x1, stride 1, no padding): grad_out is copied from NCHW into shared memory and
                       //    written by the epilogue warps into tensor memory, where the MMA reads A; no frame
    int a_tslots;      // a_tmem: tensor-memory A slots (32 columns each)
    int a_tcol;        // a_tmem: first tensor-memory column of the A slots (after the accumulators)
    int img_align_sms; // a_tmem: tiles aligned to images (one copy per chunk, never a second image) when all
                       //    units then fit in this many CTAs (the SM count); 0: never
    int simt_wide;     // FFMA frame pipeline: 8 x 8 register tiles, 128 compute threads, two CTAs per SM
    int a_box_rows;    // rows of one A tensor copy (<= 256)
    int a_nbox;        // tensor copies per A stage
    int co_v;          // channels per packed frame row
    int split;         // 1: TF32X3 (frame rows hold hi and lo halves; three K passes per channel chunk)
    int co_h;          // split: channels of one half of a frame row (a multiple of 32)
    size_t frame_bytes;
    int c2i_R;         // col2im path: input rows per band (a multiple of the stride)
    int c2i_pitch;     // col2im path: floats per band row, max((oW - 1)*s + kW, W + pw)
    int c2i_bands;     // col2im path: N * ceil(H / R)
    int acc_bufs;      // tensor-memory accumulator sets
    int acc_cols;      // columns of one set
    int tmem_cols;
    int smem_bytes;
    size_t packed_bytes;
};

dgrad_status_t choose_tiling(const Geometry &g, int precision, const dgrad_options_t *opts,
                             int sm_count, Tiling *t);

// The tcgen05 producers can copy grad_out in aligned 4-element quads of a
// channel plane when every plane starts 16-byte aligned (oH*oW % 4 == 0) and
// one A band spans only a few images (each image is one contiguous quad
// range of the band).
constexpr int kMaxBandImages = 4;
inline bool use_vec_producer(const Geometry &g, const Tiling &t) {
    const long long img = (long long)g.Hv * g.Wp;
    return t.path == DGRAD_PATH_TCGEN05 && (g.oH * g.oW) % 4 == 0 && (t.a_rows + img - 1) / img + 1 <= kMaxBandImages;
}

// FFMA path with a frame (simt_pipe_kernel): eight compute warps (8 x 4
// register tiles; `wide`: four, 8 x 8 tiles, two CTAs per SM) and one loader
// warp; a barrier block, then a ring of stages, each the band's KC/4 groups of
// a_rows 16-byte rows followed by the phase's weights (at most `taps` taps of
// KC x bn), padded to 128 bytes.
__host__ __device__ constexpr int simt_pipe_threads(bool wide) { return (wide ? 128 : 256) + 32; }
// Output positions per work unit of the FFMA gather kernel: 128, or 1024 for
// 4-channel slices (inputs with at most 4 channels: 256 threads x 4 positions)
__host__ __device__ constexpr int simt_unit_rows(int bn) { return bn == 4 ? 1024 : 128; }
constexpr int kSimtMaxStages = 6;
constexpr int kSimtPipeHeader = 1024;
__host__ __device__ constexpr int simt_stage_bytes(int a_rows, int kc, int bn, int taps) {
    return ((kc / 4) * a_rows * 16 + taps * kc * bn * 4 + 127) / 128 * 128;
}

// ---------------------------------------------------------------- kernels
// Packed weights.  One (slice sl, chunk c) is one contiguous block of
// chunk_bytes holding, for every tap t, input channel j of the slice and
// output channel co = c*kc + k of the chunk, weight[co][sl*bn + j][kh_t][kw_t]
// (0 outside the tensor), in one of two layouts:
//  layout 0 (FFMA kernel), 16-byte groups of 4 output channels:
//    wp[((((sl*n_chunks + c)*n_taps + t)*(kc/4) + k/4)*bn + j)*4 + k%4]
//  layout 1 (tcgen05 kernel, kc = 32), one 128-byte row per input channel,
//  its 16-byte chunks permuted by the 128-byte swizzle of the tensor core's
//  K-major operand layout (chunk k/4 stored at position (k/4) ^ (j % 8)):
//    wp[(((sl*n_chunks + c)*n_taps + t)*bn + j)*32 + (((k/4) ^ (j%8))*4) + k%4]
//  layout 2 (col2im path, kc = 32), one 128-byte row per GEMM column
//    r = (kh*kW + kw)*Ci + ci (rows up to bn, zero past Ci*kH*kW), swizzled
//    like layout 1: wp[(c*bn + r)*32 + (((k/4) ^ (r%8))*4) + k%4]
// Split precision (split_chunks = C > 0, n_chunks = 3C): chunk c holds output
// channels of chunk c mod C, as the TF32 low part of the weight for c < C and
// as the TF32 high part for c >= C (the three K passes hi*lo, lo*hi, hi*hi).
struct PrepackParams {
    const float *w;
    float *wp;
    int Co, Ci, kH, kW;
    int n_taps, bn, n_slices, kc, n_chunks;
    int layout;
    int round_tf32;
    int split_chunks;  // 0, or the channel chunks of one K pass (split precision)
    long long total;   // floats written
    int tap_kh[kMaxTaps];
    int tap_kw[kMaxTaps];
};

// Packed frame: V[P][k] = grad_out[n][k][y - Ph][x - Pw] at flattened
// position P = (n*Hv + y)*Wp + x (0 outside grad_out and for k >= Co),
// TF32-rounded when the plan computes in TF32; co_v channels per row.
// Split precision: row P holds hi = tf32(x) in channels [0, co_h) and
// lo = tf32(x - hi) in [co_h, 2*co_h) (co_v = 2*co_h).
// The frame is zeroed once when the plan is made; a pack writes only the
// rows of grad_out's positions (the zero rows and channels never change).
// Pack blocks: (image n, 32-channel group, segment of seg_len consecutive
// elements of the oH*oW channel plane).
struct FramePackParams {
    const float *go;
    float *v;
    int N, Co, oH, oW, Hv, Wp, Ph, Pw;
    int co_v;
    int round_tf32;
    int split;         // 1: write hi and lo halves
    int co_h;          // split: channels per half (channels >= Co are zero)
    int positions;     // N * Hv * Wp
    int seg_len;       // plane elements per pack block: a multiple of 4, <= kPackSegMax
    int segs;          // ceil(oH*oW / seg_len)
    int c_groups;      // ceil(Co / kPackChannels)
    int vec;           // 1: 16-byte grad_out loads (oH*oW % 4 == 0)
};
constexpr int kPackChannels = 32;   // channels per pack block (one 128-byte frame row segment)
constexpr int kPackSegMax = 256;    // plane elements per pack block at most

// Main-kernel MMA group entry: A window offset (bytes), accumulator column
// (bit 31: first group of its phase), B offset inside the chunk's tap block
// (bytes), instruction descriptor (N = ntaps * bn).
struct MainParams {
    CUtensorMap a_map;   // packed frame [positions][co_v], box 32 x a_box_rows, 128-byte swizzle; staged:
                         // grad_out as [N][Co][oH*oW], box stg_box x 32 x 1, no swizzle (encoded per call)
    const float *go;
    const float *wp;
    float *gi;
    uint32_t *err;
    int N, Ci, Co, H, W, oH, oW, s;
    int Ph, Pw, Hv, Wp, HvWp;
    int positions;
    int tm, bn, n_slices, kc, n_chunks, n_tiles;
    int n_work;
    int a_rows, a_stages, b_stages, b_resident, chunk_bytes;
    int tap_group, n_tgroups;
    int vec_producer;   // 1: 16-byte quad loads + register transpose; 0: 4-byte asynchronous copies
    int a_tma, a_box_rows, a_nbox;
    int a_staged, stg_box, band_rows, img_tiles;   // see Tiling
    int a_tmem, a_tslots, a_tcol;                  // see Tiling
    int prefetch_ahead; // staged: stages whose grad_out boxes are prefetched into L2 ahead of their copy
    int acc_bufs, acc_cols, tmem_cols;
    int round_tf32;
    int split_chunks;   // split precision: channel chunks of one K pass (n_chunks = 3 * split_chunks), else 0
    int co_h;           // split precision: frame channel of the first lo value
    int n_phases, n_taps;
    uint32_t idesc;
    long long timeout_ns;
    int wait_test;      // failure-detection test: the MMA warp first waits on a barrier nothing completes
    int tile_step;      // output positions per tile
    int grouped;
    int max_sub;        // largest sub-accumulator count of a phase
    int vec_w;          // epilogue stores the s column phases of a row phase together (s = 2 or 4)
    int n_mgroups;
    int xchg_bytes;
    int xchg_unit;      // the epilogue publishes a unit's boundary rows once, for all columns
    int epi_groups;     // 2: a second group of four epilogue warps takes every other unit
    PhaseDesc phase[kMaxPhases];
    TapDesc tap[kMaxTaps];
    // Fused epilogue: grad_input = (accumulate ? grad_input : 0) + m * dgrad,
    // m = (relu_in > 0) when relu_in is given (same shape as grad_input), else 1.
    const float *relu_in;
    int accumulate;
    uint4 mgroup[kMaxTaps];
    int bg_first[kMaxTaps + 1];
    int bg_tap0[kMaxTaps + 1];   // first tap of each B stage (and n_taps at the end)
};

// Kernel parameter blocks from a plan (host).  Pointers are left null.
void fill_main_params(const Geometry &g, const Tiling &t, int round_tf32, MainParams *m);
void fill_prepack_params(const Geometry &g, const Tiling &t, int round_tf32, PrepackParams *q);

// Weight pre-pack and (optional, fp may be null) frame pack in one launch;
// either part may be skipped (pp may be null).
cudaError_t launch_pack(const PrepackParams *pp, const FramePackParams *fp, cudaStream_t stream);
inline cudaError_t launch_prepack(const PrepackParams &p, cudaStream_t stream) { return launch_pack(&p, nullptr, stream); }
cudaError_t launch_simt(const MainParams &p, const Tiling &t, cudaStream_t stream);

// col2im path: P[position][(ci,kh,kw)] = sum over co of V[position][co] *
// weight[co][ci][kh][kw] on tcgen05 (V the packed frame), scattered into a
// shared-memory band of grad_input rows [r0, r0 + R) and written out.
constexpr int kC2iMaxCols = 256;
struct C2iParams {
    CUtensorMap a_map;   // the packed frame, box 32 channels x 128 positions, 128-byte swizzle
    const float *wp;     // packed weights, layout 2
    float *gi;
    uint32_t *err;
    const float *relu_in;   // fused epilogue, as MainParams
    int accumulate;
    int N, Ci, H, W, Co, kH, kW, s, ph, pw, oH, oW, Ph, Pw, Hv, Wp;
    int n_chunks, bn, ncols, R, pitch, bands_per_img, n_bands, a_stages, tmem_cols, chunk_bytes;
    uint32_t idesc;
    long long timeout_ns;
    int col_kh[kC2iMaxCols];    // kernel row of GEMM column c
    int col_off[kC2iMaxCols];   // (ci*R + kh)*pitch + kw: offset of column c in a band copy from its position's base
};
void fill_c2i_params(const Geometry &g, const Tiling &t, C2iParams *c);
cudaError_t launch_c2i(const C2iParams &p, const Tiling &t, cudaStream_t stream, bool pdl);
cudaError_t launch_tc(const MainParams &p, const Tiling &t, cudaStream_t stream, bool pdl);
// Tensor-copy mode with the fused epilogue, and the staged mode (plain and
// fused stores); called by launch_tc.
cudaError_t launch_tc_fused(const MainParams &p, const Tiling &t, cudaStream_t stream, bool pdl);
cudaError_t launch_tc_staged(const MainParams &p, const Tiling &t, cudaStream_t stream, bool pdl);
cudaError_t launch_tc_staged_fused(const MainParams &p, const Tiling &t, cudaStream_t stream, bool pdl);
cudaError_t launch_tc_tmem(const MainParams &p, const Tiling &t, cudaStream_t stream, bool pdl);

}  // namespace dgrad

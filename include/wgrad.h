/*
 * wgrad.h -- C ABI of the convolution weight gradient (wgrad) in
 * libdgrad_gb300.so, on one NVIDIA GB300 (sm_103a).
 *
 * Operation: the weight half of @simulatte/doppler 0.1.0's runConv2DBackward
 * (conv2d_backward.js: with computeGradWeight it produces gradWeight of shape
 * [outChannels, inChannels, kernelH, kernelW] from gradOutput and the forward
 * input; the shader it dispatches is not on the page).  Written from the
 * forward mapping of the same page's conv2d_backward_input.wgsl (main(),
 * "forward mapping" comment: the forward pass read input row
 * ih = oh*stride - pad + kh):
 *
 *   grad_weight[co,ci,kh,kw] = sum over n, oh, ow of
 *                              grad_out[n,co,oh,ow] * input[n,ci,ih,iw]
 *   where ih = oh*stride - pad_h + kh, iw = ow*stride - pad_w + kw, and terms
 *   whose (ih, iw) falls outside the input are absent.
 *
 * The batch is summed (a batched forward pass shares one weight tensor).
 *
 * Tensors (fp32, contiguous, row-major):
 *   grad_out    [N, Co, oH, oW]   NCHW
 *   input       [N, Ci, H, W]     NCHW, the forward pass's input
 *   grad_weight [Co, Ci, kH, kW]  OIHW, fully OVERWRITTEN
 * with oH = floor((H + 2*pad_h - kH)/stride) + 1 and likewise oW.
 *
 * Arithmetic: DGRAD_PREC_TF32 (both operands rounded to TF32, round to
 * nearest with ties away from zero; products accumulated in fp32 on the
 * tcgen05 tensor cores, the batch-and-position sum split over CTAs and
 * finished by a second, deterministic pass) or DGRAD_PREC_TF32X3 (each
 * operand v split into hi = tf32(v) and lo = tf32(v - hi), three tensor-core
 * products hi*lo + lo*hi + hi*hi per term: fp32-level accuracy, about three
 * times the tensor work and twice the frame bytes).  DGRAD_PREC_FP32 returns
 * DGRAD_ERR_UNSUPPORTED.
 *
 * Ownership, errors and streams follow dgrad.h: the caller owns the three
 * tensors; a plan owns its device workspace and is bound to the device that
 * was current when it was made; errors are returned as dgrad_status_t and
 * kernel waits are bounded (wgrad_plan_check reports a wait that ran out);
 * grad_weight overlapping an input returns DGRAD_ERR_ALIAS, a NULL or
 * non-16-byte-aligned pointer DGRAD_ERR_MISALIGNED.  Same unsupported
 * features as dgrad (dilation, groups, per-axis strides, asymmetric padding).
 */
#ifndef WGRAD_GB300_H
#define WGRAD_GB300_H

#include <stddef.h>

#include "dgrad.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct wgrad_plan_s *wgrad_plan_t;

/* Everything a wgrad plan decided. */
typedef struct {
    int N, Ci, H, W, Co, kH, kW, stride, pad_h, pad_w;
    int oH, oW;
    int precision;          /* dgrad_precision_t */
    int interleave;         /* f: images interleaved along K (32: batch-blocked frames; else 4, or 2, 1 for batches below 4) */
    int mode;               /* main kernel: 0 segment (a tensor copy per tap segment and chunk), 1 run (a tensor copy
                               per tile of adjacent taps holds a run of positions for several chunks; batch-blocked
                               frames, TF32 and split precision), 2 direct (1x1, stride 1, no padding, H*W a
                               multiple of 4, TF32: the segment kernel's tensor copies read the caller's NCHW
                               tensors, no frames; the MMA takes the TF32 part of each fp32 value instead of
                               rounding it), 3 plane (stride 1, oH = H, oW = W, W a multiple of 4, 1 < kH*kW,
                               kW <= 7, TF32, and tiles that fit: kH*round8(Co) <= 256, the kW*round8(Ci) rows in
                               tiles of 128 with all accumulators in 512 tensor-memory columns,
                               (kW-1)*round8(Ci) <= 512; no frames and no pack: K runs over the input plane's
                               positions, each kernel row of grad_out is a tensor copy shifted by whole rows, each
                               kernel column of the input a copy shifted in shared memory; the MMA takes the TF32
                               part of each value) */
    int Wf;                 /* row pitch of the position frames (grad_out columns plus the taps' column reach) */
    int Kimg;               /* GEMM K per group of f images: oH*Wf*f rounded up to a multiple of 32 */
    int Lx;                 /* length of one input-copy plane (Kimg plus the largest tap offset) */
    int n_copies;           /* phase-split, shifted copies of the input (one per row and column phase when f = 4) */
    int seg_rows;           /* GEMM rows per (tap, input-channel block) segment */
    int n_mt, n_nt, n_ks;   /* row tiles of (tap, ci), column tiles of co, splits of K */
    int slice_n;            /* output channels per column tile (MMA N) */
    int n_units, grid, stages, smem_bytes, tmem_cols;
    size_t workspace_bytes;
    double useful_flops;      /* 2*N*Co*oH*oW*Ci*kH*kW */
    double algorithmic_bytes; /* 4*(|grad_out| + |input| + |grad_weight|) */
} wgrad_plan_info_t;

/* Host-only planning (no device, no allocation): what wgrad_plan would
 * decide for this shape on `sm_count` SMs (0: 152). */
dgrad_status_t wgrad_describe(int N, int Ci, int H, int W, int Co, int kH, int kW, int stride, int pad_h,
                              int pad_w, dgrad_precision_t precision, int sm_count, wgrad_plan_info_t *info);

/* Host-only tap table of the frame modes (for tests; planned as if plane
 * mode did not exist).  Frames interleave f = *interleave
 * images along K: position (row y, column u) of image n = f*q + j sits at K
 * index (y*Wf + u)*f + j of image group q.  For tap t = kh*kW + kw: the input
 * copy it reads (copy[t]) and its K offset (offset[t], a multiple of 4).
 * Input copy c holds input row s*(y - *ty) + copy_rh[c] and column
 * s*(u - *tu + copy_shift[c]) + copy_rw[c] at frame position (y, u) (0
 * outside the input).  Arrays hold at least `cap` entries;
 * DGRAD_ERR_INVALID_ARG if kH*kW or the copy count exceeds cap. */
dgrad_status_t wgrad_describe_taps(int N, int Ci, int H, int W, int Co, int kH, int kW, int stride, int pad_h,
                                   int pad_w, int cap, int *copy, int *offset, int *copy_rh, int *copy_rw,
                                   int *copy_shift, int *n_copies, int *ty, int *tu, int *interleave);

/* Host-only run-mode table (for tests); DGRAD_ERR_UNSUPPORTED when the shape
 * runs the segment mode.  Planned as if plane mode did not exist (the table a
 * TF32 shape that runs plane mode would have in the frame modes).  hdr[15] = {groups, tiles, taps per tile (spt),
 * rows per position block, stages, positions per image group of grad_out
 * (Pg) and of the input copies (Px), chunks per unit, K splits per image
 * group, ci blocks, co tiles, image groups, chunks per stage (L), tiles per
 * unit, tile sets}; per group 6 ints {input copy, base position, taps,
 * tiles, 0, first entry in taps[]}; taps[] lists the taps group by group in
 * position order; per tile 2 ints {group, first tap in the group}.  Each
 * array holds at least `cap` entries of its kind. */
dgrad_status_t wgrad_describe_run(int N, int Ci, int H, int W, int Co, int kH, int kW, int stride, int pad_h,
                                     int pad_w, int sm_count, int cap, int *hdr, int *groups, int *taps, int *tiles);

/* Optional settings for wgrad_plan_ex; 0 = default. */
typedef struct {
    int timeout_us;   /* limit of every bounded in-kernel wait, in microseconds (0: one second) */
    int wait_test;    /* failure-detection test only: 1 makes the main kernel's MMA warp first wait on a
                         barrier that nothing ever completes, so that this bounded wait runs out after
                         timeout_us; the kernel then records DGRAD_ERR_DEVICE_TIMEOUT (read by
                         wgrad_plan_check), lets its copies land, frees its tensor memory and exits with
                         grad_weight incomplete.  Nothing faults or traps.  0 for every real use. */
} wgrad_options_t;

/* Create a plan on the current device: validate, plan the tiles and allocate
 * the workspace (position frames of grad_out and input, the partial-sum
 * tiles, an error word).  *plan_out owns that memory until
 * wgrad_plan_destroy; it is NULL on failure. */
dgrad_status_t wgrad_plan(int N, int Ci, int H, int W, int Co, int kH, int kW, int stride, int pad_h, int pad_w,
                          dgrad_precision_t precision, wgrad_plan_t *plan_out);

/* Same as wgrad_plan with options (opts may be NULL: the defaults). */
dgrad_status_t wgrad_plan_ex(int N, int Ci, int H, int W, int Co, int kH, int kW, int stride, int pad_h,
                             int pad_w, dgrad_precision_t precision, const wgrad_options_t *opts,
                             wgrad_plan_t *plan_out);

dgrad_status_t wgrad_plan_info(wgrad_plan_t plan, wgrad_plan_info_t *info);

/* grad_weight = wgrad(grad_out, input), asynchronously on `stream` (three
 * kernels: frame pack, tcgen05 main kernel, reduction; two in the direct and
 * plane modes, which read the caller's tensors and have no pack).  One plan
 * must not run on two streams at once (its workspace is shared). */
dgrad_status_t wgrad_run(wgrad_plan_t plan, const float *grad_out, const float *input, float *grad_weight,
                         void *stream);

/* After the stream has been synchronised: DGRAD_ERR_DEVICE_TIMEOUT if a
 * bounded in-kernel wait ran out since the last check (then clears it). */
dgrad_status_t wgrad_plan_check(wgrad_plan_t plan);

void wgrad_plan_destroy(wgrad_plan_t plan);

#ifdef __cplusplus
}
#endif

#endif /* WGRAD_GB300_H */

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
    int Wf;                 /* row pitch of the position frames: oW rounded up to a multiple of 4 */
    int Kimg;               /* GEMM K per image: oH*Wf rounded up to a multiple of 32 */
    int Lx;                 /* length of one input-copy plane (Kimg plus the largest tap offset) */
    int n_copies;           /* shifted, phase-split copies of the input (one per kw and row phase) */
    int seg_rows;           /* GEMM rows per (tap, input-channel block) segment */
    int n_mt, n_nt, n_ks;   /* row tiles of (tap, ci), column tiles of co, splits of K */
    int slice_n;            /* output channels per column tile (MMA N) */
    int n_units, grid, stages, smem_bytes, tmem_cols;
    size_t workspace_bytes;
    double useful_flops;      /* 2*N*Co*oH*oW*Ci*kH*kW */
    double algorithmic_bytes; /* 4*(|grad_out| + |input| + |grad_weight|) */
} wgrad_plan_info_t;

/* Host-only planning (no device, no allocation): what wgrad_plan would
 * decide for this shape on `sm_count` SMs (0: 148). */
dgrad_status_t wgrad_describe(int N, int Ci, int H, int W, int Co, int kH, int kW, int stride, int pad_h,
                              int pad_w, dgrad_precision_t precision, int sm_count, wgrad_plan_info_t *info);

/* Host-only tap table (for tests): for tap t = kh*kW + kw, the input copy it
 * reads (copy[t]) and its K offset in positions (offset[t]); for input copy
 * c, its kernel column (copy_kw[c]) and row phase (copy_rh[c]); and the
 * copies' leading zero rows (*ty).  Arrays hold at least `cap` entries;
 * DGRAD_ERR_INVALID_ARG if kH*kW or the copy count exceeds cap. */
dgrad_status_t wgrad_describe_taps(int N, int Ci, int H, int W, int Co, int kH, int kW, int stride, int pad_h,
                                   int pad_w, int cap, int *copy, int *offset, int *copy_kw, int *copy_rh,
                                   int *n_copies, int *ty);

/* Create a plan on the current device: validate, plan the tiles and allocate
 * the workspace (position frames of grad_out and input, the partial-sum
 * tiles, an error word).  *plan_out owns that memory until
 * wgrad_plan_destroy; it is NULL on failure. */
dgrad_status_t wgrad_plan(int N, int Ci, int H, int W, int Co, int kH, int kW, int stride, int pad_h, int pad_w,
                          dgrad_precision_t precision, wgrad_plan_t *plan_out);

dgrad_status_t wgrad_plan_info(wgrad_plan_t plan, wgrad_plan_info_t *info);

/* grad_weight = wgrad(grad_out, input), asynchronously on `stream` (three
 * kernels: frame pack, tcgen05 main kernel, reduction).  One plan must not
 * run on two streams at once (its workspace is shared). */
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

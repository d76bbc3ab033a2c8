/*
 * dgrad.h -- C ABI of libdgrad_gb300.so: convolution backward-data (dgrad) on
 * one NVIDIA GB300 (sm_103a).
 *
 * Operation (meganeura, src/shaders/conv2d_grad_input_gemm.wgsl, header
 * comment and Params struct; @simulatte/doppler 0.1.0,
 * conv2d_backward_input.wgsl, header comment and "forward mapping" comment):
 *
 *   grad_input[n,ci,ih,iw] = sum over (co,kh,kw) of
 *                            grad_out[n,co,oh,ow] * weight[co,ci,kh,kw]
 *   where ih = oh*stride - pad_h + kh and iw = ow*stride - pad_w + kw,
 *
 * i.e. the input-adjoint of a 2-D convolution with one stride, symmetric
 * padding pad_h (rows) and pad_w (columns), dilation 1 and one group.  Per
 * batch item it is the implicit GEMM C[Ci, H*W] = W^T[Ci, Co*kH*kW] x
 * im2col(grad_out)[Co*kH*kW, H*W] (meganeura's header comment).
 *
 * Tensors (all fp32, contiguous, row-major; layouts from meganeura's storage
 * declarations):
 *   grad_out   [N, Co, oH, oW]   NCHW
 *   weight     [Co, Ci, kH, kW]  OIHW
 *   grad_input [N, Ci, H, W]     NCHW
 * with oH = floor((H + 2*pad_h - kH)/stride) + 1 and likewise oW.  H and W are
 * the authoritative input size; input rows or columns that no term reaches are
 * written as 0.
 *
 * Semantics shared by every entry point:
 *  - grad_input is fully OVERWRITTEN (both pages store the sum, never add to
 *    the destination).  grad_out and weight are never written.
 *  - Ownership: the caller owns the three tensors.  A plan owns its device
 *    workspace (the packed weights, a device error word) and is bound to the
 *    CUDA device that was current when it was created.
 *  - Errors are returned as dgrad_status_t; nothing aborts the process and no
 *    kernel traps.  Kernel waits are bounded: a wait that runs out records
 *    DGRAD_ERR_DEVICE_TIMEOUT in the plan's device error word, which
 *    dgrad_plan_check() reports once the stream has been synchronised.
 *  - Not supported (neither page has them): dilation, groups, different row
 *    and column strides, asymmetric per-side padding, output padding.
 *  - Limits: kH*kW <= 128 kernel taps, stride <= 4, all extents and element
 *    counts below 2^31.  Larger shapes return DGRAD_ERR_UNSUPPORTED.
 *  - Streams are passed as `void *` holding a cudaStream_t (NULL = the legacy
 *    default stream) so this header needs no CUDA include.
 */
#ifndef DGRAD_GB300_H
#define DGRAD_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct dgrad_plan_s *dgrad_plan_t;

typedef enum {
    DGRAD_OK = 0,
    DGRAD_ERR_INVALID_ARG = 1,    /* a dimension <= 0, stride < 1, pad < 0, oH or oW < 1, NULL plan */
    DGRAD_ERR_UNSUPPORTED = 2,    /* outside the limits above */
    DGRAD_ERR_MISALIGNED = 3,     /* a tensor pointer is NULL or not 16-byte aligned */
    DGRAD_ERR_ALIAS = 4,          /* grad_input overlaps grad_out or weight */
    DGRAD_ERR_OOM = 5,            /* workspace allocation failed */
    DGRAD_ERR_CUDA = 6,           /* a CUDA runtime call or kernel launch failed */
    DGRAD_ERR_DEVICE_TIMEOUT = 7, /* a bounded in-kernel wait ran out (reported by dgrad_plan_check) */
    DGRAD_ERR_NO_DEVICE = 8,      /* no CUDA device, or the device is not sm_103 */
    DGRAD_ERR_WRONG_DEVICE = 9    /* the current device is not the plan's device */
} dgrad_status_t;

/* Arithmetic of the contraction.
 *  FP32:   exact fp32 products, fp32 accumulation (FFMA on the CUDA cores).
 *  TF32:   both operands rounded to TF32 (round to nearest, ties away from zero),
 *          products accumulated in fp32 on the tcgen05 tensor cores.
 *  TF32X3: split precision on the tensor cores.  Each operand x is split into
 *          hi = tf32(x) and lo = tf32(x - hi) (same rounding), so that
 *          |x - hi - lo| <= 2^-22 |x|; every product is formed as
 *          hi*lo + lo*hi + hi*hi (three TF32 MMAs, the lo*lo term dropped) and
 *          accumulated in fp32.  Each product is then off by at most about
 *          3 * 2^-22 of its size, which with fp32 accumulation gives
 *          fp32-level accuracy at three times the TF32 MMA work.  tcgen05 path
 *          only, with the packed grad_out frame (the plan's workspace holds hi
 *          and lo halves) or a source that forms hi and lo on chip (a_source
 *          3 and 4); DGRAD_PATH_SIMT, a_source = 2 and dgrad_run_noalloc
 *          return DGRAD_ERR_UNSUPPORTED for it.  Not in the pages: an
 *          accuracy variant of their contraction. */
typedef enum { DGRAD_PREC_FP32 = 0, DGRAD_PREC_TF32 = 1, DGRAD_PREC_TF32X3 = 2 } dgrad_precision_t;

/* Kernel family.  AUTO picks TCGEN05 for TF32 and TF32X3, SIMT for FP32. */
typedef enum {
    DGRAD_PATH_AUTO = 0,
    DGRAD_PATH_SIMT = 1,     /* FFMA implicit GEMM (exact fp32; also accepts TF32-rounded operands) */
    DGRAD_PATH_TCGEN05 = 2,  /* warp-specialised tcgen05/TMEM implicit GEMM (TF32 and TF32X3) */
    DGRAD_PATH_COL2IM = 3    /* for few input channels (stems, Ci <= 4): the GEMM
                                P[position][(ci,kh,kw)] = sum over co of grad_out x weight on tcgen05
                                (N = Ci*kH*kW <= 256, no per-tap slices), then col2im: every
                                P element added into a shared-memory band of grad_input (one copy
                                per epilogue warp, summed in a fixed order), bands written out
                                whole.  TF32 only; opt-in (never chosen by AUTO). */
} dgrad_path_t;

/* Optional tuning overrides for dgrad_plan_ex / dgrad_describe; 0 = automatic. */
typedef struct {
    int path;          /* dgrad_path_t */
    int tile_blocks;   /* 128-position M blocks per work unit (tcgen05 path) */
    int slice_n;       /* input channels per work unit (GEMM N), multiple of 16 */
    int chunk_k;       /* output channels per pipeline stage, multiple of 8 */
    int grid;          /* CTAs launched (persistent kernels) */
    int sm_count;      /* dgrad_describe only: SM count to plan for */
    int a_source;      /* tcgen05 path, how grad_out reaches the MMA: 0 automatic (4 where it applies,
                          else 1 when the frame fits in 2 GiB, else 2), 1 packed frame + tensor copies
                          (workspace holds a channels-last copy of grad_out, written by the pack kernel),
                          2 producer warps, 4 tensor memory (1x1 kernels, stride 1, no padding,
                          oH*oW % 4 == 0 and oH*oW >= 128; else DGRAD_ERR_UNSUPPORTED): per 32-channel
                          chunk the main kernel copies the tile's NCHW grad_out elements into shared
                          memory and its epilogue warps write them into tensor memory, where the MMA
                          reads A -- no frame and no grad_out pass, results bit for bit those of the
                          frame; 3 staged
                          (opt-in): each A stage is one tensor copy of the caller's NCHW grad_out (the
                          band's plane elements x 32 channels), transposed in shared memory by two warps
                          of the main kernel -- no frame and no grad_out pass, results bit for bit those
                          of the frame; needs oH*oW % 4 == 0 and one 128-row block whose band plus
                          alignment fits one copy (128 + largest tap shift + 3 <= 256 rows), else
                          DGRAD_ERR_UNSUPPORTED.
                          FFMA path (DGRAD_PATH_SIMT): 0 automatic (1 where the frame fits in 2 GiB and
                          every phase has at most 4 taps or the slice is 64 channels wide, else 2), 1
                          packed frame + a loader warp's
                          tensor copies into a ring of stages under mbarriers, persistent CTAs (the
                          pack kernel writes the frame, fp32), 2 every thread of the CTA gathers the
                          band from NCHW grad_out (no frame); 3 and 4 DGRAD_ERR_UNSUPPORTED */
    int group_taps;    /* tcgen05 path, taps issued as one MMA: 0 automatic (3 where it applies; for
                          one phase (stride 1) in TF32 with slice_n < 128 and kW >= 2, 1 where it fits;
                          else none), 1 the taps of one kernel row (N = taps x slice_n, sub-accumulators
                          summed with row shifts by the epilogue; DGRAD_ERR_UNSUPPORTED when that
                          cannot fit), 2 none, 3 the taps of different sub-pixel phases that read the
                          same frame shift (stride > 1; DGRAD_ERR_UNSUPPORTED when not possible) */
    int b_stages;      /* tcgen05 path, packed-weight pipeline: 0 automatic, 2..8 stream the weights
                          through that many shared-memory stages (never resident) */
    int timeout_us;    /* limit of every bounded in-kernel wait, in microseconds (0: one second) */
    int wait_test;     /* failure-detection test only, tcgen05 path: 1 makes the main
                          kernel's MMA warp first wait on a barrier that nothing ever completes, so
                          that this bounded wait runs out after timeout_us; the kernel then records
                          DGRAD_ERR_DEVICE_TIMEOUT (read by dgrad_plan_check), lets its copies land,
                          frees its tensor memory and exits with grad_input incomplete.  Nothing
                          faults or traps.  0 for every real use. */
} dgrad_options_t;

/* Everything a plan decided, for tests, benchmarks and logs. */
typedef struct {
    int N, Ci, H, W, Co, kH, kW, stride, pad_h, pad_w;
    int oH, oW;
    int precision;         /* dgrad_precision_t */
    int path;              /* dgrad_path_t actually used */
    int n_phases;          /* sub-pixel phases with at least one output (<= stride^2) */
    int n_taps;            /* kernel taps kept over all phases (taps that only ever meet padding are dropped) */
    int Ph, Pw, Hv, Wp;    /* zero-padded grad_out frame: Ph/Pw leading zero rows/cols, Hv x Wp per image */
    long long positions;   /* N*Hv*Wp flattened output positions (GEMM M before tiling) */
    int max_shift;         /* largest tap offset in flattened positions */
    int tile_blocks, slice_n, n_slices, chunk_k, n_chunks;
    long long n_work;      /* work units of the main kernel */
    int grid;              /* CTAs of the main kernel */
    int b_resident;        /* 1: packed weights stay in shared memory for the whole launch */
    int a_source;          /* 1 packed frame + tensor copies, 2 producer warps (FFMA path: the CTA's
                              own gather), 3 staged, 4 tensor memory; col2im path: 1 */
    int smem_bytes;        /* dynamic shared memory of the main kernel */
    int tmem_cols;         /* tensor-memory columns allocated per CTA (tcgen05 path) */
    int group_taps;        /* tcgen05 path: 0 one MMA per tap, 1 per kernel row of taps, 2 per shared shift */
    int tile_step;         /* output positions per work-unit tile */
    int a_stages, b_stages;/* tcgen05 path: operand pipeline stages (b_stages = channel chunks when resident) */
    size_t workspace_bytes;/* device workspace owned by the plan */
    size_t packed_weight_bytes;
    double useful_flops;   /* 2*N*Co*oH*oW*Ci*kH*kW */
    double algorithmic_bytes; /* 4*(|grad_out| + |weight| + |grad_input|) */
    int band_rows;         /* tcgen05 path: frame rows the MMAs of one A stage read (tile rows + largest shift) */
    int stg_box;           /* staged (a_source 3): plane elements per tensor copy of grad_out */
    int img_tiles;         /* staged: tiles per image (tiles never cross an image); 0 otherwise */
    int a_rows;            /* tcgen05 path: rows of one A stage in shared memory */
} dgrad_plan_info_t;

/* Create a plan on the current CUDA device: validates the shape, derives the
 * sub-pixel phase and tap tables, picks tiles and allocates the device
 * workspace (cudaMalloc).  On success *plan_out owns that memory until
 * dgrad_plan_destroy.  On failure *plan_out is set to NULL. */
dgrad_status_t dgrad_plan(int N, int Ci, int H, int W, int Co, int kH, int kW,
                          int stride, int pad_h, int pad_w,
                          dgrad_precision_t precision, dgrad_plan_t *plan_out);

/* Same as dgrad_plan with tuning overrides (opts may be NULL). */
dgrad_status_t dgrad_plan_ex(int N, int Ci, int H, int W, int Co, int kH, int kW,
                             int stride, int pad_h, int pad_w,
                             dgrad_precision_t precision, const dgrad_options_t *opts,
                             dgrad_plan_t *plan_out);

/* Host-only: the decisions dgrad_plan_ex would take for opts->sm_count SMs
 * (152, the GB300's SM count, if 0), without touching any device.  Fills *info. */
dgrad_status_t dgrad_describe(int N, int Ci, int H, int W, int Co, int kH, int kW,
                              int stride, int pad_h, int pad_w,
                              dgrad_precision_t precision, const dgrad_options_t *opts,
                              dgrad_plan_info_t *info);

/* Host-only: the sub-pixel phase and tap tables behind dgrad_describe, for
 * checking the decomposition without a device.  Writes up to `cap` phases
 * (a, b, Hq, Wq, tap_begin, tap_count, row_len: 7 ints each, into `phases`)
 * and up to `cap` taps (kh, kw, shift: 3 ints each, into `taps`); *n_phases
 * and *n_taps receive the full counts.  A phase lists its taps kernel row by
 * kernel row, row_len taps per row, the shift falling by one from each tap
 * to the next inside a row.  Phase (a, b) holds input rows ih = stride*q + a
 * and columns iw = stride*u + b, q < Hq, u < Wq; its output (n, q, u) is the
 * flattened frame position (n*Hv + q)*Wp + u, and tap t of the phase reads
 * the zero-padded grad_out frame at that position plus shift (see
 * dgrad_plan_info_t for Ph, Pw, Hv, Wp). */
dgrad_status_t dgrad_describe_taps(int N, int Ci, int H, int W, int Co, int kH, int kW,
                                   int stride, int pad_h, int pad_w, int cap,
                                   int *phases, int *n_phases, int *taps, int *n_taps);

/* Copy the plan's decisions into *info. */
dgrad_status_t dgrad_plan_info(dgrad_plan_t plan, dgrad_plan_info_t *info);

/* Compute grad_input from grad_out and weight, asynchronously on `stream`.
 * All three are DEVICE pointers on the plan's device, 16-byte aligned, shaped
 * as above.  Launches two kernels on `stream`: the pack kernel (weights, and
 * on the frame path grad_out into the plan's channels-last frame) and then
 * the main kernel.  One plan must not run on two streams at once (they would
 * share the workspace).  Returns after the launches; errors detected inside
 * the kernels surface through dgrad_plan_check. */
dgrad_status_t dgrad_run(dgrad_plan_t plan, const float *grad_out, const float *weight,
                         float *grad_input, void *stream);

/* dgrad_run with a fused epilogue, for autograd chains:
 *   grad_input = (accumulate ? grad_input : 0) + m * dgrad(grad_out, weight),
 *   m = (relu_in > 0) elementwise when relu_in is not NULL, else 1.
 * relu_in is the input of a ReLU whose output was this convolution's input
 * (same shape and layout as grad_input): the product is that ReLU's backward
 * pass (ferrotensor kernels.wgsl, section 12 "Relu", relu_backward: the
 * gradient passes where the ReLU input is > 0 and is 0 elsewhere, NaN
 * included); accumulate = 1 adds the result to what grad_input holds
 * (section 20 "Gradient Accumulation", grad += new_grad) instead of
 * overwriting it.  relu_in, when given, is a 16-byte aligned DEVICE pointer
 * that must not overlap grad_input (DGRAD_ERR_ALIAS); accumulate must be 0 or
 * 1 (else DGRAD_ERR_INVALID_ARG).  Everything else as dgrad_run, which is
 * dgrad_run_fused(plan, grad_out, weight, grad_input, NULL, 0, stream). */
dgrad_status_t dgrad_run_fused(dgrad_plan_t plan, const float *grad_out, const float *weight,
                               float *grad_input, const float *relu_in, int accumulate,
                               void *stream);

/* The stages of dgrad_run, for callers whose weights stay fixed over
 * several calls, or who time the stages apart:
 *   dgrad_prepack        packs `weight` into the plan's workspace;
 *   dgrad_run_packed     packs grad_out (frame path only) and runs the main
 *                        kernel on the weights packed last;
 *   dgrad_pack_grad_out  packs grad_out into the plan's frame (frame path;
 *                        returns DGRAD_OK and launches nothing otherwise);
 *   dgrad_run_main       the main kernel alone, on the weights packed last
 *                        and, on the frame path, the frame packed last.
 *                        grad_out must be the tensor whose frame was packed
 *                        last (the other paths read it directly).
 * dgrad_run_packed = dgrad_pack_grad_out + dgrad_run_main.  Same pointer
 * rules, stream order and errors as dgrad_run.  dgrad_run_packed or
 * dgrad_run_main before any dgrad_prepack/dgrad_run, or dgrad_run_main on
 * the frame path before any grad_out was packed, returns
 * DGRAD_ERR_INVALID_ARG.  dgrad_plan_info's a_source tells whether the plan
 * uses a frame (1) or not (2, 3, 4). */
dgrad_status_t dgrad_prepack(dgrad_plan_t plan, const float *weight, void *stream);
dgrad_status_t dgrad_run_packed(dgrad_plan_t plan, const float *grad_out, float *grad_input,
                                void *stream);
dgrad_status_t dgrad_pack_grad_out(dgrad_plan_t plan, const float *grad_out, void *stream);
dgrad_status_t dgrad_run_main(dgrad_plan_t plan, const float *grad_out, float *grad_input,
                              void *stream);

/* The same computation from HOST buffers: copies grad_out and weight to
 * device staging buffers owned by the plan (allocated on the first call),
 * runs dgrad_run, copies grad_input back and synchronises `stream` (and the
 * plan's own copy streams).  With N >= 2 the batch goes through in up to 4
 * chunks, each run by a sub-plan (made on the first call) on `stream` while
 * the next chunk is copied in and the previous one copied out on two
 * non-blocking streams the plan owns; the result is bit-for-bit that of
 * dgrad_run.  Page-locked host buffers give the fastest copies; pageable ones
 * also work. */
dgrad_status_t dgrad_run_host(dgrad_plan_t plan, const float *grad_out_host,
                              const float *weight_host, float *grad_input_host,
                              void *stream);

/* Allocation-free dgrad: the same result as dgrad_run, from DEVICE pointers,
 * without creating a plan and without allocating any device memory.  The
 * pages have no counterpart; it exists for callers that may not allocate,
 * for example code running inside a framework whose own allocator owns the
 * whole device memory budget (a second allocator would overrun or fragment
 * it), or latency-critical code that cannot accept the device-wide
 * synchronisation a cudaMalloc/cudaFree pair can cause mid-step.
 *
 * Scratch: the packed weights and the error word go into one fixed 4 MiB
 * array that the library reserves statically on every device that loads it,
 * for the life of the process.  Shapes whose packed weights need more
 * (dgrad_describe's packed_weight_bytes > 4 MiB - 256 B) are refused with
 * DGRAD_ERR_UNSUPPORTED before anything is launched.  The first call on a
 * device looks up that array's device address (cudaGetSymbolAddress, with the
 * device current) and caches it; make that first call before any stream
 * capture.  The cached address does not survive a reset of the device
 * (cudaDeviceReset, or the primary context released and made again): do not
 * call this function again in a process after such a reset.  Every call on a
 * device shares the one array and it keeps the last call's contents (each
 * call clears the error word and rewrites the packed weights), so calls whose
 * kernels can overlap on the GPU (different streams or threads) race and give
 * wrong results: serialise them.  In-kernel wait timeouts are recorded in the
 * array, which no caller can read: they are not reported (use a plan and
 * dgrad_plan_check where that matters).  Pointer rules, layouts, stream
 * semantics and the other errors are those of dgrad_run, and a DGRAD_ERR_CUDA
 * is explained by dgrad_cuda_error_string as there.  There is no frame
 * buffer, so grad_out reaches the tensor cores through producer warps: the
 * tiles are those dgrad_plan_ex would choose with a_source = 2, which can
 * differ from dgrad_plan's own choice (and run slower) where a plan would
 * use the packed frame. */
dgrad_status_t dgrad_run_noalloc(int N, int Ci, int H, int W, int Co, int kH, int kW,
                                 int stride, int pad_h, int pad_w, dgrad_precision_t precision,
                                 const float *grad_out, const float *weight, float *grad_input,
                                 void *stream);

/* Read and clear the plan's device error word.  Call after synchronising the
 * stream of the last dgrad_run.  Returns DGRAD_OK or the recorded error. */
dgrad_status_t dgrad_plan_check(dgrad_plan_t plan);

/* Free the plan's workspace (synchronises the plan's device first). NULL is a no-op. */
void dgrad_plan_destroy(dgrad_plan_t plan);

/* Static English description of a status code. */
const char *dgrad_status_string(dgrad_status_t status);

/* The CUDA runtime's message for the error behind the last
 * DGRAD_ERR_CUDA returned to the calling thread ("" if none). */
const char *dgrad_cuda_error_string(void);

#ifdef __cplusplus
}
#endif

#endif /* DGRAD_GB300_H */

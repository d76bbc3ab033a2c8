/*
 * dgrad_probe.h -- measurement helper of libdgrad_gb300.so: the FP32 FFMA
 * pipe's throughput on this GPU, the denominator of the exact-fp32 path's
 * roofline.  The pages have no counterpart (they publish no numbers and name
 * no hardware); the benchmark calls this to measure the peak it reports the
 * FFMA kernel against, instead of assuming one.
 */
#ifndef DGRAD_GB300_PROBE_H
#define DGRAD_GB300_PROBE_H

#ifdef __cplusplus
extern "C" {
#endif

/* Launch `blocks` blocks of 256 threads, each thread running 8 independent
 * chains of `iters` dependent fp32 fused multiply-adds (x = x*m + c with m,
 * c passed at run time, so nothing folds), asynchronously on `stream` (a
 * cudaStream_t as void *; NULL = legacy default stream).  Every thread
 * writes the sum of its chains to out[thread], so `out` is a DEVICE buffer
 * of blocks*256 floats (16-byte aligned, owned by the caller).  The launch
 * performs exactly blocks * 256 * 8 * iters FMAs (2 FLOP each); time it with
 * events on `stream`.  Returns 0 on success, DGRAD_ERR_INVALID_ARG (1) for
 * blocks < 1, iters not a positive multiple of 4 or a NULL out,
 * DGRAD_ERR_CUDA (6) if the launch
 * fails (dgrad_cuda_error_string says why). */
int dgrad_probe_ffma(int blocks, int iters, float *out, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* DGRAD_GB300_PROBE_H */

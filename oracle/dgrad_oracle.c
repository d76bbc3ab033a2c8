/*
 * CPU oracle for the convolution backward-data pass (dgrad).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark use it.  It shares no code, header, table or constant with the
 * CUDA library; the two meet only through the seeded input generators.
 *
 * Everything here is plain, slow and written to be checked by eye.  Inputs are
 * fp32 (as the pages' tensors are `array<f32>`) and are widened to fp64; every
 * product of two widened fp32 values is exact in fp64, so the only rounding is
 * in the fp64 additions.
 *
 * Sources (page title, then the part of the page):
 *  - meganeura, src/shaders/conv2d_grad_input_gemm.wgsl: the header comment
 *    (grad_input[n] = weight_T x im2col(grad_out[n]), C[Ci,H*W] = A[Ci,K] x
 *    B[K,H*W], K = Co*kH*kW) and the Params struct (one stride, padding_h and
 *    padding_w, NCHW / OIHW / NCHW tensors).
 *  - @simulatte/doppler 0.1.0, conv2d_backward_input.wgsl: the header comment
 *    (each input element sums the contributions of every output element it fed
 *    in the forward pass) and the "forward mapping" comment in main()
 *    (oy = (iy + pad - ky) / stride, i.e. iy = oy*stride - pad + ky).
 *
 * Shape convention (all row-major, contiguous):
 *   grad_out   [N, Co, oH, oW]
 *   weight     [Co, Ci, kH, kW]
 *   grad_input [N, Ci, H, W]
 *   oH = floor((H + 2*pad_h - kH) / stride) + 1, likewise oW.
 * H and W are authoritative; input rows or columns that no term reaches are 0.
 *
 * Every entry point returns 0 on success and -1 on an invalid shape.
 */
#include <math.h>
#include <pthread.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int N, Ci, H, W, Co, kH, kW, s, ph, pw, oH, oW;
} shape_t;

/* Forward-conv output extent: floor((in + 2p - k)/s) + 1, or 0 if negative. */
static int out_extent(int in, int k, int s, int p)
{
    int num = in + 2 * p - k;
    if (num < 0) return 0;
    return num / s + 1;
}

static int make_shape(shape_t *sh, int N, int Ci, int H, int W, int Co, int kH,
                      int kW, int s, int ph, int pw)
{
    if (N < 1 || Ci < 1 || H < 1 || W < 1 || Co < 1 || kH < 1 || kW < 1 ||
        s < 1 || ph < 0 || pw < 0)
        return -1;
    sh->N = N; sh->Ci = Ci; sh->H = H; sh->W = W; sh->Co = Co;
    sh->kH = kH; sh->kW = kW; sh->s = s; sh->ph = ph; sh->pw = pw;
    sh->oH = out_extent(H, kH, s, ph);
    sh->oW = out_extent(W, kW, s, pw);
    if (sh->oH < 1 || sh->oW < 1) return -1;
    return 0;
}

static size_t go_at(const shape_t *sh, int n, int co, int oh, int ow)
{
    return (((size_t)n * sh->Co + co) * sh->oH + oh) * sh->oW + ow;
}
static size_t w_at(const shape_t *sh, int co, int ci, int kh, int kw)
{
    return (((size_t)co * sh->Ci + ci) * sh->kH + kh) * sh->kW + kw;
}
static size_t gi_at(const shape_t *sh, int n, int ci, int ih, int iw)
{
    return (((size_t)n * sh->Ci + ci) * sh->H + ih) * sh->W + iw;
}

/* ------------------------------------------------------------------------ */
/* O1: the definition, as a direct scatter over grad_out.                    */
/*                                                                           */
/* For every grad_out element g = go[n,co,oh,ow] and every weight tap        */
/* (ci,kh,kw), the forward pass read input element (ih,iw) with              */
/* ih = oh*stride - pad_h + kh, iw = ow*stride - pad_w + kw (doppler         */
/* conv2d_backward_input.wgsl, "forward mapping").  If that element lies in  */
/* the input, the term g*w[co,ci,kh,kw] is added to grad_input there, and    */
/* its absolute value to `mag` (the sum of |terms| used for error bounds).   */
/* Elements no term reaches stay 0.                                          */
/* ------------------------------------------------------------------------ */
typedef struct {
    const shape_t *sh;
    const float *go, *w;
    double *acc, *mag;
    int n0, n1;
} scatter_job_t;

static void scatter_batch_range(const scatter_job_t *j)
{
    const shape_t *sh = j->sh;
    for (int n = j->n0; n < j->n1; ++n)
        for (int co = 0; co < sh->Co; ++co)
            for (int oh = 0; oh < sh->oH; ++oh)
                for (int ow = 0; ow < sh->oW; ++ow) {
                    double g = (double)j->go[go_at(sh, n, co, oh, ow)];
                    for (int ci = 0; ci < sh->Ci; ++ci)
                        for (int kh = 0; kh < sh->kH; ++kh) {
                            int ih = oh * sh->s - sh->ph + kh;
                            if (ih < 0 || ih >= sh->H) continue;
                            for (int kw = 0; kw < sh->kW; ++kw) {
                                int iw = ow * sh->s - sh->pw + kw;
                                if (iw < 0 || iw >= sh->W) continue;
                                double t = g * (double)j->w[w_at(sh, co, ci, kh, kw)];
                                size_t o = gi_at(sh, n, ci, ih, iw);
                                j->acc[o] += t;
                                if (j->mag) j->mag[o] += fabs(t);
                            }
                        }
                }
}

static void *scatter_thread(void *arg)
{
    scatter_batch_range((const scatter_job_t *)arg);
    return NULL;
}

int oracle_dgrad_scatter(int N, int Ci, int H, int W, int Co, int kH, int kW,
                         int stride, int pad_h, int pad_w, const float *go,
                         const float *w, double *acc, double *mag, int nthreads)
{
    shape_t sh;
    if (make_shape(&sh, N, Ci, H, W, Co, kH, kW, stride, pad_h, pad_w)) return -1;
    size_t n_gi = (size_t)N * Ci * H * W;
    memset(acc, 0, n_gi * sizeof(double));
    if (mag) memset(mag, 0, n_gi * sizeof(double));

    /* Batch items write disjoint parts of grad_input, so they may run on
     * separate threads without changing any sum. */
    if (nthreads < 1) nthreads = 1;
    if (nthreads > N) nthreads = N;
    scatter_job_t jobs[256];
    pthread_t tids[256];
    if (nthreads > 256) nthreads = 256;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].sh = &sh; jobs[t].go = go; jobs[t].w = w;
        jobs[t].acc = acc; jobs[t].mag = mag;
        jobs[t].n0 = (int)((long)N * t / nthreads);
        jobs[t].n1 = (int)((long)N * (t + 1) / nthreads);
    }
    int started = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&tids[t], NULL, scatter_thread, &jobs[t]) != 0) break;
        started = t;
    }
    scatter_batch_range(&jobs[0]);
    for (int t = 1; t <= started; ++t) pthread_join(tids[t], NULL);
    for (int t = started + 1; t < nthreads; ++t) scatter_batch_range(&jobs[t]);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* O-fwd: the forward convolution whose input-adjoint dgrad is.              */
/* y[n,co,oh,ow] = sum over (ci,kh,kw) with (ih,iw) inside the input of      */
/* x[n,ci,ih,iw] * w[co,ci,kh,kw], ih = oh*stride - pad_h + kh (same map as  */
/* O1).  fp64 in and out, so tests can feed exact unit vectors.              */
/* ------------------------------------------------------------------------ */
int oracle_conv2d_fwd(int N, int Ci, int H, int W, int Co, int kH, int kW,
                      int stride, int pad_h, int pad_w, const double *x,
                      const double *w, double *y)
{
    shape_t sh;
    if (make_shape(&sh, N, Ci, H, W, Co, kH, kW, stride, pad_h, pad_w)) return -1;
    for (int n = 0; n < N; ++n)
        for (int co = 0; co < Co; ++co)
            for (int oh = 0; oh < sh.oH; ++oh)
                for (int ow = 0; ow < sh.oW; ++ow) {
                    double sum = 0.0;
                    for (int ci = 0; ci < Ci; ++ci)
                        for (int kh = 0; kh < kH; ++kh) {
                            int ih = oh * stride - pad_h + kh;
                            if (ih < 0 || ih >= H) continue;
                            for (int kw = 0; kw < kW; ++kw) {
                                int iw = ow * stride - pad_w + kw;
                                if (iw < 0 || iw >= W) continue;
                                sum += x[gi_at(&sh, n, ci, ih, iw)] *
                                       w[w_at(&sh, co, ci, kh, kw)];
                            }
                        }
                    y[go_at(&sh, n, co, oh, ow)] = sum;
                }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Per-element gather, written from the definition: for input element        */
/* (n,ci,ih,iw) sum over (co,kh,kw) the grad_out elements whose forward      */
/* window covered it, i.e. those with oh*stride = ih + pad_h - kh for an     */
/* integer oh in [0,oH) (same for w).  Shared by O2 and O-at below.          */
/* ------------------------------------------------------------------------ */
static void gather_one(const shape_t *sh, const float *go, const float *w,
                       int n, int ci, int ih, int iw, double *acc, double *mag)
{
    double sum = 0.0, abs_sum = 0.0;
    for (int co = 0; co < sh->Co; ++co)
        for (int kh = 0; kh < sh->kH; ++kh) {
            int py = ih + sh->ph;          /* row in the padded input */
            if (py < kh) continue;
            int hy = py - kh;
            if (hy % sh->s != 0) continue; /* not on the stride lattice */
            int oh = hy / sh->s;
            if (oh >= sh->oH) continue;
            for (int kw = 0; kw < sh->kW; ++kw) {
                int px = iw + sh->pw;
                if (px < kw) continue;
                int hx = px - kw;
                if (hx % sh->s != 0) continue;
                int ow = hx / sh->s;
                if (ow >= sh->oW) continue;
                double t = (double)go[go_at(sh, n, co, oh, ow)] *
                           (double)w[w_at(sh, co, ci, kh, kw)];
                sum += t;
                abs_sum += fabs(t);
            }
        }
    *acc = sum;
    if (mag) *mag = abs_sum;
}

/* O2: the gather formulation of doppler's conv2d_backward_input.wgsl main()
 * (one result per input element; loops over output channel, then kernel row,
 * then kernel column; skips taps that fall before the padded origin, off the
 * stride lattice, or past the output edge), with a batch axis and separate
 * row/column padding added. */
int oracle_dgrad_gather(int N, int Ci, int H, int W, int Co, int kH, int kW,
                        int stride, int pad_h, int pad_w, const float *go,
                        const float *w, double *acc)
{
    shape_t sh;
    if (make_shape(&sh, N, Ci, H, W, Co, kH, kW, stride, pad_h, pad_w)) return -1;
    for (int n = 0; n < N; ++n)
        for (int ci = 0; ci < Ci; ++ci)
            for (int ih = 0; ih < H; ++ih)
                for (int iw = 0; iw < W; ++iw)
                    gather_one(&sh, go, w, n, ci, ih, iw,
                               &acc[gi_at(&sh, n, ci, ih, iw)], NULL);
    return 0;
}

/* O-at: the definition at a list of sampled input elements.  idx holds
 * 4 ints (n, ci, ih, iw) per sample. */
int oracle_dgrad_at(int N, int Ci, int H, int W, int Co, int kH, int kW,
                    int stride, int pad_h, int pad_w, const float *go,
                    const float *w, const int *idx, long n_idx, double *acc,
                    double *mag)
{
    shape_t sh;
    if (make_shape(&sh, N, Ci, H, W, Co, kH, kW, stride, pad_h, pad_w)) return -1;
    for (long i = 0; i < n_idx; ++i) {
        int n = idx[4 * i], ci = idx[4 * i + 1], ih = idx[4 * i + 2], iw = idx[4 * i + 3];
        if (n < 0 || n >= N || ci < 0 || ci >= Ci || ih < 0 || ih >= H || iw < 0 || iw >= W)
            return -1;
        gather_one(&sh, go, w, n, ci, ih, iw, &acc[i], mag ? &mag[i] : NULL);
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* O3: meganeura's implicit-GEMM index map, restated without its tiling.     */
/* C[ci, hw] = sum_k A[ci,k] * B[k,hw] with k = co*kH*kW + kh*kW + kw,       */
/* A[ci,k] = weight[co,ci,kh,kw] and B[k,hw] read from grad_out exactly as   */
/* the shader's B-tile load does: for stride 1 through the "transposed       */
/* padding" (kH-1-padding_h), for larger strides through the divisibility    */
/* test.  Kept as a cross-check only: for stride 1 it equals the definition  */
/* only when 2*pad = k-1 ("same" padding).                                   */
/* ------------------------------------------------------------------------ */
int oracle_dgrad_gemm_p1(int N, int Ci, int H, int W, int Co, int kH, int kW,
                         int stride, int pad_h, int pad_w, const float *go,
                         const float *w, double *acc)
{
    shape_t sh;
    if (make_shape(&sh, N, Ci, H, W, Co, kH, kW, stride, pad_h, pad_w)) return -1;
    int K = Co * kH * kW;
    int tp_h = kH - 1 - pad_h, tp_w = kW - 1 - pad_w;
    for (int n = 0; n < N; ++n)
        for (int ci = 0; ci < Ci; ++ci)
            for (int hw = 0; hw < H * W; ++hw) {
                int ih = hw / W, iw = hw % W;
                double sum = 0.0;
                for (int k = 0; k < K; ++k) {
                    int co = k / (kH * kW), rem = k % (kH * kW);
                    int kh = rem / kW, kw = rem % kW;
                    double a = (double)w[w_at(&sh, co, ci, kh, kw)];
                    double b = 0.0;
                    if (stride == 1) {
                        int oh = ih + tp_h - kh, ow = iw + tp_w - kw;
                        if (oh >= 0 && oh < sh.oH && ow >= 0 && ow < sh.oW)
                            b = (double)go[go_at(&sh, n, co, oh, ow)];
                    } else {
                        int hoff = ih + pad_h - kh, woff = iw + pad_w - kw;
                        if (hoff >= 0 && woff >= 0 && hoff % stride == 0 && woff % stride == 0) {
                            int oh = hoff / stride, ow = woff / stride;
                            if (oh < sh.oH && ow < sh.oW)
                                b = (double)go[go_at(&sh, n, co, oh, ow)];
                        }
                    }
                    sum += a * b;
                }
                acc[gi_at(&sh, n, ci, ih, iw)] = sum;
            }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* O-phase: the sub-pixel phase split of the strided case, restated on the   */
/* CPU so the decomposition itself is checked against the definition.       */
/*                                                                           */
/* Input row ih = stride*q + a (phase a in [0,stride)) receives kernel rows  */
/* kh with (a + pad_h - kh) divisible by stride, i.e. kh = r_a + stride*j    */
/* with r_a = (a + pad_h) mod stride, and then oh = q + c_a - j with         */
/* c_a = floor((a + pad_h) / stride).  Same for columns.  Each phase is a    */
/* dense stride-1 correlation over its own taps.                             */
/* ------------------------------------------------------------------------ */
int oracle_dgrad_phase(int N, int Ci, int H, int W, int Co, int kH, int kW,
                       int stride, int pad_h, int pad_w, const float *go,
                       const float *w, double *acc)
{
    shape_t sh;
    if (make_shape(&sh, N, Ci, H, W, Co, kH, kW, stride, pad_h, pad_w)) return -1;
    int s = stride;
    memset(acc, 0, (size_t)N * Ci * H * W * sizeof(double));
    for (int a = 0; a < s; ++a) {
        int r_a = (a + pad_h) % s, c_a = (a + pad_h) / s;
        for (int b = 0; b < s; ++b) {
            int r_b = (b + pad_w) % s, c_b = (b + pad_w) / s;
            for (int n = 0; n < N; ++n)
                for (int ci = 0; ci < Ci; ++ci)
                    for (int q = 0; s * q + a < H; ++q)
                        for (int u = 0; s * u + b < W; ++u) {
                            double sum = 0.0;
                            for (int j = 0; r_a + s * j < kH; ++j) {
                                int oh = q + c_a - j;
                                if (oh < 0 || oh >= sh.oH) continue;
                                for (int i = 0; r_b + s * i < kW; ++i) {
                                    int ow = u + c_b - i;
                                    if (ow < 0 || ow >= sh.oW) continue;
                                    for (int co = 0; co < Co; ++co)
                                        sum += (double)go[go_at(&sh, n, co, oh, ow)] *
                                               (double)w[w_at(&sh, co, ci, r_a + s * j, r_b + s * i)];
                                }
                            }
                            acc[gi_at(&sh, n, ci, s * q + a, s * u + b)] = sum;
                        }
        }
    }
    return 0;
}

/* Output extents, so callers need not restate the formula. */
int oracle_out_extent(int in, int k, int stride, int pad)
{
    if (in < 1 || k < 1 || stride < 1 || pad < 0) return 0;
    return out_extent(in, k, stride, pad);
}

/* ------------------------------------------------------------------------ */
/* O-w: the weight gradient (wgrad), the other half of doppler's            */
/* runConv2DBackward (conv2d_backward.js: with computeGradWeight it runs     */
/* one invocation per weight element, [outChannels, inChannels, kernelH,     */
/* kernelW], over gradOutput and the forward input; its shader is not on     */
/* the page).  Written from the same forward mapping as O1: the forward      */
/* pass multiplied w[co,ci,kh,kw] by x[n,ci,ih,iw] with                      */
/* ih = oh*stride - pad_h + kh, iw = ow*stride - pad_w + kw into             */
/* y[n,co,oh,ow], so                                                         */
/*   dW[co,ci,kh,kw] = sum over n, oh, ow with (ih,iw) inside the input of   */
/*                     go[n,co,oh,ow] * x[n,ci,ih,iw].                       */
/* `mag` gets the sum of |terms|.  The batch is summed (the pages' host      */
/* code has no batch axis; a batched forward pass shares one weight).        */
/* ------------------------------------------------------------------------ */
typedef struct {
    const shape_t *sh;
    const float *go, *x;
    double *acc, *mag;
    int co0, co1;
} wgrad_job_t;

static void wgrad_co_range(const wgrad_job_t *j)
{
    const shape_t *sh = j->sh;
    for (int co = j->co0; co < j->co1; ++co)
        for (int ci = 0; ci < sh->Ci; ++ci)
            for (int kh = 0; kh < sh->kH; ++kh)
                for (int kw = 0; kw < sh->kW; ++kw) {
                    double a = 0.0, m = 0.0;
                    for (int n = 0; n < sh->N; ++n)
                        for (int oh = 0; oh < sh->oH; ++oh) {
                            int ih = oh * sh->s - sh->ph + kh;
                            if (ih < 0 || ih >= sh->H) continue;
                            for (int ow = 0; ow < sh->oW; ++ow) {
                                int iw = ow * sh->s - sh->pw + kw;
                                if (iw < 0 || iw >= sh->W) continue;
                                double t = (double)j->go[go_at(sh, n, co, oh, ow)] *
                                           (double)j->x[gi_at(sh, n, ci, ih, iw)];
                                a += t;
                                m += fabs(t);
                            }
                        }
                    size_t o = w_at(sh, co, ci, kh, kw);
                    j->acc[o] = a;
                    if (j->mag) j->mag[o] = m;
                }
}

static void *wgrad_thread(void *arg)
{
    wgrad_co_range((const wgrad_job_t *)arg);
    return NULL;
}

int oracle_wgrad(int N, int Ci, int H, int W, int Co, int kH, int kW, int stride,
                 int pad_h, int pad_w, const float *go, const float *x,
                 double *acc, double *mag, int nthreads)
{
    shape_t sh;
    if (make_shape(&sh, N, Ci, H, W, Co, kH, kW, stride, pad_h, pad_w)) return -1;
    /* Output channels own disjoint parts of dW: threads split them. */
    if (nthreads < 1) nthreads = 1;
    if (nthreads > Co) nthreads = Co;
    if (nthreads > 256) nthreads = 256;
    wgrad_job_t jobs[256];
    pthread_t tids[256];
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].sh = &sh; jobs[t].go = go; jobs[t].x = x;
        jobs[t].acc = acc; jobs[t].mag = mag;
        jobs[t].co0 = (int)((long)Co * t / nthreads);
        jobs[t].co1 = (int)((long)Co * (t + 1) / nthreads);
    }
    int started = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&tids[t], NULL, wgrad_thread, &jobs[t]) != 0) break;
        started = t;
    }
    wgrad_co_range(&jobs[0]);
    for (int t = 1; t <= started; ++t) pthread_join(tids[t], NULL);
    for (int t = started + 1; t < nthreads; ++t) wgrad_co_range(&jobs[t]);
    return 0;
}

// C ABI of libdgrad_gb300 (declared in include/dgrad.h): plan creation,
// validation, launches and error reporting.
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

#include "dgrad.h"
#include "dgrad_internal.h"

constexpr int kHostChunks = 4;   // batch chunks of dgrad_run_host's copy/compute pipeline (4: 252 us e2e on
                                 // resnet_stage; 6: 255, 8: 260, 12: 266 -- per-chunk costs against fill and drain)

struct dgrad_plan_s {
    int device;
    int precision;
    dgrad::Geometry g;
    dgrad::Tiling t;
    dgrad::MainParams mp;
    dgrad::C2iParams cp;   // col2im path
    dgrad::PrepackParams pp;
    float *wp;             // packed weights (device)
    float *frame;          // packed grad_out frame (device), tensor-copy mode only
    dgrad::FramePackParams fp;
    uint32_t *err;         // device error word
    float *stage_go;       // dgrad_run_host staging (device), allocated on first use
    float *stage_w;
    float *stage_gi;
    // dgrad_run_host pipeline (made on first use): the batch in chunks of
    // chunk_n images, each run by a sub-plan while the next chunk's input and
    // the previous chunk's output are in flight on their own streams
    dgrad_options_t opts;
    int chunk_n;
    dgrad_plan_s *sub[2];          // sub-plans for chunk_n images and for the remainder
    cudaStream_t h2d, d2h;
    cudaEvent_t ev_in[kHostChunks], ev_out[kHostChunks];
    uint32_t *host_err;            // page-locked copies of the sub-plans' error words
    int host_ready;
    size_t workspace_bytes;
    int packed;            // dgrad_prepack (or dgrad_run) has run at least once
    int frame_packed;      // grad_out has been packed into the frame at least once
    // staged A source: the tensor map of the caller's grad_out, encoded for
    // the last pointer seen (re-encoded when the pointer changes)
    const float *go_map_ptr;
    CUtensorMap go_map;
};

// cuTensorMapEncodeTiled from the driver, looked up once through the
// runtime (no link-time dependency on the driver library).
// The CUDA error behind the last DGRAD_ERR_CUDA of this thread.
static thread_local cudaError_t g_last_cuda = cudaSuccess;

dgrad_status_t dgrad::cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return DGRAD_OK;
    g_last_cuda = e;
    cudaGetLastError();   // clear the (non-sticky) error
    return DGRAD_ERR_CUDA;
}

PFN_cuTensorMapEncodeTiled_v12000 dgrad::tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
        cudaGetLastError();
    });
    return fn;
}

namespace {

using dgrad::Geometry;
using dgrad::Tiling;

constexpr long long kTimeoutNs = 1000000000LL;   // bounded in-kernel waits: 1 s

using dgrad::cuda_status;

size_t go_elems(const Geometry &g) { return (size_t)g.N * g.Co * g.oH * g.oW; }
size_t w_elems(const Geometry &g) { return (size_t)g.Co * g.Ci * g.kH * g.kW; }
size_t gi_elems(const Geometry &g) { return (size_t)g.N * g.Ci * g.H * g.W; }

void fill_info(const Geometry &g, const Tiling &t, int precision, size_t ws, dgrad_plan_info_t *info) {
    std::memset(info, 0, sizeof(*info));
    info->N = g.N; info->Ci = g.Ci; info->H = g.H; info->W = g.W; info->Co = g.Co;
    info->kH = g.kH; info->kW = g.kW; info->stride = g.s; info->pad_h = g.ph; info->pad_w = g.pw;
    info->oH = g.oH; info->oW = g.oW;
    info->precision = precision;
    info->path = t.path;
    info->n_phases = g.n_phases;
    info->n_taps = g.n_taps;
    info->Ph = g.Ph; info->Pw = g.Pw; info->Hv = g.Hv; info->Wp = g.Wp;
    info->positions = g.positions;
    info->max_shift = g.max_shift;
    info->tile_blocks = t.tm; info->slice_n = t.bn; info->n_slices = t.n_slices;
    info->chunk_k = t.kc; info->n_chunks = t.n_chunks;
    info->n_work = t.n_work;
    info->grid = t.path == DGRAD_PATH_SIMT && !t.a_tma ? (int)t.n_work : t.grid;
    info->b_resident = t.b_resident;
    info->a_source = t.path == DGRAD_PATH_COL2IM ? 1 : t.a_tmem ? 4 : t.a_staged ? 3 : t.a_tma ? 1 : 2;
    info->smem_bytes = t.smem_bytes;
    info->tmem_cols = t.tmem_cols;
    info->group_taps = t.grouped ? 1 : (t.pgroup ? 2 : 0);
    info->tile_step = t.tile_step;
    info->a_stages = t.a_stages;
    info->b_stages = t.b_stages;
    info->workspace_bytes = ws;
    info->packed_weight_bytes = t.packed_bytes;
    info->useful_flops = 2.0 * g.N * g.Co * g.oH * g.oW * (double)g.Ci * g.kH * g.kW;
    info->algorithmic_bytes = 4.0 * ((double)go_elems(g) + (double)w_elems(g) + (double)gi_elems(g));
    info->band_rows = t.band_rows;
    info->stg_box = (t.a_staged || t.a_tmem) ? t.stg_box : 0;
    info->img_tiles = t.img_tiles;
    info->a_rows = t.a_rows;
}

dgrad_status_t plan_host(int N, int Ci, int H, int W, int Co, int kH, int kW, int stride, int pad_h,
                         int pad_w, dgrad_precision_t precision, const dgrad_options_t *opts, int sm_count,
                         Geometry *g, Tiling *t) {
    if (precision != DGRAD_PREC_FP32 && precision != DGRAD_PREC_TF32 && precision != DGRAD_PREC_TF32X3)
        return DGRAD_ERR_INVALID_ARG;
    dgrad_status_t st = dgrad::make_geometry(N, Ci, H, W, Co, kH, kW, stride, pad_h, pad_w, g);
    if (st != DGRAD_OK) return st;
    return dgrad::choose_tiling(*g, precision, opts, sm_count, t);
}

void fill_params(dgrad_plan_s *pl) {
    const Geometry &g = pl->g;
    const Tiling &t = pl->t;
    const int round = pl->precision != DGRAD_PREC_FP32 ? 1 : 0;
    dgrad::fill_main_params(g, t, round, &pl->mp);
    pl->mp.wp = pl->wp;
    pl->mp.err = pl->err;
    const long long tmo = pl->opts.timeout_us > 0 ? 1000LL * pl->opts.timeout_us : kTimeoutNs;
    pl->mp.timeout_ns = tmo;
    pl->mp.wait_test = pl->opts.wait_test ? 1 : 0;
    dgrad::fill_prepack_params(g, t, round, &pl->pp);
    pl->pp.wp = pl->wp;
    if (t.path == DGRAD_PATH_COL2IM) {
        dgrad::fill_c2i_params(g, t, &pl->cp);
        pl->cp.wp = pl->wp;
        pl->cp.err = pl->err;
        pl->cp.timeout_ns = tmo;
    }

    dgrad::FramePackParams &f = pl->fp;
    std::memset(&f, 0, sizeof(f));
    f.v = pl->frame;
    f.N = g.N; f.Co = g.Co; f.oH = g.oH; f.oW = g.oW; f.Hv = g.Hv; f.Wp = g.Wp; f.Ph = g.Ph; f.Pw = g.Pw;
    f.co_v = t.co_v;
    f.split = t.split;
    f.co_h = t.co_h;
    f.round_tf32 = t.split ? 0 : round;   // split: the write stage rounds both halves
    f.positions = (int)g.positions;
    // Pack blocks of 32 channels x seg_len plane elements: 256 elements
    // unless that leaves fewer than 512 blocks (then shorter segments, down
    // to 32, so that every SM gets a few; measured best of 256/512/1024).
    const long long plane = (long long)g.oH * g.oW;
    f.c_groups = (g.Co + dgrad::kPackChannels - 1) / dgrad::kPackChannels;
    f.seg_len = dgrad::kPackSegMax;
    while (f.seg_len > 32 && (long long)g.N * f.c_groups * ((plane + f.seg_len - 1) / f.seg_len) < 512)
        f.seg_len /= 2;
    f.segs = (int)((plane + f.seg_len - 1) / f.seg_len);
    f.vec = plane % 4 == 0 ? 1 : 0;
}

// Tensor map of the packed frame [positions][co_v] (fp32) by a_box_rows
// positions; rows past the frame read as zeros.  tcgen05 and col2im: boxes
// of 32 channels (128 bytes, 128-byte swizzle: the MMA's K-major operand
// layout); FFMA path: boxes of 4 channels (16 bytes, no swizzle), one per
// 4-channel group of the FFMA loop's band layout.
dgrad_status_t encode_frame_map(dgrad_plan_s *pl) {
    auto fn = dgrad::tensor_map_encoder();
    if (!fn) return DGRAD_ERR_CUDA;
    const bool ffma = pl->t.path == DGRAD_PATH_SIMT;
    const cuuint64_t dims[2] = {(cuuint64_t)pl->t.co_v, (cuuint64_t)pl->g.positions};
    const cuuint64_t strides[1] = {(cuuint64_t)pl->t.co_v * 4};
    const cuuint32_t box[2] = {ffma ? 4u : 32u, (cuuint32_t)pl->t.a_box_rows};
    const cuuint32_t es[2] = {1u, 1u};
    CUresult r = fn(&pl->mp.a_map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, pl->frame, dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, ffma ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? DGRAD_OK : DGRAD_ERR_CUDA;
}

// Staged and tensor-memory A sources: grad_out viewed as [N][Co][oH*oW]
// (fp32), boxes of stg_box plane elements x 32 channels x 1 image, no
// swizzle; channels past Co and elements past the plane read as zeros.
// Encoded on the caller's pointer (16-byte aligned; the plane stride
// oH*oW*4 is a multiple of 16 for every such plan).
dgrad_status_t encode_staged_map(dgrad_plan_s *pl, const float *grad_out) {
    if (pl->go_map_ptr == grad_out) return DGRAD_OK;
    auto fn = dgrad::tensor_map_encoder();
    if (!fn) return DGRAD_ERR_CUDA;
    const Geometry &g = pl->g;
    const cuuint64_t plane = (cuuint64_t)g.oH * g.oW;
    const cuuint64_t dims[3] = {plane, (cuuint64_t)g.Co, (cuuint64_t)g.N};
    const cuuint64_t strides[2] = {plane * 4, plane * 4 * (cuuint64_t)g.Co};
    const cuuint32_t box[3] = {(cuuint32_t)pl->t.stg_box, 32u, 1u};
    const cuuint32_t es[3] = {1u, 1u, 1u};
    CUresult r = fn(&pl->go_map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(grad_out), dims, strides,
                    box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        pl->go_map_ptr = nullptr;
        return DGRAD_ERR_CUDA;
    }
    pl->go_map_ptr = grad_out;
    return DGRAD_OK;
}

bool overlaps(const void *a, size_t abytes, const void *b, size_t bbytes) {
    uintptr_t a0 = (uintptr_t)a, a1 = a0 + abytes, b0 = (uintptr_t)b, b1 = b0 + bbytes;
    return a0 < b1 && b0 < a1;
}

bool aligned16(const void *p) { return p != nullptr && ((uintptr_t)p & 15u) == 0; }

dgrad_status_t check_device(const dgrad_plan_s *plan) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return DGRAD_ERR_CUDA;
    return dev == plan->device ? DGRAD_OK : DGRAD_ERR_WRONG_DEVICE;
}

// One pack launch: the weights (when `weight` is given) and, in tensor-copy
// mode, the grad_out frame (when `grad_out` is given).
dgrad_status_t launch_pack_on(dgrad_plan_s *plan, const float *weight, const float *grad_out, cudaStream_t s) {
    dgrad::PrepackParams pp = plan->pp;
    pp.w = weight;
    dgrad::FramePackParams fp = plan->fp;
    fp.go = grad_out;
    const bool frame = plan->frame != nullptr && grad_out != nullptr;
    dgrad_status_t st = cuda_status(dgrad::launch_pack(weight ? &pp : nullptr, frame ? &fp : nullptr, s));
    if (st != DGRAD_OK) return st;
    if (weight) plan->packed = 1;
    if (frame) plan->frame_packed = 1;
    return DGRAD_OK;
}

dgrad_status_t launch_main_on(dgrad_plan_s *plan, const float *grad_out, float *grad_input, cudaStream_t s,
                              const float *relu_in = nullptr, int accumulate = 0) {
    dgrad::MainParams mp = plan->mp;
    mp.go = grad_out;
    mp.gi = grad_input;
    mp.relu_in = relu_in;
    mp.accumulate = accumulate;
    if (plan->t.path == DGRAD_PATH_COL2IM) {
        dgrad::C2iParams cp = plan->cp;
        cp.gi = grad_input;
        cp.relu_in = relu_in;
        cp.accumulate = accumulate;
        return cuda_status(dgrad::launch_c2i(cp, plan->t, s, true));
    }
    if (plan->t.path == DGRAD_PATH_TCGEN05 && (plan->t.a_staged || plan->t.a_tmem)) {
        dgrad_status_t st = encode_staged_map(plan, grad_out);
        if (st != DGRAD_OK) return st;
        mp.a_map = plan->go_map;
    }
    cudaError_t e = plan->t.path == DGRAD_PATH_TCGEN05 ? dgrad::launch_tc(mp, plan->t, s, true)
                                                       : dgrad::launch_simt(mp, plan->t, s);
    return cuda_status(e);
}

// dgrad_run_host's pipeline: chunks of ceil(N / kHostChunks) images, two
// sub-plans (full chunk, remainder), two copy streams and their events.
dgrad_status_t make_host_pipeline(dgrad_plan_s *plan) {
    const Geometry &g = plan->g;
    plan->chunk_n = (g.N + kHostChunks - 1) / kHostChunks;   // the same split dgrad_run_host stages
    const int rem = g.N % plan->chunk_n;
    const int sizes[2] = {plan->chunk_n, rem};
    for (int i = 0; i < 2; ++i) {
        if (sizes[i] == 0 || plan->sub[i]) continue;
        dgrad_status_t st = dgrad_plan_ex(sizes[i], g.Ci, g.H, g.W, g.Co, g.kH, g.kW, g.s, g.ph, g.pw,
                                          static_cast<dgrad_precision_t>(plan->precision), &plan->opts, &plan->sub[i]);
        if (st != DGRAD_OK) return st;
    }
    // Each object is made once; after a failure the next call makes what is
    // missing and dgrad_plan_destroy releases what exists.
    if (!plan->h2d && cudaStreamCreateWithFlags(&plan->h2d, cudaStreamNonBlocking) != cudaSuccess)
        return cuda_status(cudaGetLastError());
    if (!plan->d2h && cudaStreamCreateWithFlags(&plan->d2h, cudaStreamNonBlocking) != cudaSuccess)
        return cuda_status(cudaGetLastError());
    for (int i = 0; i < kHostChunks; ++i) {
        if ((!plan->ev_in[i] && cudaEventCreateWithFlags(&plan->ev_in[i], cudaEventDisableTiming) != cudaSuccess) ||
            (!plan->ev_out[i] && cudaEventCreateWithFlags(&plan->ev_out[i], cudaEventDisableTiming) != cudaSuccess))
            return cuda_status(cudaGetLastError());
    }
    if (!plan->host_err) {
        void *h = nullptr;
        if (cudaHostAlloc(&h, 2 * sizeof(uint32_t), cudaHostAllocDefault) != cudaSuccess)
            return cuda_status(cudaGetLastError());
        plan->host_err = static_cast<uint32_t *>(h);
    }
    plan->host_ready = 1;
    return DGRAD_OK;
}

}  // namespace

extern "C" {

const char *dgrad_cuda_error_string(void) {
    return g_last_cuda == cudaSuccess ? "" : cudaGetErrorString(g_last_cuda);
}

const char *dgrad_status_string(dgrad_status_t s) {
    switch (s) {
        case DGRAD_OK: return "ok";
        case DGRAD_ERR_INVALID_ARG: return "invalid argument (shape, stride, padding or plan)";
        case DGRAD_ERR_UNSUPPORTED: return "shape outside the supported limits";
        case DGRAD_ERR_MISALIGNED: return "tensor pointer is NULL or not 16-byte aligned";
        case DGRAD_ERR_ALIAS: return "grad_input overlaps grad_out or weight";
        case DGRAD_ERR_OOM: return "device workspace allocation failed";
        case DGRAD_ERR_CUDA: return "CUDA runtime error or kernel launch failure";
        case DGRAD_ERR_DEVICE_TIMEOUT: return "a bounded in-kernel wait ran out";
        case DGRAD_ERR_NO_DEVICE: return "no CUDA device of compute capability 10.3";
        case DGRAD_ERR_WRONG_DEVICE: return "current CUDA device is not the plan's device";
    }
    return "unknown status";
}

dgrad_status_t dgrad_describe(int N, int Ci, int H, int W, int Co, int kH, int kW, int stride, int pad_h,
                              int pad_w, dgrad_precision_t precision, const dgrad_options_t *opts,
                              dgrad_plan_info_t *info) {
    if (!info) return DGRAD_ERR_INVALID_ARG;
    Geometry g;
    Tiling t;
    int sms = (opts && opts->sm_count > 0) ? opts->sm_count : 152;
    dgrad_status_t st = plan_host(N, Ci, H, W, Co, kH, kW, stride, pad_h, pad_w, precision, opts, sms, &g, &t);
    if (st != DGRAD_OK) return st;
    fill_info(g, t, precision, t.packed_bytes + 256, info);
    return DGRAD_OK;
}

dgrad_status_t dgrad_describe_taps(int N, int Ci, int H, int W, int Co, int kH, int kW, int stride, int pad_h,
                                   int pad_w, int cap, int *phases, int *n_phases, int *taps, int *n_taps) {
    if (!phases || !n_phases || !taps || !n_taps || cap < 0) return DGRAD_ERR_INVALID_ARG;
    Geometry g;
    dgrad_status_t st = dgrad::make_geometry(N, Ci, H, W, Co, kH, kW, stride, pad_h, pad_w, &g);
    if (st != DGRAD_OK) return st;
    *n_phases = g.n_phases;
    *n_taps = g.n_taps;
    for (int i = 0; i < g.n_phases && i < cap; ++i) {
        const dgrad::PhaseDesc &p = g.phase[i];
        int *o = phases + 7 * i;
        o[0] = p.a; o[1] = p.b; o[2] = p.Hq; o[3] = p.Wq; o[4] = p.tap_begin; o[5] = p.tap_count;
        o[6] = p.row_len;
    }
    for (int i = 0; i < g.n_taps && i < cap; ++i) {
        taps[3 * i] = g.tap[i].kh;
        taps[3 * i + 1] = g.tap[i].kw;
        taps[3 * i + 2] = g.tap[i].shift;
    }
    return DGRAD_OK;
}

dgrad_status_t dgrad_plan_ex(int N, int Ci, int H, int W, int Co, int kH, int kW, int stride, int pad_h,
                             int pad_w, dgrad_precision_t precision, const dgrad_options_t *opts,
                             dgrad_plan_t *plan_out) {
    if (!plan_out) return DGRAD_ERR_INVALID_ARG;
    *plan_out = nullptr;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DGRAD_ERR_NO_DEVICE;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return DGRAD_ERR_NO_DEVICE;
    if (prop.major != 10 || prop.minor != 3) return DGRAD_ERR_NO_DEVICE;

    dgrad_plan_s *pl = new (std::nothrow) dgrad_plan_s;
    if (!pl) return DGRAD_ERR_OOM;
    std::memset(pl, 0, sizeof(*pl));
    pl->device = dev;
    pl->precision = precision;
    if (opts) pl->opts = *opts;
    dgrad_status_t st = plan_host(N, Ci, H, W, Co, kH, kW, stride, pad_h, pad_w, precision, opts,
                                  prop.multiProcessorCount, &pl->g, &pl->t);
    if (st != DGRAD_OK) {
        delete pl;
        return st;
    }
    // Workspace: the error word (256 B), the packed weights, then (tensor-
    // copy mode) the packed grad_out frame, each 256-byte aligned.
    const size_t wp_bytes = (pl->t.packed_bytes + 255) & ~size_t(255);
    const bool has_frame = pl->t.a_tma && !pl->t.a_staged && !pl->t.a_tmem;
    size_t ws = 256 + wp_bytes + (has_frame ? pl->t.frame_bytes : 0);
    void *mem = nullptr;
    if (cudaMalloc(&mem, ws) != cudaSuccess) {
        cudaGetLastError();
        delete pl;
        return DGRAD_ERR_OOM;
    }
    // Zero everything once: the error word, and the frame's rows and
    // channels that no pack ever writes (its zero padding).  Completed here,
    // so that work later queued on any stream sees it.
    if (cudaMemset(mem, 0, ws) != cudaSuccess || cudaStreamSynchronize(nullptr) != cudaSuccess) {
        cudaGetLastError();
        cudaFree(mem);
        delete pl;
        return DGRAD_ERR_CUDA;
    }
    pl->err = static_cast<uint32_t *>(mem);
    pl->wp = reinterpret_cast<float *>(static_cast<uint8_t *>(mem) + 256);
    if (has_frame) pl->frame = reinterpret_cast<float *>(static_cast<uint8_t *>(mem) + 256 + wp_bytes);
    pl->workspace_bytes = ws;
    fill_params(pl);
    if (pl->frame && (st = encode_frame_map(pl)) != DGRAD_OK) {
        cudaFree(mem);
        delete pl;
        return st;
    }
    if (pl->t.path == DGRAD_PATH_COL2IM) pl->cp.a_map = pl->mp.a_map;
    *plan_out = pl;
    return DGRAD_OK;
}

dgrad_status_t dgrad_plan(int N, int Ci, int H, int W, int Co, int kH, int kW, int stride, int pad_h, int pad_w,
                          dgrad_precision_t precision, dgrad_plan_t *plan_out) {
    return dgrad_plan_ex(N, Ci, H, W, Co, kH, kW, stride, pad_h, pad_w, precision, nullptr, plan_out);
}

dgrad_status_t dgrad_plan_info(dgrad_plan_t plan, dgrad_plan_info_t *info) {
    if (!plan || !info) return DGRAD_ERR_INVALID_ARG;
    fill_info(plan->g, plan->t, plan->precision, plan->workspace_bytes, info);
    return DGRAD_OK;
}

dgrad_status_t dgrad_run(dgrad_plan_t plan, const float *grad_out, const float *weight, float *grad_input,
                         void *stream) {
    return dgrad_run_fused(plan, grad_out, weight, grad_input, nullptr, 0, stream);
}

dgrad_status_t dgrad_run_fused(dgrad_plan_t plan, const float *grad_out, const float *weight, float *grad_input,
                               const float *relu_in, int accumulate, void *stream) {
    if (!plan || (accumulate != 0 && accumulate != 1)) return DGRAD_ERR_INVALID_ARG;
    if (!aligned16(grad_out) || !aligned16(weight) || !aligned16(grad_input)) return DGRAD_ERR_MISALIGNED;
    if (relu_in && !aligned16(relu_in)) return DGRAD_ERR_MISALIGNED;
    const Geometry &g = plan->g;
    const size_t gi_bytes = gi_elems(g) * 4;
    if (overlaps(grad_input, gi_bytes, grad_out, go_elems(g) * 4) ||
        overlaps(grad_input, gi_bytes, weight, w_elems(g) * 4) ||
        (relu_in && overlaps(grad_input, gi_bytes, relu_in, gi_bytes)))
        return DGRAD_ERR_ALIAS;
    dgrad_status_t st = check_device(plan);
    if (st != DGRAD_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (g.n_taps == 0) {   // no term reaches any input element: dgrad is all zeros
        plan->packed = 1;
        return accumulate ? DGRAD_OK : cuda_status(cudaMemsetAsync(grad_input, 0, gi_bytes, s));
    }
    st = launch_pack_on(plan, weight, grad_out, s);
    if (st != DGRAD_OK) return st;
    return launch_main_on(plan, grad_out, grad_input, s, relu_in, accumulate);
}

dgrad_status_t dgrad_prepack(dgrad_plan_t plan, const float *weight, void *stream) {
    if (!plan) return DGRAD_ERR_INVALID_ARG;
    if (!aligned16(weight)) return DGRAD_ERR_MISALIGNED;
    dgrad_status_t st = check_device(plan);
    if (st != DGRAD_OK) return st;
    if (plan->g.n_taps == 0) {
        plan->packed = 1;
        return DGRAD_OK;
    }
    return launch_pack_on(plan, weight, nullptr, static_cast<cudaStream_t>(stream));
}

dgrad_status_t dgrad_run_packed(dgrad_plan_t plan, const float *grad_out, float *grad_input, void *stream) {
    if (!plan || !plan->packed) return DGRAD_ERR_INVALID_ARG;
    dgrad_status_t st = dgrad_pack_grad_out(plan, grad_out, stream);
    if (st != DGRAD_OK) return st;
    return dgrad_run_main(plan, grad_out, grad_input, stream);
}

dgrad_status_t dgrad_pack_grad_out(dgrad_plan_t plan, const float *grad_out, void *stream) {
    if (!plan) return DGRAD_ERR_INVALID_ARG;
    if (!aligned16(grad_out)) return DGRAD_ERR_MISALIGNED;
    dgrad_status_t st = check_device(plan);
    if (st != DGRAD_OK) return st;
    if (!plan->frame || plan->g.n_taps == 0) return DGRAD_OK;
    st = launch_pack_on(plan, nullptr, grad_out, static_cast<cudaStream_t>(stream));
    if (st == DGRAD_OK) plan->frame_packed = 1;
    return st;
}

dgrad_status_t dgrad_run_main(dgrad_plan_t plan, const float *grad_out, float *grad_input, void *stream) {
    if (!plan || !plan->packed) return DGRAD_ERR_INVALID_ARG;
    if (!aligned16(grad_out) || !aligned16(grad_input)) return DGRAD_ERR_MISALIGNED;
    const Geometry &g = plan->g;
    const size_t gi_bytes = gi_elems(g) * 4;
    if (overlaps(grad_input, gi_bytes, grad_out, go_elems(g) * 4)) return DGRAD_ERR_ALIAS;
    dgrad_status_t st = check_device(plan);
    if (st != DGRAD_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (g.n_taps == 0)
        return cuda_status(cudaMemsetAsync(grad_input, 0, gi_bytes, s));
    if (plan->frame && !plan->frame_packed) return DGRAD_ERR_INVALID_ARG;
    return launch_main_on(plan, grad_out, grad_input, s);
}

dgrad_status_t dgrad_run_host(dgrad_plan_t plan, const float *grad_out_host, const float *weight_host,
                              float *grad_input_host, void *stream) {
    if (!plan) return DGRAD_ERR_INVALID_ARG;
    if (!grad_out_host || !weight_host || !grad_input_host) return DGRAD_ERR_MISALIGNED;
    dgrad_status_t st = check_device(plan);
    if (st != DGRAD_OK) return st;
    const Geometry &g = plan->g;
    const size_t go_b = go_elems(g) * 4, w_b = w_elems(g) * 4, gi_b = gi_elems(g) * 4;
    // Staging: one 256-byte aligned slot per batch chunk for grad_out and for
    // grad_input (every device pointer a run gets is aligned), and the weights.
    const size_t go_img = go_b / g.N, gi_img = gi_b / g.N;
    const int chunk_n = (g.N + kHostChunks - 1) / kHostChunks;
    const int nck = (g.N + chunk_n - 1) / chunk_n;
    auto up = [](size_t b) { return (b + 255) & ~size_t(255); };
    const size_t go_slot = up(chunk_n * go_img), gi_slot = up(chunk_n * gi_img);
    if (!plan->stage_go) {
        void *m = nullptr;
        if (cudaMalloc(&m, nck * go_slot + up(w_b) + nck * gi_slot) != cudaSuccess) {
            cudaGetLastError();
            return DGRAD_ERR_OOM;
        }
        plan->stage_go = static_cast<float *>(m);
        plan->stage_w = reinterpret_cast<float *>(static_cast<uint8_t *>(m) + nck * go_slot);
        plan->stage_gi = reinterpret_cast<float *>(static_cast<uint8_t *>(m) + nck * go_slot + up(w_b));
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (g.N < 2) {   // one image: copy in, run, copy out
        if (cudaMemcpyAsync(plan->stage_go, grad_out_host, go_b, cudaMemcpyHostToDevice, s) != cudaSuccess ||
            cudaMemcpyAsync(plan->stage_w, weight_host, w_b, cudaMemcpyHostToDevice, s) != cudaSuccess)
            return cuda_status(cudaGetLastError());
        st = dgrad_run(plan, plan->stage_go, plan->stage_w, plan->stage_gi, stream);
        if (st != DGRAD_OK) return st;
        if (cudaMemcpyAsync(grad_input_host, plan->stage_gi, gi_b, cudaMemcpyDeviceToHost, s) != cudaSuccess)
            return cuda_status(cudaGetLastError());
        return cuda_status(cudaStreamSynchronize(s));
    }
    if (!plan->host_ready && (st = make_host_pipeline(plan)) != DGRAD_OK) return st;
    // Chunk i: copy in on h2d, run on the caller's stream once its copy is
    // there, copy out on d2h once its run is done; the copy engines of the
    // two directions and the SMs work on different chunks at the same time.
    // Every input copy is queued first, so that the host-to-device engine
    // never waits for the host to queue the runs.
    cudaError_t e = cudaMemcpyAsync(plan->stage_w, weight_host, w_b, cudaMemcpyHostToDevice, plan->h2d);
    for (int i = 0; e == cudaSuccess && i < nck; ++i) {
        const int n0 = i * chunk_n, nn = std::min(chunk_n, g.N - n0);
        uint8_t *dgo = reinterpret_cast<uint8_t *>(plan->stage_go) + i * go_slot;
        e = cudaMemcpyAsync(dgo, reinterpret_cast<const uint8_t *>(grad_out_host) + n0 * go_img, nn * go_img,
                            cudaMemcpyHostToDevice, plan->h2d);
        if (e == cudaSuccess) e = cudaEventRecord(plan->ev_in[i], plan->h2d);
    }
    for (int i = 0; e == cudaSuccess && i < nck; ++i) {
        const int n0 = i * chunk_n, nn = std::min(chunk_n, g.N - n0);
        dgrad_plan_s *sp = plan->sub[nn == chunk_n ? 0 : 1];
        uint8_t *dgo = reinterpret_cast<uint8_t *>(plan->stage_go) + i * go_slot;
        uint8_t *dgi = reinterpret_cast<uint8_t *>(plan->stage_gi) + i * gi_slot;
        e = cudaStreamWaitEvent(s, plan->ev_in[i], 0);
        if (e != cudaSuccess) break;
        st = dgrad_run(sp, reinterpret_cast<const float *>(dgo), plan->stage_w, reinterpret_cast<float *>(dgi), stream);
        if (st != DGRAD_OK) {
            cudaStreamSynchronize(plan->h2d);
            cudaStreamSynchronize(plan->d2h);
            return st;
        }
        e = cudaEventRecord(plan->ev_out[i], s);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(plan->d2h, plan->ev_out[i], 0);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(reinterpret_cast<uint8_t *>(grad_input_host) + n0 * gi_img, dgi, nn * gi_img,
                                cudaMemcpyDeviceToHost, plan->d2h);
    }
    // The sub-plans' error words ride behind the last output copy (which
    // waits for every run), so no extra synchronisation reads them.
    for (int i = 0; e == cudaSuccess && i < 2; ++i)
        if (plan->sub[i])
            e = cudaMemcpyAsync(&plan->host_err[i], plan->sub[i]->err, sizeof(uint32_t), cudaMemcpyDeviceToHost,
                                plan->d2h);
    const cudaError_t e1 = cudaStreamSynchronize(plan->h2d);
    const cudaError_t e2 = cudaStreamSynchronize(plan->d2h);
    const cudaError_t e3 = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_status(e);
    if (e1 != cudaSuccess) return cuda_status(e1);
    if (e2 != cudaSuccess) return cuda_status(e2);
    if (e3 != cudaSuccess) return cuda_status(e3);
    // a bounded wait that ran out in a sub-plan's kernels is reported here
    for (int i = 0; i < 2; ++i)
        if (plan->sub[i] && plan->host_err[i] != 0) {
            plan->host_err[i] = 0;
            if (cudaMemset(plan->sub[i]->err, 0, sizeof(uint32_t)) != cudaSuccess) return cuda_status(cudaGetLastError());
            return DGRAD_ERR_DEVICE_TIMEOUT;
        }
    return DGRAD_OK;
}

dgrad_status_t dgrad_plan_check(dgrad_plan_t plan) {
    if (!plan) return DGRAD_ERR_INVALID_ARG;
    uint32_t word = 0;
    if (cudaMemcpy(&word, plan->err, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return DGRAD_ERR_CUDA;
    if (word == 0) return DGRAD_OK;
    if (cudaMemset(plan->err, 0, sizeof(word)) != cudaSuccess) return DGRAD_ERR_CUDA;
    return DGRAD_ERR_DEVICE_TIMEOUT;
}

void dgrad_plan_destroy(dgrad_plan_t plan) {
    if (!plan) return;
    int cur = -1;
    cudaGetDevice(&cur);
    if (cur != plan->device) cudaSetDevice(plan->device);
    cudaDeviceSynchronize();
    cudaFree(plan->err);
    if (plan->stage_go) cudaFree(plan->stage_go);
    for (int i = 0; i < kHostChunks; ++i) {
        if (plan->ev_in[i]) cudaEventDestroy(plan->ev_in[i]);
        if (plan->ev_out[i]) cudaEventDestroy(plan->ev_out[i]);
    }
    if (plan->h2d) cudaStreamDestroy(plan->h2d);
    if (plan->d2h) cudaStreamDestroy(plan->d2h);
    if (plan->host_err) cudaFreeHost(plan->host_err);
    for (int i = 0; i < 2; ++i)
        if (plan->sub[i]) dgrad_plan_destroy(plan->sub[i]);
    if (cur >= 0 && cur != plan->device) cudaSetDevice(cur);
    delete plan;
}

}  // extern "C"

// C ABI of the weight gradient (declared in include/wgrad.h): plan geometry,
// workspace, tensor maps and the three launches.
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cstdint>
#include <cstring>
#include <new>

#include "wgrad.h"
#include "wgrad_internal.h"

struct wgrad_plan_s {
    int device;
    dgrad::WgradGeometry g;
    dgrad::WgradMainParams mp;
    dgrad::WgradPackParams pp;
    dgrad::WgradReduceParams rp;
    uint32_t *err;
    float *gf, *xc, *part;
    size_t workspace_bytes;
};

namespace dgrad {

namespace {

constexpr int kWgSplitChunks = 12;      // longest K range of one split-precision unit, in 32-position chunks
constexpr int kWgBarrierBytes = 2048;   // barrier block + alignment slack of the stage ring
constexpr long long kWgTimeoutNs = 1000000000LL;

int ceil_div(int a, int b) { return (a + b - 1) / b; }
int round_up(int a, int b) { return ceil_div(a, b) * b; }
int floor_div(int a, int b) { return a >= 0 ? a / b : -((-a + b - 1) / b); }
int pow2_at_least(int v) {
    int p = 32;
    while (p < v) p *= 2;
    return p;
}

size_t align256(size_t b) { return (b + 255) & ~size_t(255); }

}  // namespace

dgrad_status_t make_wgrad_geometry(int N, int Ci, int H, int W, int Co, int kH, int kW, int stride, int pad_h,
                                   int pad_w, int precision, int sm_count, WgradGeometry *out) {
    if (N < 1 || Ci < 1 || H < 1 || W < 1 || Co < 1 || kH < 1 || kW < 1 || stride < 1 || pad_h < 0 || pad_w < 0)
        return DGRAD_ERR_INVALID_ARG;
    if (precision != DGRAD_PREC_FP32 && precision != DGRAD_PREC_TF32 && precision != DGRAD_PREC_TF32X3)
        return DGRAD_ERR_INVALID_ARG;
    const long long nh = (long long)H + 2LL * pad_h - kH, nw = (long long)W + 2LL * pad_w - kW;
    if (nh < 0 || nw < 0) return DGRAD_ERR_INVALID_ARG;
    if (precision == DGRAD_PREC_FP32) return DGRAD_ERR_UNSUPPORTED;
    if (stride > kWgMaxRowPhases || (long long)kH * kW > kMaxTaps) return DGRAD_ERR_UNSUPPORTED;
    if (sm_count < 1) sm_count = 148;
    WgradGeometry g;
    std::memset(&g, 0, sizeof(g));
    g.N = N; g.Ci = Ci; g.H = H; g.W = W; g.Co = Co; g.kH = kH; g.kW = kW;
    g.s = stride; g.ph = pad_h; g.pw = pad_w;
    g.split = precision == DGRAD_PREC_TF32X3 ? 1 : 0;
    const int halves = g.split ? 2 : 1;
    g.oH = (int)(nh / stride) + 1;
    g.oW = (int)(nw / stride) + 1;
    g.Wf = round_up(g.oW, 4);
    if ((long long)g.oH * g.Wf > INT_MAX / 2) return DGRAD_ERR_UNSUPPORTED;
    g.Kimg = round_up(g.oH * g.Wf, 32);
    g.cpi = g.Kimg / 32;
    // Row decomposition of the taps: kh - ph = s*dh + rh.
    int dh_min = INT_MAX, dh_max = INT_MIN;
    int dh_of[kMaxTaps], rhi_of[kMaxTaps];
    g.n_rh = 0;
    for (int kh = 0; kh < kH; ++kh) {
        const int e = kh - pad_h;
        const int dh = floor_div(e, stride), rh = e - dh * stride;
        int idx = -1;
        for (int i = 0; i < g.n_rh; ++i)
            if (g.rh_list[i] == rh) idx = i;
        if (idx < 0) {
            idx = g.n_rh;
            g.rh_list[g.n_rh++] = rh;
        }
        dh_of[kh] = dh;
        rhi_of[kh] = idx;
        dh_min = std::min(dh_min, dh);
        dh_max = std::max(dh_max, dh);
    }
    g.Ty = std::max(0, -dh_min);
    const long long lx = (long long)g.Kimg + (long long)(dh_max + g.Ty) * g.Wf;
    if (lx > INT_MAX / 2) return DGRAD_ERR_UNSUPPORTED;
    g.Lx = (int)lx;
    g.n_copies = kW * g.n_rh;
    g.taps = kH * kW;
    for (int kh = 0; kh < kH; ++kh)
        for (int kw = 0; kw < kW; ++kw) {
            const int t = kh * kW + kw;
            g.tap_copy[t] = kw * g.n_rh + rhi_of[kh];
            g.tap_off[t] = (dh_of[kh] + g.Ty) * g.Wf;
        }
    // Row tiles: (tap, input-channel block) segments of seg_rows rows.
    g.seg_rows = std::min(128, round_up(Ci, 8));
    g.cpt = ceil_div(Ci, g.seg_rows);
    g.n_segs = g.taps * g.cpt;
    if (g.n_segs > kWgMaxSegs) return DGRAD_ERR_UNSUPPORTED;
    g.spt = 128 / g.seg_rows;
    g.n_mt = ceil_div(g.n_segs, g.spt);
    // Column tiles of output channels (MMA N <= 256).
    g.n_nt = ceil_div(Co, 256);
    g.bn = round_up(ceil_div(Co, g.n_nt), 16);
    // K splits.  A CTA runs units w = blockIdx.x, + grid, ...; the slowest CTA
    // runs ceil(units / grid) units of up to cps chunks each, plus about two
    // chunks' worth of time per unit for its partial tile, so the split count
    // minimises ceil(tiles * n_ks / sm) * (cps + 2) (ties: fewer splits), with
    // units of at least 8 chunks and at most eight waves of them.
    const long long total_chunks = (long long)N * g.cpi;
    if (total_chunks > INT_MAX / 2) return DGRAD_ERR_UNSUPPORTED;
    g.total_chunks = (int)total_chunks;
    const int tiles = g.n_mt * g.n_nt;
    // Split precision: the tensor cores' fp32 accumulation loses accuracy about
    // in proportion to the number of MMAs accumulated into one accumulator
    // (measured near 2e-8 relative error per MMA on random data), so a unit
    // takes at most kWgSplitChunks chunks (12 MMAs each) and the rest of the
    // sum goes to the fp32 reduction of the partial tiles.
    const int ks_lo = g.split ? ceil_div(g.total_chunks, kWgSplitChunks) : 1;
    const int ks_hi = std::max(ks_lo, std::min(std::max(1, g.total_chunks / 8), ceil_div(8 * sm_count, tiles)));
    long long best_cost = -1;
    int n_ks = ks_lo;
    for (int k = ks_lo; k <= ks_hi; ++k) {
        const int cps = ceil_div(g.total_chunks, k);
        if (ceil_div(g.total_chunks, cps) != k) continue;   // the same split as a smaller count
        const long long cost = (long long)ceil_div(tiles * k, sm_count) * (cps + 2);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            n_ks = k;
        }
    }
    g.cps = ceil_div(g.total_chunks, n_ks);
    g.n_ks = ceil_div(g.total_chunks, g.cps);
    const long long units = (long long)tiles * g.n_ks;
    if (units > INT_MAX / 2) return DGRAD_ERR_UNSUPPORTED;
    g.n_units = (int)units;
    g.grid = std::min(g.n_units, sm_count);
    const int stage_bytes = halves * (128 * 128 + g.bn * 128);
    g.stages = std::min(kWgMaxStages, (kMaxSmem - kWgBarrierBytes) / stage_bytes);
    if (g.stages < 2) return DGRAD_ERR_UNSUPPORTED;
    g.smem_bytes = kWgBarrierBytes + g.stages * stage_bytes;
    g.tmem_cols = pow2_at_least(2 * g.bn);
    g.g_elems = (size_t)halves * N * Co * g.Kimg;
    g.x_elems = (size_t)halves * g.n_copies * N * Ci * g.Lx;
    if ((g.g_elems + g.x_elems) / 4 > (size_t)INT_MAX) return DGRAD_ERR_UNSUPPORTED;   // 32-bit pack indices
    g.part_elems = (size_t)g.n_units * g.bn * 128;
    *out = g;
    return DGRAD_OK;
}

}  // namespace dgrad

namespace {

using dgrad::WgradGeometry;

void fill_wgrad_info(const WgradGeometry &g, size_t ws, wgrad_plan_info_t *info) {
    std::memset(info, 0, sizeof(*info));
    info->N = g.N; info->Ci = g.Ci; info->H = g.H; info->W = g.W; info->Co = g.Co;
    info->kH = g.kH; info->kW = g.kW; info->stride = g.s; info->pad_h = g.ph; info->pad_w = g.pw;
    info->oH = g.oH; info->oW = g.oW;
    info->precision = g.split ? DGRAD_PREC_TF32X3 : DGRAD_PREC_TF32;
    info->Wf = g.Wf; info->Kimg = g.Kimg; info->Lx = g.Lx; info->n_copies = g.n_copies;
    info->seg_rows = g.seg_rows; info->n_mt = g.n_mt; info->n_nt = g.n_nt; info->n_ks = g.n_ks;
    info->slice_n = g.bn; info->n_units = g.n_units; info->grid = g.grid; info->stages = g.stages;
    info->smem_bytes = g.smem_bytes; info->tmem_cols = g.tmem_cols;
    info->workspace_bytes = ws;
    info->useful_flops = 2.0 * g.N * g.Co * g.oH * g.oW * (double)g.Ci * g.kH * g.kW;
    info->algorithmic_bytes =
        4.0 * ((double)g.N * g.Co * g.oH * g.oW + (double)g.N * g.Ci * g.H * g.W + (double)g.Co * g.Ci * g.kH * g.kW);
}

size_t workspace_of(const WgradGeometry &g) {
    return 256 + dgrad::align256(g.g_elems * 4) + dgrad::align256(g.x_elems * 4) + dgrad::align256(g.part_elems * 4);
}

dgrad_status_t wcuda(cudaError_t e) { return dgrad::cuda_status(e); }

bool wal16(const void *p) { return p != nullptr && ((uintptr_t)p & 15u) == 0; }
bool woverlap(const void *a, size_t an, const void *b, size_t bn) {
    const uintptr_t a0 = (uintptr_t)a, a1 = a0 + an, b0 = (uintptr_t)b, b1 = b0 + bn;
    return a0 < b1 && b0 < a1;
}

dgrad_status_t encode_maps(wgrad_plan_s *pl) {
    auto fn = dgrad::tensor_map_encoder();
    if (!fn) return DGRAD_ERR_CUDA;
    const WgradGeometry &g = pl->g;
    const cuuint32_t es4[4] = {1u, 1u, 1u, 1u};
    {
        const cuuint64_t dims[4] = {(cuuint64_t)g.Lx, (cuuint64_t)g.Ci, (cuuint64_t)g.N,
                                    (cuuint64_t)g.n_copies * (g.split ? 2 : 1)};
        const cuuint64_t strides[3] = {(cuuint64_t)g.Lx * 4, (cuuint64_t)g.Lx * 4 * g.Ci,
                                       (cuuint64_t)g.Lx * 4 * g.Ci * g.N};
        const cuuint32_t box[4] = {32u, (cuuint32_t)g.seg_rows, 1u, 1u};
        if (fn(&pl->mp.x_map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, pl->xc, dims, strides, box, es4,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return DGRAD_ERR_CUDA;
    }
    {
        const cuuint64_t dims[3] = {(cuuint64_t)g.Kimg, (cuuint64_t)g.Co, (cuuint64_t)g.N * (g.split ? 2 : 1)};
        const cuuint64_t strides[2] = {(cuuint64_t)g.Kimg * 4, (cuuint64_t)g.Kimg * 4 * g.Co};
        const cuuint32_t box[3] = {32u, (cuuint32_t)g.bn, 1u};
        if (fn(&pl->mp.g_map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, pl->gf, dims, strides, box, es4,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return DGRAD_ERR_CUDA;
    }
    return DGRAD_OK;
}

void fill_wgrad_params(wgrad_plan_s *pl) {
    const WgradGeometry &g = pl->g;
    dgrad::WgradMainParams &m = pl->mp;
    m.part = pl->part;
    m.err = pl->err;
    m.n_mt = g.n_mt; m.n_nt = g.n_nt; m.n_ks = g.n_ks; m.n_units = g.n_units; m.bn = g.bn;
    m.seg_rows = g.seg_rows; m.spt = g.spt; m.n_segs = g.n_segs; m.cpi = g.cpi;
    m.total_chunks = g.total_chunks; m.cps = g.cps; m.stages = g.stages; m.tmem_cols = g.tmem_cols;
    m.idesc = dgrad::tf32_idesc(128, g.bn);
    m.split = g.split; m.N = g.N; m.n_copies = g.n_copies;
    m.timeout_ns = dgrad::kWgTimeoutNs;
    for (int sidx = 0; sidx < g.n_segs; ++sidx) {
        const int t = sidx / g.cpt;
        m.seg[sidx] = make_int4(g.tap_copy[t], (sidx - t * g.cpt) * g.seg_rows, g.tap_off[t], 0);
    }
    dgrad::WgradPackParams &q = pl->pp;
    q.gf = pl->gf; q.xc = pl->xc;
    q.N = g.N; q.Ci = g.Ci; q.H = g.H; q.W = g.W; q.Co = g.Co; q.oH = g.oH; q.oW = g.oW;
    q.s = g.s; q.pw = g.pw; q.Wf = g.Wf; q.Kimg = g.Kimg; q.Lx = g.Lx; q.Ty = g.Ty; q.n_rh = g.n_rh;
    for (int i = 0; i < dgrad::kWgMaxRowPhases; ++i) q.rh_list[i] = g.rh_list[i];
    q.split = g.split;
    q.g4 = (long long)(g.g_elems / 4 / (g.split ? 2 : 1));
    q.x4 = (long long)(g.x_elems / 4 / (g.split ? 2 : 1));
    dgrad::WgradReduceParams &r = pl->rp;
    r.part = pl->part;
    r.Co = g.Co; r.Ci = g.Ci; r.taps = g.taps; r.bn = g.bn; r.n_mt = g.n_mt; r.n_nt = g.n_nt; r.n_ks = g.n_ks;
    r.seg_rows = g.seg_rows; r.cpt = g.cpt; r.spt = g.spt; r.n_segs = g.n_segs;
    r.total = (long long)g.n_mt * g.n_nt * g.bn * 128;
}

}  // namespace

extern "C" {

dgrad_status_t wgrad_describe(int N, int Ci, int H, int W, int Co, int kH, int kW, int stride, int pad_h,
                              int pad_w, dgrad_precision_t precision, int sm_count, wgrad_plan_info_t *info) {
    if (!info) return DGRAD_ERR_INVALID_ARG;
    WgradGeometry g;
    dgrad_status_t st =
        dgrad::make_wgrad_geometry(N, Ci, H, W, Co, kH, kW, stride, pad_h, pad_w, precision, sm_count, &g);
    if (st != DGRAD_OK) return st;
    fill_wgrad_info(g, workspace_of(g), info);
    return DGRAD_OK;
}

dgrad_status_t wgrad_describe_taps(int N, int Ci, int H, int W, int Co, int kH, int kW, int stride, int pad_h,
                                   int pad_w, int cap, int *copy, int *offset, int *copy_kw, int *copy_rh,
                                   int *n_copies, int *ty) {
    if (!copy || !offset || !copy_kw || !copy_rh || !n_copies || !ty) return DGRAD_ERR_INVALID_ARG;
    WgradGeometry g;
    dgrad_status_t st =
        dgrad::make_wgrad_geometry(N, Ci, H, W, Co, kH, kW, stride, pad_h, pad_w, DGRAD_PREC_TF32, 0, &g);
    if (st != DGRAD_OK) return st;
    if (g.taps > cap || g.n_copies > cap) return DGRAD_ERR_INVALID_ARG;
    for (int t = 0; t < g.taps; ++t) {
        copy[t] = g.tap_copy[t];
        offset[t] = g.tap_off[t];
    }
    for (int c = 0; c < g.n_copies; ++c) {
        copy_kw[c] = c / g.n_rh;
        copy_rh[c] = g.rh_list[c % g.n_rh];
    }
    *n_copies = g.n_copies;
    *ty = g.Ty;
    return DGRAD_OK;
}

dgrad_status_t wgrad_plan(int N, int Ci, int H, int W, int Co, int kH, int kW, int stride, int pad_h, int pad_w,
                          dgrad_precision_t precision, wgrad_plan_t *plan_out) {
    if (!plan_out) return DGRAD_ERR_INVALID_ARG;
    *plan_out = nullptr;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DGRAD_ERR_NO_DEVICE;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return DGRAD_ERR_NO_DEVICE;
    if (prop.major != 10 || prop.minor != 3) return DGRAD_ERR_NO_DEVICE;
    wgrad_plan_s *pl = new (std::nothrow) wgrad_plan_s;
    if (!pl) return DGRAD_ERR_OOM;
    std::memset(pl, 0, sizeof(*pl));
    pl->device = dev;
    dgrad_status_t st = dgrad::make_wgrad_geometry(N, Ci, H, W, Co, kH, kW, stride, pad_h, pad_w, precision,
                                                   prop.multiProcessorCount, &pl->g);
    if (st != DGRAD_OK) {
        delete pl;
        return st;
    }
    const size_t ws = workspace_of(pl->g);
    void *mem = nullptr;
    if (cudaMalloc(&mem, ws) != cudaSuccess) {
        cudaGetLastError();
        delete pl;
        return DGRAD_ERR_OOM;
    }
    if (cudaMemset(mem, 0, 256) != cudaSuccess || cudaStreamSynchronize(nullptr) != cudaSuccess) {
        cudaGetLastError();
        cudaFree(mem);
        delete pl;
        return DGRAD_ERR_CUDA;
    }
    uint8_t *b = static_cast<uint8_t *>(mem);
    pl->err = reinterpret_cast<uint32_t *>(b);
    pl->gf = reinterpret_cast<float *>(b + 256);
    pl->xc = reinterpret_cast<float *>(b + 256 + dgrad::align256(pl->g.g_elems * 4));
    pl->part = reinterpret_cast<float *>(b + 256 + dgrad::align256(pl->g.g_elems * 4) +
                                         dgrad::align256(pl->g.x_elems * 4));
    pl->workspace_bytes = ws;
    fill_wgrad_params(pl);
    if ((st = encode_maps(pl)) != DGRAD_OK) {
        cudaFree(mem);
        delete pl;
        return st;
    }
    *plan_out = pl;
    return DGRAD_OK;
}

dgrad_status_t wgrad_plan_info(wgrad_plan_t plan, wgrad_plan_info_t *info) {
    if (!plan || !info) return DGRAD_ERR_INVALID_ARG;
    fill_wgrad_info(plan->g, plan->workspace_bytes, info);
    return DGRAD_OK;
}

dgrad_status_t wgrad_run(wgrad_plan_t plan, const float *grad_out, const float *input, float *grad_weight,
                         void *stream) {
    if (!plan) return DGRAD_ERR_INVALID_ARG;
    if (!wal16(grad_out) || !wal16(input) || !wal16(grad_weight)) return DGRAD_ERR_MISALIGNED;
    const WgradGeometry &g = plan->g;
    const size_t go_b = (size_t)g.N * g.Co * g.oH * g.oW * 4, x_b = (size_t)g.N * g.Ci * g.H * g.W * 4;
    const size_t w_b = (size_t)g.Co * g.Ci * g.kH * g.kW * 4;
    if (woverlap(grad_weight, w_b, grad_out, go_b) || woverlap(grad_weight, w_b, input, x_b)) return DGRAD_ERR_ALIAS;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return DGRAD_ERR_CUDA;
    if (dev != plan->device) return DGRAD_ERR_WRONG_DEVICE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    plan->pp.go = grad_out;
    plan->pp.x = input;
    plan->rp.dw = grad_weight;
    dgrad_status_t st = wcuda(dgrad::launch_wgrad_pack(plan->pp, s));
    if (st != DGRAD_OK) return st;
    st = wcuda(dgrad::launch_wgrad_main(plan->mp, g.grid, g.smem_bytes, s));
    if (st != DGRAD_OK) return st;
    return wcuda(dgrad::launch_wgrad_reduce(plan->rp, s));
}

dgrad_status_t wgrad_plan_check(wgrad_plan_t plan) {
    if (!plan) return DGRAD_ERR_INVALID_ARG;
    uint32_t word = 0;
    if (cudaMemcpy(&word, plan->err, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return DGRAD_ERR_CUDA;
    if (word == 0) return DGRAD_OK;
    if (cudaMemset(plan->err, 0, sizeof(word)) != cudaSuccess) return DGRAD_ERR_CUDA;
    return DGRAD_ERR_DEVICE_TIMEOUT;
}

void wgrad_plan_destroy(wgrad_plan_t plan) {
    if (!plan) return;
    int cur = -1;
    cudaGetDevice(&cur);
    if (cur != plan->device) cudaSetDevice(plan->device);
    cudaDeviceSynchronize();
    cudaFree(plan->err);
    if (cur >= 0 && cur != plan->device) cudaSetDevice(cur);
    delete plan;
}

}  // extern "C"

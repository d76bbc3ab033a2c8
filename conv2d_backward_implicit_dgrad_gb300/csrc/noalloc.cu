// dgrad_run_noalloc: the whole dgrad (weight pre-pack + main kernel) without
// any allocation, for callers that may not allocate device memory.
//
// The packed weights and the device error word live in one file-scope
// __device__ array, so each GPU that loads this library holds
// kNoAllocScratchBytes for the life of the process.  Host code never uses
// the array's name as a device pointer: on the first call on a device, with
// that device current, cudaGetSymbolAddress gives the array's device address,
// which is cached per device and handed to the kernels.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "dgrad.h"
#include "dgrad_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;   // 4 MiB per device
constexpr size_t kErrWordBytes = 256;                       // error word, then packed weights
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mutex;
void *g_scratch_addr[kMaxDevices];   // device address of g_noalloc_scratch, per device

dgrad_status_t scratch_address(int dev, unsigned char **out) {
    if (dev < 0 || dev >= kMaxDevices) return DGRAD_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return DGRAD_ERR_CUDA;
        }
        g_scratch_addr[dev] = p;
    }
    *out = static_cast<unsigned char *>(g_scratch_addr[dev]);
    return DGRAD_OK;
}

bool ranges_overlap(const void *a, size_t na, const void *b, size_t nb) {
    uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
    return a0 < b0 + nb && b0 < a0 + na;
}

bool is_aligned16(const void *p) { return p != nullptr && ((uintptr_t)p & 15u) == 0; }

}  // namespace

extern "C" dgrad_status_t dgrad_run_noalloc(int N, int Ci, int H, int W, int Co, int kH, int kW, int stride,
                                            int pad_h, int pad_w, dgrad_precision_t precision,
                                            const float *grad_out, const float *weight, float *grad_input,
                                            void *stream) {
    using namespace dgrad;
    if (precision != DGRAD_PREC_FP32 && precision != DGRAD_PREC_TF32) return DGRAD_ERR_INVALID_ARG;
    Geometry g;
    dgrad_status_t st = make_geometry(N, Ci, H, W, Co, kH, kW, stride, pad_h, pad_w, &g);
    if (st != DGRAD_OK) return st;

    int dev = -1, major = 0, minor = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DGRAD_ERR_NO_DEVICE;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return DGRAD_ERR_NO_DEVICE;
    if (major != 10 || minor != 3) return DGRAD_ERR_NO_DEVICE;

    // No frame buffer here: producer warps carry grad_out to the MMA.
    dgrad_options_t opts{};
    opts.a_source = 2;
    Tiling t;
    st = choose_tiling(g, precision, &opts, sms, &t);
    if (st != DGRAD_OK) return st;
    if (t.packed_bytes + kErrWordBytes > kNoAllocScratchBytes) return DGRAD_ERR_UNSUPPORTED;

    const size_t go_b = (size_t)N * Co * g.oH * g.oW * 4, w_b = (size_t)Co * Ci * kH * kW * 4;
    const size_t gi_b = (size_t)N * Ci * H * W * 4;
    if (!is_aligned16(grad_out) || !is_aligned16(weight) || !is_aligned16(grad_input)) return DGRAD_ERR_MISALIGNED;
    if (ranges_overlap(grad_input, gi_b, grad_out, go_b) || ranges_overlap(grad_input, gi_b, weight, w_b))
        return DGRAD_ERR_ALIAS;

    unsigned char *scratch = nullptr;
    st = scratch_address(dev, &scratch);
    if (st != DGRAD_OK) return st;
    uint32_t *err = reinterpret_cast<uint32_t *>(scratch);
    float *wp = reinterpret_cast<float *>(scratch + kErrWordBytes);
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    // The array keeps whatever the previous call left: the error word must
    // start at zero; the packed weights are rewritten in full below.
    if (cudaMemsetAsync(err, 0, sizeof(uint32_t), s) != cudaSuccess) return DGRAD_ERR_CUDA;
    if (g.n_taps == 0) return cudaMemsetAsync(grad_input, 0, gi_b, s) == cudaSuccess ? DGRAD_OK : DGRAD_ERR_CUDA;

    PrepackParams q;
    std::memset(&q, 0, sizeof(q));
    q.w = weight;
    q.wp = wp;
    q.Co = Co; q.Ci = Ci; q.kH = kH; q.kW = kW;
    q.n_taps = g.n_taps; q.bn = t.bn; q.n_slices = t.n_slices; q.kc = t.kc; q.n_chunks = t.n_chunks;
    q.round_tf32 = precision == DGRAD_PREC_TF32 ? 1 : 0;
    q.layout = t.path == DGRAD_PATH_TCGEN05 ? 1 : 0;
    q.total = (long long)(t.packed_bytes / 4);
    for (int i = 0; i < g.n_taps; ++i) {
        q.tap_kh[i] = g.tap[i].kh;
        q.tap_kw[i] = g.tap[i].kw;
    }

    MainParams m;
    std::memset(&m, 0, sizeof(m));
    m.go = grad_out; m.wp = wp; m.gi = grad_input; m.err = err;
    m.N = N; m.Ci = Ci; m.Co = Co; m.H = H; m.W = W; m.oH = g.oH; m.oW = g.oW; m.s = stride;
    m.Ph = g.Ph; m.Pw = g.Pw; m.Hv = g.Hv; m.Wp = g.Wp; m.HvWp = g.Hv * g.Wp;
    m.positions = (int)g.positions;
    m.tm = t.tm; m.bn = t.bn; m.n_slices = t.n_slices; m.kc = t.kc; m.n_chunks = t.n_chunks;
    m.n_tiles = t.n_tiles; m.n_work = (int)t.n_work;
    m.a_rows = t.a_rows; m.a_stages = t.a_stages; m.b_stages = t.b_stages; m.b_resident = t.b_resident;
    m.chunk_bytes = t.chunk_bytes;
    m.tap_group = t.tap_group; m.n_tgroups = t.n_tgroups;
    m.vec_producer = dgrad::use_vec_producer(g, t) ? 1 : 0;
    m.acc_bufs = t.acc_bufs; m.acc_cols = t.acc_cols; m.tmem_cols = t.tmem_cols;
    m.round_tf32 = q.round_tf32;
    m.n_phases = g.n_phases; m.n_taps = g.n_taps;
    m.idesc = tf32_idesc(kBlockM, t.bn);
    m.timeout_ns = 1000000000LL;
    for (int i = 0; i < g.n_phases; ++i) m.phase[i] = g.phase[i];
    for (int i = 0; i < g.n_taps; ++i) m.tap[i] = g.tap[i];

    if (launch_prepack(q, s) != cudaSuccess) return DGRAD_ERR_CUDA;
    cudaError_t e = t.path == DGRAD_PATH_TCGEN05 ? launch_tc(m, t, s, true) : launch_simt(m, t, s);
    return e == cudaSuccess ? DGRAD_OK : DGRAD_ERR_CUDA;
}

// dgrad_run_noalloc: the whole dgrad (weight pre-pack + main kernel) without
// any allocation, for callers that may not allocate device memory.
//
// The packed weights and the device error word live in one file-scope
// __device__ array, so each GPU that loads this library holds
// kNoAllocScratchBytes for the life of the process.  Host code never uses
// the array's name as a device pointer: on the first call on a device, with
// that device current, cudaGetSymbolAddress gives the array's device address,
// which is cached per device and handed to the kernels.  The cache does not
// survive a reset of the device (cudaDeviceReset, or the primary context
// being released and made again): the library's module is then loaded anew
// and the cached address is stale, so no call may follow such a reset in the
// same process.
//
// Every CUDA failure goes through dgrad::cuda_status, as in dgrad_run: the
// error is recorded for dgrad_cuda_error_string and the runtime's last error
// is cleared.
#include <cuda_runtime.h>

#include <cstdint>
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
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return dgrad::cuda_status(e);
        if (p == nullptr) return DGRAD_ERR_CUDA;
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
    if (precision != DGRAD_PREC_FP32 && precision != DGRAD_PREC_TF32 && precision != DGRAD_PREC_TF32X3)
        return DGRAD_ERR_INVALID_ARG;
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

    // No frame buffer here: producer warps carry grad_out to the MMA (so
    // split precision, which needs the frame, is rejected by the tiling).
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
    st = cuda_status(cudaMemsetAsync(err, 0, sizeof(uint32_t), s));
    if (st != DGRAD_OK) return st;
    if (g.n_taps == 0) return cuda_status(cudaMemsetAsync(grad_input, 0, gi_b, s));

    const int round = precision == DGRAD_PREC_TF32 ? 1 : 0;
    PrepackParams q;
    fill_prepack_params(g, t, round, &q);
    q.w = weight;
    q.wp = wp;

    MainParams m;
    fill_main_params(g, t, round, &m);
    m.go = grad_out; m.wp = wp; m.gi = grad_input; m.err = err;
    m.timeout_ns = 1000000000LL;

    st = cuda_status(launch_prepack(q, s));
    if (st != DGRAD_OK) return st;
    return cuda_status(t.path == DGRAD_PATH_TCGEN05 ? launch_tc(m, t, s, true) : launch_simt(m, t, s));
}

// Backward + SGD for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc when they run the backward pass: their
// device memory is owned by another allocator (a framework's caching
// allocator that has reserved the device, or a fixed pool handed out at
// start-up), or their rules forbid any device allocation once set-up is over
// (latency-critical serving loops).  They cannot hand tbe_backward_sgd a
// workspace of their own.  tbe_backward_sgd_noalloc runs the same kernels with
// the workspace placed in a file-scope static device array instead, so the
// call itself allocates nothing.
//
// The array has a fixed size (kStaticScratchBytes); a batch whose workspace
// would not fit is rejected before anything is launched.  Every GPU that
// loads this library keeps the array until the process exits.  All calls on a
// device share one array, so two calls whose GPU work overlaps (other
// streams, other host threads) race on it; callers must order them.
#include <nvtx3/nvToolsExt.h>

#include <mutex>

#include "../../include/tbe.h"
#include "tbe_internal.cuh"

namespace {

constexpr size_t kStaticScratchBytes = size_t(32) << 20;
constexpr int kMaxDevices = 64;

// The scratch itself.  Host code never dereferences or passes this name to a
// kernel: on the host it is only a stand-in for the symbol, and its device
// address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_tbe_scratch[kStaticScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (the first call on a device does this, with that device
// current) and cached.
int scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TBE_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return TBE_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_tbe_scratch);
        if (e != cudaSuccess || p == nullptr) return TBE_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return TBE_OK;
}

int backward_sgd_static(tbe_handle* h, const void* indices, const void* offsets, int32_t index_dtype,
                        int64_t num_indices, int32_t batch_size, const float* per_sample_weights,
                        const float* grad_out, float lr, void* stream);

}  // namespace

extern "C" int tbe_backward_sgd_noalloc(tbe_handle* h, const void* indices, const void* offsets,
                                        int32_t index_dtype, int64_t num_indices, int32_t batch_size,
                                        const float* per_sample_weights, const float* grad_out,
                                        float lr, void* stream) {
    nvtxRangePushA("tbe_backward_sgd_noalloc");
    const int rc = backward_sgd_static(h, indices, offsets, index_dtype, num_indices, batch_size,
                                       per_sample_weights, grad_out, lr, stream);
    nvtxRangePop();
    return rc;
}

namespace {

int backward_sgd_static(tbe_handle* h, const void* indices, const void* offsets, int32_t index_dtype,
                        int64_t num_indices, int32_t batch_size, const float* per_sample_weights,
                        const float* grad_out, float lr, void* stream) {
    if (!h || num_indices < 0 || batch_size < 0) return TBE_ERR_INVALID_ARG;
    // Reject a batch whose workspace does not fit before launching anything.
    const size_t need = tbe_backward_workspace_bytes(h, num_indices, batch_size);
    if (need == 0 || need > kStaticScratchBytes) return TBE_ERR_WORKSPACE_TOO_SMALL;
    void* scratch = nullptr;
    const int rc = scratch_address(&scratch);
    if (rc != TBE_OK) return rc;
    // The existing backward path clears the parts of the workspace that must
    // start at zero (the counter block, the radix digit histograms, the first
    // bag of every key tile) on `stream` before its kernels run, and its
    // kernels reset the per-run chunk counters they use, so the previous
    // call's contents do no harm.  It also refuses, before launching
    // anything, a call made while a device other than the handle's is
    // current (the scratch looked up above is then simply not used).
    return tbe_backward_sgd(h, indices, offsets, index_dtype, num_indices, batch_size,
                            per_sample_weights, grad_out, lr, scratch, kStaticScratchBytes, stream);
}

}  // namespace

// lmhead_static.cu -- spec_lmhead_argmax_static: the LM head with fused argmax, for callers
// that cannot allocate device memory.
//
// Some callers have no way to provide a workspace: an engine that hands its whole HBM budget
// to its own pool before the first step and forbids later allocations, or glue code that
// can only pass the tensors of the call (hidden rows, weight, outputs). This entry point
// runs the same kernel as spec_lmhead_argmax, with the kernel's scratch (a launch counter
// and the per-CTA argmax keys) in a file-scope device array instead of a caller workspace.
//
// The scratch array is the library's: every call on a device uses the same array, so two
// calls in flight at the same time (for instance on two streams without an ordering between
// them) race on it and may return wrong ids. Order such calls on one stream or with events.
//
// The first call on a device looks the array up and zeroes its counter (a synchronous
// cudaMemset), so that first call should be made before any stream capture; later calls on
// that device only launch. Every completed call leaves the counter at zero again.
#include <mutex>

#include "common.cuh"

namespace spec {
namespace {

// header (the launch counter, which must read zero when a call starts) + 64-bit keys for up
// to 1024 CTAs x 64 rows
constexpr size_t kScratchBytes = SPEC_LMHEAD_STATIC_SCRATCH_BYTES;
static_assert(kScratchBytes == 256 + (size_t)1024 * 64 * 8, "scratch size");
static __device__ __align__(256) unsigned char g_lmhead_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void *g_scratch_ptr[kMaxDevices];  // per device, looked up once

int scratch_of_current_device(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SPEC_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return SPEC_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_lmhead_scratch) != cudaSuccess || p == nullptr) return SPEC_ERR_CUDA;
        if (cudaMemset(p, 0, 256) != cudaSuccess) return SPEC_ERR_CUDA;  // the counter starts at zero
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return SPEC_OK;
}

}  // namespace
}  // namespace spec

SPEC_API int spec_lmhead_argmax_static(const void *hidden, const void *W, int M, int V, int H, const int32_t *d2t,
                                       int d2t_limit, int32_t *ids, float *max_logit, int32_t *dev_err,
                                       spec_stream_t stream) {
    const size_t need = spec_lmhead_workspace(M, V, H);
    if (need == 0) return SPEC_ERR_ARG;
    if (need > spec::kScratchBytes) return SPEC_ERR_WORKSPACE;  // more rows x CTAs than the scratch holds
    void *scratch = nullptr;
    const int st = spec::scratch_of_current_device(&scratch);
    if (st) return st;
    return spec_lmhead_argmax(hidden, W, M, V, H, d2t, d2t_limit, ids, max_logit, scratch, spec::kScratchBytes,
                              dev_err, stream);
}

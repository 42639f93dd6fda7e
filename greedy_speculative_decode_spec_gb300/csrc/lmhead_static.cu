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
// Every call looks the array up in the current context (cudaGetSymbolAddress allocates
// nothing); the first call in a context, or after the module was reloaded there (a device
// reset), zeroes its counter with a synchronous cudaMemset, so that call should be made
// before any stream capture; later calls only launch. Every completed call leaves the counter
// and the keys at zero again.
#include <cuda.h>

#include <mutex>

#include "common.cuh"

namespace spec {
namespace {

// header (the launch counter, which must read zero when a call starts) + 64-bit keys for up
// to 1024 CTAs x 64 rows
constexpr size_t kScratchBytes = SPEC_LMHEAD_STATIC_SCRATCH_BYTES;
static_assert(kScratchBytes == 256 + (size_t)1024 * 64 * 8, "scratch size");
static __device__ __align__(256) unsigned char g_lmhead_scratch[kScratchBytes];

// contexts seen so far and the scratch address each had when its counter was zeroed
constexpr int kMaxContexts = 64;
std::mutex g_setup_mu;
struct Seen {
    CUcontext ctx;
    void *ptr;
};
Seen g_seen[kMaxContexts];
int g_n_seen = 0;

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
CtxGetCurrentFn ctx_get_current() {
    static CtxGetCurrentFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(f);
    }
    return fn;
}

int scratch_of_current_context(void **out) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_lmhead_scratch) != cudaSuccess || p == nullptr) return SPEC_ERR_CUDA;
    CtxGetCurrentFn get = ctx_get_current();
    CUcontext ctx = nullptr;
    if (!get || get(&ctx) != CUDA_SUCCESS || ctx == nullptr) return SPEC_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mu);
    int i = 0;
    while (i < g_n_seen && g_seen[i].ctx != ctx) ++i;
    if (i == g_n_seen || g_seen[i].ptr != p) {  // a new context, or the module was reloaded in it
        if (cudaMemset(p, 0, kScratchBytes) != cudaSuccess) return SPEC_ERR_CUDA;
        if (i == g_n_seen) {
            if (g_n_seen == kMaxContexts) return SPEC_ERR_UNSUPPORTED;
            ++g_n_seen;
        }
        g_seen[i].ctx = ctx;
        g_seen[i].ptr = p;
    }
    *out = p;
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
    const int st = spec::scratch_of_current_context(&scratch);
    if (st) return st;
    return spec_lmhead_argmax(hidden, W, M, V, H, d2t, d2t_limit, ids, max_logit, scratch, spec::kScratchBytes,
                              dev_err, stream);
}

// common.cuh -- helpers shared by the kernels of libspecverify (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "spec_verify.h"

#define SPEC_API extern "C" __attribute__((visibility("default")))

namespace spec {

// ---- host side -----------------------------------------------------------------------

inline int launch_status() {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

// Launches `kernel` so that it may be scheduled while the kernel before it in the stream is
// still finishing (programmatic dependent launch): the kernel must call grid_dep_wait()
// before it reads anything an earlier kernel wrote. Falls back to an ordinary launch where
// the attribute is not available.
template <typename... KArgs, typename... Args>
inline int launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...) == cudaSuccess) return SPEC_OK;
    (void)cudaGetLastError();
    kernel<<<grid, block, smem, s>>>(static_cast<KArgs>(args)...);
    return launch_status();
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

inline int log2i(int x) {
    int r = 0;
    while ((1 << r) < x) ++r;
    return r;
}

// Validates a pool descriptor; returns SPEC_OK or an error code.
// The descriptor's shape fields (no pointer is looked at).
inline int check_kv_shape(const spec_kv_desc *kv) {
    if (!kv) return SPEC_ERR_NULL;
    if (kv->num_pages < 1 || kv->max_pages < 1 || kv->n_kv_heads < 1) return SPEC_ERR_ARG;
    if (!is_pow2(kv->page_size) || kv->page_size > 1024) return SPEC_ERR_ARG;
    if (kv->head_dim != 64 && kv->head_dim != 128 && kv->head_dim != 256) return SPEC_ERR_UNSUPPORTED;
    if (kv->kv_dtype != SPEC_KV_BF16 && kv->kv_dtype != SPEC_KV_FP8_E4M3) return SPEC_ERR_UNSUPPORTED;
    return SPEC_OK;
}

inline int check_kv_desc(const spec_kv_desc *kv) {
    if (!kv || !kv->k_pool || !kv->v_pool || !kv->page_table) return SPEC_ERR_NULL;
    const int st = check_kv_shape(kv);
    if (st) return st;
    if (kv->kv_dtype == SPEC_KV_FP8_E4M3 && (!kv->k_scale || !kv->v_scale)) return SPEC_ERR_NULL;
    if (!aligned16(kv->k_pool) || !aligned16(kv->v_pool)) return SPEC_ERR_ALIGN;
    return SPEC_OK;
}

// Plain-old-data copy of the descriptor passed to kernels by value.
struct KvView {
    void *k_pool, *v_pool;
    const float *k_scale, *v_scale;
    const int32_t *page_table;
    int num_pages, max_pages, page_size, log2_page, n_kv_heads, head_dim, kv_dtype;
};

inline KvView make_view(const spec_kv_desc *kv) {
    KvView v;
    v.k_pool = kv->k_pool;
    v.v_pool = kv->v_pool;
    v.k_scale = kv->k_scale;
    v.v_scale = kv->v_scale;
    v.page_table = kv->page_table;
    v.num_pages = kv->num_pages;
    v.max_pages = kv->max_pages;
    v.page_size = kv->page_size;
    v.log2_page = log2i(kv->page_size);
    v.n_kv_heads = kv->n_kv_heads;
    v.head_dim = kv->head_dim;
    v.kv_dtype = kv->kv_dtype;
    return v;
}

// Limit (ns) of the pipeline waits inside the tcgen05 kernels launched from now on; the
// waits that drain a kernel's own copies and MMAs before it exits always allow a second.
extern uint64_t g_wait_ns;
constexpr uint64_t DEFAULT_WAIT_NS = 1000000000ull;

// ---- device side ---------------------------------------------------------------------

__device__ __forceinline__ void raise_error(int32_t *err, int bit) {
    if (err) atomicOr(err, bit);
}

// Page holding position p of page-table row b, or a negative SPEC_DEVERR_* bit.
__device__ __forceinline__ int page_of(const KvView &kv, int b, int p) {
    if (p < 0) return -SPEC_DEVERR_POS;
    int pi = p >> kv.log2_page;
    if (pi >= kv.max_pages) return -SPEC_DEVERR_COVER;
    int pg = __ldg(kv.page_table + (size_t)b * kv.max_pages + pi);
    if (pg < 0 || pg >= kv.num_pages) return -SPEC_DEVERR_PAGE;
    return pg;
}

// Element offset of (page, kv head g, slot) in a pool.
__device__ __forceinline__ size_t pool_offset(const KvView &kv, int page, int g, int slot) {
    return (((size_t)page * kv.n_kv_heads + g) * kv.page_size + slot) * kv.head_dim;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Monotone map of a float to an unsigned key (larger float -> larger key); -0 and +0
// must be made equal by the caller (add +0.0f with round-to-nearest first).
__device__ __forceinline__ uint32_t float_key(float f) {
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_float(uint32_t k) {
    uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
    return __uint_as_float(u);
}

}  // namespace spec

// hpool.cu -- f1: the remembered hidden-row pool of the draft head.
//
// span-02 engine/crates/model/src/spec.rs, `Spec::body_inner`: each branch b owns a slot
// hslot[b] of a pool of hidden rows; a step starts by gathering h0[b] = hpool[hslot[b]] (the
// draft head's input row of the branch) and ends, after the acceptance has written the
// bonus token's hidden row into h0, by scattering it back, hpool[hslot[b]] = h0[b]. Both are
// row copies on the device, so a step captured in a CUDA graph keeps this state without a
// host round trip.
//
// One CTA per row, 16-byte copies when the row length and both bases allow them, else
// 2-byte copies. A slot outside [0, n_slots) raises SPEC_DEVERR_SLOT and its row is skipped.
#include "common.cuh"

namespace spec {

template <bool GATHER>
__global__ void __launch_bounds__(128) hpool_copy_kernel(uint16_t *dst, const uint16_t *__restrict__ src,
                                                         const int32_t *__restrict__ hslot, int H, int n_slots,
                                                         bool vec, int32_t *err) {
    const int b = blockIdx.x;
    const int s = __ldg(hslot + b);
    if (s < 0 || s >= n_slots) {
        if (threadIdx.x == 0) raise_error(err, SPEC_DEVERR_SLOT);
        return;
    }
    // gather: dst row b <- pool row s; scatter: pool row s <- src row b
    uint16_t *d = dst + (size_t)(GATHER ? b : s) * H;
    const uint16_t *r = src + (size_t)(GATHER ? s : b) * H;
    if (vec) {
        const int n = H / 8;
        for (int i = threadIdx.x; i < n; i += blockDim.x)
            reinterpret_cast<uint4 *>(d)[i] = __ldg(reinterpret_cast<const uint4 *>(r) + i);
    } else {
        for (int i = threadIdx.x; i < H; i += blockDim.x) d[i] = r[i];
    }
}

static int hpool_launch(bool gather, void *dst, const void *src, const int32_t *hslot, int B, int H, int n_slots,
                        int32_t *dev_err, spec_stream_t stream) {
    if (!dst || !src || !hslot) return SPEC_ERR_NULL;
    if (B < 1 || H < 1 || n_slots < 1) return SPEC_ERR_ARG;
    const bool vec = (H % 8) == 0 && ((uintptr_t)dst % 16) == 0 && ((uintptr_t)src % 16) == 0;
    if (gather)
        hpool_copy_kernel<true><<<B, 128, 0, (cudaStream_t)stream>>>(
            (uint16_t *)dst, (const uint16_t *)src, hslot, H, n_slots, vec, dev_err);
    else
        hpool_copy_kernel<false><<<B, 128, 0, (cudaStream_t)stream>>>(
            (uint16_t *)dst, (const uint16_t *)src, hslot, H, n_slots, vec, dev_err);
    return launch_status();
}

}  // namespace spec

SPEC_API int spec_h_gather(void *h_out, const void *hpool, const int32_t *hslot, int B, int H, int n_slots,
                           int32_t *dev_err, spec_stream_t stream) {
    return spec::hpool_launch(true, h_out, hpool, hslot, B, H, n_slots, dev_err, stream);
}

SPEC_API int spec_h_scatter(void *hpool, const void *h_in, const int32_t *hslot, int B, int H, int n_slots,
                            int32_t *dev_err, spec_stream_t stream) {
    return spec::hpool_launch(false, hpool, h_in, hslot, B, H, n_slots, dev_err, stream);
}

// mtp_input.cu -- a5: the MTP / NextN draft head's input stage.
//
// oxinfer src/qwen_mtp.rs, module documentation: for main-model position i the extra
// layer takes x = fc([rmsnorm_emb(embed(x_{i+1})), rmsnorm_hidden(h_i)]) with fc of shape
// [H, 2H], the embedding half first. memra-engine src/spec.rs, `mtp_head_forward_dev`:
// embedding gather, the two RMSNorms and the eh_proj matmul on the device.
//
// Kernel 1 (one block per row): gather E[tok], both RMSNorms in fp32 with a fixed
// reduction order, the two halves rounded to bf16 into c[m] = [e ; h] (workspace).
// Kernel 2: x = c . W_fc^T through the skinny GEMM, stored as bf16.
#include "common.cuh"
#include "gemm.cuh"

namespace spec {

__device__ __forceinline__ float block_sum_256(float v, float *red) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float s = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) s += red[w];  // fixed order
    return s;
}

__global__ void __launch_bounds__(256) mtp_norm_concat_kernel(const int32_t *tok, const uint16_t *E,
                                                              const uint16_t *h, const float *g_emb,
                                                              const float *g_hid, float eps, int H, int V,
                                                              uint16_t *concat, int32_t *err) {
    __shared__ float red[8];
    const int m = blockIdx.x;
    const int t = __ldg(tok + m);
    uint16_t *c = concat + (size_t)m * 2 * H;
    for (int half = 0; half < 2; ++half) {
        const uint16_t *src;
        const float *gain;
        if (half == 0) {
            if (t < 0 || t >= V) {
                if (threadIdx.x == 0) raise_error(err, SPEC_DEVERR_TOKEN);
                for (int i = threadIdx.x; i < H; i += blockDim.x) c[i] = 0;
                continue;
            }
            src = E + (size_t)t * H;
            gain = g_emb;
        } else {
            src = h + (size_t)m * H;
            gain = g_hid;
        }
        float ss = 0.f;
        for (int i = threadIdx.x; i < H; i += blockDim.x) {
            const float x = __uint_as_float((uint32_t)src[i] << 16);
            ss = fmaf(x, x, ss);
        }
        ss = block_sum_256(ss, red);
        const float inv = 1.0f / sqrtf(ss / (float)H + eps);
        for (int i = threadIdx.x; i < H; i += blockDim.x) {
            const float x = __uint_as_float((uint32_t)src[i] << 16);
            __nv_bfloat16 b = __float2bfloat16_rn(x * inv * __ldg(gain + i));
            c[half * H + i] = *reinterpret_cast<uint16_t *>(&b);
        }
    }
}

static size_t concat_bytes(int M, int H) { return (((size_t)M * 2 * H * 2) + 255) & ~(size_t)255; }

}  // namespace spec

SPEC_API size_t spec_mtp_input_workspace(int M, int H) {
    if (M < 1 || M > 256 || H < 64 || (H % 64)) return 0;
    return 256 + spec::concat_bytes(M, H) + spec::gemm_store_ws_bytes(M, H, 2 * H);
}

SPEC_API int spec_mtp_input(const int32_t *tok, const void *E, const void *h, const float *g_emb,
                            const float *g_hid, float eps, const void *W_fc, int M, int H, int V, void *x_out,
                            void *ws, size_t ws_bytes, int32_t *dev_err, spec_stream_t stream) {
    if (!tok || !E || !h || !g_emb || !g_hid || !W_fc || !x_out) return SPEC_ERR_NULL;
    if (M < 1 || M > 256 || H < 64 || (H % 64) || V < 1 || !(eps >= 0.f)) return SPEC_ERR_ARG;
    const size_t need = spec_mtp_input_workspace(M, H);
    if (!ws || ws_bytes < need) return SPEC_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) || !spec::aligned16(E) || !spec::aligned16(h) ||
        !spec::aligned16(W_fc) || !spec::aligned16(x_out))
        return SPEC_ERR_ALIGN;
    cudaStream_t s = (cudaStream_t)stream;
    uint16_t *concat = (uint16_t *)((char *)ws + 256);
    spec::mtp_norm_concat_kernel<<<M, 256, 0, s>>>(tok, (const uint16_t *)E, (const uint16_t *)h, g_emb, g_hid, eps,
                                                   H, V, concat, dev_err);
    int st = spec::launch_status();
    if (st) return st;
    char *gws = (char *)ws + 256 + spec::concat_bytes(M, H);
    return spec::gemm_store_bf16(concat, W_fc, M, H, 2 * H, x_out, gws, spec::gemm_store_ws_bytes(M, H, 2 * H), s);
}

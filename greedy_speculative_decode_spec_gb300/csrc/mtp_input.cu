// mtp_input.cu -- a5: the MTP / NextN draft head's input stage.
//
// oxinfer src/qwen_mtp.rs, module documentation: for main-model position i the extra
// layer takes x = fc([rmsnorm_emb(embed(x_{i+1})), rmsnorm_hidden(h_i)]) with fc of shape
// [H, 2H], the embedding half first. memra-engine src/spec.rs, `mtp_head_forward_dev`:
// embedding gather, the two RMSNorms and the eh_proj matmul on the device.
//
// Kernel 1 (one block per row and half): gather E[tok], the RMSNorms in fp32 with a fixed
// reduction order, the two halves rounded to bf16 into c[m] = [e ; h] (workspace).
// Kernel 2: x = c . W_fc^T through the skinny GEMM, stored as bf16.
#include "common.cuh"
#include "gemm.cuh"

namespace spec {

// One block per (row m, half): half 0 normalises E[tok[m]], half 1 normalises h[m]. Each
// thread holds up to MAXC 8-element chunks of the vector in registers (16-byte loads), so
// the vector is read once; longer vectors are re-read for the second pass.
constexpr int NC_THREADS = 256, NC_MAXC = 8;
__global__ void __launch_bounds__(NC_THREADS) mtp_norm_concat_kernel(const int32_t *tok, const uint16_t *E,
                                                                     const uint16_t *h, const float *g_emb,
                                                                     const float *g_hid, float eps, int H, int V,
                                                                     uint16_t *concat, int32_t *err) {
    __shared__ float red[NC_THREADS / 32];
    const int m = blockIdx.x >> 1, half = blockIdx.x & 1;
    uint16_t *c = concat + (size_t)m * 2 * H + (size_t)half * H;
    const int nch = H / 8;  // 8-element chunks
    const uint16_t *src;
    const float *gain;
    if (half == 0) {
        const int t = __ldg(tok + m);
        if (t < 0 || t >= V) {
            if (threadIdx.x == 0) raise_error(err, SPEC_DEVERR_TOKEN);
            for (int i = threadIdx.x; i < nch; i += NC_THREADS) reinterpret_cast<uint4 *>(c)[i] = make_uint4(0, 0, 0, 0);
            return;
        }
        src = E + (size_t)t * H;
        gain = g_emb;
    } else {
        src = h + (size_t)m * H;
        gain = g_hid;
    }
    const uint4 *src4 = reinterpret_cast<const uint4 *>(src);
    uint4 v[NC_MAXC];
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < NC_MAXC; ++k) {
        const int i = threadIdx.x + k * NC_THREADS;
        v[k] = i < nch ? __ldg(src4 + i) : make_uint4(0, 0, 0, 0);
    }
    for (int i = threadIdx.x + NC_MAXC * NC_THREADS; i < nch; i += NC_THREADS) {  // H > 16384 only
        const uint4 w = __ldg(src4 + i);
        const uint32_t q[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) ss = fmaf(bf16_lo(q[e]), bf16_lo(q[e]), fmaf(bf16_hi(q[e]), bf16_hi(q[e]), ss));
    }
#pragma unroll
    for (int k = 0; k < NC_MAXC; ++k) {
        const uint32_t q[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) ss = fmaf(bf16_lo(q[e]), bf16_lo(q[e]), fmaf(bf16_hi(q[e]), bf16_hi(q[e]), ss));
    }
    // block sum, fixed order
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, off);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < NC_THREADS / 32; ++w) tot += red[w];
    const float inv = 1.0f / sqrtf(tot / (float)H + eps);
    auto emit = [&](int i, const uint4 &w) {
        const uint32_t q[4] = {w.x, w.y, w.z, w.w};
        const float4 g0 = __ldg(reinterpret_cast<const float4 *>(gain) + 2 * i);
        const float4 g1 = __ldg(reinterpret_cast<const float4 *>(gain) + 2 * i + 1);
        const float gg[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const __nv_bfloat162 b = __floats2bfloat162_rn(bf16_lo(q[e]) * inv * gg[2 * e], bf16_hi(q[e]) * inv * gg[2 * e + 1]);
            o[e] = *reinterpret_cast<const uint32_t *>(&b);
        }
        reinterpret_cast<uint4 *>(c)[i] = make_uint4(o[0], o[1], o[2], o[3]);
    };
#pragma unroll
    for (int k = 0; k < NC_MAXC; ++k) {
        const int i = threadIdx.x + k * NC_THREADS;
        if (i < nch) emit(i, v[k]);
    }
    for (int i = threadIdx.x + NC_MAXC * NC_THREADS; i < nch; i += NC_THREADS) emit(i, __ldg(src4 + i));
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
    if (!spec::aligned16(g_emb) || !spec::aligned16(g_hid)) return SPEC_ERR_ALIGN;
    spec::mtp_norm_concat_kernel<<<2 * M, spec::NC_THREADS, 0, s>>>(tok, (const uint16_t *)E, (const uint16_t *)h, g_emb, g_hid, eps,
                                                   H, V, concat, dev_err);
    int st = spec::launch_status();
    if (st) return st;
    char *gws = (char *)ws + 256 + spec::concat_bytes(M, H);
    return spec::gemm_store_bf16(concat, W_fc, M, H, 2 * H, x_out, gws, spec::gemm_store_ws_bytes(M, H, 2 * H), s);
}

// lmhead.cu -- a3: LM head with a fused per-row argmax, and the skinny GEMM it shares
// with the MTP fc.
//
// span-02 engine/crates/model/src/spec.rs, `Spec::body_inner`: `lm_head_argmax` turns
// the verify rows' hidden states into target ids on the device; `greedy_logprob`: the
// first maximum wins. flashrt-structures decode_loop/whole_step.py,
// `generate_speculative`: argmax of the fp32 logits. memra-engine src/spec.rs: only the
// ids cross to the host, never the logits.
//
// logit[m][v] = sum_h hidden[m][h] * W[v][h]. Every logit is accumulated by one thread
// in ascending h order, the same program for every (m, v) and every M, so a row's
// logits do not depend on the batch it is in and equal W rows give equal logits.
// The argmax key packs (orderable fp32 logit, inverted index) into 64 bits: the
// largest key is the largest logit and, among equal logits, the lowest index.
#include "common.cuh"
#include "gemm.cuh"

namespace spec {

constexpr int TV = 64;   // vocab rows per block
constexpr int TM = 16;   // hidden rows per pass
constexpr int TK = 64;   // K chunk

enum Epi { EPI_ARGMAX = 0, EPI_LOGITS = 1, EPI_STORE = 2 };

__device__ __forceinline__ unsigned long long pack_key(float logit, int v) {
    const float canon = __fadd_rn(logit, 0.0f);  // -0 -> +0
    return ((unsigned long long)float_key(canon) << 32) | (unsigned)(0xFFFFFFFFu - (unsigned)v);
}

template <int EPI>
__global__ void __launch_bounds__(256) skinny_simt_kernel(const uint16_t *__restrict__ A, const uint16_t *__restrict__ W,
                                                          int M, int N, int K, float *logits,
                                                          unsigned long long *partial, uint16_t *out) {
    __shared__ float ws[TV][TK + 1];
    __shared__ float as[TM][TK + 1];
    __shared__ unsigned long long best[TM][TV];
    const int t = threadIdx.x;
    const int tv = t % TV, tm = t / TV;  // tm in 0..3, 4 rows each
    const int v0 = blockIdx.x * TV;
    const int v = v0 + tv;
    for (int m0 = 0; m0 < M; m0 += TM) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        for (int k0 = 0; k0 < K; k0 += TK) {
            // W tile: 64 x 64 elements, 16 per thread
            for (int i = t; i < TV * TK; i += 256) {
                const int rr = i / TK, cc = i % TK;
                const int gv = v0 + rr, gk = k0 + cc;
                float x = 0.f;
                if (gv < N && gk < K) x = __uint_as_float((uint32_t)W[(size_t)gv * K + gk] << 16);
                ws[rr][cc] = x;
            }
            for (int i = t; i < TM * TK; i += 256) {
                const int rr = i / TK, cc = i % TK;
                const int gm = m0 + rr, gk = k0 + cc;
                float x = 0.f;
                if (gm < M && gk < K) x = __uint_as_float((uint32_t)A[(size_t)gm * K + gk] << 16);
                as[rr][cc] = x;
            }
            __syncthreads();
#pragma unroll 8
            for (int kk = 0; kk < TK; ++kk) {
                const float w = ws[tv][kk];
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[i] = fmaf(w, as[tm * 4 + i][kk], acc[i]);
            }
            __syncthreads();
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int m = m0 + tm * 4 + i;
            if (EPI == EPI_STORE) {
                if (m < M && v < N) {
                    __nv_bfloat16 b = __float2bfloat16_rn(acc[i]);
                    out[(size_t)m * N + v] = *reinterpret_cast<uint16_t *>(&b);
                }
                continue;
            }
            if (EPI == EPI_LOGITS && m < M && v < N) logits[(size_t)m * N + v] = acc[i];
            best[tm * 4 + i][tv] = (v < N) ? pack_key(acc[i], v) : 0ull;
        }
        if (EPI != EPI_STORE) {
            __syncthreads();
            if (t < TM && m0 + t < M) {
                unsigned long long bk = 0ull;
                for (int j = 0; j < TV; ++j) bk = best[t][j] > bk ? best[t][j] : bk;
                partial[(size_t)blockIdx.x * M + m0 + t] = bk;
            }
            __syncthreads();
        }
    }
}

// Reduce the per-block partial keys of each row (one thread per row).
__global__ void argmax_final_kernel(const unsigned long long *partial, int n_parts, int M,
                                    const int32_t *d2t, int d2t_limit, int32_t *ids, float *max_logit,
                                    int32_t *err) {
    const int m = blockIdx.x * blockDim.x + threadIdx.x;
    if (m >= M) return;
    unsigned long long bk = 0ull;
    for (int p = 0; p < n_parts; ++p) {
        const unsigned long long k = partial[(size_t)p * M + m];
        bk = k > bk ? k : bk;
    }
    int id = (int)(0xFFFFFFFFu - (unsigned)(bk & 0xFFFFFFFFull));
    if (max_logit) max_logit[m] = key_float((uint32_t)(bk >> 32));
    if (d2t) {
        const int t = d2t[id];
        if (t < 0 || t >= d2t_limit) {
            raise_error(err, SPEC_DEVERR_D2T);
            id = -1;
        } else {
            id = t;
        }
    }
    ids[m] = id;
}

static size_t lmhead_ws_bytes(int M, int V) {
    const size_t tiles = (size_t)(V + TV - 1) / TV;
    return 256 + tiles * (size_t)M * sizeof(unsigned long long);
}

static int lmhead_run(const void *hidden, const void *W, int M, int V, int H, const int32_t *d2t,
                      int d2t_limit, int32_t *ids, float *max_logit, float *logits, void *ws,
                      size_t ws_bytes, int32_t *dev_err, cudaStream_t s) {
    if (!hidden || !W || !ids) return SPEC_ERR_NULL;
    if (M < 1 || M > 256 || V < 1 || H < 8 || (H & 7)) return SPEC_ERR_ARG;
    if (d2t && d2t_limit < 1) return SPEC_ERR_ARG;
    if (!ws || ws_bytes < lmhead_ws_bytes(M, V)) return SPEC_ERR_WORKSPACE;
    if (!aligned16(hidden) || !aligned16(W) || (reinterpret_cast<uintptr_t>(ws) & 255u)) return SPEC_ERR_ALIGN;
    unsigned long long *partial = (unsigned long long *)((char *)ws + 256);
    const int tiles = (V + TV - 1) / TV;
    if (logits)
        skinny_simt_kernel<EPI_LOGITS><<<tiles, 256, 0, s>>>((const uint16_t *)hidden, (const uint16_t *)W, M, V, H,
                                                              logits, partial, nullptr);
    else
        skinny_simt_kernel<EPI_ARGMAX><<<tiles, 256, 0, s>>>((const uint16_t *)hidden, (const uint16_t *)W, M, V, H,
                                                              nullptr, partial, nullptr);
    argmax_final_kernel<<<(M + 127) / 128, 128, 0, s>>>(partial, tiles, M, d2t, d2t_limit, ids, max_logit, dev_err);
    return launch_status();
}

size_t gemm_store_ws_bytes(int M, int N, int K) {
    (void)M;
    (void)N;
    (void)K;
    return 256;
}

int gemm_store_bf16(const void *A, const void *W, int M, int N, int K, void *out, void *ws, size_t ws_bytes,
                    cudaStream_t s) {
    (void)ws;
    (void)ws_bytes;
    const int tiles = (N + TV - 1) / TV;
    skinny_simt_kernel<EPI_STORE><<<tiles, 256, 0, s>>>((const uint16_t *)A, (const uint16_t *)W, M, N, K, nullptr,
                                                         nullptr, (uint16_t *)out);
    return launch_status();
}

}  // namespace spec

SPEC_API size_t spec_lmhead_workspace(int M, int V, int H) {
    if (M < 1 || M > 256 || V < 1 || H < 8) return 0;
    return spec::lmhead_ws_bytes(M, V);
}

SPEC_API int spec_lmhead_argmax(const void *hidden, const void *W, int M, int V, int H, const int32_t *d2t,
                                int d2t_limit, int32_t *ids, float *max_logit, void *ws, size_t ws_bytes,
                                int32_t *dev_err, spec_stream_t stream) {
    return spec::lmhead_run(hidden, W, M, V, H, d2t, d2t_limit, ids, max_logit, nullptr, ws, ws_bytes, dev_err,
                            (cudaStream_t)stream);
}

SPEC_API int spec_lmhead_logits(const void *hidden, const void *W, int M, int V, int H, float *logits,
                                int32_t *ids, void *ws, size_t ws_bytes, spec_stream_t stream) {
    if (!logits) return SPEC_ERR_NULL;
    return spec::lmhead_run(hidden, W, M, V, H, nullptr, 0, ids, nullptr, logits, ws, ws_bytes, nullptr,
                            (cudaStream_t)stream);
}

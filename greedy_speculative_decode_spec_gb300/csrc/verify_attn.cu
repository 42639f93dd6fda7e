// verify_attn.cu -- a2: causal GQA verify attention over paged KV (split-KV flash-decode).
//
// Row r = b*(k+1)+j (position p = pos[b]+j) and q head h attend keys 0..p of branch b
// (kv head h / G): span-02 engine/crates/model/src/spec.rs, module documentation
// (kv_hi = position, rejected-row KV beyond pos is never attended); memra-engine
// src/spec.rs, `full_attn_verify` (row r sees keys [0, base_len + r + 1), one launch for
// all rows); memra-engine `MtpScratch` (split count fixed by capacity, not by the current
// length, so one program serves every length bit for bit).
//
// Split-KV: keys are cut at fixed multiples of SPLIT_KEYS positions. A work unit is
// (branch, kv head, split); it produces, for every query vector of the group (the
// (k+1)*G rows x heads that share the kv head), the partial max m, sum l and
// unnormalised output o over its keys. A combine pass merges the splits of each query in
// ascending order. A row's result depends only on its own keys and the fixed split
// boundaries, so it is identical whatever B, k or batch it is verified in.
// Keys beyond a row's position are excluded by the loop bound (never multiplied by a
// zero weight), so NaN in unattended slots cannot leak.
#include <cuda_fp8.h>
#include <math.h>

#include "common.cuh"

namespace spec {

constexpr int SPLIT_KEYS = 1024;
constexpr float LOG2E = 1.4426950408889634f;

struct AttnArgs {
    KvView kv;
    const int32_t *pos;
    int B, k, Hq, G, n_splits, max_pos;
    const uint16_t *q;  // [R][Hq][d]
    float scale_log2;   // scale * log2(e)
    float *ws_ml;       // [units][n_q][2]   (m in log2 units, l)
    float *ws_o;        // [units][n_q][d]
    uint16_t *out;      // [R][Hq][d]
    int32_t *err;
};

template <int D>
__device__ __forceinline__ void load_k_lane(const AttnArgs &a, int page, int g, int slot, int lane,
                                            float (&x)[D / 32], bool is_v) {
    constexpr int E = D / 32;
    const size_t off = pool_offset(a.kv, page, g, slot) + (size_t)lane * E;
    if (a.kv.kv_dtype == SPEC_KV_BF16) {
        const uint16_t *src = reinterpret_cast<const uint16_t *>(is_v ? a.kv.v_pool : a.kv.k_pool) + off;
#pragma unroll
        for (int e = 0; e < E; e += 2) {
            uint32_t w = *reinterpret_cast<const uint32_t *>(src + e);
            x[e] = bf16_lo(w);
            x[e + 1] = bf16_hi(w);
        }
    } else {
        const uint8_t *src = reinterpret_cast<const uint8_t *>(is_v ? a.kv.v_pool : a.kv.k_pool) + off;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            __nv_fp8_e4m3 c;
            c.__x = src[e];
            x[e] = float(c);
        }
    }
}

// One warp per query vector of the unit (strided over the block's warps).
template <int D>
__global__ void __launch_bounds__(256) attn_split_kernel(AttnArgs a) {
    constexpr int E = D / 32;
    const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_q = (a.k + 1) * a.G;
    const size_t unit = ((size_t)b * a.kv.n_kv_heads + g) * a.n_splits + split;
    const int pos_b = __ldg(a.pos + b);
    const bool bad_pos = pos_b < 0 || pos_b + a.k + 1 > a.max_pos;
    if (bad_pos && split == 0 && g == 0 && threadIdx.x == 0) raise_error(a.err, SPEC_DEVERR_POS);
    const int s0 = split * SPLIT_KEYS;
    for (int qi = warp; qi < n_q; qi += blockDim.x >> 5) {
        const int j = qi / a.G, hi = qi % a.G;
        const int h = g * a.G + hi;
        const int r = b * (a.k + 1) + j;
        float *ml = a.ws_ml + (unit * n_q + qi) * 2;
        float *o_ws = a.ws_o + (unit * n_q + qi) * D;
        // keys of this row inside this split: [s0, min(s0 + SPLIT, p + 1))
        const int p = pos_b + j;
        const int nv = bad_pos ? -1 : min(SPLIT_KEYS, p + 1 - s0);
        float qv[E];
        {
            const uint16_t *qp = a.q + ((size_t)r * a.Hq + h) * D + lane * E;
#pragma unroll
            for (int e = 0; e < E; e += 2) {
                uint32_t w = *reinterpret_cast<const uint32_t *>(qp + e);
                qv[e] = bf16_lo(w);
                qv[e + 1] = bf16_hi(w);
            }
        }
        float m = -INFINITY, l = 0.f, o[E];
#pragma unroll
        for (int e = 0; e < E; ++e) o[e] = 0.f;
        bool failed = bad_pos;
        for (int t = 0; t < nv; ++t) {
            const int key = s0 + t;
            const int page = page_of(a.kv, b, key);
            if (page < 0) {
                if (lane == 0) raise_error(a.err, -page);
                failed = true;
                break;
            }
            const int slot = key & (a.kv.page_size - 1);
            float kx[E];
            load_k_lane<D>(a, page, g, slot, lane, kx, false);
            float dot = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) dot = fmaf(qv[e], kx[e], dot);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xFFFFFFFFu, dot, off);
            float sk = 1.f, sv = 1.f;
            if (a.kv.kv_dtype != SPEC_KV_BF16) {
                const size_t sidx = (size_t)page * a.kv.n_kv_heads + g;
                sk = __ldg(a.kv.k_scale + sidx);
                sv = __ldg(a.kv.v_scale + sidx);
            }
            const float s = dot * sk * a.scale_log2;
            const float m_new = fmaxf(m, s);
            const float corr = exp2f(m - m_new);
            const float w = exp2f(s - m_new);
            l = l * corr + w;
            float vx[E];
            load_k_lane<D>(a, page, g, slot, lane, vx, true);
            const float wv = w * sv;
#pragma unroll
            for (int e = 0; e < E; ++e) o[e] = fmaf(wv, vx[e], o[e] * corr);
            m = m_new;
        }
        if (lane == 0) {
            ml[0] = m;
            ml[1] = failed ? -1.f : (nv > 0 ? l : 0.f);
        }
#pragma unroll
        for (int e = 0; e < E; ++e) o_ws[lane * E + e] = o[e];
    }
}

// One warp per (row, q head): merge the splits in ascending order.
template <int D>
__global__ void __launch_bounds__(256) attn_combine_kernel(AttnArgs a) {
    constexpr int E = D / 32;
    const int warp_global = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    const int R = a.B * (a.k + 1);
    if (warp_global >= R * a.Hq) return;
    const int r = warp_global / a.Hq, h = warp_global % a.Hq;
    const int b = r / (a.k + 1), j = r % (a.k + 1);
    const int g = h / a.G, hi = h % a.G;
    const int n_q = (a.k + 1) * a.G;
    const int qi = j * a.G + hi;
    const size_t unit0 = ((size_t)b * a.kv.n_kv_heads + g) * a.n_splits;
    float M = -INFINITY;
    bool failed = false;
    for (int s = 0; s < a.n_splits; ++s) {
        const float *ml = a.ws_ml + ((unit0 + s) * n_q + qi) * 2;
        const float l = ml[1];
        if (l < 0.f) failed = true;
        if (l > 0.f) M = fmaxf(M, ml[0]);
    }
    if (failed || M == -INFINITY) return;  // error already raised; output left unwritten
    float L = 0.f, o[E];
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] = 0.f;
    for (int s = 0; s < a.n_splits; ++s) {
        const float *ml = a.ws_ml + ((unit0 + s) * n_q + qi) * 2;
        const float l = ml[1];
        if (!(l > 0.f)) continue;
        const float w = exp2f(ml[0] - M);
        L = fmaf(l, w, L);
        const float *os = a.ws_o + ((unit0 + s) * n_q + qi) * D + lane * E;
#pragma unroll
        for (int e = 0; e < E; ++e) o[e] = fmaf(w, os[e], o[e]);
    }
    const float inv = 1.f / L;
    uint16_t *dst = a.out + ((size_t)r * a.Hq + h) * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; e += 2) {
        __nv_bfloat162 v = __floats2bfloat162_rn(o[e] * inv, o[e + 1] * inv);
        *reinterpret_cast<__nv_bfloat162 *>(dst + e) = v;
    }
}

static size_t ws_bytes_for(int B, int Hkv, int n_splits, int n_q, int d) {
    const size_t units = (size_t)B * Hkv * n_splits;
    size_t ml = units * n_q * 2 * sizeof(float);
    ml = (ml + 255) & ~(size_t)255;
    return ml + units * n_q * d * sizeof(float);
}

}  // namespace spec

SPEC_API size_t spec_verify_attn_workspace(const spec_kv_desc *kv, int B, int k, int n_q_heads,
                                           int max_pos) {
    if (spec::check_kv_desc(kv) || B < 1 || k < 0 || k > SPEC_KMAX || n_q_heads < 1 || max_pos < 1) return 0;
    if (n_q_heads % kv->n_kv_heads) return 0;
    const int G = n_q_heads / kv->n_kv_heads;
    const int n_splits = (max_pos + spec::SPLIT_KEYS - 1) / spec::SPLIT_KEYS;
    return spec::ws_bytes_for(B, kv->n_kv_heads, n_splits, (k + 1) * G, kv->head_dim);
}

SPEC_API int spec_verify_attn(const spec_kv_desc *kvd, const int32_t *pos, int B, int k, int n_q_heads,
                              const void *q, float scale, void *out, void *ws, size_t ws_bytes,
                              int max_pos, int32_t *dev_err, spec_stream_t stream) {
    int st = spec::check_kv_desc(kvd);
    if (st) return st;
    if (!pos || !q || !out) return SPEC_ERR_NULL;
    if (B < 1 || k < 0 || k > SPEC_KMAX || n_q_heads < 1 || max_pos < k + 1) return SPEC_ERR_ARG;
    if (n_q_heads % kvd->n_kv_heads) return SPEC_ERR_ARG;
    const size_t need = spec_verify_attn_workspace(kvd, B, k, n_q_heads, max_pos);
    if (!ws || ws_bytes < need) return SPEC_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return SPEC_ERR_ALIGN;
    if (!spec::aligned16(q) || !spec::aligned16(out)) return SPEC_ERR_ALIGN;
    spec::AttnArgs a;
    a.kv = spec::make_view(kvd);
    a.pos = pos;
    a.B = B;
    a.k = k;
    a.Hq = n_q_heads;
    a.G = n_q_heads / kvd->n_kv_heads;
    a.n_splits = (max_pos + spec::SPLIT_KEYS - 1) / spec::SPLIT_KEYS;
    a.max_pos = max_pos;
    a.q = (const uint16_t *)q;
    a.scale_log2 = scale * spec::LOG2E;
    const int n_q = (k + 1) * a.G;
    const size_t units = (size_t)B * kvd->n_kv_heads * a.n_splits;
    size_t ml = units * n_q * 2 * sizeof(float);
    ml = (ml + 255) & ~(size_t)255;
    a.ws_ml = (float *)ws;
    a.ws_o = (float *)((char *)ws + ml);
    a.out = (uint16_t *)out;
    a.err = dev_err;
    cudaStream_t s = (cudaStream_t)stream;
    dim3 grid(a.n_splits, kvd->n_kv_heads, B);
    if (grid.y > 65535 || grid.z > 65535) return SPEC_ERR_ARG;
    const int R = B * (k + 1);
    const int cblocks = (R * n_q_heads + 7) / 8;
    switch (kvd->head_dim) {
        case 64:
            spec::attn_split_kernel<64><<<grid, 256, 0, s>>>(a);
            spec::attn_combine_kernel<64><<<cblocks, 256, 0, s>>>(a);
            break;
        case 128:
            spec::attn_split_kernel<128><<<grid, 256, 0, s>>>(a);
            spec::attn_combine_kernel<128><<<cblocks, 256, 0, s>>>(a);
            break;
        default:
            spec::attn_split_kernel<256><<<grid, 256, 0, s>>>(a);
            spec::attn_combine_kernel<256><<<cblocks, 256, 0, s>>>(a);
            break;
    }
    return spec::launch_status();
}

// kv_append.cu -- a1: write the new K/V rows of the verify step into the paged pool.
//
// span-02 engine/crates/model/src/spec.rs, module documentation: the verify forward
// appends the KV of its B(k+1) rows in place at pos..pos+k of each branch's own pages;
// `SpecReq`: the slot of position p is page pages[p / page_size].
// memra-engine src/spec.rs, `full_attn_verify`: all T verify rows are appended in one
// launch before the attention (instead of one launch per row).
//
// One thread moves 16 bytes of one (row, kv head) vector: 8 bf16 values, copied as
// they are (bf16 pool) or quantised to 8 E4M3 codes with the page's scale (FP8 pool):
// code = cvt.rn.satfinite.e4m3(x / scale), the division in IEEE fp32.
#include <cuda_fp8.h>

#include "common.cuh"

namespace spec {

struct RowMap {
    // verify form: row r -> branch r / (k+1), position pos[branch] + r % (k+1)
    const int32_t *pos;
    int kp1;
    // general form: row r -> (row_branch[r], row_pos[r])
    const int32_t *row_branch, *row_pos;
};

__global__ void __launch_bounds__(256) kv_write_kernel(KvView kv, RowMap map, int n_rows,
                                                       const uint4 *__restrict__ k_rows,
                                                       const uint4 *__restrict__ v_rows,
                                                       int32_t *err) {
    const int vec_per_head = kv.head_dim >> 3;  // 16-byte vectors per (row, head)
    const long long total = (long long)n_rows * kv.n_kv_heads * vec_per_head;
    long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= total) return;
    const int c = (int)(i % vec_per_head);
    const long long pair = i / vec_per_head;
    const int g = (int)(pair % kv.n_kv_heads);
    const int row = (int)(pair / kv.n_kv_heads);
    int b, p;
    if (map.row_branch) {
        b = __ldg(map.row_branch + row);
        p = __ldg(map.row_pos + row);
    } else {
        b = row / map.kp1;
        p = __ldg(map.pos + b) + row % map.kp1;
    }
    const int page = page_of(kv, b, p);
    if (page < 0) {
        if (c == 0 && g == 0) raise_error(err, -page);
        return;
    }
    const int slot = p & (kv.page_size - 1);
    const size_t dst = pool_offset(kv, page, g, slot) + (size_t)c * 8;  // element index
    const uint4 kk = __ldg(k_rows + pair * vec_per_head + c);
    const uint4 vv = __ldg(v_rows + pair * vec_per_head + c);
    if (kv.kv_dtype == SPEC_KV_BF16) {
        reinterpret_cast<uint4 *>(kv.k_pool)[dst >> 3] = kk;
        reinterpret_cast<uint4 *>(kv.v_pool)[dst >> 3] = vv;
        return;
    }
    const size_t sidx = (size_t)page * kv.n_kv_heads + g;
    const float sk = __ldg(kv.k_scale + sidx), sv = __ldg(kv.v_scale + sidx);
    const uint32_t kw[4] = {kk.x, kk.y, kk.z, kk.w};
    const uint32_t vw[4] = {vv.x, vv.y, vv.z, vv.w};
    uint32_t ko[2], vo[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t kp = 0, vp = 0;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const uint32_t wk = kw[2 * h + q], wv = vw[2 * h + q];
            float2 fk = make_float2(__fdiv_rn(bf16_lo(wk), sk), __fdiv_rn(bf16_hi(wk), sk));
            float2 fv = make_float2(__fdiv_rn(bf16_lo(wv), sv), __fdiv_rn(bf16_hi(wv), sv));
            // low byte <- .x (the lower-addressed element), high byte <- .y
            const uint32_t pk = __nv_cvt_float2_to_fp8x2(fk, __NV_SATFINITE, __NV_E4M3);
            const uint32_t pv = __nv_cvt_float2_to_fp8x2(fv, __NV_SATFINITE, __NV_E4M3);
            kp |= (pk & 0xFFFFu) << (16 * q);
            vp |= (pv & 0xFFFFu) << (16 * q);
        }
        ko[h] = kp;
        vo[h] = vp;
    }
    reinterpret_cast<uint2 *>(kv.k_pool)[dst >> 3] = make_uint2(ko[0], ko[1]);
    reinterpret_cast<uint2 *>(kv.v_pool)[dst >> 3] = make_uint2(vo[0], vo[1]);
}

static int launch_write(const spec_kv_desc *kvd, RowMap map, int n_rows, const void *k_rows,
                        const void *v_rows, int32_t *dev_err, cudaStream_t stream) {
    int st = check_kv_desc(kvd);
    if (st) return st;
    if (n_rows < 0) return SPEC_ERR_ARG;
    if (n_rows == 0) return SPEC_OK;
    if (!k_rows || !v_rows) return SPEC_ERR_NULL;
    if (!aligned16(k_rows) || !aligned16(v_rows)) return SPEC_ERR_ALIGN;
    KvView kv = make_view(kvd);
    const long long total = (long long)n_rows * kv.n_kv_heads * (kv.head_dim / 8);
    const int threads = 256;
    const long long blocks = (total + threads - 1) / threads;
    if (blocks > 0x7FFFFFFF) return SPEC_ERR_ARG;
    kv_write_kernel<<<(unsigned)blocks, threads, 0, stream>>>(kv, map, n_rows, (const uint4 *)k_rows,
                                                                (const uint4 *)v_rows, dev_err);
    return launch_status();
}

}  // namespace spec

SPEC_API int spec_kv_append(const spec_kv_desc *kv, const int32_t *pos, int B, int k,
                            const void *k_new, const void *v_new, int32_t *dev_err,
                            spec_stream_t stream) {
    if (!pos) return SPEC_ERR_NULL;
    if (B < 1 || k < 0 || k > SPEC_KMAX) return SPEC_ERR_ARG;
    spec::RowMap map{pos, k + 1, nullptr, nullptr};
    return spec::launch_write(kv, map, B * (k + 1), k_new, v_new, dev_err, (cudaStream_t)stream);
}

SPEC_API int spec_kv_write_rows(const spec_kv_desc *kv, const int32_t *row_branch,
                                const int32_t *row_pos, int n_rows, const void *k_rows,
                                const void *v_rows, int32_t *dev_err, spec_stream_t stream) {
    if (n_rows > 0 && (!row_branch || !row_pos)) return SPEC_ERR_NULL;
    spec::RowMap map{nullptr, 1, row_branch, row_pos};
    return spec::launch_write(kv, map, n_rows, k_rows, v_rows, dev_err, (cudaStream_t)stream);
}

// tree.cu -- f2: the greedy tree walk and the KV compaction of the accepted path.
//
// DSSD-dev `_star_cycle` / `_set_rows`: the k+1 verify rows of a branch form a tree (row 0
// the root, parent[j] < j); the walk starts at the root and repeatedly moves to the first
// child (in row order) whose draft token equals the current row's target argmax; the
// accepted drafts are emitted in walk order, then the last row's target (the bonus). The
// accepted rows' K/V were written at their own slots pos_b + row; compaction moves the i-th
// accepted row to slot pos_b + i, so that the committed prefix is contiguous again (DSSD-dev
// `_star_cycle`: the accepted child's K/V is copied to slot pos0 + 1). A chain (parent[j] =
// j - 1) walks like spec_accept and compacts nothing.
#include <cuda_fp8.h>

#include "common.cuh"

namespace spec {

// one warp per branch: lane c (1..k) holds row c's parent and draft
__global__ void __launch_bounds__(128) accept_tree_kernel(const int32_t *__restrict__ drafts,
                                                          const int32_t *__restrict__ ids, const int32_t *pos,
                                                          const int32_t *__restrict__ parent, int B, int k,
                                                          int32_t *out_tokens, int32_t *out_n, int32_t *out_accepted,
                                                          int32_t *out_pos, int32_t *out_next, int32_t *out_path,
                                                          int32_t *err) {
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (b >= B) return;
    const int32_t *tgt = ids + (size_t)b * (k + 1);
    int par = -1, d = -1;
    if (lane >= 1 && lane <= k) {
        par = __ldg(parent + (size_t)b * (k + 1) + lane);
        d = __ldg(drafts + (size_t)b * k + lane - 1);
    }
    // a parent outside [0, c) is an error; such a row is never walked to (c > cur = parent)
    const unsigned bad = __ballot_sync(0xFFFFFFFFu, lane >= 1 && lane <= k && (par < 0 || par >= lane));
    if (bad && lane == 0) raise_error(err, SPEC_DEVERR_TREE);
    int32_t *toks = out_tokens + (size_t)b * (k + 1);
    int32_t *path = out_path + (size_t)b * (k + 1);
    int cur = 0, a = 0;
    for (;;) {
        const int32_t t = __ldg(tgt + cur);
        const unsigned m = __ballot_sync(0xFFFFFFFFu, lane > cur && lane <= k && par == cur && d == t);
        if (!m) break;
        const int next = __ffs(m) - 1;
        if (lane == next) {
            toks[a] = d;
            path[a + 1] = next;
        }
        ++a;
        cur = next;
    }
    const int32_t bonus = __ldg(tgt + cur);
    __syncwarp();
    if (lane == 0) {
        toks[a] = bonus;
        path[0] = 0;
        out_n[b] = a + 1;
        out_accepted[b] = a;
        out_pos[b] = pos[b] + a + 1;  // out_pos may be pos
        out_next[b] = bonus;
    }
    if (lane > a && lane <= k) {
        toks[lane] = -1;
        path[lane] = -1;
    }
}

// one CTA per branch; the accepted rows move in ascending order (a path's rows increase,
// so no source is overwritten before it is read), one barrier between moves
__global__ void __launch_bounds__(256) kv_compact_kernel(KvView kv, const int32_t *pos,
                                                         const int32_t *__restrict__ path,
                                                         const int32_t *__restrict__ accepted, int k,
                                                         int32_t *err) {
    const int b = blockIdx.x;
    const int a = __ldg(accepted + b);
    const int base = pos[b];
    const int n_el = kv.n_kv_heads * kv.head_dim;
    for (int i = 1; i <= a && i <= k; ++i) {
        const int src_row = __ldg(path + (size_t)b * (k + 1) + i);
        if (src_row == i) continue;
        if (src_row < i || src_row > k) {
            if (threadIdx.x == 0) raise_error(err, SPEC_DEVERR_TREE);
            continue;
        }
        const int sp = page_of(kv, b, base + src_row), dp = page_of(kv, b, base + i);
        if (sp < 0 || dp < 0) {
            if (threadIdx.x == 0) raise_error(err, sp < 0 ? -sp : -dp);
            continue;
        }
        const int ss = (base + src_row) & (kv.page_size - 1), ds = (base + i) & (kv.page_size - 1);
        if (kv.kv_dtype == SPEC_KV_BF16) {
            const int nv = n_el / 8;  // 16-byte vectors of one position (all kv heads)
            for (int e = threadIdx.x; e < 2 * nv; e += blockDim.x) {
                const int which = e / nv, v = e % nv, g = v / (kv.head_dim / 8), c = v % (kv.head_dim / 8);
                uint4 *pool = reinterpret_cast<uint4 *>(which ? kv.v_pool : kv.k_pool);
                pool[(pool_offset(kv, dp, g, ds) >> 3) + c] = pool[(pool_offset(kv, sp, g, ss) >> 3) + c];
            }
        } else {
            // decode with the source page's scale, re-encode with the destination page's
            for (int e = threadIdx.x; e < 2 * n_el; e += blockDim.x) {
                const int which = e / n_el, v = e % n_el, g = v / kv.head_dim, c = v % kv.head_dim;
                uint8_t *pool = reinterpret_cast<uint8_t *>(which ? kv.v_pool : kv.k_pool);
                const float *scale = which ? kv.v_scale : kv.k_scale;
                const uint8_t code = pool[pool_offset(kv, sp, g, ss) + c];
                const __half_raw hr = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)code, __NV_E4M3);
                const float x = __half2float(*reinterpret_cast<const __half *>(&hr)) *
                                __ldg(scale + (size_t)sp * kv.n_kv_heads + g);
                const float y = __fdiv_rn(x, __ldg(scale + (size_t)dp * kv.n_kv_heads + g));
                pool[pool_offset(kv, dp, g, ds) + c] = (uint8_t)__nv_cvt_float_to_fp8(y, __NV_SATFINITE, __NV_E4M3);
            }
        }
        __syncthreads();
    }
}

}  // namespace spec

SPEC_API int spec_accept_tree(const int32_t *drafts, const int32_t *ids, const int32_t *pos,
                              const int32_t *parent, int B, int k, int32_t *out_tokens, int32_t *out_n,
                              int32_t *out_accepted, int32_t *out_pos, int32_t *out_next, int32_t *out_path,
                              int32_t *dev_err, spec_stream_t stream) {
    if (!ids || !pos || !parent || !out_tokens || !out_n || !out_accepted || !out_pos || !out_next || !out_path)
        return SPEC_ERR_NULL;
    if (k > 0 && !drafts) return SPEC_ERR_NULL;
    if (B < 1 || k < 0 || k > SPEC_KMAX) return SPEC_ERR_ARG;
    const int warps = 4;
    spec::accept_tree_kernel<<<(B + warps - 1) / warps, warps * 32, 0, (cudaStream_t)stream>>>(
        drafts, ids, pos, parent, B, k, out_tokens, out_n, out_accepted, out_pos, out_next, out_path, dev_err);
    return spec::launch_status();
}

SPEC_API int spec_kv_compact(const spec_kv_desc *kvd, const int32_t *pos, const int32_t *path,
                             const int32_t *accepted, int B, int k, int32_t *dev_err, spec_stream_t stream) {
    int st = spec::check_kv_desc(kvd);
    if (st) return st;
    if (!pos || !path || !accepted) return SPEC_ERR_NULL;
    if (B < 1 || k < 0 || k > SPEC_KMAX) return SPEC_ERR_ARG;
    if (k == 0) return SPEC_OK;
    spec::kv_compact_kernel<<<B, 256, 0, (cudaStream_t)stream>>>(spec::make_view(kvd), pos, path, accepted, k,
                                                                   dev_err);
    return spec::launch_status();
}

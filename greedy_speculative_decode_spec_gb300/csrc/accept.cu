// accept.cu -- a4: greedy chain acceptance, one warp per branch.
//
// span-02 engine/crates/model/src/spec.rs, module documentation: a token is emitted
// only if it equals the target's argmax at the verify row before it; rollback is the
// position advance alone. DSSD-dev dssd/fast.py, `generate_spec`: stop at the first
// draft that differs from its row's target, then append target[accepted] (the
// correction, or the bonus after a full acceptance). flashrt-structures
// decode_loop/whole_step.py, `generate_speculative`: the prefix match runs on the
// device and pos advances by accepted + 1.
//
// Lane i < k compares draft i with the target of row i; the first mismatching lane
// (a ballot) is the accepted count a. Lanes 0..k write the emitted tokens.
#include "common.cuh"

namespace spec {

__global__ void __launch_bounds__(128) accept_kernel(const int32_t *__restrict__ drafts,
                                                     const int32_t *__restrict__ ids,
                                                     const int32_t *__restrict__ pos, int B, int k,
                                                     int32_t *out_tokens, int32_t *out_n,
                                                     int32_t *out_accepted, int32_t *out_pos,
                                                     int32_t *out_next, const uint16_t *hidden, int H,
                                                     uint16_t *h_out) {
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (b >= B) return;
    const int32_t *tgt = ids + (size_t)b * (k + 1);
    bool mismatch = false;
    int32_t d = -1;
    if (lane < k) {
        d = __ldg(drafts + (size_t)b * k + lane);
        mismatch = d != __ldg(tgt + lane);
    }
    const unsigned bad = __ballot_sync(0xFFFFFFFFu, mismatch);
    const int a = bad ? (__ffs(bad) - 1) : k;
    const int32_t bonus = __ldg(tgt + a);
    if (lane <= k) out_tokens[(size_t)b * (k + 1) + lane] = lane < a ? d : (lane == a ? bonus : -1);
    if (lane == 0) {
        out_n[b] = a + 1;
        out_accepted[b] = a;
        out_pos[b] = __ldg(pos + b) + a + 1;
        out_next[b] = bonus;
    }
    if (h_out) {
        // the next draft step's hidden state: the target row that produced the bonus
        const uint16_t *src = hidden + ((size_t)b * (k + 1) + a) * H;
        uint16_t *dst = h_out + (size_t)b * H;
        if ((H & 7) == 0) {
            const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
            uint4 *d4 = reinterpret_cast<uint4 *>(dst);
            for (int i = lane; i < H / 8; i += 32) d4[i] = __ldg(s4 + i);
        } else {
            for (int i = lane; i < H; i += 32) dst[i] = src[i];
        }
    }
}

}  // namespace spec

SPEC_API int spec_accept(const int32_t *drafts, const int32_t *ids, const int32_t *pos, int B, int k,
                         int32_t *out_tokens, int32_t *out_n, int32_t *out_accepted, int32_t *out_pos,
                         int32_t *out_next, const void *hidden, int H, void *h_out,
                         spec_stream_t stream) {
    if (!ids || !pos || !out_tokens || !out_n || !out_accepted || !out_pos || !out_next) return SPEC_ERR_NULL;
    if (k > 0 && !drafts) return SPEC_ERR_NULL;
    if (B < 1 || k < 0 || k > SPEC_KMAX) return SPEC_ERR_ARG;
    const bool gather = hidden || h_out;
    if (gather) {
        if (!hidden || !h_out) return SPEC_ERR_NULL;
        if (H < 1) return SPEC_ERR_ARG;
        if ((H & 7) == 0 && (!spec::aligned16(hidden) || !spec::aligned16(h_out))) return SPEC_ERR_ALIGN;
    }
    const int warps = 4;
    const int blocks = (B + warps - 1) / warps;
    spec::accept_kernel<<<blocks, warps * 32, 0, (cudaStream_t)stream>>>(
        drafts, ids, pos, B, k, out_tokens, out_n, out_accepted, out_pos, out_next,
        (const uint16_t *)hidden, gather ? H : 0, (uint16_t *)h_out);
    return spec::launch_status();
}

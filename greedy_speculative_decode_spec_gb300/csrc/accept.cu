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
//
// Device-resident step state: out_pos may be the pos array itself (the branch's position
// is read once, by the lane that writes it), so a loop captured in a CUDA graph advances its
// positions on the device, and out_next / h_out give the next step's first fed token and
// its draft-head hidden row without a host round trip (span-02 spec.rs, module
// documentation: the state stays on the device between steps; flashrt-structures
// decode_loop/whole_step.py, `generate_speculative`: pos advances by accepted + 1 on the
// device).
//
// With a stop set and a budget (spec_accept_stop): the run drafts[0..a) ++ [ids[a]] is
// cut right after its first token in the stop set and then to at most the branch's budget
// (DSSD-dev dssd/fast.py, `_commit`: the committed tokens are appended until the stop rule
// fires on one, which is kept, or the generation limit is reached; span-02
// engine/crates/model/src/spec.rs, `Spec::body_inner`: a small stop-id buffer whose unused
// entries are -1, and a token limit). Lane i <= a tests run token i against the stop ids;
// a second ballot gives the first stop.
#include <climits>

#include "common.cuh"

namespace spec {

__global__ void __launch_bounds__(128) accept_kernel(const int32_t *__restrict__ drafts,
                                                     const int32_t *__restrict__ ids,
                                                     const int32_t *pos, int B, int k,
                                                     int32_t *out_tokens, int32_t *out_n,
                                                     int32_t *out_accepted, int32_t *out_pos,
                                                     int32_t *out_next, const uint16_t *hidden, int H,
                                                     uint16_t *h_out, const int32_t *__restrict__ stop,
                                                     int n_stop, const int32_t *__restrict__ budget,
                                                     int32_t *out_done) {
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
    const int32_t tok = lane < a ? d : (lane == a ? bonus : -1);  // run token `lane`
    // the first run token in the stop set, then the budget
    bool is_stop = false;
    if (lane <= a)
        for (int j = 0; j < n_stop; ++j) {
            const int32_t sid = __ldg(stop + j);
            is_stop |= sid >= 0 && sid == tok;
        }
    const unsigned hits = __ballot_sync(0xFFFFFFFFu, is_stop);
    int n = hits ? __ffs(hits) : a + 1;  // tokens kept
    bool stopped = hits != 0;
    int cap = INT_MAX;
    if (budget) {
        cap = __ldg(budget + b);
        cap = cap < 0 ? 0 : cap;
        if (n > cap) {
            n = cap;
            stopped = false;  // the stop token was cut off
        }
    }
    const int32_t last = __shfl_sync(0xFFFFFFFFu, tok, n > 0 ? n - 1 : 0);
    if (lane <= k) out_tokens[(size_t)b * (k + 1) + lane] = lane < n ? tok : -1;
    if (lane == 0) {
        out_n[b] = n;
        out_accepted[b] = a < n ? a : n;
        out_pos[b] = pos[b] + n;  // pos may be out_pos: the position advances in place
        out_next[b] = n > 0 ? last : -1;
        if (out_done) out_done[b] = (stopped || (budget && n == cap)) ? 1 : 0;
    }
    if (h_out && n > 0) {
        // the next draft step's hidden state: the target row that produced the last kept
        // token (the bonus when nothing was cut)
        const uint16_t *src = hidden + ((size_t)b * (k + 1) + (n - 1)) * H;
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
        (const uint16_t *)hidden, gather ? H : 0, (uint16_t *)h_out, nullptr, 0, nullptr, nullptr);
    return spec::launch_status();
}

SPEC_API int spec_accept_stop(const int32_t *drafts, const int32_t *ids, const int32_t *pos, int B, int k,
                              const int32_t *stop_ids, int n_stop, const int32_t *budget, int32_t *out_tokens,
                              int32_t *out_n, int32_t *out_accepted, int32_t *out_pos, int32_t *out_next,
                              int32_t *out_done, const void *hidden, int H, void *h_out, spec_stream_t stream) {
    if (!ids || !pos || !out_tokens || !out_n || !out_accepted || !out_pos || !out_next) return SPEC_ERR_NULL;
    if (k > 0 && !drafts) return SPEC_ERR_NULL;
    if (B < 1 || k < 0 || k > SPEC_KMAX) return SPEC_ERR_ARG;
    if (n_stop < 0 || n_stop > SPEC_MAX_STOP) return SPEC_ERR_ARG;
    if (n_stop > 0 && !stop_ids) return SPEC_ERR_NULL;
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
        (const uint16_t *)hidden, gather ? H : 0, (uint16_t *)h_out, stop_ids, n_stop, budget, out_done);
    return spec::launch_status();
}

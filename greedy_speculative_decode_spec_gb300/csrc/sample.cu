// sample.cu -- f4: speculative sampling acceptance (the random numbers are inputs).
//
// oxinfer `speculative_accept`: a draft token d drawn from the draft distribution q is kept
// with probability min(1, p(d) / q(d)); otherwise it is replaced by a token drawn from the
// normalised max(0, p - q), or from p when that residual is all zero. DSSD-dev
// `_sample_verify`: walk the chain, stop at the first rejection, and after a full
// acceptance draw the bonus token from the last row's p. Here p_j = softmax(logits_j / T)
// and q_j are given per verify row; u_acc[b][i] decides draft i (kept when p >= q or
// u < p / q) and u_res[b] is the one draw of the step: the smallest index t whose running
// sum of the weights exceeds u * (their total), taken in index order.
//
// One CTA of 1024 threads per branch. Per verify row: the maximum of the logits (one pass,
// warp max reductions), the softmax denominator (one pass; each thread sums exp2 of its
// elements with a compensated fp32 sum, the 1024 partial sums are added in fp64), then the
// draft's probability on one thread. A draw: each thread owns a contiguous chunk of the
// vocabulary and sums its weights (compensated), the chunk sums are scanned in fp64, and the
// thread whose chunk crosses u * total walks it in fp64. The decisions are taken in fp32
// probabilities with fp64 sums; they can differ from an all-fp64 evaluation only where the
// test value lies within the fp32 rounding of a boundary.
#include <climits>
#include <math.h>

#include "common.cuh"

namespace spec {

constexpr int SMP_THREADS = 1024;
constexpr int SMP_WARPS = SMP_THREADS / 32;

struct SampleArgs {
    const int32_t *drafts;  // [B][k]
    const float *logits;    // [B*(k+1)][V]
    const float *q;         // [B][k][V]
    const int32_t *pos;     // [B]
    int B, k, V;
    float inv_t_log2;       // log2(e) / temperature
    const float *u_acc;     // [B][k]
    const float *u_res;     // [B]
    int32_t *out_tokens, *out_n, *out_accepted, *out_pos, *out_next;
    int32_t *err;
};

__device__ __forceinline__ float smp_warp_max(float v) {
    float r;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}

__device__ __forceinline__ double smp_warp_sum(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// compensated (Kahan) fp32 accumulation
struct KSum {
    float s = 0.f, c = 0.f;
    __device__ __forceinline__ void add(float x) {
        const float y = x - c;
        const float t = s + y;
        c = (t - s) - y;
        s = t;
    }
    __device__ __forceinline__ double value() const { return (double)s - (double)c; }
};

// block-wide maximum / fp64 sum through shared scratch (red: SMP_WARPS doubles)
__device__ float block_max(float v, float *redf) {
    v = smp_warp_max(v);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) redf[w] = v;
    __syncthreads();
    float r = l < SMP_WARPS ? redf[l] : -INFINITY;
    return smp_warp_max(r);
}

__device__ double block_sum(double v, double *red) {
    v = smp_warp_sum(v);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) red[w] = v;
    __syncthreads();
    double r = l < SMP_WARPS ? red[l] : 0.0;
    return smp_warp_sum(r);
}

// Softmax statistics of one row: the maximum logit and the fp64 sum of exp2((z - mx) * c).
__device__ void row_stats(const float *z, int V, float c, float *redf, double *red, float &mx, double &den) {
    float m = -INFINITY;
    for (int t = threadIdx.x; t < V; t += SMP_THREADS) m = fmaxf(m, __ldg(z + t));
    mx = block_max(m, redf);
    KSum ks;
    for (int t = threadIdx.x; t < V; t += SMP_THREADS) ks.add(exp2f((__ldg(z + t) - mx) * c));
    den = block_sum(ks.value(), red);
}

// Inverse-CDF draw over the weights w_t = max(0, p_t - q_t) (q != nullptr, falling back to
// p_t when they are all zero) or w_t = p_t, with p_t = exp2((z_t - mx) * c) / den: the
// smallest t whose running sum exceeds u * sum(w) (the last t with w_t > 0 if rounding puts
// the limit past the total). scan: SMP_THREADS + 1 doubles of shared scratch.
__device__ int draw_index(const float *z, const float *q, int V, float mx, float c, double den, float u,
                          float *redf, double *red, double *scan, int *s_found) {
    const float inv = (float)(1.0 / den);
    const int chunk = (V + SMP_THREADS - 1) / SMP_THREADS;
    const int t0 = min(V, (int)threadIdx.x * chunk), t1 = min(V, t0 + chunk);
    auto weight = [&](int t, bool use_q) -> float {
        const float p = exp2f((__ldg(z + t) - mx) * c) * inv;
        return use_q ? fmaxf(p - __ldg(q + t), 0.f) : p;
    };
    bool use_q = q != nullptr;
    KSum ks;
    for (int t = t0; t < t1; ++t) ks.add(weight(t, use_q));
    double S = ks.value();
    double total = block_sum(S, red);
    if (use_q && !(total > 0.0)) {  // the residual is all zero: draw from p
        use_q = false;
        KSum kp;
        for (int t = t0; t < t1; ++t) kp.add(weight(t, false));
        S = kp.value();
        total = block_sum(S, red);
    }
    // exclusive prefix of the chunk sums (fp64): warp scan, then the warp totals
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    double incl = S;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (l >= o) incl += y;
    }
    __syncthreads();
    if (l == 31) red[w] = incl;
    if (threadIdx.x == 0) *s_found = INT_MAX;
    __syncthreads();
    if (w == 0) {
        double v = l < SMP_WARPS ? red[l] : 0.0, vi = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double y = __shfl_up_sync(0xFFFFFFFFu, vi, o);
            if (l >= o) vi += y;
        }
        if (l < SMP_WARPS) red[l] = vi - v;  // exclusive prefix of the warps
    }
    __syncthreads();
    const double excl = red[w] + (incl - S);
    scan[threadIdx.x] = excl;
    if (threadIdx.x == SMP_THREADS - 1) scan[SMP_THREADS] = excl + S;
    __syncthreads();
    const double lim = (double)u * total;
    if (excl <= lim && lim < scan[threadIdx.x + 1]) {
        double run = excl;
        int pick = -1, last_pos = -1;
        for (int t = t0; t < t1; ++t) {
            const double wt = (double)weight(t, use_q);
            if (wt > 0.0) last_pos = t;
            run += wt;
            if (run > lim) {
                pick = t;
                break;
            }
        }
        if (pick < 0) pick = last_pos;  // rounding: the chunk ended at the limit
        if (pick >= 0) atomicMin(s_found, pick);
    }
    __syncthreads();
    int found = *s_found;
    if (found == INT_MAX) {
        // the limit lies past the total: the last index with a positive weight
        int last = -1;
        for (int t = t0; t < t1; ++t)
            if (weight(t, use_q) > 0.f) last = t;
        found = (int)block_max((float)last, redf);
        found = found < 0 ? 0 : found;
    }
    __syncthreads();
    return found;
}

__global__ void __launch_bounds__(SMP_THREADS) sample_accept_kernel(SampleArgs a) {
    __shared__ float redf[SMP_WARPS];
    __shared__ double red[SMP_WARPS];
    __shared__ double scan[SMP_THREADS + 1];
    __shared__ int s_found, s_keep;
    const int b = blockIdx.x;
    const int k = a.k, V = a.V;
    const float c = a.inv_t_log2;
    int acc = k, last = -1;
    for (int i = 0; i < k; ++i) {
        const float *z = a.logits + ((size_t)b * (k + 1) + i) * V;
        const float *qi = a.q + ((size_t)b * k + i) * V;
        float mx;
        double den;
        row_stats(z, V, c, redf, red, mx, den);
        if (threadIdx.x == 0) {
            const int d = __ldg(a.drafts + (size_t)b * k + i);
            // a draft is a sample of q: one outside [0, V) or with q(d) <= 0 (or NaN) is
            // reported and rejected
            const double qd = (d >= 0 && d < V) ? (double)__ldg(qi + d) : 0.0;
            int keep = 0;
            if (!(qd > 0.0)) {
                raise_error(a.err, SPEC_DEVERR_TOKEN);
            } else {
                const double pd = (double)exp2f((__ldg(z + d) - mx) * c) / den;
                keep = (pd >= qd || (double)__ldg(a.u_acc + (size_t)b * k + i) < pd / qd) ? 1 : 0;
            }
            s_keep = keep;
        }
        __syncthreads();
        const int keep = s_keep;
        __syncthreads();
        if (!keep) {
            acc = i;
            last = draw_index(z, qi, V, mx, c, den, __ldg(a.u_res + b), redf, red, scan, &s_found);
            break;
        }
    }
    if (acc == k) {  // every draft kept: the bonus token from the last row's p
        const float *z = a.logits + ((size_t)b * (k + 1) + k) * V;
        float mx;
        double den;
        row_stats(z, V, c, redf, red, mx, den);
        last = draw_index(z, nullptr, V, mx, c, den, __ldg(a.u_res + b), redf, red, scan, &s_found);
    }
    const int t = threadIdx.x;
    if (t <= k)
        a.out_tokens[(size_t)b * (k + 1) + t] = t < acc ? __ldg(a.drafts + (size_t)b * k + t) : (t == acc ? last : -1);
    if (t == 0) {
        a.out_n[b] = acc + 1;
        a.out_accepted[b] = acc;
        a.out_pos[b] = a.pos[b] + acc + 1;  // out_pos may be pos
        a.out_next[b] = last;
    }
}

}  // namespace spec

SPEC_API int spec_accept_sample(const int32_t *drafts, const float *logits, const float *q, const int32_t *pos,
                                int B, int k, int V, float temperature, const float *u_acc, const float *u_res,
                                int32_t *out_tokens, int32_t *out_n, int32_t *out_accepted, int32_t *out_pos,
                                int32_t *out_next, int32_t *dev_err, spec_stream_t stream) {
    if (!logits || !pos || !u_res || !out_tokens || !out_n || !out_accepted || !out_pos || !out_next)
        return SPEC_ERR_NULL;
    if (k > 0 && (!drafts || !q || !u_acc)) return SPEC_ERR_NULL;
    if (B < 1 || k < 0 || k > SPEC_KMAX || V < 1) return SPEC_ERR_ARG;
    if (!(temperature > 0.f) || !isfinite(temperature)) return SPEC_ERR_ARG;
    spec::SampleArgs a;
    a.drafts = drafts;
    a.logits = logits;
    a.q = q;
    a.pos = pos;
    a.B = B;
    a.k = k;
    a.V = V;
    a.inv_t_log2 = (float)(1.4426950408889634 / (double)temperature);
    a.u_acc = u_acc;
    a.u_res = u_res;
    a.out_tokens = out_tokens;
    a.out_n = out_n;
    a.out_accepted = out_accepted;
    a.out_pos = out_pos;
    a.out_next = out_next;
    a.err = dev_err;
    spec::sample_accept_kernel<<<B, spec::SMP_THREADS, 0, (cudaStream_t)stream>>>(a);
    return spec::launch_status();
}

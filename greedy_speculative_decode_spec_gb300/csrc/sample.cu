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
// A verify row of a 151936-entry vocabulary is 600 KB of fp32 logits, so the work is spread
// over the whole GPU, in chunks of SMP_CHUNK entries, in two launches:
//  1. row statistics, one CTA per (verify row, chunk): the chunk's largest logit m_c and the
//     sum of exp2(z c - m_c c), c = log2(e) / T (the hardware exp2, per-thread sums taken
//     pairwise). Every verify row is read, all at once (rather than one after another up to
//     the first rejection);
//  2. the walk and the draw weights, one CTA per (branch, chunk): the branch's rows' maxima
//     M (over chunks) and denominators S = sum_c s_c * 2^((m_c - M) c) (the factor in fp32,
//     the sum a double-float, in a fixed order), every draft's decision at once (the walk
//     stops at the first draft not kept), then the chunk's sums of the draw weights of the
//     decisive row (the residual and p);
//  3. the draw, by the branch's last CTA of step 2 to finish: the chunk whose running sum
//     crosses u * total (in chunk order), then the index inside it (each thread owns a
//     contiguous run of SMP_PER entries; a scan of the runs' sums; the crossing run is
//     walked entry by entry).
// Probabilities are fp32 (exp2f); every sum is kept as a double-float (an unevaluated pair of
// fp32 values, about 48 significant bits: Knuth's TwoSum and an fma-based TwoProduct give the
// exact rounding error of each addition and product), from compensated or pairwise fp32
// partial sums, in a fixed order: GB300's fp64 pipe is narrow, so per-thread fp64 would bound
// these kernels.
// A decision can differ from an exact evaluation only where its test value lies within that
// rounding (about 2^-24 relative, from the fp32 probabilities) of a boundary.
#include <climits>
#include <math.h>

#include "common.cuh"
#include "sm100.cuh"

namespace spec {

constexpr int SMP_T = 256;                  // threads per CTA
constexpr int SMP_W = SMP_T / 32;
constexpr int SMP_PER = 32;                 // entries per thread
constexpr int SMP_CHUNK = SMP_T * SMP_PER;  // entries per CTA

struct SampleArgs {
    const int32_t *drafts;  // [B][k]
    const float *logits;    // [B*(k+1)][V]
    const float *q;         // [B][k][V]
    const int32_t *pos;     // [B]
    int B, k, V, NC;        // NC: chunks per row
    bool vec;               // rows start on 16-byte boundaries (V % 4 == 0, aligned base)
    float inv_t_log2;       // log2(e) / temperature
    const float *u_acc;     // [B][k]
    const float *u_res;     // [B]
    int32_t *out_tokens, *out_n, *out_accepted, *out_pos, *out_next;
    int32_t *err;
};

// Workspace: per (row, chunk) the statistics; per (branch, chunk) the draw-weight sums and
// the last index with a positive weight; per branch a count of its finished walk CTAs (zero
// before a call; the branch's last CTA sets it back to zero).
struct SampleWs {
    float2 *s, *wq, *wp;  // double-floats (hi, lo)
    float *m;
    int32_t *lq, *lp;
    uint32_t *cnt;  // per branch: the walk CTAs done (zero between calls)
};
__host__ __device__ inline size_t sample_ws_layout(int B, int k, int V, uint8_t *base, SampleWs *w) {
    const size_t NC = (size_t)((V + SMP_CHUNK - 1) / SMP_CHUNK), R = (size_t)B * (k + 1);
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = (o + bytes + 255) & ~(size_t)255;
        return base ? base + at : nullptr;
    };
    uint8_t *s = take(R * NC * 8), *wq = take((size_t)B * NC * 8), *wp = take((size_t)B * NC * 8);  // float2
    uint8_t *m = take(R * NC * 4);
    uint8_t *lq = take((size_t)B * NC * 4), *lp = take((size_t)B * NC * 4), *cnt = take((size_t)B * 4);
    if (w) {
        w->s = reinterpret_cast<float2 *>(s);
        w->wq = reinterpret_cast<float2 *>(wq);
        w->wp = reinterpret_cast<float2 *>(wp);
        w->m = reinterpret_cast<float *>(m);
        w->lq = reinterpret_cast<int32_t *>(lq);
        w->lp = reinterpret_cast<int32_t *>(lp);
        w->cnt = reinterpret_cast<uint32_t *>(cnt);
    }
    return o;
}

__device__ __forceinline__ float smp_warp_max(float v) {
    float r;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}

// Double-float arithmetic. A value is hi + lo with |lo| <= ulp(hi) / 2; every sum here is of
// non-negative terms, so no addition cancels.
struct DF {
    float hi, lo;
};
__device__ __forceinline__ DF df_fast(float s, float e) {  // |s| >= |e|: the pair renormalised
    const float h = s + e;
    return {h, e - (h - s)};
}
// a + b: TwoSum gives the exact error of hi + hi (the same in either order); the low parts
// are added as one commutative sum, so df_add(a, b) == df_add(b, a) bit for bit
__device__ __forceinline__ DF df_add(DF a, DF b) {
    const float s = a.hi + b.hi;
    const float bb = s - a.hi;
    const float err = (a.hi - (s - bb)) + (b.hi - bb);
    return df_fast(s, err + (a.lo + b.lo));
}
__device__ __forceinline__ DF df_addf(DF a, float b) { return df_add(a, DF{b, 0.f}); }
// a * b (b fp32): the product's exact error by an fma
__device__ __forceinline__ DF df_mulf(DF a, float b) {
    const float p = a.hi * b;
    return df_fast(p, fmaf(a.lo, b, fmaf(a.hi, b, -p)));
}
__device__ __forceinline__ bool df_less(DF a, DF b) { return a.hi < b.hi || (a.hi == b.hi && a.lo < b.lo); }
__device__ __forceinline__ DF df_shfl_xor(DF v, int o) {
    return {__shfl_xor_sync(0xFFFFFFFFu, v.hi, o), __shfl_xor_sync(0xFFFFFFFFu, v.lo, o)};
}
__device__ __forceinline__ DF df_shfl_up(DF v, int o) {
    return {__shfl_up_sync(0xFFFFFFFFu, v.hi, o), __shfl_up_sync(0xFFFFFFFFu, v.lo, o)};
}
// xor butterfly: partners add the same two values (df_add commutes), so every lane ends
// with the same sum
__device__ __forceinline__ DF df_warp_sum(DF v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = df_add(v, df_shfl_xor(v, o));
    return v;
}

// compensated (Kahan) fp32 accumulation of one thread's terms
struct KSum {
    float s = 0.f, c = 0.f;
    __device__ __forceinline__ void add(float x) {
        const float y = x - c;
        const float t = s + y;
        c = (t - s) - y;
        s = t;
    }
    __device__ __forceinline__ DF value() const { return df_fast(s, -c); }
};

// block-wide maximum / double-float sum (every thread gets the result)
__device__ float block_max(float v, float *redf) {
    v = smp_warp_max(v);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) redf[w] = v;
    __syncthreads();
    return smp_warp_max(l < SMP_W ? redf[l] : -INFINITY);
}

__device__ DF block_sum(DF v, DF *red) {
    v = df_warp_sum(v);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) red[w] = v;
    __syncthreads();
    return df_warp_sum(l < SMP_W ? red[l] : DF{0.f, 0.f});
}

// The SMP_PER entries of a row that thread `threadIdx.x` of a CTA owns in chunk ch:
// contiguous (CONTIG: base + tid*SMP_PER + j, the order the draw walks) or spread for
// coalesced loads (base + (j/4*SMP_T + tid)*4 + j%4); entries past V read as `fill`.
template <bool CONTIG>
__device__ __forceinline__ void load_run(const float *row, int ch, int V, bool vec, float fill, float (&x)[SMP_PER]) {
    const int base = ch * SMP_CHUNK;
    if (vec) {
#pragma unroll
        for (int j = 0; j < SMP_PER; j += 4) {
            const int t = CONTIG ? base + threadIdx.x * SMP_PER + j : base + ((j / 4) * SMP_T + threadIdx.x) * 4;
            float4 v = make_float4(fill, fill, fill, fill);
            if (t < V) v = __ldg(reinterpret_cast<const float4 *>(row + t));  // V % 4 == 0: t + 3 < V
            x[j] = v.x;
            x[j + 1] = v.y;
            x[j + 2] = v.z;
            x[j + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < SMP_PER; ++j) {
            const int t = CONTIG ? base + threadIdx.x * SMP_PER + j : base + j * SMP_T + threadIdx.x;
            x[j] = t < V ? __ldg(row + t) : fill;
        }
    }
}

// p_t = exp2((z_t - M) * c) * inv (inv = 1/S rounded to fp32), the one definition the weight
// sums and the draw's walk share
__device__ __forceinline__ float prob(float z, float M, float c, float inv) { return exp2f((z - M) * c) * inv; }

// ---- 1: per (row, chunk) maximum and sum of exp2((z - m_c) * c) ----
__global__ void __launch_bounds__(SMP_T) sample_stats_kernel(SampleArgs a, SampleWs ws) {
    __shared__ float redf[SMP_W];
    __shared__ DF red[SMP_W];
    const int ch = blockIdx.x, r = blockIdx.y;
    float x[SMP_PER];
    load_run<false>(a.logits + (size_t)r * a.V, ch, a.V, a.vec, -INFINITY, x);
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < SMP_PER; ++j) m = fmaxf(m, x[j]);
    m = block_max(m, redf);
    // the thread's terms exp2(z c - m c) (one fma and one exp2 each; padding gives 0), summed
    // pairwise (31 additions in a fixed tree): this kernel streams every verify row, so it
    // keeps its instruction count low
    const float c = a.inv_t_log2, mc = m * c;
#pragma unroll
    for (int j = 0; j < SMP_PER; ++j) x[j] = sm100::ex2_approx(fmaf(x[j], c, -mc));
#pragma unroll
    for (int w = SMP_PER / 2; w >= 1; w >>= 1)
#pragma unroll
        for (int j = 0; j < w; ++j) x[j] += x[j + w];
    const DF s = block_sum(DF{x[0], 0.f}, red);
    if (threadIdx.x == 0) {
        ws.m[(size_t)r * a.NC + ch] = m;
        ws.s[(size_t)r * a.NC + ch] = make_float2(s.hi, s.lo);
    }
    sm100::grid_dep_launch();  // the walk kernel may be scheduled
}

// ---- 3: the draw and the outputs, by the branch's last walk CTA (the other CTAs' sums are
// read from L2) ----
__device__ void draw_branch(const SampleArgs &a, const SampleWs &ws, int b, int acc, float M, float inv, float *redf,
                            DF *red) {
    __shared__ int s_ch, s_use, s_found, s_last;
    __shared__ DF s_base, s_lim;
    const int k = a.k, V = a.V, NC = a.NC, tid = threadIdx.x;
    const float c = a.inv_t_log2;
    const float2 *wq = ws.wq + (size_t)b * NC, *wp = ws.wp + (size_t)b * NC;
    const int32_t *lq = ws.lq + (size_t)b * NC, *lp = ws.lp + (size_t)b * NC;
    if (tid < 32) {
        // warp 0 over the chunks' sums (read from L2: the other CTAs wrote them), 32 chunks at
        // a time; the first 32 stay in registers
        const int lane = tid;
        const float2 z2 = make_float2(0.f, 0.f);
        const float2 q0 = lane < NC ? __ldcg(wq + lane) : z2, p0 = lane < NC ? __ldcg(wp + lane) : z2;
        const int lq0 = lane < NC ? __ldcg(lq + lane) : -1, lp0 = lane < NC ? __ldcg(lp + lane) : -1;
        // the totals (lane-strided, then the butterfly: a fixed order)
        DF tq{q0.x, q0.y}, tp{p0.x, p0.y};
        for (int j = lane + 32; j < NC; j += 32) {
            const float2 u = __ldcg(wq + j), v = __ldcg(wp + j);
            tq = df_add(tq, DF{u.x, u.y});
            tp = df_add(tp, DF{v.x, v.y});
        }
        tq = df_warp_sum(tq);
        tp = df_warp_sum(tp);
        // the residual (after a rejection) unless it is all zero, else p
        const bool use_q = acc < k && tq.hi > 0.f;
        const DF lim = df_mulf(use_q ? tq : tp, __ldg(a.u_res + b));
        // the chunk whose running sum (in chunk order) crosses the limit, run <= lim < run + w:
        // an inclusive warp scan per 32 chunks, carried over
        DF run{0.f, 0.f};
        int pick = -1, last = -1;
        DF base{0.f, 0.f};
        for (int j0 = 0; j0 < NC; j0 += 32) {
            const int j = j0 + lane;
            float2 wv;
            int lv;
            if (j0 == 0) {
                wv = use_q ? q0 : p0;
                lv = use_q ? lq0 : lp0;
            } else {
                wv = j < NC ? __ldcg((use_q ? wq : wp) + j) : z2;
                lv = j < NC ? __ldcg((use_q ? lq : lp) + j) : -1;
            }
            last = max(last, __reduce_max_sync(0xFFFFFFFFu, lv));
            DF incl{wv.x, wv.y};
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const DF v = df_shfl_up(incl, o);
                if (lane >= o) incl = df_add(v, incl);
            }
            DF excl = df_shfl_up(incl, 1);
            if (lane == 0) excl = DF{0.f, 0.f};
            const DF lo = df_add(run, excl), hi = df_add(run, incl);
            const unsigned hit = __ballot_sync(0xFFFFFFFFu, j < NC && !df_less(lim, lo) && df_less(lim, hi));
            if (hit) {
                const int src = __ffs(hit) - 1;
                pick = j0 + src;
                base = DF{__shfl_sync(0xFFFFFFFFu, lo.hi, src), __shfl_sync(0xFFFFFFFFu, lo.lo, src)};
                break;
            }
            const DF tot = DF{__shfl_sync(0xFFFFFFFFu, incl.hi, 31), __shfl_sync(0xFFFFFFFFu, incl.lo, 31)};
            run = df_add(run, tot);
        }
        if (lane == 0) {
            s_use = use_q ? 1 : 0;
            s_lim = lim;
            s_ch = pick;
            s_base = base;
            s_last = last < 0 ? 0 : last;  // the limit past the total: the last positive weight
            s_found = INT_MAX;
        }
    }
    __syncthreads();
    int tok = s_last;
    const int ch = s_ch;
    const bool use_q = s_use != 0;
    if (ch >= 0) {
        const float *z = a.logits + ((size_t)b * (k + 1) + acc) * V;
        float x[SMP_PER], y[SMP_PER];
        load_run<true>(z, ch, V, a.vec, -INFINITY, x);
        if (use_q) load_run<true>(a.q + ((size_t)b * k + acc) * V, ch, V, a.vec, 0.f, y);
        float wt[SMP_PER];
        KSum ks;
#pragma unroll
        for (int j = 0; j < SMP_PER; ++j) {
            const float p = prob(x[j], M, c, inv);
            wt[j] = use_q ? fmaxf(p - y[j], 0.f) : p;
            ks.add(wt[j]);
        }
        // exclusive scan of the runs' sums: warp scan, then the warp totals in order
        const DF St = ks.value();
        const int wi = tid >> 5, l = tid & 31;
        DF incl = St, excl{0.f, 0.f};
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const DF v = df_shfl_up(incl, o);
            if (l >= o) incl = df_add(v, incl);
        }
        {
            const DF v = df_shfl_up(incl, 1);
            if (l >= 1) excl = v;
        }
        if (l == 31) red[wi] = incl;
        __syncthreads();
        DF r = s_base;
        for (int i = 0; i < wi; ++i) r = df_add(r, red[i]);
        r = df_add(r, excl);
        const DF lim = s_lim;
        const int t0 = ch * SMP_CHUNK + tid * SMP_PER;
        int lastpos = -1;
        if (!df_less(lim, r) && df_less(lim, df_add(r, St))) {
            int pk = -1;
            for (int j = 0; j < SMP_PER; ++j) {
                if (wt[j] > 0.f) lastpos = t0 + j;
                r = df_addf(r, wt[j]);
                if (df_less(lim, r)) {
                    pk = t0 + j;
                    break;
                }
            }
            if (pk < 0) pk = lastpos;  // rounding: the run ended at the limit
            if (pk >= 0) atomicMin(&s_found, pk);
        }
        // the chunk's last positive weight, for a limit that the runs' own sums put past it
#pragma unroll
        for (int j = 0; j < SMP_PER; ++j)
            if (wt[j] > 0.f) lastpos = t0 + j;
        lastpos = (int)block_max((float)lastpos, redf);
        const int found = s_found;
        tok = found != INT_MAX ? found : (lastpos >= 0 ? lastpos : s_last);
    }
    const int t = tid;
    if (t <= k)
        a.out_tokens[(size_t)b * (k + 1) + t] = t < acc ? __ldg(a.drafts + (size_t)b * k + t) : (t == acc ? tok : -1);
    if (t == 0) {
        a.out_n[b] = acc + 1;
        a.out_accepted[b] = acc;
        a.out_pos[b] = a.pos[b] + acc + 1;  // out_pos may be pos
        a.out_next[b] = tok;
    }
}

// ---- 2: the walk, then this chunk's draw-weight sums of the decisive row ----
__global__ void __launch_bounds__(SMP_T) sample_walk_kernel(SampleArgs a, SampleWs ws) {
    __shared__ float redf[SMP_W];
    __shared__ DF red[SMP_W];
    __shared__ float sM[SPEC_KMAX + 1];
    __shared__ DF sS[SPEC_KMAX + 1];
    __shared__ int s_acc;
    __shared__ float s_inv;
    const int ch = blockIdx.x, b = blockIdx.y, k = a.k, V = a.V, NC = a.NC;
    const float c = a.inv_t_log2;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // the decisions' inputs first (their loads overlap the merge below): per draft its id, q(d)
    // and logit z(d); a draft is a sample of q, so one outside [0, V) or with q(d) <= 0 (or NaN)
    // is rejected, and reported if the walk reaches it
    float qd = 0.f, ud = 0.f, zd = 0.f;
    if (warp == 0 && lane < k) {
        const int d = __ldg(a.drafts + (size_t)b * k + lane);
        ud = __ldg(a.u_acc + (size_t)b * k + lane);
        if (d >= 0 && d < V) {
            qd = __ldg(a.q + ((size_t)b * k + lane) * V + d);
            zd = __ldg(a.logits + ((size_t)b * (k + 1) + lane) * V + d);
        }
    }
    sm100::grid_dep_wait();  // the row statistics
    // each row's M and S from its chunks, one warp per row (lane-strided, then the
    // butterfly: a fixed order)
    for (int i = warp; i <= k; i += SMP_W) {
        const size_t r0 = ((size_t)b * (k + 1) + i) * NC;
        float m = -INFINITY;
        for (int j = lane; j < NC; j += 32) m = fmaxf(m, ws.m[r0 + j]);
        m = smp_warp_max(m);
        DF sum{0.f, 0.f};
        for (int j = lane; j < NC; j += 32) {
            const float2 sc = ws.s[r0 + j];
            sum = df_add(sum, df_mulf(DF{sc.x, sc.y}, exp2f((ws.m[r0 + j] - m) * c)));
        }
        sum = df_warp_sum(sum);
        if (lane == 0) {
            sM[i] = m;
            sS[i] = sum;
        }
    }
    __syncthreads();
    if (warp == 0) {
        // every draft's decision at once; the walk stops at the first one not kept
        int keep = 1;
        bool bad = false;
        if (lane < k) {
            if (!(qd > 0.f)) {
                keep = 0;
                bad = true;
            } else {
                // p(d) = e / S: kept when p(d) >= q(d) or u < p(d) / q(d), tested as e >= q(d) S
                // or u q(d) S < e (q(d) > 0, S > 0)
                const DF e{exp2f((zd - sM[lane]) * c), 0.f};
                const DF qS = df_mulf(sS[lane], qd);
                keep = (!df_less(e, qS) || df_less(df_mulf(qS, ud), e)) ? 1 : 0;
            }
        }
        const unsigned rej = __ballot_sync(0xFFFFFFFFu, lane < k && !keep);
        const int acc = rej ? __ffs(rej) - 1 : k;
        if (ch == 0 && lane == acc && bad) raise_error(a.err, SPEC_DEVERR_TOKEN);
        if (lane == 0) {
            s_acc = acc;
            s_inv = 1.f / (sS[acc].hi + sS[acc].lo);  // 1/S rounded to fp32
        }
    }
    __syncthreads();
    const int acc = s_acc;
    const float M = sM[acc], inv = s_inv;
    const float *z = a.logits + ((size_t)b * (k + 1) + acc) * V;
    const float *qr = acc < k ? a.q + ((size_t)b * k + acc) * V : nullptr;
    // this chunk's sums (spread entries for coalesced loads: a sum's order is free; the draw
    // walks its chunk with sums of its own) and the last index with a positive weight
    float x[SMP_PER], y[SMP_PER];
    load_run<false>(z, ch, V, a.vec, -INFINITY, x);
    if (qr) load_run<false>(qr, ch, V, a.vec, 0.f, y);
    KSum kq, kp;
    int lq = -1, lp = -1;
#pragma unroll
    for (int j = 0; j < SMP_PER; ++j) {
        const int t = a.vec ? ch * SMP_CHUNK + ((j / 4) * SMP_T + threadIdx.x) * 4 + (j & 3)
                            : ch * SMP_CHUNK + j * SMP_T + threadIdx.x;
        const float p = prob(x[j], M, c, inv);  // 0 past V
        kp.add(p);
        if (p > 0.f) lp = max(lp, t);
        if (qr) {
            const float w = fmaxf(p - y[j], 0.f);
            kq.add(w);
            if (w > 0.f) lq = max(lq, t);
        }
    }
    const DF sq = block_sum(kq.value(), red);
    const DF sp = block_sum(kp.value(), red);
    lq = (int)block_max((float)lq, redf);  // indices < 2^24: exact in fp32
    lp = (int)block_max((float)lp, redf);
    // publish this chunk's sums; the branch's last CTA to finish draws
    __shared__ int s_lastcta;
    if (threadIdx.x == 0) {
        const size_t o = (size_t)b * NC + ch;
        ws.wq[o] = make_float2(sq.hi, sq.lo);
        ws.wp[o] = make_float2(sp.hi, sp.lo);
        ws.lq[o] = lq;
        ws.lp[o] = lp;
        __threadfence();
        const bool last = atomicAdd(ws.cnt + b, 1u) == (unsigned)NC - 1;
        if (last) ws.cnt[b] = 0u;  // no other CTA of the branch touches it again in this call
        s_lastcta = last ? 1 : 0;
    }
    __syncthreads();
    if (!s_lastcta) return;
    __threadfence();
    draw_branch(a, ws, b, acc, M, inv, redf, red);
}

}  // namespace spec

SPEC_API size_t spec_accept_sample_workspace(int B, int k, int V) {
    if (B < 1 || k < 0 || k > SPEC_KMAX || V < 1) return 0;
    return spec::sample_ws_layout(B, k, V, nullptr, nullptr);
}

SPEC_API int spec_accept_sample(const int32_t *drafts, const float *logits, const float *q, const int32_t *pos,
                                int B, int k, int V, float temperature, const float *u_acc, const float *u_res,
                                int32_t *out_tokens, int32_t *out_n, int32_t *out_accepted, int32_t *out_pos,
                                int32_t *out_next, void *workspace, size_t ws_bytes, int32_t *dev_err,
                                spec_stream_t stream) {
    if (!logits || !pos || !u_res || !out_tokens || !out_n || !out_accepted || !out_pos || !out_next)
        return SPEC_ERR_NULL;
    if (k > 0 && (!drafts || !q || !u_acc)) return SPEC_ERR_NULL;
    if (B < 1 || k < 0 || k > SPEC_KMAX || V < 1 || V >= (1 << 24)) return SPEC_ERR_ARG;
    if (!(temperature > 0.f) || !isfinite(temperature)) return SPEC_ERR_ARG;
    spec::SampleWs ws;
    const size_t need = spec::sample_ws_layout(B, k, V, reinterpret_cast<uint8_t *>(workspace), &ws);
    if (!workspace || ws_bytes < need) return SPEC_ERR_WORKSPACE;
    if (((uintptr_t)workspace % 16) != 0) return SPEC_ERR_ALIGN;
    spec::SampleArgs a;
    a.drafts = drafts;
    a.logits = logits;
    a.q = q;
    a.pos = pos;
    a.B = B;
    a.k = k;
    a.V = V;
    a.NC = (V + spec::SMP_CHUNK - 1) / spec::SMP_CHUNK;
    a.vec = (V % 4) == 0 && ((uintptr_t)logits % 16) == 0 && (k == 0 || ((uintptr_t)q % 16) == 0);
    a.inv_t_log2 = (float)(1.4426950408889634 / (double)temperature);
    a.u_acc = u_acc;
    a.u_res = u_res;
    a.out_tokens = out_tokens;
    a.out_n = out_n;
    a.out_accepted = out_accepted;
    a.out_pos = out_pos;
    a.out_next = out_next;
    a.err = dev_err;
    const cudaStream_t s = (cudaStream_t)stream;
    spec::sample_stats_kernel<<<dim3(a.NC, B * (k + 1)), spec::SMP_T, 0, s>>>(a, ws);
    const int st = spec::launch_status();
    if (st != SPEC_OK) return st;
    // may start while the statistics finish (it waits for them before reading them)
    return spec::launch_pdl(spec::sample_walk_kernel, dim3(a.NC, B), dim3(spec::SMP_T), 0, s, a, ws);
}

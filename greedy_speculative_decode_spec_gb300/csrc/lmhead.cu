// lmhead.cu -- a3: LM head with a fused per-row argmax, and the skinny GEMM it shares
// with the MTP fc (a5).
//
// span-02 engine/crates/model/src/spec.rs, `Spec::body_inner`: `lm_head_argmax` turns
// the verify rows' hidden states into target ids on the device; `greedy_logprob`: the
// first maximum wins. flashrt-structures decode_loop/whole_step.py,
// `generate_speculative`: argmax of the fp32 logits. memra-engine src/spec.rs: only the
// ids cross to the host, never the logits.
//
// GB300 design. The weight W [V, H] is the big operand and is streamed from HBM exactly
// once; the M <= 256 hidden rows are the small one. The MMA therefore runs "swap-AB":
//   D[128 vocab rows x N rows] = W_tile[128 x K] . hidden[N x K]^T
// with the vocab tile as the tcgen05 M = 128 side and the verify rows (padded to 16) as
// N. A persistent CTA per SM owns a contiguous run of vocab tiles. Warp 0 streams
// 64-wide K chunks of W and of the hidden rows into a shared-memory ring with TMA
// (128-byte swizzle); warp 1 issues tcgen05.mma into one of two TMEM accumulators;
// warps 2..5 read the finished accumulator with tcgen05.ld while the next tile is being
// multiplied. Every logit of every row goes through the same K order, whatever M is, so
// a row's logits do not depend on its batch and equal W rows give equal logits.
//
// Argmax: each (orderable fp32 logit, inverted vocab index) pair packs into 64 bits, so
// the maximum key is the largest logit and, among equal logits, the lowest index. A warp
// reduces its 32 vocab rows per column with one redux.sync + ballot; the four lane
// quadrants and the CTA's tiles merge with 64-bit max; each CTA folds its keys into one
// global 64-bit maximum per row (atomicMax) and the last CTA to finish (atomic counter)
// reads them back, zeroes them for the next call, applies d2t and writes the ids. Logits
// never reach HBM.
//
// Every pipeline wait is bounded (1 s); on a timeout the kernel raises
// SPEC_DEVERR_TIMEOUT, lets the loads and MMAs already issued land, frees TMEM and exits.
#include <cuda.h>

#include "common.cuh"
#include "gemm.cuh"
#include "sm100.cuh"

namespace spec {

using namespace sm100;

constexpr int TC_BM = 128;            // W rows per tile (MMA M)
constexpr int TC_BK = 64;             // K elements per pipeline stage (128 bytes of bf16)
constexpr int TC_THREADS = 192;       // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr uint32_t W_STAGE_BYTES = TC_BM * TC_BK * 2;
constexpr uint64_t WAIT_NS = 1000000000ull;
constexpr int MAX_SPLITS = 8;
constexpr int MAX_CTAS = 1024;
constexpr int SMEM_LIMIT = 227 * 1024;

enum TcEpi { TC_ARGMAX = 0, TC_LOGITS = 1, TC_PARTIAL = 2 };

struct TcParams {
    int M, N_pad, V, K;
    int n_tiles, n_kc, splits, stages;
    int tps;                        // W tiles per stage (1 or 2): the hidden chunk of a stage serves them all
    int n_groups;                   // groups of tps tiles
    uint32_t w_stage_bytes, a_stage_bytes, tmem_cols;
    float *logits;                  // TC_LOGITS: [M][V]
    float *partial;                 // TC_PARTIAL: [splits][M][V]
    unsigned long long *keys;       // argmax: [M] running maxima (zero between calls)
    unsigned int *counter;          // argmax: last-CTA detection (zero between calls)
    const int32_t *d2t;
    int d2t_limit;
    int32_t *ids;
    float *max_logit;
    int32_t *err;
    uint64_t wait_ns;               // pipeline-wait limit (drains: WAIT_NS)
};

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

template <int EPI>
__global__ void __launch_bounds__(TC_THREADS, 1)
    tc_skinny_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_a,
                     TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sw = smem_u32(smem);
    const uint32_t sa = sw + p.stages * p.w_stage_bytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + p.stages * (p.w_stage_bytes + p.a_stage_bytes));
    const uint32_t full0 = smem_u32(bars);
    const uint32_t empty0 = full0 + 8 * p.stages;
    const uint32_t tfull0 = empty0 + 8 * p.stages;
    const uint32_t tempty0 = tfull0 + 16;
    const uint32_t drain = tempty0 + 16;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * p.stages + 5);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile int *last_flag = reinterpret_cast<volatile int *>(tmem_slot + 2);
    unsigned long long *cand = reinterpret_cast<unsigned long long *>(tmem_slot + 4);  // [2][tps][4][N_pad]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull0 + 8 * a, 1);
            mbar_init(tempty0 + 8 * a, 4);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        *last_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmap_w);
        prefetch_tmap(&tmap_a);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), p.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int G = gridDim.x;
    const int n_work = p.n_groups * p.splits;
    const int wb = (int)(((long long)blockIdx.x * n_work) / G);
    const int we = (int)(((long long)(blockIdx.x + 1) * n_work) / G);

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            const uint32_t tx = p.w_stage_bytes + p.a_stage_bytes;
            uint32_t it = 0, s = 0, ph = 0;  // stages issued; the next stage and its phase parity
            bool ok = true;
            for (int w = wb; w < we && ok; ++w) {
                const int grp = w / p.splits, sp = w % p.splits;
                const int kb = sp * p.n_kc / p.splits, ke = (sp + 1) * p.n_kc / p.splits;
                for (int kc = kb; kc < ke; ++kc, ++it) {
                    if (!mbar_wait(empty0 + 8 * s, ph ^ 1u, abort_flag, p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(full0 + 8 * s, tx);
                    // one box of tps * 128 W rows (rows past V read as zeros)
                    tma_load_2d(sw + s * p.w_stage_bytes, &tmap_w, kc * TC_BK, grp * TC_BM * p.tps, full0 + 8 * s);
                    tma_load_2d(sa + s * p.a_stage_bytes, &tmap_a, kc * TC_BK, 0, full0 + 8 * s);
                    if (++s == (uint32_t)p.stages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok) {
                *abort_flag = 1;
                raise_error(p.err, SPEC_DEVERR_TIMEOUT);
            }
            // let the loads still in flight land before the CTA can exit
            for (uint32_t j = 0; j < (uint32_t)p.stages && j < it; ++j) {
                if (s == 0) {
                    s = (uint32_t)p.stages;
                    ph ^= 1u;
                }
                --s;
                mbar_wait(full0 + 8 * s, ph, nullptr, WAIT_NS);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(TC_BM, p.N_pad);
            uint32_t it = 0, t = 0, s = 0, ph = 0;
            bool ok = true;
            for (int w = wb; w < we && ok; ++w, ++t) {
                const uint32_t acc = t & 1u, use = t >> 1;
                if (!mbar_wait(tempty0 + 8 * acc, (use & 1u) ^ 1u, abort_flag, p.wait_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem + acc * (uint32_t)(p.tps * p.N_pad);  // tile i: + i * N_pad
                const int sp = w % p.splits;
                const int kb = sp * p.n_kc / p.splits, ke = (sp + 1) * p.n_kc / p.splits;
                for (int kc = kb; kc < ke; ++kc, ++it) {
                    if (!mbar_wait(full0 + 8 * s, ph, abort_flag, p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_base = sw + s * p.w_stage_bytes, b_base = sa + s * p.a_stage_bytes;
                    const uint64_t wa0 = desc_kmajor_sw128(a_base), hb0 = desc_kmajor_sw128(b_base);
                    for (int i = 0; i < p.tps; ++i) {
#pragma unroll
                        for (int k = 0; k < TC_BK / 16; ++k)
                            mma_bf16(d_tmem + i * p.N_pad, desc_advance(wa0, i * W_STAGE_BYTES + 32 * k),
                                     desc_advance(hb0, 32 * k), idesc, (kc > kb || k > 0) ? 1u : 0u);
                    }
                    mma_commit(empty0 + 8 * s);
                    if (++s == (uint32_t)p.stages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (ok) mma_commit(tfull0 + 8 * acc);
            }
            if (!ok) {
                *abort_flag = 1;
                raise_error(p.err, SPEC_DEVERR_TIMEOUT);
            }
            // every MMA issued by this thread completes before TMEM is released
            mma_commit(drain);
            mbar_wait(drain, 0, nullptr, WAIT_NS);
            // and every arrive those MMAs' commits send is delivered before the CTA may exit:
            // wait for the last phase of each stage's "empty" barrier (a late arrive would
            // land in shared memory this CTA no longer owns)
            for (uint32_t j = 0; j < (uint32_t)p.stages && j < it; ++j) {
                if (s == 0) {
                    s = (uint32_t)p.stages;
                    ph ^= 1u;
                }
                --s;
                mbar_wait(empty0 + 8 * s, ph, nullptr, WAIT_NS);
            }
        }
    } else {
        // ---------------- epilogue: 4 warps, one TMEM lane quadrant each ----------------
        const int q = warp & 3;
        const int etid = threadIdx.x - 64;
        unsigned long long running[2] = {0ull, 0ull};
        uint32_t t = 0;
        bool ok = true;
        for (int w = wb; w < we; ++w, ++t) {
            const uint32_t acc = t & 1u, use = t >> 1;
            if (!mbar_wait(tfull0 + 8 * acc, use & 1u, abort_flag, p.wait_ns)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int grp = w / p.splits, sp = w % p.splits;
            for (int i = 0; i < p.tps; ++i) {
                const int tile = grp * p.tps + i;
                const int v = tile * TC_BM + q * 32 + lane;
                const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + (acc * p.tps + i) * (uint32_t)p.N_pad;
                unsigned long long *cq = cand + (((size_t)acc * p.tps + i) * 4 + q) * p.N_pad;
                for (int c0 = 0; c0 < p.N_pad; c0 += 16) {
                    uint32_t r[16];
                    tmem_ld16(taddr + c0, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int m = c0 + j;
                        if (m >= p.M) break;
                        const float x = __uint_as_float(r[j]);
                        if (EPI == TC_PARTIAL) {
                            if (v < p.V) p.partial[((size_t)sp * p.M + m) * p.V + v] = x;
                            continue;
                        }
                        if (EPI == TC_LOGITS && v < p.V) p.logits[(size_t)m * p.V + v] = x;
                        const uint32_t key = v < p.V ? float_key(__fadd_rn(x, 0.0f)) : 0u;
                        const uint32_t best = __reduce_max_sync(0xFFFFFFFFu, key);
                        const uint32_t who = __ballot_sync(0xFFFFFFFFu, key == best);
                        if (lane == 0) {
                            const uint32_t vw = (uint32_t)(tile * TC_BM + q * 32 + __ffs(who) - 1);
                            cq[m] = ((unsigned long long)best << 32) | (0xFFFFFFFFu - vw);
                        }
                    }
                }
            }
            tc_fence_before();
            if (EPI != TC_PARTIAL) {
                epi_bar();
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int m = etid + 128 * i;
                    if (m < p.M) {
                        unsigned long long b = running[i];
                        for (int qq = 0; qq < 4 * p.tps; ++qq) {
                            const unsigned long long c = cand[((size_t)acc * p.tps * 4 + qq) * p.N_pad + m];
                            b = c > b ? c : b;
                        }
                        running[i] = b;
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty0 + 8 * acc);
        }
        if (!ok) {
            *abort_flag = 1;
            raise_error(p.err, SPEC_DEVERR_TIMEOUT);
        }
        if (EPI != TC_PARTIAL) {
            // every CTA folds its keys into one 64-bit maximum per row in global memory as it
            // finishes (order-independent, so the result is unique); the last CTA reads them
            for (int i = 0; i < 2; ++i) {
                const int m = etid + 128 * i;
                if (m < p.M) atomicMax(p.keys + m, running[i]);
            }
            __threadfence();
            epi_bar();
            if (etid == 0) {
                const unsigned prev = atomicAdd(p.counter, 1u);
                if (prev >= (unsigned)G) raise_error(p.err, SPEC_DEVERR_INTERNAL);  // counter not zeroed
                *last_flag = (prev == (unsigned)G - 1u) ? 1 : 0;
            }
            epi_bar();
            if (*last_flag) {
                __threadfence();
                for (int m = etid; m < p.M; m += 128) {
                    const unsigned long long b = atomicExch(p.keys + m, 0ull);  // read, and zero for the next call
                    int id = (int)(0xFFFFFFFFu - (uint32_t)(b & 0xFFFFFFFFull));
                    if (p.max_logit) p.max_logit[m] = key_float((uint32_t)(b >> 32));
                    if (id < 0 || id >= p.V) {
                        // cannot happen when every CTA published its keys; never index with it
                        raise_error(p.err, SPEC_DEVERR_INTERNAL);
                        p.ids[m] = -1;
                        continue;
                    }
                    if (p.d2t) {
                        const int tgt = __ldg(p.d2t + id);
                        if (tgt < 0 || tgt >= p.d2t_limit) {
                            raise_error(p.err, SPEC_DEVERR_D2T);
                            id = -1;
                        } else {
                            id = tgt;
                        }
                    }
                    p.ids[m] = id;
                }
                if (etid == 0) atomicExch(p.counter, 0u);
            }
        }
    }
    // ---------------- teardown ----------------
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, p.tmem_cols);
    }
}

// out[m][n] = bf16( sum_s partial[s][m][n] ), splits summed in ascending order.
__global__ void splitk_reduce_bf16_kernel(const float *__restrict__ partial, int splits, int M, int N,
                                          uint16_t *__restrict__ out) {
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    const size_t total = (size_t)M * N;
    if (i >= total) return;
    float s = 0.f;
    for (int k = 0; k < splits; ++k) s += __ldcg(partial + (size_t)k * total + i);
    __nv_bfloat16 b = __float2bfloat16_rn(s);
    out[i] = *reinterpret_cast<uint16_t *>(&b);
}

// ---- host side ---------------------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// 2-D bf16 row-major [rows][cols] map with a (64 x box_rows) box and 128-byte swizzle.
static bool make_map(CUtensorMap *map, const void *base, int rows, int cols, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)TC_BK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    return n;
}

struct TcPlan {
    TcParams p;
    int grid;
    size_t smem;
};

static int plan(int M, int V, int K, int splits, TcPlan &pl) {
    TcParams &p = pl.p;
    p = TcParams{};
    p.M = M;
    p.wait_ns = g_wait_ns;
    p.N_pad = ((M + 15) / 16) * 16;
    p.V = V;
    p.K = K;
    p.n_tiles = (V + TC_BM - 1) / TC_BM;
    p.n_kc = (K + TC_BK - 1) / TC_BK;
    p.splits = splits < 1 ? 1 : (splits > p.n_kc ? p.n_kc : splits);
    p.a_stage_bytes = (uint32_t)p.N_pad * TC_BK * 2;
    // Two W tiles per stage when both accumulators of both fit TMEM (N_pad <= 128): the
    // stage's hidden chunk then serves 256 W rows, which halves the hidden-row traffic per
    // weight byte (a pure TMA stream of 128-row boxes plus a hidden box ran ~12 % slower than
    // the W boxes alone; 256-row boxes with the hidden box ran within 1 % of it)
    p.tps = (p.N_pad <= 128 && V >= 2 * TC_BM) ? 2 : 1;
    p.n_groups = (p.n_tiles + p.tps - 1) / p.tps;
    p.w_stage_bytes = W_STAGE_BYTES * (uint32_t)p.tps;
    uint32_t cols = 32;
    while (cols < 2u * (uint32_t)(p.tps * p.N_pad)) cols <<= 1;
    p.tmem_cols = cols;
    const size_t fixed = 1024 + 8 * 64 + 64 + (size_t)2 * p.tps * 4 * p.N_pad * 8;
    const size_t stage = p.w_stage_bytes + p.a_stage_bytes;
    int stages = (int)((SMEM_LIMIT - fixed) / stage);
    const int max_stages = p.tps == 2 ? 6 : 8;
    if (stages > max_stages) stages = max_stages;
    if (stages < 2) return SPEC_ERR_UNSUPPORTED;
    p.stages = stages;
    pl.smem = fixed + (size_t)stages * stage;
    const int sms = sm_count();
    if (sms < 1) return SPEC_ERR_CUDA;
    const int work = p.n_groups * p.splits;
    int g = work < sms ? work : sms;
    if (g > MAX_CTAS) g = MAX_CTAS;
    pl.grid = g;
    return SPEC_OK;
}

template <int EPI>
static int launch_tc(const void *A, const void *W, TcPlan &pl, cudaStream_t s) {
    CUtensorMap mw, ma;
    if (!make_map(&mw, W, pl.p.V, pl.p.K, TC_BM * pl.p.tps) || !make_map(&ma, A, pl.p.M, pl.p.K, pl.p.N_pad))
        return SPEC_ERR_CUDA;
    // Always the same ceiling, never the launch's own size: a CUDA graph may hold launches
    // of this kernel with different shared-memory sizes, and lowering the attribute for a
    // later launch would leave an earlier captured one above the function's maximum.
    if (cudaFuncSetAttribute(tc_skinny_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_LIMIT) !=
        cudaSuccess)
        return SPEC_ERR_CUDA;
    tc_skinny_kernel<EPI><<<pl.grid, TC_THREADS, pl.smem, s>>>(mw, ma, pl.p);
    return launch_status();
}

static size_t lmhead_ws_bytes(int M, int V) {
    const size_t tiles = (size_t)(V + TC_BM - 1) / TC_BM;
    const size_t ctas = tiles < (size_t)MAX_CTAS ? tiles : (size_t)MAX_CTAS;
    return 256 + ctas * (size_t)M * sizeof(unsigned long long);
}

static int lmhead_run(const void *hidden, const void *W, int M, int V, int H, const int32_t *d2t, int d2t_limit,
                      int32_t *ids, float *max_logit, float *logits, void *ws, size_t ws_bytes, int32_t *dev_err,
                      cudaStream_t s) {
    if (!hidden || !W || !ids) return SPEC_ERR_NULL;
    if (M < 1 || M > 256 || V < 1 || H < 8 || (H & 7)) return SPEC_ERR_ARG;
    if (d2t && d2t_limit < 1) return SPEC_ERR_ARG;
    if (!ws || ws_bytes < lmhead_ws_bytes(M, V)) return SPEC_ERR_WORKSPACE;
    if (!aligned16(hidden) || !aligned16(W) || (reinterpret_cast<uintptr_t>(ws) & 255u)) return SPEC_ERR_ALIGN;
    TcPlan pl;
    int st = plan(M, V, H, 1, pl);
    if (st) return st;
    TcParams &p = pl.p;
    p.counter = (unsigned int *)ws;
    p.keys = (unsigned long long *)((char *)ws + 256);
    p.logits = logits;
    p.d2t = d2t;
    p.d2t_limit = d2t_limit;
    p.ids = ids;
    p.max_logit = max_logit;
    p.err = dev_err;
    return logits ? launch_tc<TC_LOGITS>(hidden, W, pl, s) : launch_tc<TC_ARGMAX>(hidden, W, pl, s);
}

size_t gemm_store_ws_bytes(int M, int N, int K) {
    (void)K;
    return (size_t)MAX_SPLITS * M * N * sizeof(float);
}

int gemm_store_bf16(const void *A, const void *W, int M, int N, int K, void *out, void *ws, size_t ws_bytes,
                    cudaStream_t s) {
    if (M < 1 || M > 256 || N < 1 || K < 8 || (K & 7)) return SPEC_ERR_ARG;
    if (ws_bytes < gemm_store_ws_bytes(M, N, K)) return SPEC_ERR_WORKSPACE;
    const int sms = sm_count();
    if (sms < 1) return SPEC_ERR_CUDA;
    TcPlan pl;
    int st = plan(M, N, K, 1, pl);  // for the number of tile groups
    if (st) return st;
    int splits = sms / pl.p.n_groups;
    if (splits < 1) splits = 1;
    if (splits > MAX_SPLITS) splits = MAX_SPLITS;
    st = plan(M, N, K, splits, pl);
    if (st) return st;
    pl.p.partial = (float *)ws;
    st = launch_tc<TC_PARTIAL>(A, W, pl, s);
    if (st) return st;
    const size_t total = (size_t)M * N;
    splitk_reduce_bf16_kernel<<<(unsigned)((total + 255) / 256), 256, 0, s>>>((const float *)ws, pl.p.splits, M, N,
                                                                             (uint16_t *)out);
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

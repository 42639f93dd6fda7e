// verify_attn.cu -- a2: causal GQA verify attention over paged KV (split-KV flash-decode
// on tcgen05 tensor cores).
//
// Row r = b*(k+1)+j (position p = pos[b]+j) and q head h attend keys 0..p of branch b
// (kv head h / G): span-02 engine/crates/model/src/spec.rs, module documentation
// (kv_hi = position, rejected-row KV beyond pos is never attended); memra-engine
// src/spec.rs, `full_attn_verify` (row r sees keys [0, base_len + r + 1), all verify
// rows in one launch); memra-engine `MtpScratch` (split count fixed by capacity, not by
// the current length, so one program serves every length bit for bit).
//
// Work unit = (branch b, kv head g, split of SPLIT_KEYS positions). The (k+1)*G query
// vectors that share kv head g form the N side of the MMAs, the keys the M side:
//     S^T[128 keys x N] = K_tile[128 x d] . Q^T            (tcgen05, fp32 in TMEM)
//     O^T[d x N]       += V_tile^T[d x 128] . P^T[128 x N]  (V read MN-major)
// A persistent CTA per SM walks its units. Warp 0 gathers each 128-key K / V tile from
// the branch's pages with TMA (one box per page and 64-element column block, 128-byte
// swizzle) into a shared-memory ring; for FP8 pools it gathers the raw E4M3 bytes and
// warps 6..9 convert them to f16 operand tiles (E4M3 is exact in f16). Warp 1 issues the
// MMAs. Warps 2..5 do the softmax in two passes over the split, whose S tiles all stay in
// TMEM: pass A takes each column's maximum over the split's keys (one cross-lane
// reduction per column per split), pass B writes P = exp2(s - m) to shared memory for
// P.V and sums it per thread (one cross-lane sum per column per split). O accumulates in
// TMEM without rescaling; only when a split's S tiles do not fit in TMEM at once is it
// processed in chunks, with O rescaled between chunks. Keys beyond a row's position are
// set to -inf by select, never multiplied; V rows past the branch's last position are
// zeroed. A combine pass merges the splits of each (row, head) in ascending order.
// Tile and split boundaries sit at fixed key positions, every column of an MMA is
// computed independently of the others, and masked keys contribute exact zeros, so a
// row's output is identical whatever B, k or batch it is verified in.
// Every pipeline wait is bounded (1 s): on a timeout the kernel raises
// SPEC_DEVERR_TIMEOUT, lets issued copies and MMAs land, frees TMEM and exits.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <math.h>

#include "common.cuh"
#include "sm100.cuh"

namespace spec {

using namespace sm100;

constexpr int SPLIT_KEYS = 1024;
constexpr int TILE_KEYS = 128;
constexpr float LOG2E = 1.4426950408889634f;
constexpr float P_SCALE_FP8 = 1024.0f;   // f16 P is stored x 2^10 to stay clear of f16 subnormals
constexpr uint64_t ATT_WAIT_NS = 1000000000ull;
constexpr int ATT_SMEM_LIMIT = 227 * 1024;
constexpr int MAX_NPAD = 64;      // query vectors per (branch, kv head), padded to 16
constexpr int MAX_TS = 8;         // = SPLIT_KEYS / TILE_KEYS
constexpr uint32_t P_BUF = TILE_KEYS * 128;  // one P buffer: 128 keys x 64 columns, MN-major

struct AttnTcParams {
    KvView kv;
    const int32_t *pos;
    int B, k, Hq, G, n_q, N_pad, n_splits, max_pos, n_units;
    const uint16_t *q;     // bf16 [R][Hq][d]
    float scale_log2;      // softmax scale * log2(e)
    float *ws_ml;          // [units][n_q][2]  (m in log2 units, l)
    float *ws_o;           // [units][n_q][d]
    int32_t *err;
    int NS, NR;            // operand / raw ring depth
    int TS, OB;            // S tiles held in TMEM at once (a chunk), O buffers (1 or 2)
    uint32_t tmem_cols;
    uint32_t off_q, off_p, off_raw, off_bar, off_small;  // shared-memory offsets
};

template <int D, bool FP8>
struct AttnShape {
    static constexpr int NATOM = D / 64;                    // 128-byte column blocks of a 16-bit row
    static constexpr int OP_ATOMS = NATOM < 2 ? 2 : NATOM;  // V^T needs 2 blocks for M = 128
    static constexpr uint32_t OP_STAGE = OP_ATOMS * TILE_KEYS * 128;
    static constexpr uint32_t RAW_STAGE = FP8 ? TILE_KEYS * D : 0;
    static constexpr int NB = D <= 128 ? 1 : 2;            // 128-row blocks of d for P.V
    static constexpr int THREADS = FP8 ? 320 : 192;
};

struct UnitInfo {
    int b, g, split, pos_b, kv_end, s0, T, n_chunks;
    bool bad_pos;
};

__device__ __forceinline__ UnitInfo unit_info(const AttnTcParams &p, int u) {
    UnitInfo ui;
    ui.split = u % p.n_splits;
    ui.g = (u / p.n_splits) % p.kv.n_kv_heads;
    ui.b = u / (p.n_splits * p.kv.n_kv_heads);
    ui.pos_b = __ldg(p.pos + ui.b);
    ui.bad_pos = ui.pos_b < 0 || ui.pos_b + p.k + 1 > p.max_pos;
    ui.kv_end = ui.pos_b + p.k + 1;
    ui.s0 = ui.split * SPLIT_KEYS;
    int n = ui.bad_pos ? 0 : ui.kv_end - ui.s0;
    n = n < 0 ? 0 : (n > SPLIT_KEYS ? SPLIT_KEYS : n);
    ui.T = (n + TILE_KEYS - 1) / TILE_KEYS;
    ui.n_chunks = (ui.T + p.TS - 1) / p.TS;
    return ui;
}

// byte offset of 16-bit element (row, col) in a K-major, 128-byte-swizzled operand whose
// 64-column blocks are `block_bytes` apart
__device__ __forceinline__ uint32_t sw128_off(int row, int col, uint32_t block_bytes) {
    const int blk = col >> 6, c = col & 63;
    return blk * block_bytes + row * 128 + ((((c >> 3) ^ (row & 7)) & 7) << 4) + ((c & 7) << 1);
}

__device__ __forceinline__ float warp_max(float v) {
    // orderable-key maximum over the warp
    uint32_t u = __float_as_uint(v);
    uint32_t k = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    k = __reduce_max_sync(0xFFFFFFFFu, k);
    u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
    return __uint_as_float(u);
}

// Every lane waits; the verdict is made uniform across the warp so that no lane can
// leave a loop that the others stay in.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag) {
    const bool r = mbar_wait(bar, parity, abort_flag, ATT_WAIT_NS);
    return __all_sync(0xFFFFFFFFu, r);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
    return v;
}

template <int D, bool FP8>
__global__ void __launch_bounds__(AttnShape<D, FP8>::THREADS, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                   AttnTcParams p) {
    using S_ = AttnShape<D, FP8>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t s_op = smem_u32(smem);
    const uint32_t s_q = s_op + p.off_q, s_p = s_op + p.off_p, s_rawb = s_op + p.off_raw;
    uint8_t *g_q = smem + p.off_q;
    uint8_t *g_p = smem + p.off_p;
    const int N_pad = p.N_pad, n_q = p.n_q, TS = p.TS;
    // barrier map
    const uint32_t op_full = s_op + p.off_bar, op_empty = op_full + 8 * p.NS;
    const uint32_t raw_full = op_empty + 8 * p.NS, raw_empty = raw_full + 8 * p.NR;
    const uint32_t sfull = raw_empty + 8 * p.NR, sfree = sfull + 8 * TS;   // per S slot
    const uint32_t pfull = sfree + 8 * TS, pfree = pfull + 16;             // P double buffer
    const uint32_t ochunk = pfree + 16, ofree = ochunk + 8, qready = ofree + 16, drain = qready + 8;
    uint8_t *small = smem + p.off_small;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(small);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(small + 4);
    volatile int *fail_flag = reinterpret_cast<volatile int *>(small + 8);
    volatile int *corr_flag = reinterpret_cast<volatile int *>(small + 12);
    float *red_max = reinterpret_cast<float *>(small + 64);  // [4][N_pad]
    float *red_sum = red_max + 4 * N_pad;                    // [4][N_pad]
    float *cor = red_sum + 4 * N_pad;                        // [N_pad]
    float *mnew = cor + N_pad;
    float *mrun = mnew + N_pad;
    float *lrun = mrun + N_pad;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.NS; ++s) {
            mbar_init(op_full + 8 * s, FP8 ? 4 : 1);
            mbar_init(op_empty + 8 * s, 1);
        }
        for (int s = 0; s < p.NR; ++s) {
            mbar_init(raw_full + 8 * s, 1);
            mbar_init(raw_empty + 8 * s, 4);
        }
        for (int s = 0; s < TS; ++s) {
            mbar_init(sfull + 8 * s, 1);
            mbar_init(sfree + 8 * s, 4);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(pfull + 8 * a, 4);
            mbar_init(pfree + 8 * a, 1);
            mbar_init(ofree + 8 * a, 4);
        }
        mbar_init(ochunk, 1);
        mbar_init(qready, 4);
        mbar_init(drain, 1);
        *abort_flag = 0;
        *fail_flag = 0;
        *corr_flag = 0;
        fence_mbar_init();
    }
    if (D == 64) {
        // the second 64-row block of every V^T operand must read zeros
        for (uint32_t i = threadIdx.x; i < (uint32_t)p.NS * S_::OP_STAGE / 16; i += blockDim.x)
            reinterpret_cast<uint4 *>(smem)[i] = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&map_k);
        prefetch_tmap(&map_v);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), p.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t t_o = tmem + (uint32_t)(TS * N_pad);  // S slots first, then O buffers

    const int BR = p.kv.page_size < TILE_KEYS ? p.kv.page_size : TILE_KEYS;  // rows per gather box
    const int n_chunks_tile = TILE_KEYS / BR;

    if (warp == 0) {
        // ================= producer: page-gathered loads, per chunk K tiles then V tiles =================
        uint32_t gi = 0;
        bool ok = true;
        const uint32_t per_box = FP8 ? (uint32_t)(BR * D) : (uint32_t)(BR * 128 * S_::NATOM);
        for (int u = blockIdx.x; u < p.n_units && ok; u += gridDim.x) {
            const UnitInfo ui = unit_info(p, u);
            for (int ch = 0; ch < ui.n_chunks && ok; ++ch) {
                const int t0 = ch * TS, t1 = min(ui.T, t0 + TS);
                for (int kv = 0; kv < 2 && ok; ++kv) {
                    const CUtensorMap *map = kv ? &map_v : &map_k;
                    for (int t = t0; t < t1; ++t, ++gi) {
                        const int key0 = ui.s0 + t * TILE_KEYS;
                        int rows[4];  // box row of chunk lane, lane+32, ... (<= 128 chunks)
                        uint32_t nvalid = 0;
#pragma unroll
                        for (int rr = 0; rr < 4; ++rr) {
                            const int c = rr * 32 + lane;
                            const int kc = key0 + c * BR;
                            int row0 = -1;
                            if (c < n_chunks_tile && kc < ui.kv_end) {
                                const int pg = page_of(p.kv, ui.b, kc);
                                if (pg >= 0)
                                    row0 = (pg * p.kv.n_kv_heads + ui.g) * p.kv.page_size +
                                           (kc & (p.kv.page_size - 1));
                                else if (kv == 0)
                                    raise_error(p.err, -pg);
                            }
                            rows[rr] = row0;
                            nvalid += __popc(__ballot_sync(0xFFFFFFFFu, row0 >= 0));
                        }
                        uint32_t dst_base, bar;
                        if (FP8) {
                            const uint32_t s = gi % p.NR, ph = (gi / p.NR) & 1u;
                            if (!warp_wait(raw_empty + 8 * s, ph ^ 1u, abort_flag)) { ok = false; break; }
                            dst_base = s_rawb + s * S_::RAW_STAGE;
                            bar = raw_full + 8 * s;
                        } else {
                            const uint32_t s = gi % p.NS, ph = (gi / p.NS) & 1u;
                            if (!warp_wait(op_empty + 8 * s, ph ^ 1u, abort_flag)) { ok = false; break; }
                            dst_base = s_op + s * S_::OP_STAGE;
                            bar = op_full + 8 * s;
                        }
                        if (BR < 8) {
                            // pages smaller than one 8-row swizzle atom: gather with plain copies
                            // (a TMA box would not start on a 1024-byte boundary)
                            const uint8_t *pool = reinterpret_cast<const uint8_t *>(kv ? p.kv.v_pool : p.kv.k_pool);
                            uint8_t *dst = smem + (dst_base - s_op);
                            constexpr int CH = FP8 ? D / 16 : D / 8;  // 16-byte pieces per row
                            for (int i = lane; i < TILE_KEYS * CH; i += 32) {
                                const int row = i / CH, chn = i % CH;
                                const int key = key0 + row;
                                if (key >= ui.kv_end) continue;
                                const int pg = page_of(p.kv, ui.b, key);
                                if (pg < 0) continue;
                                const size_t elem = ((size_t)(pg * p.kv.n_kv_heads + ui.g) * p.kv.page_size +
                                                     (key & (p.kv.page_size - 1))) * D;
                                if (FP8) {
                                    *reinterpret_cast<uint4 *>(dst + row * D + chn * 16) =
                                        __ldg(reinterpret_cast<const uint4 *>(pool + elem + chn * 16));
                                } else {
                                    *reinterpret_cast<uint4 *>(dst + sw128_off(row, chn * 8, TILE_KEYS * 128)) =
                                        __ldg(reinterpret_cast<const uint4 *>(pool + 2 * elem + chn * 16));
                                }
                            }
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(bar);
                            __syncwarp();
                            continue;
                        }
                        if (lane == 0) {
                            if (nvalid) mbar_arrive_expect_tx(bar, nvalid * per_box);
                            else mbar_arrive(bar);
                        }
#pragma unroll
                        for (int rr = 0; rr < 4; ++rr) {
                            if (rr * 32 >= n_chunks_tile) break;
                            for (int cc = 0; cc < 32; ++cc) {
                                const int c = rr * 32 + cc;
                                if (c >= n_chunks_tile) break;
                                const int row0 = __shfl_sync(0xFFFFFFFFu, rows[rr], cc);
                                if (lane == 0 && row0 >= 0) {
                                    if (FP8) {
                                        tma_load_2d(dst_base + c * BR * D, map, 0, row0, bar);
                                    } else {
#pragma unroll
                                        for (int a = 0; a < S_::NATOM; ++a)
                                            tma_load_2d(dst_base + a * (TILE_KEYS * 128) + c * BR * 128, map, a * 64,
                                                        row0, bar);
                                    }
                                }
                            }
                        }
                        __syncwarp();
                    }
                }
            }
        }
        if (!ok) {
            *abort_flag = 1;
            if (lane == 0) raise_error(p.err, SPEC_DEVERR_TIMEOUT);
        }
        // let copies still in flight land before the CTA may exit
        if (lane == 0) {
            const uint32_t depth = FP8 ? p.NR : p.NS;
            const uint32_t n_last = gi < depth ? gi : depth;
            for (uint32_t j = 0; j < n_last; ++j) {
                const uint32_t i2 = gi - 1 - j;
                mbar_wait((FP8 ? raw_full : op_full) + 8 * (i2 % depth), (i2 / depth) & 1u, nullptr, ATT_WAIT_NS);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ================= MMA issuer =================
        const uint32_t idesc_s = idesc_f16kind(128, N_pad, FP8, false, false);
        const uint32_t idesc_pv = idesc_f16kind(128, N_pad, FP8, true, true);
        const uint32_t qblk = (uint32_t)N_pad * 128;
        uint32_t gi = 0, gt = 0, ul = 0;
        uint32_t slot_use[MAX_TS];
#pragma unroll
        for (int s = 0; s < MAX_TS; ++s) slot_use[s] = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < p.n_units && ok; u += gridDim.x) {
            const UnitInfo ui = unit_info(p, u);
            if (ui.T == 0) continue;
            const uint32_t ob = p.OB == 2 ? (ul & 1u) : 0u;
            const uint32_t ob_use = p.OB == 2 ? (ul >> 1) : ul;
            if (!warp_wait(qready, ul & 1u, abort_flag) ||
                !warp_wait(ofree + 8 * ob, (ob_use & 1u) ^ 1u, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            for (int ch = 0; ch < ui.n_chunks && ok; ++ch) {
                const int t0 = ch * TS, t1 = min(ui.T, t0 + TS);
                // S of every tile of the chunk
                for (int t = t0; t < t1; ++t, ++gi) {
                    const int slot = t - t0;
                    uint32_t su = 0;
#pragma unroll
                    for (int s = 0; s < MAX_TS; ++s)
                        if (s == slot) su = slot_use[s];
                    const uint32_t st = gi % p.NS;
                    if (!warp_wait(op_full + 8 * st, (gi / p.NS) & 1u, abort_flag) ||
                        !warp_wait(sfree + 8 * slot, (su & 1u) ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (lane == 0) {
                        const uint32_t a_base = s_op + st * S_::OP_STAGE;
#pragma unroll
                        for (int ks = 0; ks < D / 16; ++ks) {
                            const uint32_t blk = ks >> 2, off = (ks & 3) * 32;
                            mma_bf16(tmem + slot * N_pad, desc_kmajor_sw128(a_base + blk * (TILE_KEYS * 128) + off),
                                     desc_kmajor_sw128(s_q + blk * qblk + off), idesc_s, ks > 0 ? 1u : 0u);
                        }
                        mma_commit(op_empty + 8 * st);
                        mma_commit(sfull + 8 * slot);
                    }
                    __syncwarp();
#pragma unroll
                    for (int s = 0; s < MAX_TS; ++s)
                        if (s == slot) slot_use[s] = su + 1;
                }
                if (!ok) break;
                // P.V of every tile of the chunk, in order
                for (int t = t0; t < t1; ++t, ++gi, ++gt) {
                    const uint32_t st = gi % p.NS;
                    if (!warp_wait(op_full + 8 * st, (gi / p.NS) & 1u, abort_flag)) { ok = false; break; }
                    const int key0 = ui.s0 + t * TILE_KEYS;
                    const int nvk = ui.kv_end - key0;  // valid keys in this tile
                    if (nvk < TILE_KEYS) {
                        // keys past the branch's last position: zero their V rows (NaN-safe P.V)
                        uint4 *vb = reinterpret_cast<uint4 *>(smem + st * S_::OP_STAGE);
                        const int rows = TILE_KEYS - nvk;
                        for (int i = lane; i < rows * S_::NATOM * 8; i += 32) {
                            const int a = i / (rows * 8), rem = i % (rows * 8);
                            const int r = nvk + rem / 8, c = rem % 8;
                            vb[(a * TILE_KEYS * 128 + r * 128) / 16 + c] = make_uint4(0, 0, 0, 0);
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                    }
                    const uint32_t pb = gt & 1u;
                    if (!warp_wait(pfull + 8 * pb, (gt >> 1) & 1u, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    if (lane == 0) {
                        const uint32_t vbase = s_op + st * S_::OP_STAGE, pbase = s_p + pb * P_BUF;
#pragma unroll
                        for (int nb = 0; nb < S_::NB; ++nb) {
#pragma unroll
                            for (int ks = 0; ks < TILE_KEYS / 16; ++ks) {
                                const uint64_t ad = desc_mnmajor_sw128(vbase + (2 * nb) * (TILE_KEYS * 128) + ks * 2048,
                                                                       TILE_KEYS * 128);
                                const uint64_t bd = desc_mnmajor_sw128(pbase + ks * 2048, P_BUF);
                                mma_bf16(t_o + (ob * S_::NB + nb) * N_pad, ad, bd, idesc_pv, (t > 0 || ks > 0) ? 1u : 0u);
                            }
                        }
                        mma_commit(op_empty + 8 * st);
                        mma_commit(pfree + 8 * pb);
                    }
                    __syncwarp();
                }
                if (!ok) break;
                if (lane == 0) mma_commit(ochunk);
                __syncwarp();
            }
            if (!ok) break;
            ++ul;
        }
        if (!ok) {
            *abort_flag = 1;
            if (lane == 0) raise_error(p.err, SPEC_DEVERR_TIMEOUT);
        }
        if (lane == 0) {
            mma_commit(drain);
            mbar_wait(drain, 0, nullptr, ATT_WAIT_NS);
            // every arrive sent by this thread's commits is delivered before the CTA may exit:
            // the last phase of each operand stage's "empty" barrier and of both P buffers'
            // "free" barriers (the others were waited on by their consumers)
            const uint32_t n_last = gi < (uint32_t)p.NS ? gi : (uint32_t)p.NS;
            for (uint32_t j = 0; j < n_last; ++j) {
                const uint32_t i2 = gi - 1 - j;
                mbar_wait(op_empty + 8 * (i2 % p.NS), (i2 / p.NS) & 1u, nullptr, ATT_WAIT_NS);
            }
            for (uint32_t j = 0; j < 2 && j < gt; ++j) {
                const uint32_t t2 = gt - 1 - j;
                mbar_wait(pfree + 8 * (t2 & 1u), (t2 >> 1) & 1u, nullptr, ATT_WAIT_NS);
            }
        }
        __syncwarp();
    } else if (warp < 6) {
        // ================= softmax / output: 4 warps, TMEM lane quadrant = warp % 4 =================
        // The named-barrier sequence below does not depend on `ok`: after a failed wait a warp
        // keeps stepping through the barriers and only skips the work, so no warp is left
        // waiting at a barrier that another warp will never reach.
        const int q = warp & 3;
        const int etid = threadIdx.x - 64;  // 0..127
        const int kk = q * 32 + lane;       // key within a tile / d row within a 128-block
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        const uint32_t qblk = (uint32_t)N_pad * 128;
        uint32_t gt = 0, gch = 0, ul = 0;
        uint32_t slot_use[MAX_TS];
#pragma unroll
        for (int s = 0; s < MAX_TS; ++s) slot_use[s] = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < p.n_units; u += gridDim.x) {
            const UnitInfo ui = unit_info(p, u);
            float *ml = p.ws_ml + (size_t)u * n_q * 2;
            if (ui.T == 0) {
                if (ui.bad_pos && ui.split == 0 && ui.g == 0 && etid == 0) raise_error(p.err, SPEC_DEVERR_POS);
                for (int c = etid; c < n_q; c += 128) {
                    ml[2 * c] = -INFINITY;
                    ml[2 * c + 1] = ui.bad_pos ? -1.f : 0.f;
                }
                continue;
            }
            // ---- Q of (b, g): rows j*G + i -> q[b*(k+1)+j][g*G+i][:], zero padding rows ----
            for (int i = etid; i < N_pad * (D / 8); i += 128) {
                const int row = i / (D / 8), cc = i % (D / 8);
                uint4 v = make_uint4(0, 0, 0, 0);
                if (row < n_q) {
                    const int j = row / p.G, hi = row % p.G;
                    const uint16_t *src = p.q + ((size_t)(ui.b * (p.k + 1) + j) * p.Hq + ui.g * p.G + hi) * D + cc * 8;
                    v = __ldg(reinterpret_cast<const uint4 *>(src));
                    if (FP8) {
                        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
                        uint32_t h[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            __half2 hh = __floats2half2_rn(bf16_lo(w[e]), bf16_hi(w[e]));
                            h[e] = *reinterpret_cast<uint32_t *>(&hh);
                        }
                        v = make_uint4(h[0], h[1], h[2], h[3]);
                    }
                }
                *reinterpret_cast<uint4 *>(g_q + sw128_off(row, cc * 8, qblk)) = v;
            }
            fence_proxy_async_smem();
            if (etid < N_pad) {
                mrun[etid] = -INFINITY;
                lrun[etid] = 0.f;
            }
            if (etid == 0) *fail_flag = 0;
            __syncwarp();
            if (lane == 0) mbar_arrive(qready);
            named_bar(1, 128);
            const uint32_t ob = p.OB == 2 ? (ul & 1u) : 0u;
            bool failed = false;
            for (int ch = 0; ch < ui.n_chunks; ++ch) {
                const int t0 = ch * TS, t1 = min(ui.T, t0 + TS);
                // ---- pass A: each column's maximum over the chunk's keys ----
                float mth[MAX_NPAD];
#pragma unroll
                for (int c = 0; c < MAX_NPAD; ++c) mth[c] = -INFINITY;
                for (int t = t0; t < t1; ++t) {
                    const int slot = t - t0;
                    uint32_t su = 0;
#pragma unroll
                    for (int s = 0; s < MAX_TS; ++s)
                        if (s == slot) su = slot_use[s];
                    // this key is seen by the columns [cth, cend): rows j with key <= pos_b + j
                    const int key = ui.s0 + t * TILE_KEYS + kk;
                    int cth = 0, cend = 0;
                    float ksc = 1.f;
                    if (key < ui.kv_end) {
                        const int pg = page_of(p.kv, ui.b, key);
                        if (pg < 0) failed = true;
                        else if (FP8) ksc = __ldg(p.kv.k_scale + (size_t)pg * p.kv.n_kv_heads + ui.g);
                        const int J = key - ui.pos_b;
                        cth = J > 0 ? J * p.G : 0;
                        cend = n_q;
                    }
                    if (ok) ok = warp_wait(sfull + 8 * slot, su & 1u, abort_flag);
                    if (!ok) continue;
                    tc_fence_after();
                    const float sl = p.scale_log2 * ksc;
#pragma unroll
                    for (int c0 = 0; c0 < MAX_NPAD; c0 += 16) {
                        if (c0 < n_q) {
                            uint32_t r[16];
                            tmem_ld16(tmem + lane_base + slot * N_pad + c0, r);
                            tmem_ld_wait();
#pragma unroll
                            for (int j = 0; j < 16; ++j) {
                                const int c = c0 + j;
                                const float v = __uint_as_float(r[j]) * sl;
                                if (c >= cth && c < cend) mth[c] = fmaxf(mth[c], v);
                            }
                        }
                    }
                }
#pragma unroll
                for (int c = 0; c < MAX_NPAD; ++c) {
                    if (c < n_q) {
                        const float mx = warp_max(mth[c]);
                        if (lane == 0) red_max[q * N_pad + c] = mx;
                    }
                }
                named_bar(1, 128);
                if (etid < n_q) {
                    const float mt = fmaxf(fmaxf(red_max[etid], red_max[N_pad + etid]),
                                           fmaxf(red_max[2 * N_pad + etid], red_max[3 * N_pad + etid]));
                    const float mo = mrun[etid];
                    const float mn = fmaxf(mo, mt);
                    const float cr = (mn == -INFINITY) ? 1.f : exp2f(mo - mn);
                    cor[etid] = cr;
                    mnew[etid] = mn;
                    mrun[etid] = mn;
                    if (ch > 0 && cr != 1.f) *corr_flag = 1;
                }
                named_bar(1, 128);
                // ---- a later chunk whose maximum grew: rescale O once all earlier P.V are done ----
                if (ch > 0 && *corr_flag) {
                    if (ok) ok = warp_wait(ochunk, (gch - 1) & 1u, abort_flag);
                    if (ok) {
                        tc_fence_after();
#pragma unroll
                        for (int nb = 0; nb < S_::NB; ++nb) {
                            const uint32_t o_addr = t_o + lane_base + (ob * S_::NB + nb) * N_pad;
                            for (int c0 = 0; c0 < n_q; c0 += 16) {
                                uint32_t r[16];
                                tmem_ld16(o_addr + c0, r);
                                tmem_ld_wait();
#pragma unroll
                                for (int j = 0; j < 16; ++j)
                                    r[j] = __float_as_uint(__uint_as_float(r[j]) * cor[c0 + j]);
                                tmem_st16(o_addr + c0, r);
                            }
                        }
                        tmem_st_wait();
                        tc_fence_before();
                    }
                }
                // ---- pass B: P = exp2(s - m) for P.V, per-thread sums ----
                float lth[MAX_NPAD];
#pragma unroll
                for (int c = 0; c < MAX_NPAD; ++c) lth[c] = 0.f;
                for (int t = t0; t < t1; ++t, ++gt) {
                    const int slot = t - t0;
                    const int key = ui.s0 + t * TILE_KEYS + kk;
                    int cth = 0, cend = 0;
                    float ksc = 1.f, vsc = 1.f;
                    if (key < ui.kv_end) {
                        if (FP8) {
                            const int pg = page_of(p.kv, ui.b, key);
                            if (pg >= 0) {
                                const size_t si = (size_t)pg * p.kv.n_kv_heads + ui.g;
                                ksc = __ldg(p.kv.k_scale + si);
                                vsc = __ldg(p.kv.v_scale + si) * P_SCALE_FP8;
                            }
                        }
                        const int J = key - ui.pos_b;
                        cth = J > 0 ? J * p.G : 0;
                        cend = n_q;
                    }
                    const uint32_t pb = gt & 1u;
                    if (ok) ok = warp_wait(pfree + 8 * pb, ((gt >> 1) & 1u) ^ 1u, abort_flag);
                    if (!ok) continue;
                    const float sl = p.scale_log2 * ksc;
                    // this key's row of P (MN-major: the columns are contiguous, 128-byte swizzle)
                    uint8_t *prow = g_p + pb * P_BUF + kk * 128;
                    const int swz = kk & 7;
#pragma unroll
                    for (int c0 = 0; c0 < MAX_NPAD; c0 += 16) {
                        if (c0 < N_pad) {
                            uint32_t pk[8];
                            if (c0 < n_q) {
                                uint32_t r[16];
                                tmem_ld16(tmem + lane_base + slot * N_pad + c0, r);
                                float mv[16];
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    const float4 m4 = reinterpret_cast<const float4 *>(mnew + c0)[e];
                                    mv[4 * e] = m4.x;
                                    mv[4 * e + 1] = m4.y;
                                    mv[4 * e + 2] = m4.z;
                                    mv[4 * e + 3] = m4.w;
                                }
                                tmem_ld_wait();
#pragma unroll
                                for (int j = 0; j < 16; j += 2) {
                                    const int c = c0 + j;
                                    float a = ex2_approx(fmaf(__uint_as_float(r[j]), sl, -mv[j]));
                                    float b = ex2_approx(fmaf(__uint_as_float(r[j + 1]), sl, -mv[j + 1]));
                                    a = (c >= cth && c < cend) ? a : 0.f;
                                    b = (c + 1 >= cth && c + 1 < cend) ? b : 0.f;
                                    lth[c] += a;
                                    lth[c + 1] += b;
                                    if (FP8) {
                                        const __half2 h = __floats2half2_rn(a * vsc, b * vsc);
                                        pk[j >> 1] = *reinterpret_cast<const uint32_t *>(&h);
                                    } else {
                                        const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
                                        pk[j >> 1] = *reinterpret_cast<const uint32_t *>(&h);
                                    }
                                }
                            } else {
#pragma unroll
                                for (int e = 0; e < 8; ++e) pk[e] = 0u;
                            }
                            const int ch0 = c0 >> 3;
                            *reinterpret_cast<uint4 *>(prow + (((ch0 ^ swz) & 7) << 4)) =
                                make_uint4(pk[0], pk[1], pk[2], pk[3]);
                            *reinterpret_cast<uint4 *>(prow + ((((ch0 + 1) ^ swz) & 7) << 4)) =
                                make_uint4(pk[4], pk[5], pk[6], pk[7]);
                        }
                    }
                    tc_fence_before();
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(sfree + 8 * slot);
                        mbar_arrive(pfull + 8 * pb);
                    }
                }
#pragma unroll
                for (int s = 0; s < MAX_TS; ++s)
                    if (s < t1 - t0) slot_use[s] += 1;
                // ---- one cross-lane sum per column ----
#pragma unroll
                for (int c = 0; c < MAX_NPAD; ++c) {
                    if (c < n_q) {
                        const float sm = warp_sum(lth[c]);
                        if (lane == 0) red_sum[q * N_pad + c] = sm;
                    }
                }
                named_bar(1, 128);
                if (etid < n_q)
                    lrun[etid] = lrun[etid] * cor[etid] + ((red_sum[etid] + red_sum[N_pad + etid]) +
                                                           (red_sum[2 * N_pad + etid] + red_sum[3 * N_pad + etid]));
                if (etid == 0) *corr_flag = 0;
                ++gch;
                named_bar(1, 128);
            }
            if (failed) *fail_flag = 1;
            // the unit's last P.V, then its partial
            if (ok) {
                ok = warp_wait(ochunk, (gch - 1) & 1u, abort_flag);
                if (ok) tc_fence_after();
            }
            named_bar(1, 128);
            if (ok) {
                float *o_ws = p.ws_o + (size_t)u * n_q * D;
                const float oscale = FP8 ? 1.f / P_SCALE_FP8 : 1.f;
#pragma unroll
                for (int nb = 0; nb < S_::NB; ++nb) {
                    const uint32_t o_addr = t_o + lane_base + (ob * S_::NB + nb) * N_pad;
                    const int drow = nb * 128 + kk;
                    for (int c0 = 0; c0 < n_q; c0 += 16) {
                        uint32_t r[16];
                        tmem_ld16(o_addr + c0, r);
                        tmem_ld_wait();
                        if (drow < D) {
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                if (c0 + j < n_q) o_ws[(size_t)(c0 + j) * D + drow] = __uint_as_float(r[j]) * oscale;
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(ofree + 8 * ob);
            }
            const bool unit_failed = *fail_flag != 0;
            for (int c = etid; c < n_q; c += 128) {
                ml[2 * c] = mrun[c];
                ml[2 * c + 1] = (unit_failed || !ok) ? -1.f : lrun[c];
            }
            if (unit_failed && etid == 0) raise_error(p.err, SPEC_DEVERR_PAGE);
            ++ul;
            named_bar(1, 128);
        }
        if (!ok) {
            *abort_flag = 1;
            if (etid == 0) raise_error(p.err, SPEC_DEVERR_TIMEOUT);
        }
    } else if (FP8) {
        // ================= E4M3 -> f16 operand conversion: warps 6..9 =================
        const int ctid = threadIdx.x - 192;  // 0..127
        uint32_t gi = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < p.n_units && ok; u += gridDim.x) {
            const UnitInfo ui = unit_info(p, u);
            for (int i = 0; i < 2 * ui.T; ++i, ++gi) {
                const uint32_t rs = gi % p.NR, os = gi % p.NS;
                if (!warp_wait(raw_full + 8 * rs, (gi / p.NR) & 1u, abort_flag) ||
                    !warp_wait(op_empty + 8 * os, ((gi / p.NS) & 1u) ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                const uint8_t *raw = smem + p.off_raw + rs * S_::RAW_STAGE;
                uint8_t *op = smem + os * S_::OP_STAGE;
                constexpr int CPR = D / 16;  // 16-byte chunks per raw row
                for (int chn = ctid; chn < TILE_KEYS * CPR; chn += 128) {
                    const int row = chn / CPR, cc = chn % CPR;
                    const uint4 v = *reinterpret_cast<const uint4 *>(raw + row * D + cc * 16);
                    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
                    uint32_t h[8];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[e] & 0xFFFFu), __NV_E4M3);
                        __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[e] >> 16), __NV_E4M3);
                        h[2 * e] = (uint32_t)lo.x | ((uint32_t)lo.y << 16);
                        h[2 * e + 1] = (uint32_t)hi.x | ((uint32_t)hi.y << 16);
                    }
                    *reinterpret_cast<uint4 *>(op + sw128_off(row, cc * 16, TILE_KEYS * 128)) =
                        make_uint4(h[0], h[1], h[2], h[3]);
                    *reinterpret_cast<uint4 *>(op + sw128_off(row, cc * 16 + 8, TILE_KEYS * 128)) =
                        make_uint4(h[4], h[5], h[6], h[7]);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(op_full + 8 * os);
                    mbar_arrive(raw_empty + 8 * rs);
                }
            }
        }
        if (!ok) {
            *abort_flag = 1;
            if (ctid == 0) raise_error(p.err, SPEC_DEVERR_TIMEOUT);
        }
    }
    // ================= teardown =================
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, p.tmem_cols);
    }
}

// One warp per (row, q head): merge the splits in ascending order.
template <int D>
__global__ void __launch_bounds__(256) attn_combine_kernel(const float *__restrict__ ws_ml,
                                                           const float *__restrict__ ws_o, int B, int k, int Hq,
                                                           int G, int Hkv, int n_splits, uint16_t *out) {
    constexpr int E = D / 32;
    const int warp_global = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    const int R = B * (k + 1);
    if (warp_global >= R * Hq) return;
    const int r = warp_global / Hq, h = warp_global % Hq;
    const int b = r / (k + 1), j = r % (k + 1);
    const int g = h / G, hi = h % G;
    const int n_q = (k + 1) * G;
    const int qi = j * G + hi;
    const size_t unit0 = ((size_t)b * Hkv + g) * n_splits;
    float M = -INFINITY;
    bool failed = false;
    for (int s = 0; s < n_splits; ++s) {
        const float *ml = ws_ml + ((unit0 + s) * n_q + qi) * 2;
        const float l = ml[1];
        if (l < 0.f) failed = true;
        if (l > 0.f) M = fmaxf(M, ml[0]);
    }
    if (failed || M == -INFINITY) return;  // error already raised; output left unwritten
    float L = 0.f, o[E];
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] = 0.f;
    for (int s = 0; s < n_splits; ++s) {
        const float *ml = ws_ml + ((unit0 + s) * n_q + qi) * 2;
        const float l = ml[1];
        if (!(l > 0.f)) continue;
        const float w = exp2f(ml[0] - M);
        L = fmaf(l, w, L);
        const float *os = ws_o + ((unit0 + s) * n_q + qi) * D;
#pragma unroll
        for (int e = 0; e < E; ++e) o[e] = fmaf(w, __ldg(os + lane + 32 * e), o[e]);
    }
    const float inv = 1.f / L;
    uint16_t *dst = out + ((size_t)r * Hq + h) * D;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        __nv_bfloat16 v = __float2bfloat16_rn(o[e] * inv);
        dst[lane + 32 * e] = *reinterpret_cast<uint16_t *>(&v);
    }
}

// ---- host side ---------------------------------------------------------------------------

typedef CUresult (*EncodeTiledFnA)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFnA encode_fn_attn() {
    static EncodeTiledFnA fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFnA>(ptr);
    }
    return fn;
}

// The pool viewed as [num_pages * Hkv * page_size rows][d] with a (box_cols x box_rows) box.
static bool make_pool_map(CUtensorMap *map, const void *base, const KvView &kv, bool fp8, int box_rows) {
    EncodeTiledFnA fn = encode_fn_attn();
    if (!fn) return false;
    const cuuint64_t rows = (cuuint64_t)kv.num_pages * kv.n_kv_heads * kv.page_size;
    const int esz = fp8 ? 1 : 2;
    cuuint64_t dims[2] = {(cuuint64_t)kv.head_dim, rows};
    cuuint64_t strides[1] = {(cuuint64_t)kv.head_dim * esz};
    cuuint32_t box[2] = {(cuuint32_t)(fp8 ? kv.head_dim : 64), (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base),
              dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              fp8 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static int attn_sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    return n;
}

template <int D, bool FP8>
static int launch_attn_tc(AttnTcParams &p, cudaStream_t s) {
    using S_ = AttnShape<D, FP8>;
    const int NATOM = S_::NATOM;
    p.off_q = 0;  // set below
    const uint32_t q_bytes = NATOM * p.N_pad * 128, p_bytes = 2 * P_BUF;  // P: 2 buffers
    const uint32_t small = 64 + 12 * p.N_pad * 4 + 64;
    const uint32_t bars = 8 * 64;
    const uint32_t fixed = 1024 + q_bytes + p_bytes + small + bars;
    const uint32_t per = S_::OP_STAGE + S_::RAW_STAGE;
    int depth = (int)((ATT_SMEM_LIMIT - fixed) / per);
    depth = depth > 6 ? 6 : depth;
    if (depth >= 2) {
        p.NS = depth;
        p.NR = FP8 ? depth : 0;
    } else if (FP8 && ATT_SMEM_LIMIT >= fixed + 2 * S_::OP_STAGE + S_::RAW_STAGE) {
        // two operand stages are the minimum (the next K tile loads while the current V
        // tile is in use); the raw ring takes what is left
        p.NS = 2;
        p.NR = (int)((ATT_SMEM_LIMIT - fixed - 2 * S_::OP_STAGE) / (S_::RAW_STAGE ? S_::RAW_STAGE : 1));
        p.NR = p.NR > 2 ? 2 : p.NR;
    } else {
        return SPEC_ERR_UNSUPPORTED;
    }
    p.off_q = p.NS * S_::OP_STAGE;
    p.off_p = p.off_q + q_bytes;
    p.off_raw = p.off_p + p_bytes;
    p.off_bar = p.off_raw + p.NR * S_::RAW_STAGE;
    p.off_small = p.off_bar + bars;
    const size_t smem = 1024 + p.off_small + small;
    CUtensorMap mk, mv;
    const int box_rows = p.kv.page_size < TILE_KEYS ? p.kv.page_size : TILE_KEYS;
    if (!make_pool_map(&mk, p.kv.k_pool, p.kv, FP8, box_rows) || !make_pool_map(&mv, p.kv.v_pool, p.kv, FP8, box_rows))
        return SPEC_ERR_CUDA;
    // a fixed ceiling (see the skinny GEMM launcher): graphs may mix launch sizes
    if (cudaFuncSetAttribute(attn_tc_kernel<D, FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize, ATT_SMEM_LIMIT) !=
        cudaSuccess)
        return SPEC_ERR_CUDA;
    const int sms = attn_sm_count();
    if (sms < 1) return SPEC_ERR_CUDA;
    const int grid = p.n_units < sms ? p.n_units : sms;
    attn_tc_kernel<D, FP8><<<grid, S_::THREADS, smem, s>>>(mk, mv, p);
    return launch_status();
}

static size_t ws_bytes_for(int B, int Hkv, int n_splits, int n_q, int d) {
    const size_t units = (size_t)B * Hkv * n_splits;
    size_t ml = units * n_q * 2 * sizeof(float);
    ml = (ml + 255) & ~(size_t)255;
    return ml + units * n_q * d * sizeof(float);
}

}  // namespace spec

SPEC_API size_t spec_verify_attn_workspace(const spec_kv_desc *kv, int B, int k, int n_q_heads, int max_pos) {
    if (spec::check_kv_desc(kv) || B < 1 || k < 0 || k > SPEC_KMAX || n_q_heads < 1 || max_pos < 1) return 0;
    if (n_q_heads % kv->n_kv_heads) return 0;
    const int G = n_q_heads / kv->n_kv_heads;
    const int n_splits = (max_pos + spec::SPLIT_KEYS - 1) / spec::SPLIT_KEYS;
    return spec::ws_bytes_for(B, kv->n_kv_heads, n_splits, (k + 1) * G, kv->head_dim);
}

SPEC_API int spec_verify_attn(const spec_kv_desc *kvd, const int32_t *pos, int B, int k, int n_q_heads,
                              const void *q, float scale, void *out, void *ws, size_t ws_bytes, int max_pos,
                              int32_t *dev_err, spec_stream_t stream) {
    int st = spec::check_kv_desc(kvd);
    if (st) return st;
    if (!pos || !q || !out) return SPEC_ERR_NULL;
    if (B < 1 || k < 0 || k > SPEC_KMAX || n_q_heads < 1 || max_pos < k + 1) return SPEC_ERR_ARG;
    if (n_q_heads % kvd->n_kv_heads) return SPEC_ERR_ARG;
    const size_t need = spec_verify_attn_workspace(kvd, B, k, n_q_heads, max_pos);
    if (!ws || ws_bytes < need) return SPEC_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return SPEC_ERR_ALIGN;
    if (!spec::aligned16(q) || !spec::aligned16(out)) return SPEC_ERR_ALIGN;
    const int G = n_q_heads / kvd->n_kv_heads;
    const int n_q = (k + 1) * G;
    const int N_pad = ((n_q + 15) / 16) * 16;
    const int NB = kvd->head_dim <= 128 ? 1 : 2;
    if (N_pad > spec::MAX_NPAD) return SPEC_ERR_UNSUPPORTED;
    // TMEM: TS S tiles of N_pad columns + OB output buffers of NB*N_pad columns <= 512
    int OB = 2, TS = (512 - 2 * NB * N_pad) / N_pad;
    if (TS < spec::MAX_TS) {
        OB = 1;
        TS = (512 - NB * N_pad) / N_pad;
    }
    TS = TS > spec::MAX_TS ? spec::MAX_TS : TS;
    if (TS < 1) return SPEC_ERR_UNSUPPORTED;
    spec::AttnTcParams p{};
    p.kv = spec::make_view(kvd);
    p.pos = pos;
    p.B = B;
    p.k = k;
    p.Hq = n_q_heads;
    p.G = G;
    p.n_q = n_q;
    p.N_pad = N_pad;
    p.n_splits = (max_pos + spec::SPLIT_KEYS - 1) / spec::SPLIT_KEYS;
    p.max_pos = max_pos;
    p.n_units = B * kvd->n_kv_heads * p.n_splits;
    p.q = (const uint16_t *)q;
    p.scale_log2 = scale * spec::LOG2E;
    const size_t units = (size_t)p.n_units;
    size_t ml = units * n_q * 2 * sizeof(float);
    ml = (ml + 255) & ~(size_t)255;
    p.ws_ml = (float *)ws;
    p.ws_o = (float *)((char *)ws + ml);
    p.err = dev_err;
    p.TS = TS;
    p.OB = OB;
    uint32_t cols = 32;
    while (cols < (uint32_t)(TS * N_pad + OB * NB * N_pad)) cols <<= 1;
    p.tmem_cols = cols;
    cudaStream_t s = (cudaStream_t)stream;
    const bool fp8 = kvd->kv_dtype == SPEC_KV_FP8_E4M3;
    switch (kvd->head_dim * 2 + (fp8 ? 1 : 0)) {
        case 128: st = spec::launch_attn_tc<64, false>(p, s); break;
        case 129: st = spec::launch_attn_tc<64, true>(p, s); break;
        case 256: st = spec::launch_attn_tc<128, false>(p, s); break;
        case 257: st = spec::launch_attn_tc<128, true>(p, s); break;
        case 512: st = spec::launch_attn_tc<256, false>(p, s); break;
        default: st = spec::launch_attn_tc<256, true>(p, s); break;
    }
    if (st) return st;
    const int R = B * (k + 1);
    const int cblocks = (R * n_q_heads + 7) / 8;
    switch (kvd->head_dim) {
        case 64:
            spec::attn_combine_kernel<64><<<cblocks, 256, 0, s>>>(p.ws_ml, p.ws_o, B, k, n_q_heads, G,
                                                                  kvd->n_kv_heads, p.n_splits, (uint16_t *)out);
            break;
        case 128:
            spec::attn_combine_kernel<128><<<cblocks, 256, 0, s>>>(p.ws_ml, p.ws_o, B, k, n_q_heads, G,
                                                                   kvd->n_kv_heads, p.n_splits, (uint16_t *)out);
            break;
        default:
            spec::attn_combine_kernel<256><<<cblocks, 256, 0, s>>>(p.ws_ml, p.ws_o, B, k, n_q_heads, G,
                                                                   kvd->n_kv_heads, p.n_splits, (uint16_t *)out);
            break;
    }
    return spec::launch_status();
}

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
// Work unit = (branch b, kv head g, split of split_keys positions). The n_q = (k+1)*G
// query vectors that share kv head g sit on the 128 TMEM lanes (the M side of the MMAs,
// query i on lane i of each copy, see below); the keys of a 128-key tile are the columns:
//     S[q][key]  = Q . K_tile^T                 (tcgen05, fp32 in TMEM, double-buffered)
//     O[q][d]   += P[q][key] . V_tile[key][d]   (tcgen05, fp32 in TMEM)
// so every softmax quantity of a query (its running maximum and sum) lives in the lanes'
// threads: no cross-lane reductions, only an exchange of partial maxima between the warps
// that hold copies of the same queries. One pass per tile with a lazily raised maximum: a row's
// running maximum m only moves when a tile's maximum exceeds it by more than RESCALE_TAU
// (log2 units), so P = 2^(s - m) <= 2^RESCALE_TAU and O is rescaled (in TMEM, by the row's
// own thread) only on such a move; the final O / l does not depend on which m was used.
//
// A persistent CTA per SM walks its units with warp-specialised roles:
//   warps 0-3  gather K and V rows with 16-byte cp.async copies into the swizzled operand
//              ring (bf16), one warp per SM sub-partition (cp.async issue is throughput-
//              bound per sub-partition); for FP8 pools warps 0, 1 gather E4M3 rows into a raw
//              ring (by TMA boxes of one page-run each when pages hold >= 64 positions) and
//              warps 2, 3 convert them to f16 exactly (and Q bf16 -> f16 in place);
//   warps 4-7  softmax, one per TMEM lane quadrant (a warp reaches only the lanes of its
//              own quadrant, and quadrant w % 4 is also SM sub-partition w % 4): Q is loaded
//              in copies, four when the n_q queries fit one quadrant and two when they span
//              two, so that every quadrant holds the queries and the S MMA computes each
//              copy's scores at no extra cost (M = 128 either way); each warp takes its
//              copy's share of the tile's key columns (when four copies would leave the
//              operand ring too shallow, two copies on one quadrant each, and two warps idle);
//   warp 8     per unit: takes the next work unit, fills the page-table entries (and FP8
//              scales) into a shared table, and loads the Q copies by 3-D TMA boxes;
//   warp 9     issues S = Q . K^T of each tile as soon as its keys and an S buffer are there
//              (TMEM allocation is also this warp's);
//   warp 10    issues O += P . V of each tile as soon as its P is there, so the softmax of
//              one tile overlaps the MMAs of its neighbours.
// The page scales of FP8 pools are applied by the softmax: K's to the scores, V's to P (the
// row sum stays unscaled), so S and O come out in the pool's true units.
// Keys beyond a row's position get P = 0 by select, never by multiplication, and V rows
// past the branch's last position are zeroed before P.V, so NaN in unused pool slots
// cannot reach a result. Tile and split boundaries sit at fixed key positions and every
// MMA row is computed independently of the others, so a row's output is identical
// whatever B, k or batch it is verified in. A combine pass merges the splits of each
// (row, head) in ascending order; it and this kernel are programmatic dependent launches
// that wait on the device (griddepcontrol.wait) for the kernel before them.
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

constexpr int SPLIT_KEYS = 1024;  // largest split; the split size is split_keys_for(Hkv)
constexpr int TILE_KEYS = 128;
constexpr float LOG2E = 1.4426950408889634f;
constexpr float RESCALE_TAU = 8.0f;   // P <= 2^8: exact range for bf16 and f16 alike
constexpr uint64_t ATT_WAIT_NS = 1000000000ull;
constexpr int ATT_SMEM_LIMIT = 227 * 1024;
constexpr int MAX_NPAD = 64;          // query vectors per (branch, kv head), padded to 16
constexpr int MAX_RPAD = 128;         // TMEM lanes holding the copies of the query layout

// Per-unit table the producer warp fills: the page of each page-sized run of the split's
// keys (-1 if the table entry is invalid), the page's FP8 K / V scales, and the error
// bits of any invalid entry. Used for pages of >= 8 positions.
constexpr int UT_ENTRIES = SPLIT_KEYS / 8;
struct UnitTable {
    int32_t page[UT_ENTRIES];
    float ksc[UT_ENTRIES];
    float vsc[UT_ENTRIES];
    int32_t bad;
    int32_t iter;          // the unit's index in the walk order, or -1: no more units
    int32_t pad_[30];
};

// Split size in positions, a function of the model's KV-head count only (never of B, k or
// the context length, so a row's split boundaries are the same in every batch): few KV
// heads give few work units per branch, so their splits are shorter.
__host__ __device__ constexpr int split_keys_for(int n_kv_heads) {
    return n_kv_heads <= 2 ? 256 : (n_kv_heads <= 4 ? 512 : SPLIT_KEYS);
}

struct AttnTcParams {
    KvView kv;
    const int32_t *pos;
    int B, k, Hq, G, n_q, n_splits, max_pos, n_units, split_keys;
    // query layout on the TMEM lanes: draft rows j < J1 on lanes [0, J1*G), the rest (if
    // split) on lanes [32, 32 + (k+1-J1)*G); R_pad = rows of a Q buffer (all copies)
    int J1, split, R_pad;
    // copies of the query layout on the TMEM lanes (copy c starts at lane 32*qpc*c), so that
    // every lane quadrant, and with it every SM sub-partition, holds the queries; PR = rows
    // of P (copy 0's layout, padded to 16)
    int copies, qpc, PR;
    // FP8 pools: rows per TMA box of the K / V gather (one page-run: min(page size, 128));
    // 0 = the rows are gathered by 16-byte cp.async copies
    int tma_rows;
    const uint16_t *q;     // bf16 [R][Hq][d]
    float scale_log2;      // softmax scale * log2(e)
    unsigned int *sched;   // [2]: next unit to hand out, CTAs done (zero between calls)
    float *ws_ml;          // [units][n_q][2]  (m in log2 units, l)
    float *ws_o;           // [units][n_q][d]
    int32_t *err;
    int NS, NR;            // operand / raw ring depth (sub-tiles)
    int OB;                // O buffers in TMEM (1 or 2)
    int QB;                // Q buffers in shared memory (1 or 2)
    uint32_t off_q, off_p, off_op, off_raw, off_ut, off_bar, off_small;  // shared-memory offsets
};

// The CTA's mbarriers, as byte offsets from the barrier region (one definition for the
// kernel and the host plan, which checks that they fit BAR_BYTES).
struct BarMap {
    uint32_t op_full, op_empty, raw_full, raw_empty, sfull, sfree, pfull, pfree, odone, ofree;
    uint32_t qfull, qconv, qfree, ufull, ufree, drain, xfull, lfull, lfin, end;
};
__host__ __device__ inline BarMap bar_map(int NS, int NR) {
    BarMap m;
    uint32_t o = 0;
    m.op_full = o;   o += 8 * NS;  // operand ring: full / empty per stage
    m.op_empty = o;  o += 8 * NS;
    m.raw_full = o;  o += 8 * NR;  // FP8 raw ring
    m.raw_empty = o; o += 8 * NR;
    m.sfull = o;     o += 16;      // S double buffer
    m.sfree = o;     o += 16;
    m.pfull = o;     o += 16;      // P double buffer
    m.pfree = o;     o += 16;
    m.odone = o;     o += 8;       // P.V completions
    m.ofree = o;     o += 16;      // O buffers
    m.qfull = o;     o += 16;      // Q buffers
    m.qconv = o;     o += 16;
    m.qfree = o;     o += 16;
    m.ufull = o;     o += 16;      // unit tables
    m.ufree = o;     o += 16;
    m.drain = o;     o += 16;      // one per MMA issuer
    m.xfull = o;     o += 32;      // softmax exchanges: row maxima, row sums
    m.lfull = o;     o += 32;
    m.lfin = o;      o += 16;      // the loaders have issued every copy of a unit
    m.end = o;
    return m;
}
constexpr uint32_t BAR_BYTES = 8 * 64;

// A ring stage holds one sub-tile: 128 keys x SUB_COLS columns of d (d = 256 tiles are
// two sub-tiles, the halves of d: S accumulates over both, and each half of O reads its
// own half of V).
template <int D, bool FP8>
struct AttnShape {
    static constexpr int NATOM = D / 64;                   // 128-byte column blocks of a 16-bit row
    static constexpr int SUB_COLS = D < 128 ? D : 128;
    static constexpr int NSUB = D / SUB_COLS;              // sub-tiles per tile
    static constexpr int NATOM_SUB = SUB_COLS / 64;        // column blocks per sub-tile
    static constexpr uint32_t OP_STAGE = NATOM_SUB * TILE_KEYS * 128;
    static constexpr uint32_t RAW_STAGE = FP8 ? TILE_KEYS * SUB_COLS : 0;
    static constexpr int THREADS = 352;
};

struct UnitInfo {
    int b, g, split, pos_b, kv_end, s0, T;
    bool bad_pos;
};

// The scheduler hands out units split-major (every (branch, head) pair's first split, then
// every pair's second split, ...), which puts each pair's short last split late;
// `u` (the workspace slot) stays (branch, head, split)-major for the combine pass.
__device__ __forceinline__ UnitInfo unit_info(const AttnTcParams &p, int iter, int &u) {
    UnitInfo ui;
    const int pairs = p.B * p.kv.n_kv_heads;
    ui.split = iter / pairs;
    ui.g = (iter % pairs) % p.kv.n_kv_heads;
    ui.b = (iter % pairs) / p.kv.n_kv_heads;
    u = (ui.b * p.kv.n_kv_heads + ui.g) * p.n_splits + ui.split;
    ui.pos_b = __ldg(p.pos + ui.b);
    ui.bad_pos = ui.pos_b < 0 || ui.pos_b + p.k + 1 > p.max_pos;
    ui.kv_end = ui.pos_b + p.k + 1;
    ui.s0 = ui.split * p.split_keys;
    int n = ui.bad_pos ? 0 : ui.kv_end - ui.s0;
    n = n < 0 ? 0 : (n > p.split_keys ? p.split_keys : n);
    ui.T = (n + TILE_KEYS - 1) / TILE_KEYS;
    return ui;
}

// byte offset of 16-bit element (row, col) in a K-major, 128-byte-swizzled operand whose
// 64-column blocks are `block_bytes` apart
__device__ __forceinline__ uint32_t sw128_off(int row, int col, uint32_t block_bytes) {
    const int blk = col >> 6, c = col & 63;
    return blk * block_bytes + row * 128 + ((((c >> 3) ^ (row & 7)) & 7) << 4);
}

// Every lane waits; the verdict is made uniform across the warp so that no lane can
// leave a loop that the others stay in.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag) {
    const bool r = mbar_wait(bar, parity, abort_flag, ATT_WAIT_NS);
    return __all_sync(0xFFFFFFFFu, r);
}

__device__ __forceinline__ uint32_t pack2(float a, float b, bool f16) {
    if (f16) {
        const __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<const uint32_t *>(&h);
    }
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

template <int D, bool FP8>
__global__ void __launch_bounds__(AttnShape<D, FP8>::THREADS, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap map_q0, const __grid_constant__ CUtensorMap map_q1,
                   const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                   AttnTcParams p) {
    using S_ = AttnShape<D, FP8>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t s_base = smem_u32(smem);
    const int R_pad = p.R_pad, n_q = p.n_q;
    // Q buffers keep R_pad rows and P buffers PR rows per 64-column block; the M = 128 MMAs
    // also read the rows after those, which fall on the following memory: those rows only
    // feed TMEM lanes no thread reads.
    const uint32_t QATOM = (uint32_t)R_pad * 128, QBUF = S_::NATOM * QATOM;
    const uint32_t PATOM = (uint32_t)p.PR * 128, PBUF = 2 * PATOM;
    const uint32_t s_q = s_base + p.off_q, s_p = s_base + p.off_p, s_op = s_base + p.off_op;
    const uint32_t s_raw = s_base + p.off_raw;
    uint8_t *g_p = smem + p.off_p;
    UnitTable *tables = reinterpret_cast<UnitTable *>(smem + p.off_ut);  // [2]
    // barrier map
    const BarMap bm = bar_map(p.NS, p.NR);
    const uint32_t bar0 = s_base + p.off_bar;
    const uint32_t op_full = bar0 + bm.op_full, op_empty = bar0 + bm.op_empty;
    const uint32_t raw_full = bar0 + bm.raw_full, raw_empty = bar0 + bm.raw_empty;
    const uint32_t sfull = bar0 + bm.sfull, sfree = bar0 + bm.sfree;
    const uint32_t pfull = bar0 + bm.pfull, pfree = bar0 + bm.pfree;
    const uint32_t odone = bar0 + bm.odone, ofree = bar0 + bm.ofree;
    const uint32_t qfull = bar0 + bm.qfull, qconv = bar0 + bm.qconv, qfree = bar0 + bm.qfree;
    const uint32_t ufull = bar0 + bm.ufull, ufree = bar0 + bm.ufree;
    const uint32_t drain = bar0 + bm.drain;
    const uint32_t xfull = bar0 + bm.xfull, lfull = bar0 + bm.lfull;
    const uint32_t lfin = bar0 + bm.lfin;
    uint8_t *small = smem + p.off_small;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(small);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(small + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_act = p.copies * p.qpc;  // softmax warps with queries
    const bool small_pages = p.kv.page_size < 8;  // more than UT_ENTRIES pages per split
    const int log2P = p.kv.log2_page;

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.NS; ++s) {
            // bf16: each loader thread's copies arrive; FP8: each converter warp
            // FP8: each converter warp arrives; bf16: each loader thread's copies
            mbar_init(op_full + 8 * s, FP8 ? 2 : 128);
            mbar_init(op_empty + 8 * s, 1);
        }
        for (int s = 0; s < p.NR; ++s) {
            mbar_init(raw_full + 8 * s, p.tma_rows ? 2 : 64);  // each FP8 loader warp / thread arrives
            mbar_init(raw_empty + 8 * s, 2);  // the converter warps
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(sfull + 8 * a, 1);
            mbar_init(sfree + 8 * a, n_act);
            mbar_init(pfull + 8 * a, n_act);
            mbar_init(pfree + 8 * a, 1);
            mbar_init(ofree + 8 * a, n_act);
            mbar_init(qfull + 8 * a, 1);
            mbar_init(qconv + 8 * a, 2);
            mbar_init(qfree + 8 * a, 1);
            mbar_init(ufull + 8 * a, 1);
            mbar_init(ufree + 8 * a, n_act + (FP8 ? 2 : 4) + 1);  // softmax, loader and P.V warps
            mbar_init(drain + 8 * a, 1);
            mbar_init(lfin + 8 * a, FP8 ? 2 : 4);
        }
        mbar_init(odone, 1);
        for (int i = 0; i < 4; ++i) {
            mbar_init(xfull + 8 * i, p.copies);  // the copies of one lane quadrant's queries
            mbar_init(lfull + 8 * i, p.copies);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 8 && lane == 0) {
        prefetch_tmap(&map_q0);
        if (p.split) prefetch_tmap(&map_q1);
        if (FP8 && p.tma_rows) {
            prefetch_tmap(&map_k);
            prefetch_tmap(&map_v);
        }
    }
    if (warp == 9) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // the set-up above overlaps the end of the previous kernel in the stream; nothing it wrote
    // (the KV pool, Q, the positions) is read before this point
    grid_dep_wait();
    const uint32_t tmem = *tmem_slot;
    const uint32_t t_s = tmem;        // S buffers: columns [0, 128) and [128, 256)
    const uint32_t t_o = tmem + 256;  // O buffers: D columns each

    if (warp == 8) {
        // ================= producer: per unit, the page table entries and Q =================
        // Units are handed out dynamically: the producer takes the next index of the
        // split-major walk from a global counter, skips empty units, and publishes the unit
        // in the shared table that every other role waits on (-1 ends their loops). It takes
        // a unit only once a table is free and the loaders have issued every copy of the
        // previous unit, so that a CTA holds little more than the work in its rings and the
        // last units go to whichever CTAs run out of work first.
        uint32_t ua = 0;
        bool ok = true;
        for (;;) {
            const uint32_t ub = ua & 1u, uph = (ua >> 1) & 1u;
            UnitTable *tab = tables + ub;
            if (!warp_wait(ufree + 8 * ub, uph ^ 1u, abort_flag)) { ok = false; break; }
            if (ua > 0 && !warp_wait(lfin + 8 * ((ua - 1) & 1u), ((ua - 1) >> 1) & 1u, abort_flag)) {
                ok = false;
                break;
            }
            int it_u = -1, u = 0;
            UnitInfo ui;
            for (;;) {
                int cand = 0;
                if (lane == 0) cand = (int)atomicAdd(p.sched, 1u);
                cand = __shfl_sync(0xFFFFFFFFu, cand, 0);
                if (cand >= p.n_units) break;
                ui = unit_info(p, cand, u);
                if (ui.T > 0) {
                    it_u = cand;
                    break;
                }
                if (ui.bad_pos && ui.split == 0 && ui.g == 0 && lane == 0) raise_error(p.err, SPEC_DEVERR_POS);
            }
            if (it_u < 0) {
                if (lane == 0) tab->iter = -1;
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(ufull + 8 * ub);
                    // no new work for this CTA: the combine pass may be scheduled
                    grid_dep_launch();
                }
                break;
            }
            int badbits = 0;
            if (!small_pages) {
                const int nkeys = min(ui.kv_end - ui.s0, p.split_keys);
                const int nent = (nkeys + p.kv.page_size - 1) >> log2P;
                for (int e = lane; e < nent; e += 32) {
                    const int pg = page_of(p.kv, ui.b, ui.s0 + (e << log2P));
                    float ks = 1.f, vs = 1.f;
                    if (pg < 0) {
                        badbits |= -pg;
                    } else if (FP8) {
                        const size_t si = (size_t)pg * p.kv.n_kv_heads + ui.g;
                        ks = __ldg(p.kv.k_scale + si);
                        vs = __ldg(p.kv.v_scale + si);
                    }
                    tab->page[e] = pg < 0 ? -1 : pg;
                    tab->ksc[e] = ks;
                    tab->vsc[e] = vs;
                }
            } else {
                // pages smaller than 8 positions: the loaders look each row up themselves;
                // only the error bits are gathered here
                const int nkeys = min(ui.kv_end - ui.s0, p.split_keys);
                for (int e = lane; e < nkeys; e += 32) {
                    const int pg = page_of(p.kv, ui.b, ui.s0 + e);
                    if (pg < 0) badbits |= -pg;
                }
            }
            badbits = __reduce_or_sync(0xFFFFFFFFu, badbits);
            if (lane == 0) {
                tab->bad = badbits;
                tab->iter = it_u;
                if (badbits) raise_error(p.err, badbits);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(ufull + 8 * ub);
            // ---- Q of (b, g): one 3-D box per 64-column block lands as rows j*G + i ----
            const uint32_t qs = p.QB == 2 ? ub : 0u, qph = p.QB == 2 ? uph : (ua & 1u);  // Q buffer, phase
            if (!warp_wait(qfree + 8 * qs, qph ^ 1u, abort_flag)) { ok = false; break; }
            if (lane == 0) {
                mbar_arrive_expect_tx(qfull + 8 * qs, (uint32_t)(p.copies * S_::NATOM * n_q * 128));
                for (int c = 0; c < p.copies; ++c) {
                    const uint32_t dst = s_q + qs * QBUF + (uint32_t)(c * p.qpc * 32 * 128);
#pragma unroll
                    for (int a = 0; a < S_::NATOM; ++a) {
                        tma_load_3d(dst + a * QATOM, &map_q0, a * 64, ui.g * p.G, ui.b * (p.k + 1), qfull + 8 * qs);
                        if (p.split)
                            tma_load_3d(dst + a * QATOM + 32 * 128, &map_q1, a * 64, ui.g * p.G,
                                        ui.b * (p.k + 1) + p.J1, qfull + 8 * qs);
                    }
                }
            }
            __syncwarp();
            ++ua;
        }
        if (!ok) {
            *abort_flag = 1;
            if (lane == 0) raise_error(p.err, SPEC_DEVERR_TIMEOUT);
        }
        // the last CTA to finish handing out units leaves the counters zero for the next call
        if (lane == 0) {
            __threadfence();
            if (atomicAdd(p.sched + 1, 1u) == gridDim.x - 1) {
                atomicExch(p.sched, 0u);
                atomicExch(p.sched + 1, 0u);
            }
        }
        // the Q copies still in flight land before the CTA may exit
        if (lane == 0) {
            for (uint32_t j = 0; j < (uint32_t)p.QB && j < ua; ++j) {
                const uint32_t i2 = ua - 1 - j;
                mbar_wait(qfull + 8 * (p.QB == 2 ? (i2 & 1u) : 0u), p.QB == 2 ? (i2 >> 1) & 1u : i2 & 1u, nullptr,
                          ATT_WAIT_NS);
            }
        }
        __syncwarp();
    } else if (warp == 9 || warp == 10) {
        // ================= MMA issuers: warp 9 S = Q . K^T, warp 10 O += P . V =================
        // Two issuing threads, so that S of a tile goes to the tensor pipe as soon as its keys
        // and an S buffer are there and P.V as soon as P is: the issue, commit and wait
        // instructions of both MMA chains take longer than the tensor pipe needs for them.
        // Each thread's commits track its own MMAs.
        const bool s_role = warp == 9;
        const uint32_t idesc_s = idesc_f16kind(128, TILE_KEYS, FP8, false, false);
        const uint32_t idesc_pv = idesc_f16kind(128, S_::SUB_COLS, FP8, false, true);
        uint32_t gt = 0, ua = 0, gbase = 0;  // tiles, active units, first sub-tile of the unit
        bool ok = true;
        for (;;) {
            const uint32_t ub = ua & 1u, uph = (ua >> 1) & 1u;
            if (!warp_wait(ufull + 8 * ub, uph, abort_flag)) { ok = false; break; }
            const int it_u = tables[ub].iter;
            if (it_u < 0) break;
            int u;
            const UnitInfo ui = unit_info(p, it_u, u);
            __syncwarp();
            if (!s_role && lane == 0) mbar_arrive(ufree + 8 * ub);  // done with the unit table
            if (s_role) {
                const uint32_t qs = p.QB == 2 ? ub : 0u, qph = p.QB == 2 ? uph : (ua & 1u);  // Q buffer, phase
                if (!warp_wait((FP8 ? qconv : qfull) + 8 * qs, qph, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t q_addr = s_q + qs * QBUF;
                for (int t = 0; t < ui.T; ++t) {
                    // S(t) = Q . K_t^T into S buffer t & 1 (of the CTA's tile count)
                    const uint32_t g_t = gt + (uint32_t)t, sb = g_t & 1u;
                    if (!warp_wait(sfree + 8 * sb, ((g_t >> 1) & 1u) ^ 1u, abort_flag)) { ok = false; break; }
#pragma unroll
                    for (int h = 0; h < S_::NSUB; ++h) {
                        const uint32_t g = gbase + (uint32_t)(t * 2 * S_::NSUB + h), st = g % p.NS;
                        if (!warp_wait(op_full + 8 * st, (g / p.NS) & 1u, abort_flag)) { ok = false; break; }
                        fence_proxy_async_smem();  // cp.async data -> tensor core reads
                        tc_fence_after();
                        if (lane == 0) {
                            const uint32_t kb = s_op + st * S_::OP_STAGE;
#pragma unroll
                            for (int kl = 0; kl < S_::SUB_COLS / 16; ++kl) {
                                const int ks = h * (S_::SUB_COLS / 16) + kl;  // k step over all of d
                                mma_bf16(t_s + sb * TILE_KEYS,
                                         desc_kmajor_sw128(q_addr + (ks >> 2) * QATOM + (ks & 3) * 32),
                                         desc_kmajor_sw128(kb + (kl >> 2) * (TILE_KEYS * 128) + (kl & 3) * 32),
                                         idesc_s, ks > 0 ? 1u : 0u);
                            }
                            mma_commit(op_empty + 8 * st);
                        }
                        __syncwarp();
                    }
                    if (!ok) break;
                    if (lane == 0) {
                        mma_commit(sfull + 8 * sb);
                        // the unit's last S: its Q buffer is free once these MMAs complete
                        if (t == ui.T - 1) mma_commit(qfree + 8 * qs);
                    }
                    __syncwarp();
                }
            } else {
                const uint32_t ob = p.OB == 2 ? (ua & 1u) : 0u;
                const uint32_t ob_use = p.OB == 2 ? (ua >> 1) : ua;
                if (!warp_wait(ofree + 8 * ob, (ob_use & 1u) ^ 1u, abort_flag)) { ok = false; break; }
                tc_fence_after();
                for (int t = 0; t < ui.T; ++t) {
                    // O += P(t) . V_t
                    const uint32_t g_t = gt + (uint32_t)t, pb = g_t & 1u;
                    if (!warp_wait(pfull + 8 * pb, (g_t >> 1) & 1u, abort_flag)) { ok = false; break; }
                    const int nvk = ui.kv_end - (ui.s0 + t * TILE_KEYS);  // valid keys in this tile
#pragma unroll
                    for (int nb = 0; nb < S_::NSUB; ++nb) {
                        const uint32_t g = gbase + (uint32_t)(t * 2 * S_::NSUB + S_::NSUB + nb), st = g % p.NS;
                        if (!warp_wait(op_full + 8 * st, (g / p.NS) & 1u, abort_flag)) { ok = false; break; }
                        fence_proxy_async_smem();  // cp.async data -> tensor core reads
                        if (nvk < TILE_KEYS) {
                            // keys past the branch's last position: zero their V rows (NaN-safe P.V)
                            uint4 *vb = reinterpret_cast<uint4 *>(smem + p.off_op + st * S_::OP_STAGE);
                            const int rows = TILE_KEYS - nvk;
                            for (int i = lane; i < rows * S_::NATOM_SUB * 8; i += 32) {
                                const int a = i / (rows * 8), rem = i % (rows * 8);
                                const int r = nvk + rem / 8, c = rem % 8;
                                vb[(a * TILE_KEYS * 128 + r * 128) / 16 + c] = make_uint4(0, 0, 0, 0);
                            }
                            fence_proxy_async_smem();
                            __syncwarp();
                        }
                        tc_fence_after();
                        if (lane == 0) {
                            const uint32_t vb = s_op + st * S_::OP_STAGE, pa = s_p + pb * PBUF;
#pragma unroll
                            for (int ks = 0; ks < TILE_KEYS / 16; ++ks)
                                mma_bf16(t_o + ob * D + nb * 128, desc_kmajor_sw128(pa + (ks >> 2) * PATOM + (ks & 3) * 32),
                                         desc_mnmajor_sw128(vb + ks * 2048, TILE_KEYS * 128), idesc_pv,
                                         (t > 0 || ks > 0) ? 1u : 0u);
                            mma_commit(op_empty + 8 * st);
                        }
                        __syncwarp();
                    }
                    if (!ok) break;
                    if (lane == 0) {
                        mma_commit(pfree + 8 * pb);
                        mma_commit(odone);
                    }
                    __syncwarp();
                }
            }
            if (!ok) break;
            gbase += (uint32_t)(2 * S_::NSUB * ui.T);
            gt += (uint32_t)ui.T;
            ++ua;
        }
        if (!ok) {
            *abort_flag = 1;
            if (lane == 0) raise_error(p.err, SPEC_DEVERR_TIMEOUT);
        }
        if (lane == 0) {
            mma_commit(drain + 8 * (s_role ? 0 : 1));
            mbar_wait(drain + 8 * (s_role ? 0 : 1), 0, nullptr, ATT_WAIT_NS);
            // every arrive sent by the commits of either issuer is delivered before the CTA
            // may exit: the last phase of each operand stage's "empty" barrier, of both P and
            // Q buffers' "free" barriers and of the P.V completion barrier
            const uint32_t n_last = gbase < (uint32_t)p.NS ? gbase : (uint32_t)p.NS;
            for (uint32_t j = 0; j < n_last; ++j) {
                const uint32_t i2 = gbase - 1 - j;
                mbar_wait(op_empty + 8 * (i2 % p.NS), (i2 / p.NS) & 1u, nullptr, ATT_WAIT_NS);
            }
            for (uint32_t j = 0; j < 2 && j < gt; ++j) {
                const uint32_t t2 = gt - 1 - j;
                mbar_wait(pfree + 8 * (t2 & 1u), (t2 >> 1) & 1u, nullptr, ATT_WAIT_NS);
            }
            for (uint32_t j = 0; j < (uint32_t)p.QB && j < ua; ++j) {
                const uint32_t i2 = ua - 1 - j;
                mbar_wait(qfree + 8 * (p.QB == 2 ? (i2 & 1u) : 0u), p.QB == 2 ? (i2 >> 1) & 1u : i2 & 1u, nullptr,
                          ATT_WAIT_NS);
            }
            if (gt > 0) mbar_wait(odone, (gt - 1) & 1u, nullptr, ATT_WAIT_NS);
        }
        __syncwarp();
    } else if (warp >= 4 && warp < 8) {
        // ================= softmax: one warp per TMEM lane quadrant =================
        // The queries are held in p.copies copies on the TMEM lanes (a copy spans p.qpc lane
        // quadrants), so that each of the four SM sub-partitions has a warp that can read
        // their scores. A warp takes the tile's 32-key quarters of its copy (copy c owns
        // quarters [c*nqw, (c+1)*nqw)); the copies exchange only the row's partial maxima per
        // tile, and each warp keeps one partial row sum per quarter, added once per unit in a
        // fixed order. P is written for the rows of copy 0, whose lanes of O the P.V MMA
        // accumulates; only copy 0's warps rescale and read out O.
        const int qd = warp & 3;                     // TMEM lane quadrant
        const int QPC = p.qpc, C = p.copies;         // quadrants per copy, copies
        const int cpy = qd / QPC, qq = qd % QPC;     // this warp's copy, quadrant within it
        const int nqw = 4 / C;                       // 32-key quarters per warp (1 or 2)
        const int kq0 = cpy * nqw;                   // first quarter of this warp
        const bool owner = cpy == 0;                 // copy 0: the rows of O
        const bool active = cpy < C;                 // quadrants past the last copy idle
        const int prow_i = qq * 32 + lane;           // row of P, lane of O (copy 0)
        int myq;                                     // the query this lane holds
        bool vrow;
        if (p.split) {
            myq = qq == 0 ? lane : p.J1 * p.G + lane;
            vrow = lane < (qq == 0 ? p.J1 : p.k + 1 - p.J1) * p.G;
        } else {
            myq = qq * 32 + lane;
            vrow = myq < n_q;
        }
        const int jrow = vrow ? myq / p.G : 0;  // the row's draft index j
        const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
        const uint32_t olane_base = (uint32_t)(qq * 32) << 16;  // copy 0's lanes of O
        const float sl = p.scale_log2;
        constexpr int QC = 32;  // key columns per quarter
        // row-maximum exchange [2 tiles][qq][copy][32], then row-sum exchange
        // [2 units][qq][quarter][32]
        float *xch = reinterpret_cast<float *>(small + 64);
        uint32_t gs = 0, gp = 0, ua = 0;
        bool ok = true;
        while (active && ok) {
            const uint32_t ub = ua & 1u, uph = (ua >> 1) & 1u;
            const uint32_t ob = p.OB == 2 ? (ua & 1u) : 0u;
            if (!warp_wait(ufull + 8 * ub, uph, abort_flag)) { ok = false; break; }
            const UnitTable *tab = tables + ub;
            const int it_u = tab->iter;
            if (it_u < 0) break;
            int u;
            const UnitInfo ui = unit_info(p, it_u, u);
            float *ml = p.ws_ml + (size_t)u * n_q * 2;
            const bool failed = tab->bad != 0;
            float m = -INFINITY;             // running maximum (log2 units)
            float lq[2] = {0.f, 0.f};        // this warp's partial sums, one per quarter
            // key offsets (from the split's start) this row sees: [0, climit0]; a lane without
            // a query treats every key as seen (its row of P only feeds an unread row of O)
            const int climit0 = vrow ? ui.pos_b + jrow - ui.s0 : (1 << 30);
            for (int t = 0; t < ui.T; ++t, ++gs, ++gp) {
                const uint32_t sb = gs & 1u, pb = gp & 1u;
                if (ok) ok = warp_wait(sfull + 8 * sb, (gs >> 1) & 1u, abort_flag);
                if (!ok) continue;
                tc_fence_after();
                uint32_t sv[2][2][16];  // [quarter of this warp][16-column block][column]
#pragma unroll
                for (int i = 0; i < 2; ++i)
                    if (i < nqw) {
#pragma unroll
                        for (int c = 0; c < 2; ++c)
                            tmem_ld16(t_s + lane_base + sb * TILE_KEYS + QC * (kq0 + i) + c * 16, sv[i][c]);
                    }
                // FP8 pools: the scores come from E4M3 codes and P multiplies E4M3 codes of V.
                // A quarter's K scale joins the softmax scale and its V scale multiplies P (the
                // row sum stays unscaled); with pages shorter than a quarter the scales are
                // applied per key.
                float slk[2] = {sl, sl}, vmul[2] = {1.f, 1.f};
                const bool percol = FP8 && (small_pages || p.kv.page_size < QC);
                if (FP8 && !percol) {
#pragma unroll
                    for (int i = 0; i < 2; ++i)
                        if (i < nqw) {
                            const int e = (t * TILE_KEYS + QC * (kq0 + i)) >> log2P;
                            slk[i] = sl * tab->ksc[e];
                            vmul[i] = tab->vsc[e];
                        }
                }
                auto col_scales = [&](int qi, int c, float &ks, float &vs) {
                    const int key = ui.s0 + t * TILE_KEYS + QC * (kq0 + qi) + c;
                    ks = 0.f;
                    vs = 0.f;
                    if (key >= ui.kv_end) return;
                    if (!small_pages) {
                        const int e = (key - ui.s0) >> log2P;
                        ks = tab->ksc[e];
                        vs = tab->vsc[e];
                    } else {
                        const int pg = page_of(p.kv, ui.b, key);
                        if (pg >= 0) {
                            ks = __ldg(p.kv.k_scale + (size_t)pg * p.kv.n_kv_heads + ui.g);
                            vs = __ldg(p.kv.v_scale + (size_t)pg * p.kv.n_kv_heads + ui.g);
                        }
                    }
                };
                tmem_ld_wait();
                if (percol) {
#pragma unroll
                    for (int i = 0; i < 2; ++i)
                        if (i < nqw) {
#pragma unroll
                            for (int c = 0; c < QC; ++c) {
                                float ks, vs;
                                col_scales(i, c, ks, vs);
                                sv[i][c >> 4][c & 15] = __float_as_uint(__uint_as_float(sv[i][c >> 4][c & 15]) * ks);
                            }
                        }
                }
                // ---- pass 1: partial maximum of s*slk over the seen columns of each quarter ----
                float pm = -INFINITY;
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    if (i >= nqw) continue;
                    // columns c (of this quarter) with QC*(kq0+i) + c <= climit are seen
                    const int climit = climit0 - t * TILE_KEYS - QC * (kq0 + i);
                    const bool all_seen = __all_sync(0xFFFFFFFFu, climit >= QC - 1);
                    float acc[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[e] = -INFINITY;
                    const float sgn = slk[i] >= 0.f ? 1.f : -1.f;
                    if (all_seen) {
#pragma unroll
                        for (int c = 0; c < QC; ++c)
                            acc[c & 7] = fmaxf(acc[c & 7], sgn * __uint_as_float(sv[i][c >> 4][c & 15]));
                    } else {
#pragma unroll
                        for (int c = 0; c < QC; ++c)
                            if (c <= climit) acc[c & 7] = fmaxf(acc[c & 7], sgn * __uint_as_float(sv[i][c >> 4][c & 15]));
                    }
                    float q = fmaxf(fmaxf(fmaxf(acc[0], acc[1]), fmaxf(acc[2], acc[3])),
                                    fmaxf(fmaxf(acc[4], acc[5]), fmaxf(acc[6], acc[7])));
                    // q = max of sgn*s: the quarter's maximum of s*slk is q*|slk|
                    q = (q == -INFINITY || q == INFINITY) ? -INFINITY : q * (sgn * slk[i]);
                    pm = fmaxf(pm, q);
                }
                // ---- the row's maximum: exchange with the other copies ----
                float mx = pm;
                if (C > 1) {
                    float *xt = xch + sb * 128 + qq * C * 32;
                    xt[cpy * 32 + lane] = pm;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(xfull + 8 * (qq * 2 + sb));
                    ok = warp_wait(xfull + 8 * (qq * 2 + sb), (gs >> 1) & 1u, abort_flag);
                    if (!ok) continue;
                    for (int c = 0; c < C; ++c) mx = fmaxf(mx, xt[c * 32 + lane]);
                }
                if (!vrow) mx = -INFINITY;
                // ---- the P buffer is free once P.V of tile t-2 is done ----
                ok = warp_wait(pfree + 8 * pb, ((gp >> 1) & 1u) ^ 1u, abort_flag);
                if (!ok) continue;
                // ---- lazily raised maximum; a move rescales l and the row of O ----
                const float mnew = (mx > m + RESCALE_TAU) ? mx : m;
                const bool resc = mnew != m && m != -INFINITY;
                if (__any_sync(0xFFFFFFFFu, resc)) {
                    const float f = resc ? ex2_approx(m - mnew) : 1.f;
                    lq[0] *= f;
                    lq[1] *= f;
                    if (owner) {
                        // O is written by P.V of tile t-1 (the one before it is done: see above)
                        ok = warp_wait(odone, (gp - 1) & 1u, abort_flag);
                        if (!ok) continue;
                        tc_fence_after();
                        const uint32_t orow = t_o + olane_base + ob * D;
#pragma unroll 1
                        for (int c0 = 0; c0 < D; c0 += 32) {
                            uint32_t r[2][16];
#pragma unroll
                            for (int e = 0; e < 2; ++e) tmem_ld16(orow + c0 + 16 * e, r[e]);
                            tmem_ld_wait();
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
#pragma unroll
                                for (int j = 0; j < 16; ++j) r[e][j] = __float_as_uint(__uint_as_float(r[e][j]) * f);
                                tmem_st16(orow + c0 + 16 * e, r[e]);
                            }
                        }
                        tmem_st_wait();
                    }
                }
                m = mnew;
                // ---- pass 2: P = 2^(s*slk - m) of this warp's quarters, into copy 0's rows ----
                uint8_t *prow = g_p + pb * PBUF + prow_i * 128;
                const int swz = prow_i & 7;
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    if (i >= nqw) continue;
                    const int kq = kq0 + i;
                    const int climit = climit0 - t * TILE_KEYS - QC * kq;
                    const bool all_seen = __all_sync(0xFFFFFFFFu, climit >= QC - 1);
                    float lacc[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) lacc[e] = 0.f;
                    uint8_t *pq = prow + (kq >> 1) * PATOM;
#pragma unroll
                    for (int c0 = 0; c0 < QC; c0 += 16) {
                        const uint32_t(&r)[16] = sv[i][c0 >> 4];
                        uint32_t pk[8];
                        if (all_seen && !percol) {
#pragma unroll
                            for (int j = 0; j < 16; j += 2) {
                                const float a = ex2_approx(fmaf(__uint_as_float(r[j]), slk[i], -m));
                                const float b = ex2_approx(fmaf(__uint_as_float(r[j + 1]), slk[i], -m));
                                lacc[j >> 1] += a + b;
                                pk[j >> 1] = FP8 ? pack2(a * vmul[i], b * vmul[i], true) : pack2(a, b, false);
                            }
                        } else {
#pragma unroll
                            for (int j = 0; j < 16; j += 2) {
                                float a = ex2_approx(fmaf(__uint_as_float(r[j]), slk[i], -m));
                                float b = ex2_approx(fmaf(__uint_as_float(r[j + 1]), slk[i], -m));
                                a = (c0 + j <= climit) ? a : 0.f;
                                b = (c0 + j + 1 <= climit) ? b : 0.f;
                                lacc[j >> 1] += a + b;
                                float va = vmul[i], vb = vmul[i];
                                if (percol) {
                                    float ks;
                                    col_scales(i, c0 + j, ks, va);
                                    col_scales(i, c0 + j + 1, ks, vb);
                                }
                                pk[j >> 1] = FP8 ? pack2(a * va, b * vb, true) : pack2(a, b, false);
                            }
                        }
                        // 16-byte chunk (within the 128-byte row of the 64-key block) of keys c0..c0+7
                        const int ch0 = (kq & 1) * 4 + (c0 >> 3);
                        if (prow_i < p.PR) {
                            *reinterpret_cast<uint4 *>(pq + (((ch0 ^ swz) & 7) << 4)) =
                                make_uint4(pk[0], pk[1], pk[2], pk[3]);
                            *reinterpret_cast<uint4 *>(pq + ((((ch0 + 1) ^ swz) & 7) << 4)) =
                                make_uint4(pk[4], pk[5], pk[6], pk[7]);
                        }
                    }
                    lq[i] += ((lacc[0] + lacc[1]) + (lacc[2] + lacc[3])) + ((lacc[4] + lacc[5]) + (lacc[6] + lacc[7]));
                }
                tc_fence_before();
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(sfree + 8 * sb);
                    mbar_arrive(pfull + 8 * pb);
                }
            }
            // the unit table is no longer read
            __syncwarp();
            if (ok && lane == 0) mbar_arrive(ufree + 8 * ub);
            // ---- copy 0: the unit's last P.V (P.V of the tile before it is done first) ----
            if (owner) {
                if (ok) ok = warp_wait(pfree + 8 * (gp & 1u), ((gp >> 1) & 1u) ^ 1u, abort_flag);
                if (ok) ok = warp_wait(odone, (gp - 1) & 1u, abort_flag);
                if (ok) {
                    tc_fence_after();
                    float *orow_g = p.ws_o + ((size_t)u * n_q + myq) * D;
                    const uint32_t orow = t_o + olane_base + ob * D;
#pragma unroll 1
                    for (int c0 = 0; c0 < D; c0 += 32) {
                        uint32_t r[2][16];
#pragma unroll
                        for (int e = 0; e < 2; ++e) tmem_ld16(orow + c0 + 16 * e, r[e]);
                        tmem_ld_wait();
                        if (vrow) {
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                reinterpret_cast<float4 *>(orow_g + c0)[e] =
                                    make_float4(__uint_as_float(r[e >> 2][4 * (e & 3)]),
                                                __uint_as_float(r[e >> 2][4 * (e & 3) + 1]),
                                                __uint_as_float(r[e >> 2][4 * (e & 3) + 2]),
                                                __uint_as_float(r[e >> 2][4 * (e & 3) + 3]));
                        }
                    }
                    tc_fence_before();
                }
            }
            __syncwarp();
            if (ok && lane == 0) mbar_arrive(ofree + 8 * ob);
            // ---- the row's sum: the quarters' partial sums, in quarter order ----
            const uint32_t lb = qq * 2 + (ua & 1u);
            float *lx = xch + 256 + (ua & 1u) * 256 + qq * 128;
#pragma unroll
            for (int i = 0; i < 2; ++i)
                if (i < nqw) lx[(kq0 + i) * 32 + lane] = lq[i];
            __syncwarp();
            if (lane == 0) mbar_arrive(lfull + 8 * lb);
            const bool lok = warp_wait(lfull + 8 * lb, (ua >> 1) & 1u, abort_flag);
            if (owner && vrow) {
                const float l = (lx[lane] + lx[32 + lane]) + (lx[64 + lane] + lx[96 + lane]);
                ml[2 * myq] = m;
                ml[2 * myq + 1] = (failed || !ok || !lok) ? -1.f : l;
            }
            if (!lok) ok = false;
            ++ua;
        }
        if (!ok) {
            *abort_flag = 1;
            if (qd == 0 && lane == 0) raise_error(p.err, SPEC_DEVERR_TIMEOUT);
        }
    } else if (!FP8 || warp < 2) {
        // ================= loaders: K / V gather (bf16: warps 0..3; FP8: warps 0, 1) =================
        // Each thread copies its own 16-byte pieces of every sub-tile with cp.async and lets the
        // copies arrive on the stage's barrier by themselves when they land
        // (cp.async.mbarrier.arrive.noinc), so a sub-tile is visible to its consumer as soon as
        // its data is in shared memory and no loader ever holds data back. bf16 rows go straight
        // into the swizzled operand stage (the MMA warp fences for the async proxy after its
        // wait); E4M3 rows go to the raw ring, which the converter warps turn into operand
        // stages. A loader waits only for a free stage.
        constexpr int NT = FP8 ? 64 : 128;           // loader threads
        const int ltid = warp * 32 + lane;  // warps 0..3 (one per SM sub-partition)
        constexpr int ESZ = FP8 ? 1 : 2;
        constexpr int CH = S_::SUB_COLS * ESZ / 16;  // 16-byte pieces per row of a sub-tile
        constexpr int RPS = NT / CH;                 // rows per step of the loader threads
        constexpr int NPIECE = TILE_KEYS / RPS;      // pieces per thread per sub-tile
        const int pch = ltid % CH, prow0 = ltid / CH;
        const size_t row_bytes = (size_t)D * ESZ;
        const uint32_t depth = FP8 ? (uint32_t)p.NR : (uint32_t)p.NS;
        const uint32_t full_base = FP8 ? raw_full : op_full, empty_base = FP8 ? raw_empty : op_empty;
        const uint32_t ring_base = FP8 ? s_raw : s_op;
        const uint32_t stage_bytes = FP8 ? S_::RAW_STAGE : S_::OP_STAGE;
        uint32_t gi = 0, ua = 0;  // sub-tiles issued, active units
        bool ok = true;
        for (;;) {
            const uint32_t ub = ua & 1u, uph = (ua >> 1) & 1u;
            const UnitTable *tab = tables + ub;
            if (!warp_wait(ufull + 8 * ub, uph, abort_flag)) { ok = false; break; }
            const int it_u = tab->iter;
            if (it_u < 0) break;
            int u;
            const UnitInfo ui = unit_info(p, it_u, u);
            ++ua;
            for (int t = 0; t < ui.T && ok; ++t) {
                const int key0 = ui.s0 + t * TILE_KEYS;
                for (int it = 0; it < 2 * S_::NSUB; ++it) {
                    const int kv = it / S_::NSUB, h = it % S_::NSUB;  // K or V, half of d
                    const uint8_t *pool = reinterpret_cast<const uint8_t *>(kv ? p.kv.v_pool : p.kv.k_pool);
                    const uint32_t s = gi % depth;
                    if (!warp_wait(empty_base + 8 * s, ((gi / depth) & 1u) ^ 1u, abort_flag)) { ok = false; break; }
                    const uint32_t dst_base = ring_base + s * stage_bytes;
                    if (FP8 && p.tma_rows) {
                        // one TMA box per page-run of rows into the raw stage; loader warp w
                        // issues runs w, w + 2, ... and announces their bytes on the stage's
                        // barrier. Runs past the branch's last position or of an invalid page
                        // are not loaded.
                        const int BR = p.tma_rows, nruns = TILE_KEYS / BR;
                        const CUtensorMap *map = kv ? &map_v : &map_k;
                        if (lane == 0) {
                            uint32_t bytes = 0;
                            for (int r = warp; r < nruns; r += 2) {
                                if (key0 + r * BR >= ui.kv_end) break;
                                if (tab->page[(t * TILE_KEYS + r * BR) >> log2P] >= 0) bytes += (uint32_t)(BR * S_::SUB_COLS);
                            }
                            mbar_arrive_expect_tx(full_base + 8 * s, bytes);
                            for (int r = warp; r < nruns; r += 2) {
                                const int kr = key0 + r * BR;
                                if (kr >= ui.kv_end) break;
                                const int pg = tab->page[(t * TILE_KEYS + r * BR) >> log2P];
                                if (pg < 0) continue;
                                const int row = (pg * p.kv.n_kv_heads + ui.g) * p.kv.page_size + (kr & (p.kv.page_size - 1));
                                tma_load_2d(dst_base + (uint32_t)(r * BR) * S_::SUB_COLS, map, h * S_::SUB_COLS, row,
                                            full_base + 8 * s);
                            }
                        }
                        __syncwarp();
                        ++gi;
                        continue;
                    }
                    const uint8_t *src_col = pool + (size_t)h * S_::SUB_COLS * ESZ + pch * 16;
                    // rows past the branch's last position, or of an invalid page, stay unloaded.
                    // Per group of 8 pieces: the page lookups and offsets first (independent
                    // loads), then the copies.
                    constexpr int GRP = NPIECE < 8 ? NPIECE : 8;
#pragma unroll
                    for (int k0 = 0; k0 < NPIECE; k0 += GRP) {
                        uint32_t rowi[GRP];  // row index in the pool viewed as [num_pages * Hkv * P][d]
                        uint32_t valid = 0;
                        if (!small_pages) {
                            int pgk[GRP];
#pragma unroll
                            for (int k = 0; k < GRP; ++k) {  // (key - s0) < split_keys: inside the table
                                const int e = (t * TILE_KEYS + (k0 + k) * RPS + prow0) >> log2P;
                                pgk[k] = tab->page[e];
                            }
#pragma unroll
                            for (int k = 0; k < GRP; ++k) {
                                const int key = key0 + (k0 + k) * RPS + prow0;
                                const int pg = key < ui.kv_end ? pgk[k] : -1;
                                valid |= (pg >= 0 ? 1u : 0u) << k;
                                rowi[k] = (uint32_t)(pg * p.kv.n_kv_heads + ui.g) * (uint32_t)p.kv.page_size +
                                          (uint32_t)(key & (p.kv.page_size - 1));
                            }
                        } else {
                            for (int k = 0; k < GRP; ++k) {
                                const int key = key0 + (k0 + k) * RPS + prow0;
                                const int pg = key < ui.kv_end ? page_of(p.kv, ui.b, key) : -1;
                                valid |= (pg >= 0 ? 1u : 0u) << k;
                                rowi[k] = (uint32_t)(pg * p.kv.n_kv_heads + ui.g) * (uint32_t)p.kv.page_size +
                                          (uint32_t)(key & (p.kv.page_size - 1));
                            }
                        }
#pragma unroll
                        for (int k = 0; k < GRP; ++k) {
                            const int row = (k0 + k) * RPS + prow0;
                            const uint32_t dst =
                                FP8 ? dst_base + row * S_::SUB_COLS + pch * 16
                                    : dst_base + (pch >> 3) * (TILE_KEYS * 128) + row * 128 +
                                          ((((pch & 7) ^ (row & 7)) & 7) << 4);
                            if ((valid >> k) & 1u) cp_async16(dst, src_col + (size_t)rowi[k] * row_bytes);
                        }
                    }
                    cp_async_arrive(full_base + 8 * s);
                    ++gi;
                }
            }
            // the unit's table is no longer read by this warp
            __syncwarp();
            if (ok && lane == 0) {
                mbar_arrive(lfin + 8 * ub);
                mbar_arrive(ufree + 8 * ub);
            }
        }
        // every copy lands before the CTA may exit (TMA boxes: the last phase of each stage)
        cp_async_wait_all();
        if (FP8 && p.tma_rows && lane == 0) {
            const uint32_t n_last = gi < depth ? gi : depth;
            for (uint32_t j = 0; j < n_last; ++j) {
                const uint32_t i2 = gi - 1 - j;
                mbar_wait(full_base + 8 * (i2 % depth), (i2 / depth) & 1u, nullptr, ATT_WAIT_NS);
            }
        }
        __syncwarp();
        if (!ok) {
            *abort_flag = 1;
            if (ltid == 0) raise_error(p.err, SPEC_DEVERR_TIMEOUT);
        }
    } else {
        // ================= FP8 converters, warps 2, 3: E4M3 -> f16 operand stages =================
        // E4M3 is exact in f16 (the page scales are applied by the softmax). Per unit the bf16
        // Q is first converted to f16 in place, then every landed raw sub-tile in ring order.
        const int ctid = (warp - 2) * 32 + lane;  // 0..63
        constexpr int CCH = S_::SUB_COLS / 16;     // 16-byte raw pieces per row
        constexpr int NPC = TILE_KEYS * CCH / 64;  // pieces per converter thread per sub-tile
        uint32_t gc = 0, ua = 0;                   // sub-tiles converted, active units
        bool ok = true;
        for (;;) {
            const uint32_t ub = ua & 1u, uph = (ua >> 1) & 1u;
            if (!warp_wait(ufull + 8 * ub, uph, abort_flag)) { ok = false; break; }
            const int it_u = tables[ub].iter;
            if (it_u < 0) break;
            int u;
            const UnitInfo ui = unit_info(p, it_u, u);
            // ---- Q arrives as bf16; the f16-kind MMA needs f16 on both sides ----
            const uint32_t qs = p.QB == 2 ? ub : 0u, qph = p.QB == 2 ? uph : (ua & 1u);  // Q buffer, phase
            if (!warp_wait(qfull + 8 * qs, qph, abort_flag)) { ok = false; break; }
            uint8_t *qb = smem + p.off_q + qs * QBUF;
            for (int i = ctid; i < S_::NATOM * R_pad * 8; i += 64) {
                const int a = i / (R_pad * 8), rem = i % (R_pad * 8);
                uint4 *ptr = reinterpret_cast<uint4 *>(qb + a * QATOM + rem * 16);
                const uint4 v = *ptr;
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
                uint32_t hq[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) hq[e] = pack2(bf16_lo(w[e]), bf16_hi(w[e]), true);
                *ptr = make_uint4(hq[0], hq[1], hq[2], hq[3]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(qconv + 8 * qs);
            ++ua;
            // ---- the unit's K / V sub-tiles ----
            const uint32_t n_sub = (uint32_t)(2 * S_::NSUB * ui.T);
            for (uint32_t i = 0; i < n_sub; ++i, ++gc) {
                const uint32_t rs = gc % p.NR, os = gc % p.NS;
                if (!warp_wait(raw_full + 8 * rs, (gc / p.NR) & 1u, abort_flag) ||
                    !warp_wait(op_empty + 8 * os, ((gc / p.NS) & 1u) ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                const uint8_t *raw = smem + p.off_raw + rs * S_::RAW_STAGE;
                uint8_t *op = smem + p.off_op + os * S_::OP_STAGE;
#pragma unroll
                for (int k = 0; k < NPC; ++k) {
                    const int piece = k * 64 + ctid;
                    const int row = piece / CCH, pc = piece % CCH;
                    const uint4 v = *reinterpret_cast<const uint4 *>(raw + row * S_::SUB_COLS + pc * 16);
                    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
                    uint32_t hv[8];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[e] & 0xFFFFu), __NV_E4M3);
                        const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[e] >> 16), __NV_E4M3);
                        hv[2 * e] = (uint32_t)lo.x | ((uint32_t)lo.y << 16);
                        hv[2 * e + 1] = (uint32_t)hi.x | ((uint32_t)hi.y << 16);
                    }
                    *reinterpret_cast<uint4 *>(op + sw128_off(row, pc * 16, TILE_KEYS * 128)) =
                        make_uint4(hv[0], hv[1], hv[2], hv[3]);
                    *reinterpret_cast<uint4 *>(op + sw128_off(row, pc * 16 + 8, TILE_KEYS * 128)) =
                        make_uint4(hv[4], hv[5], hv[6], hv[7]);
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
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// One CTA of 8 warps per (row, q head): merge the row's splits. Only the branch's
// non-empty splits were computed (split s holds keys from s * split_keys on); among them,
// splits the row does not reach (l = 0) are skipped, so the result depends only on the
// row's own splits, not on the batch's split count. The maximum over the splits is reduced
// in parallel; warp w sums the splits s = w, w+8, ... in ascending order, and the 8 partial
// sums are added in warp order.
constexpr int CMB_WARPS = 8;
template <int D>
__global__ void __launch_bounds__(CMB_WARPS * 32) attn_combine_kernel(const float *__restrict__ ws_ml,
                                                                      const float *__restrict__ ws_o,
                                                                      const int32_t *__restrict__ pos, int B, int k,
                                                                      int Hq, int G, int Hkv, int n_splits,
                                                                      int split_keys, int max_pos, uint16_t *out) {
    constexpr int E = D / 32;  // columns per lane
    __shared__ float red_m[CMB_WARPS];
    __shared__ int red_f[CMB_WARPS];
    __shared__ float part_o[CMB_WARPS][D];
    __shared__ float part_l[CMB_WARPS];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    grid_dep_wait();  // the split kernel's partial results
    const int r = blockIdx.x / Hq, h = blockIdx.x % Hq;
    const int b = r / (k + 1), j = r % (k + 1);
    const int g = h / G, hi = h % G;
    const int n_q = (k + 1) * G;
    const int qi = j * G + hi;
    const size_t unit0 = ((size_t)b * Hkv + g) * n_splits;
    const int pos_b = __ldg(pos + b);
    if (pos_b < 0 || pos_b + k + 1 > max_pos) return;  // error raised by the split kernel
    const int n_used = (pos_b + k + split_keys) / split_keys;  // splits holding keys 0..pos_b+k
    // ---- the maximum over the non-empty splits; any failed split fails the row ----
    float M = -INFINITY;
    int failed = 0;
    for (int s = threadIdx.x; s < n_used; s += CMB_WARPS * 32) {
        const float *ml = ws_ml + ((unit0 + s) * n_q + qi) * 2;
        const float l = ml[1];
        if (l < 0.f) failed = 1;
        if (l > 0.f) M = fmaxf(M, ml[0]);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, off));
        failed |= __shfl_xor_sync(0xFFFFFFFFu, failed, off);
    }
    if (lane == 0) {
        red_m[warp] = M;
        red_f[warp] = failed;
    }
    __syncthreads();
    M = -INFINITY;
    failed = 0;
#pragma unroll
    for (int w = 0; w < CMB_WARPS; ++w) {
        M = fmaxf(M, red_m[w]);
        failed |= red_f[w];
    }
    if (failed || M == -INFINITY) return;  // error already raised; output left unwritten
    // ---- this warp's splits ----
    float L = 0.f, o[E];
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] = 0.f;
    for (int s = warp; s < n_used; s += CMB_WARPS) {
        const float *ml = ws_ml + ((unit0 + s) * n_q + qi) * 2;
        const float l = ml[1];
        if (!(l > 0.f)) continue;
        const float w = exp2f(ml[0] - M);
        L = fmaf(l, w, L);
        const float *os = ws_o + ((unit0 + s) * n_q + qi) * D + lane * E;
        if (E % 4 == 0) {
#pragma unroll
            for (int e = 0; e < E; e += 4) {
                const float4 v = __ldg(reinterpret_cast<const float4 *>(os + e));
                o[e] = fmaf(w, v.x, o[e]);
                o[e + 1] = fmaf(w, v.y, o[e + 1]);
                o[e + 2] = fmaf(w, v.z, o[e + 2]);
                o[e + 3] = fmaf(w, v.w, o[e + 3]);
            }
        } else {
#pragma unroll
            for (int e = 0; e < E; ++e) o[e] = fmaf(w, __ldg(os + e), o[e]);
        }
    }
#pragma unroll
    for (int e = 0; e < E; ++e) part_o[warp][lane * E + e] = o[e];
    if (lane == 0) part_l[warp] = L;
    __syncthreads();
    // ---- the warps' partial sums, in warp order ----
    float Lt = 0.f;
#pragma unroll
    for (int w = 0; w < CMB_WARPS; ++w) Lt += part_l[w];
    const float inv = 1.f / Lt;
    uint16_t *dst = out + ((size_t)r * Hq + h) * D;
    for (int c = threadIdx.x; c < D; c += CMB_WARPS * 32) {
        float acc = 0.f;
#pragma unroll
        for (int w = 0; w < CMB_WARPS; ++w) acc += part_o[w][c];
        __nv_bfloat16 v = __float2bfloat16_rn(acc * inv);
        dst[c] = *reinterpret_cast<uint16_t *>(&v);
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

static int attn_sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    return n;
}

// Q [R][Hq][d] viewed as a 3-D tensor (d, Hq, R): a (64, G, J) box at (a*64, g*G, b*(k+1) + j0)
// holds the J*G query vectors of (branch b, kv head g) with draft rows j0..j0+J-1, in row
// order (j - j0)*G + i.
static bool make_q_map(CUtensorMap *map, const void *q, int R, int Hq, int d, int G, int J) {
    EncodeTiledFnA fn = encode_fn_attn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)Hq, (cuuint64_t)R};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)Hq * d * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)J};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// An FP8 K or V pool viewed as a 2-D byte tensor (d, num_pages * Hkv * P): a box of
// box_rows rows of one raw sub-tile row's width (min(d, 128) bytes) is one page-run of a
// (page, kv head), landing unswizzled in the raw ring.
static bool make_kv_map(CUtensorMap *map, const void *pool, uint64_t rows, int d, int box_rows) {
    EncodeTiledFnA fn = encode_fn_attn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)d};
    cuuint32_t box[2] = {(cuuint32_t)(d < 128 ? d : 128), (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(pool), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Shared-memory plan, in this order (every block 1024-aligned): the Q buffer(s), 2 P
// buffers, the operand ring, the raw ring (FP8), 2 unit tables, barriers, flags. The M =
// 128 MMAs read up to (128 - R_pad) rows past the last Q block and (128 - PR) past the last
// P block; the operand ring that follows is always larger than that.
template <int D, bool FP8>
static int plan_rings(AttnTcParams &p, int QB) {
    using S_ = AttnShape<D, FP8>;
    const uint32_t q_bytes = QB * S_::NATOM * p.R_pad * 128, p_bytes = 2 * 2 * p.PR * 128;
    const uint32_t ut_bytes = 2 * (uint32_t)sizeof(UnitTable);
    const uint32_t bars = BAR_BYTES, small = 64 + 3072;
    const uint32_t fixed = 1024 + q_bytes + p_bytes + ut_bytes + bars + small;
    const uint32_t raw_row = FP8 ? S_::RAW_STAGE : 0;
    if (ATT_SMEM_LIMIT < fixed + 2 * S_::OP_STAGE + 2 * raw_row) return SPEC_ERR_UNSUPPORTED;
    const uint32_t avail = ATT_SMEM_LIMIT - fixed;
    if (!FP8) {
        p.NS = (int)(avail / S_::OP_STAGE);
        p.NS = p.NS > 6 ? 6 : p.NS;
        p.NR = 0;
    } else {
        // the raw ring holds the bytes in flight from HBM, the operand ring converted
        // sub-tiles waiting for their MMA: one stage more than two tiles' worth, so that the
        // converter (which works in ring order) never waits on V of a tile behind its softmax
        p.NS = 2 * S_::NSUB + 1;
        if (avail < p.NS * S_::OP_STAGE + 4 * raw_row) p.NS = 2 * S_::NSUB;
        if (avail < p.NS * S_::OP_STAGE + 2 * raw_row) p.NS = 2;
        p.NR = (int)((avail - p.NS * S_::OP_STAGE) / (raw_row ? raw_row : 1u));
        p.NR = p.NR > 8 ? 8 : p.NR;
        if (p.NR < 2) return SPEC_ERR_UNSUPPORTED;
    }
    p.QB = QB;
    return SPEC_OK;
}

// The plan for `copies` copies of the query layout: two Q buffers let a unit's Q load
// during the previous unit; one is used instead when that buys a deeper ring (the bytes in
// flight per SM).
template <int D, bool FP8>
static int plan_copies(AttnTcParams &p, int copies) {
    p.copies = copies;
    p.R_pad = (copies - 1) * p.qpc * 32 + p.PR;
    if (p.R_pad > MAX_RPAD) return SPEC_ERR_UNSUPPORTED;
    AttnTcParams p1 = p;
    const int st2 = plan_rings<D, FP8>(p, 2);
    const int st1 = plan_rings<D, FP8>(p1, 1);
    if (st2 && st1) return st2;
    // FP8: the raw ring first (bytes in flight), then the operand ring (converted stages)
    if (st2 || (FP8 ? (p1.NR > p.NR || (p1.NR == p.NR && p1.NS > p.NS)) : p1.NS > p.NS)) p = p1;
    return SPEC_OK;
}

// Four copies (queries within one lane quadrant) put a softmax warp on every SM
// sub-partition; two copies are used when four leave the operand ring too shallow to issue
// S of the next tile ahead of P.V (long head dims), or when the queries span two quadrants.
template <int D, bool FP8>
static int plan_attn(AttnTcParams &p, size_t *smem_bytes) {
    using S_ = AttnShape<D, FP8>;
    int st = SPEC_ERR_UNSUPPORTED;
    if (p.qpc == 1) {
        AttnTcParams p4 = p;
        st = plan_copies<D, FP8>(p4, 4);
        if (!st && p4.NS >= 2 * S_::NSUB) {
            p = p4;
        } else {
            AttnTcParams p2 = p;
            const int st2 = plan_copies<D, FP8>(p2, 2);
            if (!st2) {
                p = p2;
                st = SPEC_OK;
            } else if (!st) {
                p = p4;
            }
        }
    } else {
        st = plan_copies<D, FP8>(p, 2);
    }
    if (st) return st;
    if (bar_map(p.NS, p.NR).end > BAR_BYTES) return SPEC_ERR_UNSUPPORTED;
    p.OB = 256 + 2 * D <= 512 ? 2 : 1;
    const uint32_t q_bytes = p.QB * S_::NATOM * p.R_pad * 128, p_bytes = 2 * 2 * p.PR * 128;
    const uint32_t ut_bytes = 2 * (uint32_t)sizeof(UnitTable);
    const uint32_t bars = BAR_BYTES, small = 64 + 3072;
    p.off_q = 0;
    p.off_p = p.off_q + q_bytes;
    p.off_op = p.off_p + p_bytes;
    p.off_raw = p.off_op + p.NS * S_::OP_STAGE;
    p.off_ut = p.off_raw + p.NR * S_::RAW_STAGE;
    p.off_bar = p.off_ut + ut_bytes;
    p.off_small = p.off_bar + bars;
    *smem_bytes = 1024 + p.off_small + small;
    return SPEC_OK;
}

template <int D, bool FP8>
static int launch_attn_tc(AttnTcParams &p, cudaStream_t s) {
    using S_ = AttnShape<D, FP8>;
    size_t smem = 0;
    const int st = plan_attn<D, FP8>(p, &smem);
    if (st) return st;
    CUtensorMap mq0, mq1, mk, mv;
    if (!make_q_map(&mq0, p.q, p.B * (p.k + 1), p.Hq, D, p.G, p.J1)) return SPEC_ERR_CUDA;
    if (!make_q_map(&mq1, p.q, p.B * (p.k + 1), p.Hq, D, p.G, p.split ? p.k + 1 - p.J1 : p.J1)) return SPEC_ERR_CUDA;
    // FP8 pools with pages of at least 64 positions: K / V rows go to the raw ring by TMA
    // boxes of one page-run each, so the two loader warps issue a few boxes per sub-tile
    // instead of 16-byte copies (measured faster there; shorter runs make boxes too small
    // for the TMA issue rate, and on bf16 pools the branch's registers cost the cp.async
    // gather more than the boxes gained). A pool too large for 32-bit row coordinates also
    // takes the cp.async path.
    p.tma_rows = 0;
    mk = mq0;
    mv = mq0;
    const uint64_t pool_rows = (uint64_t)p.kv.num_pages * p.kv.n_kv_heads * p.kv.page_size;
    if (FP8 && p.kv.page_size >= 64 && pool_rows < (1ull << 31)) {
        const int br = p.kv.page_size < TILE_KEYS ? p.kv.page_size : TILE_KEYS;
        if (make_kv_map(&mk, p.kv.k_pool, pool_rows, D, br) && make_kv_map(&mv, p.kv.v_pool, pool_rows, D, br))
            p.tma_rows = br;
    }
    // a fixed ceiling (see the skinny GEMM launcher): graphs may mix launch sizes
    if (cudaFuncSetAttribute(attn_tc_kernel<D, FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize, ATT_SMEM_LIMIT) !=
        cudaSuccess)
        return SPEC_ERR_CUDA;
    const int sms = attn_sm_count();
    if (sms < 1) return SPEC_ERR_CUDA;
    const int grid = p.n_units < sms ? p.n_units : sms;
    return launch_pdl(attn_tc_kernel<D, FP8>, dim3(grid), dim3(S_::THREADS), smem, s, mq0, mq1, mk, mv, p);
}

// workspace: a 256-byte header (the unit scheduler's counters: zero before the first call,
// left zero by every call), the (m, l) pairs, the partial outputs
static size_t ws_bytes_for(int B, int Hkv, int n_splits, int n_q, int d) {
    const size_t units = (size_t)B * Hkv * n_splits;
    size_t ml = units * n_q * 2 * sizeof(float);
    ml = (ml + 255) & ~(size_t)255;
    return 256 + ml + units * n_q * d * sizeof(float);
}

// The launch parameters that depend only on the shapes (the caller checks the descriptor
// and fills in the pointers).
static int attn_setup(const spec_kv_desc *kvd, int B, int k, int n_q_heads, int max_pos, AttnTcParams &p) {
    if (B < 1 || k < 0 || k > SPEC_KMAX || n_q_heads < 1 || max_pos < k + 1) return SPEC_ERR_ARG;
    if (n_q_heads % kvd->n_kv_heads) return SPEC_ERR_ARG;
    const int G = n_q_heads / kvd->n_kv_heads;
    const int n_q = (k + 1) * G;
    const int N_pad = ((n_q + 15) / 16) * 16;
    // more than 32 query vectors need two TMEM lane quadrants: the draft rows are then split
    // in two halves of at most 32 lanes each when they fit (otherwise the vectors run
    // contiguously over both quadrants); PR = the lanes of one copy of that layout
    const int J1 = (k + 2) / 2;
    const bool split = n_q > 32 && k >= 1 && J1 * G <= 32 && (k + 1 - J1) * G <= 32;
    p = AttnTcParams{};
    p.kv = make_view(kvd);
    p.B = B;
    p.k = k;
    p.Hq = n_q_heads;
    p.G = G;
    p.n_q = n_q;
    p.J1 = split ? J1 : k + 1;
    p.split = split ? 1 : 0;
    p.PR = split ? 32 + (((k + 1 - J1) * G + 15) / 16) * 16 : N_pad;
    p.qpc = n_q > 32 ? 2 : 1;
    p.split_keys = split_keys_for(kvd->n_kv_heads);
    p.n_splits = (max_pos + p.split_keys - 1) / p.split_keys;
    p.max_pos = max_pos;
    p.n_units = B * kvd->n_kv_heads * p.n_splits;
    return N_pad > MAX_NPAD ? SPEC_ERR_UNSUPPORTED : SPEC_OK;
}

static int plan_dispatch(AttnTcParams &p, size_t *smem) {
    switch (p.kv.head_dim * 2 + (p.kv.kv_dtype == SPEC_KV_FP8_E4M3 ? 1 : 0)) {
        case 128: return plan_attn<64, false>(p, smem);
        case 129: return plan_attn<64, true>(p, smem);
        case 256: return plan_attn<128, false>(p, smem);
        case 257: return plan_attn<128, true>(p, smem);
        case 512: return plan_attn<256, false>(p, smem);
        default: return plan_attn<256, true>(p, smem);
    }
}

}  // namespace spec

SPEC_API int spec_verify_attn_plan(const spec_kv_desc *kvd, int B, int k, int n_q_heads, int max_pos, int32_t *out,
                                   int n_out) {
    if (!out || n_out < SPEC_ATTN_PLAN_FIELDS) return SPEC_ERR_ARG;
    int st = spec::check_kv_shape(kvd);
    if (st) return st;
    spec::AttnTcParams p;
    st = spec::attn_setup(kvd, B, k, n_q_heads, max_pos, p);
    if (st) return st;
    size_t smem = 0;
    st = spec::plan_dispatch(p, &smem);
    if (st) return st;
    const bool fp8 = kvd->kv_dtype == SPEC_KV_FP8_E4M3;
    const uint64_t pool_rows = (uint64_t)kvd->num_pages * kvd->n_kv_heads * kvd->page_size;
    const int tma_rows = fp8 && kvd->page_size >= 64 && pool_rows < (1ull << 31)
                             ? (kvd->page_size < spec::TILE_KEYS ? kvd->page_size : spec::TILE_KEYS)
                             : 0;
    const int32_t v[SPEC_ATTN_PLAN_FIELDS] = {(int32_t)smem, p.copies, p.qpc, p.R_pad, p.PR, p.NS, p.NR, p.QB, p.OB,
                                              p.split_keys, p.n_splits, p.n_units, p.split, tma_rows,
                                              (int32_t)spec::bar_map(p.NS, p.NR).end, (int32_t)spec::BAR_BYTES};
    for (int i = 0; i < SPEC_ATTN_PLAN_FIELDS; ++i) out[i] = v[i];
    return SPEC_OK;
}

SPEC_API size_t spec_verify_attn_workspace(const spec_kv_desc *kv, int B, int k, int n_q_heads, int max_pos) {
    if (spec::check_kv_desc(kv) || B < 1 || k < 0 || k > SPEC_KMAX || n_q_heads < 1 || max_pos < 1) return 0;
    if (n_q_heads % kv->n_kv_heads) return 0;
    const int G = n_q_heads / kv->n_kv_heads;
    const int sk = spec::split_keys_for(kv->n_kv_heads);
    const int n_splits = (max_pos + sk - 1) / sk;
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
    spec::AttnTcParams p;
    st = spec::attn_setup(kvd, B, k, n_q_heads, max_pos, p);
    if (st) return st;
    const int G = p.G, n_q = p.n_q;
    p.pos = pos;
    p.q = (const uint16_t *)q;
    p.scale_log2 = scale * spec::LOG2E;
    const size_t units = (size_t)p.n_units;
    size_t ml = units * n_q * 2 * sizeof(float);
    ml = (ml + 255) & ~(size_t)255;
    p.sched = (unsigned int *)ws;
    p.ws_ml = (float *)((char *)ws + 256);
    p.ws_o = (float *)((char *)ws + 256 + ml);
    p.err = dev_err;
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
    const int cblocks = R * n_q_heads;
    constexpr int CT = spec::CMB_WARPS * 32;
    uint16_t *o16 = (uint16_t *)out;
    const float *wml = p.ws_ml, *wo = p.ws_o;
    const int Hkv = kvd->n_kv_heads, ns = p.n_splits, sk = p.split_keys;
    switch (kvd->head_dim) {
        case 64:
            return spec::launch_pdl(spec::attn_combine_kernel<64>, dim3(cblocks), dim3(CT), 0, s, wml, wo, pos, B, k,
                                    n_q_heads, G, Hkv, ns, sk, max_pos, o16);
        case 128:
            return spec::launch_pdl(spec::attn_combine_kernel<128>, dim3(cblocks), dim3(CT), 0, s, wml, wo, pos, B, k,
                                    n_q_heads, G, Hkv, ns, sk, max_pos, o16);
        default:
            return spec::launch_pdl(spec::attn_combine_kernel<256>, dim3(cblocks), dim3(CT), 0, s, wml, wo, pos, B, k,
                                    n_q_heads, G, Hkv, ns, sk, max_pos, o16);
    }
}

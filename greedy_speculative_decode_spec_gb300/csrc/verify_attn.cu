// verify_attn.cu -- a2: causal GQA verify attention over paged KV (split-KV flash-decode
// on tcgen05 tensor cores, with the split merge in the same kernel).
//
// Row r = b*(k+1)+j (position p = pos[b]+j) and q head h attend keys 0..p of branch b
// (kv head h / G): span-02 engine/crates/model/src/spec.rs, module documentation
// (kv_hi = position, rejected-row KV beyond pos is never attended); memra-engine
// src/spec.rs, `full_attn_verify` (row r sees keys [0, base_len + r + 1), all verify
// rows in one launch); memra-engine `MtpScratch` (split count fixed by capacity, not by
// the current length, so one program serves every length bit for bit).
//
// Work unit = (branch b, kv head g, split of split_keys positions). The n_q = (k+1)*G
// query vectors that share kv head g are the narrow side of every MMA ("swap-AB"): the
// 128 keys of a tile sit on the TMEM lanes and the queries on the columns,
//     S^T[key][q]  = K_tile[key][:] . Q[q][:]            (M = 128 keys, N = NQ >= n_q)
//     O^T[d][q]   += V_tile^T[d][key] . P^T[key][q]      (M = 128 head-dim lanes)
//     L[*][q]     += ones[*][key] . P^T[key][q]          (the row sums, on every lane; the
//                                                         ones operand is held in TMEM)
// so the tensor work per tile scales with the real query count, not with a 128-row
// padding. FP8 pools feed their E4M3 K codes straight into kind::f8f6f4 MMAs: each query
// is split into two E4M3 terms (q * sigma = hi + lo, sigma a power of two per query), exact
// for every element within 2^10 of the query's largest one; V codes times their page
// scale are rounded to f16 for the P.V product (P in f16 too), or to bf16 (P in bf16) for a
// unit with a V page scale outside [2^-14, 128]. The K page scales are applied by the
// softmax to the scores.
//
// Softmax: a thread owns one key of the tile (its TMEM lane) and all query columns. One
// pass per tile with a lazily raised maximum: per tile the four softmax warps exchange
// their column maxima through shared memory; a column's running maximum m only moves when
// the tile's maximum exceeds it by more than RESCALE_TAU (log2 units), so P = 2^(s - m) <=
// 2^RESCALE_TAU, and O and L are rescaled in TMEM only on such a move. Every decision is
// taken per column from that column's own scores, so a query's result does not depend on
// the other queries of the batch.
//
// A persistent CTA per SM walks work units handed out by a global counter, with
// warp-specialised roles:
//   warps 0-3  softmax (warp w reads TMEM lane quadrant w: keys 32w..32w+31 of S, head-dim
//              lanes 32w.. of O) and each unit's epilogue, deferred until the next unit's
//              first P has been handed off;
//   warps 4-7  bf16 pools: warps 4-5 gather K rows, warps 6-7 V rows, with 16-byte cp.async
//              copies (zero fill past the branch's last position) into the 128-byte-swizzled
//              K and V rings; FP8 pools: turn the raw E4M3 V sub-tiles into scaled bf16 rows
//              of the V ring (one warp per SM sub-partition);
//   warp 8     per unit: takes the next work unit, fills the page table entries (and FP8
//              scales) into a shared table, loads Q by TMA boxes;
//   warp 9     issues S = K . Q^T of each tile (TMEM allocation is also this warp's);
//   warp 10    issues O += V^T . P^T and L += 1 . P^T of each tile;
//   warp 11    FP8 pools: TMA boxes of one page-run each, lane 0 K (straight into the MMA
//              layout), lane 1 V (into the raw ring), each lane on its own loop; no role for
//              bf16 pools.
// Keys beyond a row's position get P = 0 by select, never by multiplication, and V rows
// past the branch's last position are zero, so NaN in unused pool slots cannot reach a
// result. Tile and split boundaries sit at fixed key positions, and every MMA column is
// computed independently of the others, so a row's output is identical whatever B, k or
// batch it is verified in.
//
// Split merge: each unit writes its (m, l, O) partial, and a second kernel (a programmatic
// dependent launch) merges them per (row, head) with a summation order fixed by split
// positions alone: splits in groups of COMBINE_GROUP consecutive ones, each group summed in
// ascending order, then the groups in ascending order (skipping splits a row does not
// reach), so that any number of warps can share the work without changing a bit.
// Every pipeline wait is bounded (1 s unless a test shortens it): on a timeout the kernel
// raises SPEC_DEVERR_TIMEOUT, lets issued copies and MMAs land, frees TMEM and exits.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <math.h>

#include "common.cuh"
#include "sm100.cuh"

namespace spec {

using namespace sm100;

constexpr int SPLIT_KEYS = 2048;     // largest split; the split size is split_keys_for(Hkv, dtype)
constexpr int TILE_KEYS = 128;
constexpr int COMBINE_GROUP = 8;     // splits summed in order before the groups are
constexpr int MAX_NQ = 128;          // query vectors per (branch, kv head), padded to 16
constexpr float LOG2E = 1.4426950408889634f;
constexpr float RESCALE_TAU = 8.0f;  // P <= 2^8: exact range for bf16 and f16 alike
// FP8 pools: the converted V and P are f16 when every V page scale of the unit lies in
// [2^-14, 128] (the scale is an f16 normal, and |code * scale| <= 448 * 128 < 65504, so no
// converted value overflows), bf16 otherwise; f16 keeps three more mantissa bits of both,
// and the conversion is one f16 multiply
constexpr float VF16_MIN_SCALE = 6.103515625e-05f;
constexpr float VF16_MAX_SCALE = 128.0f;
constexpr uint64_t ATT_WAIT_NS = 1000000000ull;
constexpr int ATT_SMEM_LIMIT = 227 * 1024;
constexpr int ATT_THREADS = 384;

struct UnitInfo {
    int b, g, split, rank, pos_b, kv_end, s0, T, n_used, u;  // u: the unit's workspace slot
    bool bad_pos;
};

// Per-unit table the producer warp fills: the unit itself (computed once, read by every
// role), the error bits of any invalid page-table entry, and then, for pages of >= 8
// positions, E = ceil(split_keys / page_size) entries each of: the page of each page-sized
// run of the split's keys (-1 if the entry is invalid), and the page's FP8 K and V scales.
// The plan sizes E; a table is the header followed by its three arrays.
struct alignas(16) UnitTable {
    UnitInfo ui;
    int32_t bad;
    int32_t vf16;          // FP8: the unit's P.V runs in f16 (every V page scale keeps code * scale in range)
    int32_t iter;          // the unit's index in the walk order, or -1: no more units
};
// the arrays (and the softmax scratch that follows the two tables) are read with 16-byte
// vector loads
static_assert(sizeof(UnitTable) % 16 == 0, "unit table size must keep 16-byte alignment");
struct UnitTabView {
    UnitTable *h;
    int32_t *page;
    float *ksc, *vsc;
};
__host__ __device__ constexpr uint32_t unit_table_stride(int entries) {
    return (uint32_t)((sizeof(UnitTable) + 12u * (uint32_t)entries + 15u) & ~15u);
}
__device__ __forceinline__ UnitTabView unit_tab(uint8_t *base, uint32_t ub, int entries) {
    UnitTabView v;
    uint8_t *t = base + ub * unit_table_stride(entries);
    v.h = reinterpret_cast<UnitTable *>(t);
    v.page = reinterpret_cast<int32_t *>(t + sizeof(UnitTable));
    v.ksc = reinterpret_cast<float *>(v.page + entries);
    v.vsc = v.ksc + entries;
    return v;
}

// Split size in positions, a function of the KV pool's shape only (its KV-head count and
// element type; never of B, k or the context length, so a row's split boundaries are the
// same in every batch): few KV heads give few work units per branch, so their splits are
// shorter; with more, a split holds about 512 KB of K and V at a head dimension of 128
// (2048 E4M3 positions, 1024 bf16 ones), long enough that a unit's fixed costs are small
// against its tiles, short enough that the units balance across the SMs.
__host__ __device__ constexpr int split_keys_for(int n_kv_heads, bool fp8) {
    return n_kv_heads <= 2 ? 256 : (n_kv_heads <= 4 ? 512 : (fp8 ? SPLIT_KEYS : SPLIT_KEYS / 2));
}

template <int D, bool FP8>
struct AttnShape {
    static constexpr int SUB = D < 128 ? D : 128;          // head-dim columns per sub-tile
    static constexpr int NSUB = D / SUB;                    // sub-tiles per tile (d halves for 256)
    static constexpr uint32_t OP_STAGE = TILE_KEYS * SUB * 2;  // 16-bit sub-tile: 128 keys x SUB
    static constexpr uint32_t F8_STAGE = TILE_KEYS * SUB;      // E4M3 sub-tile
    static constexpr uint32_t K_STAGE = FP8 ? F8_STAGE : OP_STAGE;  // a K ring stage
    static constexpr int KSTEP = FP8 ? 32 : 16;             // K elements per MMA of S
    static constexpr int K8ROW = SUB;                       // bytes per E4M3 row of a sub-tile
    static constexpr int NATOM_Q = D / 64;                  // 128-byte column blocks of a bf16 Q row
    static constexpr int Q8ROW = D < 128 ? 64 : 128;        // bytes per row of an E4M3 Q block
    static constexpr int NQ8 = D / Q8ROW;                   // E4M3 Q column blocks
};

struct AttnParams {
    KvView kv;
    const int32_t *pos;
    const int32_t *anc;    // tree verify: [B*(k+1)] ancestor masks over the verify slots; null: a chain
    int B, k, Hq, G, n_q, NQ, n_splits, max_pos, n_units, split_keys;
    int TPI;               // tiles per softmax iteration (a tile group)
    // FP8 pools: rows per TMA box of the K / V gather (one page-run: min(page size, 128))
    int tma_rows;
    const uint16_t *q;     // bf16 [R][Hq][d]
    const float *qinv_g;   // FP8: [B*Hkv][NQ] 1/sigma of every query column (the split's scale)
    uint8_t *q8_g;         // FP8: [B*Hkv][2][NQ][d] the split queries' E4M3 terms (hi, lo)
    uint16_t *out;         // bf16 [R][Hq][d]
    float scale_log2;      // softmax scale * log2(e)
    unsigned int *sched;   // [2]: next unit to hand out, CTAs done (zero between calls)
    float *ws_ml;          // [units][NQ][2]  (m in log2 units, l)
    float *ws_o;           // [units][NQ][d]
    int32_t *err;
    uint64_t wait_ns;      // pipeline-wait limit
    int NK, NV, NR, NSB, NPB, QB, OB;  // K, bf16 V and (FP8) raw V ring stages; S, P, Q, O buffers
    int ut_entries;        // page-table entries per unit table (0 for pages of < 8 positions)
    uint32_t off_q, off_q8, off_p, off_k, off_v, off_raw, off_ut, off_sx, off_bar, off_small;
    uint32_t t_o;          // first TMEM column of the O / L buffers
    uint32_t t_one;        // first TMEM column of the ones operand (8 bf16 columns, then 8 f16)
};

// The CTA's mbarriers, as byte offsets from the barrier region (one definition for the
// kernel and the host plan, which checks that they fit BAR_BYTES).
struct BarMap {
    uint32_t kfull, kempty, vfull, vempty, rfull, rempty, sfull, sfree, pfull, pfree, ofree;
    uint32_t qfull, qfree, ufull, ufree, lfin, drain, xbar, end;
};
__host__ __device__ inline BarMap bar_map(int NK, int NV, int NR, int NSB, int NPB) {
    BarMap m;
    uint32_t o = 0;
    m.kfull = o;    o += 8 * NK;   // K ring
    m.kempty = o;   o += 8 * NK;
    m.vfull = o;    o += 8 * NV;   // bf16 V ring
    m.vempty = o;   o += 8 * NV;
    m.rfull = o;    o += 8 * NR;   // FP8 raw V ring
    m.rempty = o;   o += 8 * NR;
    m.sfull = o;    o += 8 * NSB;
    m.sfree = o;    o += 8 * NSB;
    m.pfull = o;    o += 8 * NPB;
    m.pfree = o;    o += 8 * NPB;
    m.ofree = o;    o += 16;
    m.qfull = o;    o += 16;
    m.qfree = o;    o += 16;
    m.ufull = o;    o += 16;
    m.ufree = o;    o += 16;
    m.lfin = o;     o += 16;
    m.drain = o;    o += 16;
    m.xbar = o;     o += 16;   // softmax column-maximum exchange, by group parity
    m.end = o;
    return m;
}
constexpr uint32_t BAR_BYTES = 8 * 96;

// The scheduler hands out units by rank, the rank of a split being its distance from its
// pair's last split: first every (branch, head) pair's split of rank n_splits - 1 (only the
// longest pairs have one), ..., last every pair's rank-0 split, its last and only partial
// one. Long pairs thus start first and the short partial units come last, where they fill
// the gaps of the grid's final wave; walk entries with no split (rank >= the pair's split
// count) are empty. `u` (the workspace slot) is (branch, head, split)-major, so a merge
// group's partials are contiguous.
static __device__ __noinline__ UnitInfo unit_info(const AttnParams &p, int iter) {
    UnitInfo ui;
    const int pairs = p.B * p.kv.n_kv_heads;
    ui.rank = p.n_splits - 1 - iter / pairs;
    ui.g = (iter % pairs) % p.kv.n_kv_heads;
    ui.b = (iter % pairs) / p.kv.n_kv_heads;
    ui.pos_b = __ldg(p.pos + ui.b);
    ui.bad_pos = ui.pos_b < 0 || ui.pos_b + p.k + 1 > p.max_pos;
    ui.kv_end = ui.pos_b + p.k + 1;
    ui.n_used = ui.bad_pos ? 0 : (ui.kv_end + p.split_keys - 1) / p.split_keys;
    ui.split = ui.n_used - 1 - ui.rank;  // < 0: no such split
    ui.u = (ui.b * p.kv.n_kv_heads + ui.g) * p.n_splits + (ui.split < 0 ? 0 : ui.split);
    ui.s0 = ui.split * p.split_keys;
    int n = ui.split < 0 ? 0 : ui.kv_end - ui.s0;
    n = n > p.split_keys ? p.split_keys : n;
    ui.T = (n + TILE_KEYS - 1) / TILE_KEYS;
    return ui;
}

// byte offset of 16-bit element (row, col) in a K-major (or, read the other way, MN-major)
// 128-byte-swizzled tile whose 64-column blocks are `block_bytes` apart
__device__ __forceinline__ uint32_t sw128_off(int row, int col, uint32_t block_bytes) {
    const int blk = col >> 6, c = col & 63;
    return blk * block_bytes + row * 128 + ((((c >> 3) ^ (row & 7)) & 7) << 4);
}

// Every lane waits; the verdict is made uniform across the warp so that no lane can
// leave a loop that the others stay in. SLEEP > 0: the warp is not latency-critical and
// sleeps about SLEEP ns between probes, so that it does not take issue slots from the
// softmax warp of its SM sub-partition.
template <uint32_t SLEEP = 0>
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag, uint64_t ns) {
    const bool r = SLEEP ? mbar_wait_sleep(bar, parity, abort_flag, ns, SLEEP) : mbar_wait(bar, parity, abort_flag, ns);
    return __all_sync(0xFFFFFFFFu, r);
}
// A position in a ring of n stages: the stage and the parity of its current use (kept by
// increments, so that no loop divides by a run-time ring size).
struct RingPos {
    uint32_t s = 0, ph = 0;
    __device__ __forceinline__ void next(int n) {
        if (++s == (uint32_t)n) {
            s = 0;
            ph ^= 1u;
        }
    }
    __device__ __forceinline__ void prev(int n) {
        if (s == 0) {
            s = (uint32_t)n;
            ph ^= 1u;
        }
        --s;
    }
};
// Waits (drain, bounded) for the last min(used, n) completed phases of a ring's barriers,
// walking back from the position after the last use.
__device__ __noinline__ void drain_ring(uint32_t bar0, RingPos r, int n, uint32_t used) {
    for (uint32_t j = 0; j < (uint32_t)n && j < used; ++j) {
        r.prev(n);
        mbar_wait(bar0 + 8 * r.s, r.ph, nullptr, ATT_WAIT_NS);
    }
}
// tiles before a unit's end at which its K stream lets the producer take the next unit
constexpr int NEXT_UNIT_LEAD = 6;
constexpr uint32_t SLEEP_LOAD = 128;  // loaders, converters, producer
constexpr uint32_t SLEEP_MMA = 32;    // MMA issuers
// FP8 TMA lanes (polling probes): a failed probe sleeps, so that the polling warp leaves
// the issue slots of its SM sub-partition to the softmax and converter warps there
// (long-context FP8: 264 -> 246 us per call against busy polling)
constexpr uint32_t SLEEP_POLL = 20;

// The wait of the two FP8 TMA lanes, which share a warp but run their own loops: non-blocking
// probes (a probe never holds the warp, so the other lane's path keeps being issued), a
// sleep after each failed one, bounded like every other wait. Inline: an out-of-line call
// made from the two divergent lanes serialises them, so that one lane's sleep stalls the
// other.
__device__ __forceinline__ bool lane_poll_wait(uint32_t bar, uint32_t parity, volatile int *abort, uint64_t timeout_ns) {
    const uint64_t t0 = globaltimer();
    for (uint32_t i = 1;; ++i) {
        if (mbar_test(bar, parity)) return true;
        __nanosleep(SLEEP_POLL);
        if ((i & 7u) == 0) {
            if (abort != nullptr && *abort) return false;
            if (globaltimer() - t0 > timeout_ns) return false;
        }
    }
}

__device__ __forceinline__ uint32_t pack2(float a, float b, bool f16) {
    if (f16) {
        const __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<const uint32_t *>(&h);
    }
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// The weight of a partial result with maximum m against the merged maximum M: exactly 1
// when m is the maximum (so a merge of one partial reproduces it bit for bit).
__device__ __forceinline__ float merge_weight(float m, float M) { return m == M ? 1.f : ex2_approx(m - M); }

template <int D, bool FP8>
__global__ void __launch_bounds__(ATT_THREADS, 1)
    attn_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                const __grid_constant__ CUtensorMap map_v, AttnParams p) {
    using S_ = AttnShape<D, FP8>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t s_base = smem_u32(smem);
    const int NQ = p.NQ, n_q = p.n_q;
    const uint32_t QATOM = (uint32_t)NQ * 128, QBUF = S_::NATOM_Q * QATOM;      // bf16 Q
    const uint32_t Q8ATOM = (uint32_t)NQ * S_::Q8ROW, Q8PART = S_::NQ8 * Q8ATOM;  // one E4M3 Q part
    const uint32_t PTILE = (uint32_t)NQ * 256;                                  // a tile's P^T: [NQ/16][128 keys][32 B]
    const uint32_t PBUF = (uint32_t)p.TPI * PTILE;                              // a tile group's
    const uint32_t s_q = s_base + p.off_q, s_q8 = s_base + p.off_q8, s_p = s_base + p.off_p;
    const uint32_t s_k = s_base + p.off_k, s_v = s_base + p.off_v;
    const uint32_t s_raw = s_base + p.off_raw;
    uint8_t *ut_base = smem + p.off_ut;  // [2] unit tables
    const int UTE = p.ut_entries;
    const BarMap bm = bar_map(p.NK, p.NV, p.NR, p.NSB, p.NPB);
    const uint32_t bar0 = s_base + p.off_bar;
    const uint32_t kfull = bar0 + bm.kfull, kempty = bar0 + bm.kempty;
    const uint32_t vfull = bar0 + bm.vfull, vempty = bar0 + bm.vempty;
    const uint32_t rfull = bar0 + bm.rfull, rempty = bar0 + bm.rempty;
    const uint32_t sfull = bar0 + bm.sfull, sfree = bar0 + bm.sfree;
    const uint32_t pfull = bar0 + bm.pfull, pfree = bar0 + bm.pfree;
    const uint32_t ofree = bar0 + bm.ofree;
    const uint32_t qfull = bar0 + bm.qfull, qfree = bar0 + bm.qfree;
    const uint32_t ufull = bar0 + bm.ufull, ufree = bar0 + bm.ufree, lfin = bar0 + bm.lfin;
    const uint32_t drain = bar0 + bm.drain, xbar = bar0 + bm.xbar;
    uint8_t *small = smem + p.off_small;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(small);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(small + 4);
    // softmax scratch: column-maximum exchange [2 exchange slots][4 warps][NQ], then per warp
    // its copy of the running maxima [2 unit parities][4][NQ] (a unit's maxima outlive it
    // until its deferred epilogue), the rescale factors and the column limits [4][NQ], then
    // the E4M3 Q scales [2 unit tables][NQ], then per exchange slot and warp whether a running
    // maximum must move
    float *sx_red = reinterpret_cast<float *>(smem + p.off_sx);
    float *sx_m = sx_red + 8 * NQ;
    float *sx_f = sx_m + 8 * NQ;
    int *sx_msk = reinterpret_cast<int *>(sx_f + 4 * NQ);
    float *sx_qinv = reinterpret_cast<float *>(sx_msk + 4 * NQ);
    int *sx_need = reinterpret_cast<int *>(sx_qinv + 2 * NQ);  // [2 exchange slots][4 warps]
    // per query column q = j*G + i: its draft row j (-1 for padding) and its output offset
    // (j*Hq + i)*D from the (branch, kv head)'s first output
    int *sx_colj = sx_need + 8;
    int *sx_coloff = sx_colj + NQ;
    const uint64_t wns = p.wait_ns;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool small_pages = p.kv.page_size < 8;  // no page-table entries: per-row lookups
    const int log2P = p.kv.log2_page;

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.NK; ++s) {
            mbar_init(kfull + 8 * s, FP8 ? 1 : 64);  // FP8: the TMA bytes; bf16: each K loader thread
            mbar_init(kempty + 8 * s, 1);            // an S MMA commit
        }
        for (int s = 0; s < p.NV; ++s) {
            mbar_init(vfull + 8 * s, FP8 ? 4 : 64);  // FP8: each converter warp; bf16: each V loader thread
            mbar_init(vempty + 8 * s, 1);            // a P.V commit
        }
        for (int s = 0; s < p.NR; ++s) {
            mbar_init(rfull + 8 * s, 1);             // the TMA bytes
            mbar_init(rempty + 8 * s, 4);            // each converter warp
        }
        for (int s = 0; s < p.NSB; ++s) {
            mbar_init(sfull + 8 * s, 1);
            mbar_init(sfree + 8 * s, 4);
        }
        for (int s = 0; s < p.NPB; ++s) {
            mbar_init(pfull + 8 * s, 4);
            mbar_init(pfree + 8 * s, 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(ofree + 8 * a, 4);
            mbar_init(qfull + 8 * a, 1);
            mbar_init(qfree + 8 * a, 1);
            mbar_init(ufull + 8 * a, 1);
            // softmax 4, both MMA issuers, bf16 loaders 4 / FP8 converters 4 and the two TMA lanes
            mbar_init(ufree + 8 * a, FP8 ? 12 : 10);
            mbar_init(lfin + 8 * a, FP8 ? 1 : 2);  // the K stream: FP8 its TMA lane, bf16 its two loader warps
            mbar_init(drain + 8 * a, 1);
            mbar_init(xbar + 8 * a, 4);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    for (int q = threadIdx.x; q < NQ; q += ATT_THREADS) {
        sx_colj[q] = q < n_q ? q / p.G : -1;
        sx_coloff[q] = q < n_q ? ((q / p.G) * p.Hq + q % p.G) * D : 0;
    }
    // bf16 Q rows n_q..NQ-1 (never written by the Q loads) are zero, so the padding columns
    // of S hold finite zeros
    if (!FP8 && NQ > n_q) {
        const int per = (NQ - n_q) * 8;  // 16-byte pieces per (buffer, column block)
        for (int i = threadIdx.x; i < p.QB * S_::NATOM_Q * per; i += ATT_THREADS) {
            const int blk = i / per, r = i % per;
            *reinterpret_cast<uint4 *>(smem + p.off_q + blk * QATOM + n_q * 128 + r * 16) = make_uint4(0, 0, 0, 0);
        }
    }
    if (warp == 8 && lane == 0) {
        prefetch_tmap(&map_q);
        if (FP8) {
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
    const uint32_t t_o0 = tmem + p.t_o;  // O buffers: [OB][NSUB + 1][NQ] columns (the last NQ: L)

    if (warp == 8) {
        // ================= producer: per unit, the page table entries and Q =================
        // Units are handed out dynamically: the producer takes the next index of the
        // rank-ordered walk from a global counter, skips empty units, and publishes the unit
        // in the shared table that every other role waits on (-1 ends their loops). It takes
        // a unit only once a table is free and the K loads are issuing the last
        // NEXT_UNIT_LEAD tiles of the previous unit: late enough that a CTA holds little more
        // than the work in its rings (the last units go to whichever CTAs run out of work
        // first), early enough that the next unit's table and Q are ready when the loaders
        // get to it.
        uint32_t ua = 0;
        RingPos qr;  // Q buffers
        bool ok = true;
        for (;;) {
            const uint32_t ub = ua & 1u, uph = (ua >> 1) & 1u;
            const UnitTabView tv = unit_tab(ut_base, ub, UTE);
            UnitTable *tab = tv.h;
            if (!warp_wait<SLEEP_LOAD>(ufree + 8 * ub, uph ^ 1u, abort_flag, wns)) { ok = false; break; }
            if (ua > 0 && !warp_wait<SLEEP_LOAD>(lfin + 8 * ((ua - 1) & 1u), ((ua - 1) >> 1) & 1u, abort_flag, wns)) {
                ok = false;
                break;
            }
            int it_u = -1;
            UnitInfo ui;
            for (;;) {
                int cand = 0;
                if (lane == 0) cand = (int)atomicAdd(p.sched, 1u);
                cand = __shfl_sync(0xFFFFFFFFu, cand, 0);
                if (cand >= p.n_units) break;
                ui = unit_info(p, cand);
                if (ui.T > 0) {
                    it_u = cand;
                    break;
                }
                if (ui.bad_pos && ui.rank == 0 && ui.g == 0 && lane == 0) raise_error(p.err, SPEC_DEVERR_POS);
            }
            if (it_u < 0) {
                if (lane == 0) tab->iter = -1;
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(ufull + 8 * ub);
                    // no new work for this CTA: the next kernel in the stream may be scheduled
                    grid_dep_launch();
                }
                break;
            }
            int badbits = 0;
            bool v_big = false;  // some V page scale of the unit is too large for an f16 P.V
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
                        v_big |= !(vs >= VF16_MIN_SCALE && vs <= VF16_MAX_SCALE);
                    }
                    tv.page[e] = pg < 0 ? -1 : pg;
                    tv.ksc[e] = ks;
                    tv.vsc[e] = vs;
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
            v_big = __any_sync(0xFFFFFFFFu, v_big);
            if (FP8) {  // the unit's query scales (1/sigma per column), read by the softmax
                const float *qi = p.qinv_g + (size_t)(ui.b * p.kv.n_kv_heads + ui.g) * NQ;
                for (int q = lane; q < NQ; q += 32) sx_qinv[ub * NQ + q] = __ldg(qi + q);
            }
            if (lane == 0) {
                tab->ui = ui;
                tab->bad = badbits;
                tab->vf16 = FP8 && !v_big ? 1 : 0;
                tab->iter = it_u;
                if (badbits) raise_error(p.err, badbits);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(ufull + 8 * ub);
            // ---- Q of (b, g) ----
            // bf16: one 3-D box per 64-column block lands as rows j*G + i. FP8: the two E4M3
            // parts (hi, lo) of the split queries, one 2-D box per 128-byte column block each
            // (the split kernel wrote them as [pair][part][NQ][d] bytes).
            const uint32_t qs = qr.s;
            if (!warp_wait<SLEEP_LOAD>(qfree + 8 * qs, qr.ph ^ 1u, abort_flag, wns)) { ok = false; break; }
            if (lane == 0) {
                if (FP8) {
                    mbar_arrive_expect_tx(qfull + 8 * qs, (uint32_t)(2 * NQ * D));
                    const int row0 = (ui.b * p.kv.n_kv_heads + ui.g) * 2 * NQ;
#pragma unroll
                    for (int part = 0; part < 2; ++part)
#pragma unroll
                        for (int a = 0; a < S_::NQ8; ++a)
                            tma_load_2d(s_q8 + (qs * 2 + part) * Q8PART + a * Q8ATOM, &map_q, a * S_::Q8ROW,
                                        row0 + part * NQ, qfull + 8 * qs);
                } else {
                    mbar_arrive_expect_tx(qfull + 8 * qs, (uint32_t)(S_::NATOM_Q * n_q * 128));
#pragma unroll
                    for (int a = 0; a < S_::NATOM_Q; ++a)
                        tma_load_3d(s_q + qs * QBUF + a * QATOM, &map_q, a * 64, ui.g * p.G, ui.b * (p.k + 1),
                                    qfull + 8 * qs);
                }
            }
            __syncwarp();
            ++ua;
            qr.next(p.QB);
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
        if (lane == 0) drain_ring(qfull, qr, p.QB, ua);
        __syncwarp();
    } else if (warp == 9) {
        // ================= MMA issuer: S^T = K . Q^T =================
        const uint32_t idesc = FP8 ? idesc_f8_e4m3(128, NQ) : idesc_f16kind(128, NQ, false, false, false);
        uint32_t gs = 0, ua = 0, gk = 0;  // tile groups, active units, K sub-tiles consumed
        RingPos kr, sr, qr;               // K ring, S buffers, Q buffers
        bool ok = true;
        for (;;) {
            const uint32_t ub = ua & 1u, uph = (ua >> 1) & 1u;
            if (!warp_wait<SLEEP_MMA>(ufull + 8 * ub, uph, abort_flag, wns)) { ok = false; break; }
            const UnitTable *tab = unit_tab(ut_base, ub, UTE).h;
            const int it_u = tab->iter;
            if (it_u < 0) break;
            const UnitInfo ui = tab->ui;
            __syncwarp();
            if (lane == 0) mbar_arrive(ufree + 8 * ub);
            const uint32_t qs = qr.s;
            if (!warp_wait<SLEEP_MMA>(qfull + 8 * qs, qr.ph, abort_flag, wns)) { ok = false; break; }
            tc_fence_after();
            for (int t0 = 0; t0 < ui.T; t0 += p.TPI, ++gs, sr.next(p.NSB)) {
                // a group of up to TPI tiles: each tile's S into its own NQ columns of the group's
                // S buffer, one "full" signal for the group
                const uint32_t sb = sr.s;
                const int nt = min(p.TPI, ui.T - t0);
                if (!warp_wait<SLEEP_MMA>(sfree + 8 * sb, sr.ph ^ 1u, abort_flag, wns)) {
                    ok = false;
                    break;
                }
#pragma unroll 1
                for (int i = 0; i < nt && ok; ++i) {
#pragma unroll
                    for (int h = 0; h < S_::NSUB; ++h) {
                        const uint32_t st = kr.s;
                        if (!warp_wait<SLEEP_MMA>(kfull + 8 * st, kr.ph, abort_flag, wns)) { ok = false; break; }
                        kr.next(p.NK);
                        ++gk;
                        if (!FP8) fence_proxy_async_smem();  // cp.async data -> tensor core reads
                        tc_fence_after();
                        if (lane == 0) {
                            const uint32_t kb = s_k + st * S_::K_STAGE;
                            const uint32_t d_s = tmem + (sb * (uint32_t)p.TPI + (uint32_t)i) * (uint32_t)NQ;
                            if (FP8) {
                                // S = K . (hi + lo)^T: both E4M3 parts accumulate into one S
                                const uint64_t ka0 = desc_kmajor(kb, S_::K8ROW, 8 * S_::K8ROW);
                                const uint64_t qa0 = desc_kmajor(s_q8 + qs * 2 * Q8PART, S_::Q8ROW, 8 * S_::Q8ROW);
#pragma unroll
                                for (int part = 0; part < 2; ++part) {
#pragma unroll
                                    for (int kl = 0; kl < S_::SUB / 32; ++kl) {
                                        const int ks = h * (S_::SUB / 32) + kl;  // 32-byte step over all of d
                                        const uint32_t qoff = S_::Q8ROW == 128 ? (ks >> 2) * Q8ATOM + (ks & 3) * 32
                                                                               : (uint32_t)ks * 32;
                                        mma_f8(d_s, desc_advance(ka0, kl * 32), desc_advance(qa0, part * Q8PART + qoff), idesc,
                                               (h > 0 || part > 0 || kl > 0) ? 1u : 0u);
                                    }
                                }
                            } else {
                                const uint64_t ka0 = desc_kmajor(kb, 128, 1024), qb0 = desc_kmajor(s_q + qs * QBUF, 128, 1024);
#pragma unroll
                                for (int kl = 0; kl < S_::SUB / 16; ++kl) {
                                    const int ks = h * (S_::SUB / 16) + kl;  // 16-element step over all of d
                                    mma_bf16(d_s, desc_advance(ka0, (kl >> 2) * (TILE_KEYS * 128) + (kl & 3) * 32),
                                             desc_advance(qb0, (ks >> 2) * QATOM + (ks & 3) * 32), idesc, ks > 0 ? 1u : 0u);
                                }
                            }
                            mma_commit(kempty + 8 * st);
                        }
                        __syncwarp();
                    }
                }
                if (!ok) break;
                if (lane == 0) {
                    mma_commit(sfull + 8 * sb);
                    // the unit's last S: its Q buffers are free once these MMAs complete
                    if (t0 + nt == ui.T) mma_commit(qfree + 8 * qs);
                }
                __syncwarp();
            }
            if (!ok) break;
            ++ua;
            qr.next(p.QB);
        }
        if (!ok) {
            *abort_flag = 1;
            if (lane == 0) raise_error(p.err, SPEC_DEVERR_TIMEOUT);
        }
        if (lane == 0) {
            mma_commit(drain);
            mbar_wait(drain, 0, nullptr, ATT_WAIT_NS);
            // every arrive sent by this issuer's commits is delivered before the CTA may exit:
            // the last phases of the K ring's "empty" barriers, of the S buffers' "full" and of
            // the Q buffers' "free" (only commits that were issued are waited for, so a CTA that
            // gave up on a wait also leaves at once)
            drain_ring(kempty, kr, p.NK, gk);
            drain_ring(sfull, sr, p.NSB, gs);
            drain_ring(qfree, qr, p.QB, ua);
        }
        __syncwarp();
    } else if (warp == 10) {
        // ================= MMA issuer: O^T += V^T . P^T, L += 1 . P^T =================
        // bf16 operands, or f16 ones for FP8 units whose V and P are f16
        const uint32_t idesc_pv_b = idesc_f16kind(128, NQ, false, true, true), idesc_l_b = idesc_f16kind(128, NQ, false, false, true);
        const uint32_t idesc_pv_h = idesc_f16kind(128, NQ, true, true, true), idesc_l_h = idesc_f16kind(128, NQ, true, false, true);
        // V's MN-major descriptor: 64-column blocks 128 keys x 128 bytes apart; a 64-wide
        // head dimension repeats its one block on lanes 64..127 (never read)
        const uint32_t v_lbo = S_::SUB == 128 ? TILE_KEYS * 128 : 0;
        uint32_t gp = 0, gv = 0, ua = 0;  // tile groups, V sub-tiles consumed, units
        RingPos pr, vr, orr;              // P buffers, V ring, O buffers
        bool ok = true;
        for (;;) {
            const uint32_t ub = ua & 1u, uph = (ua >> 1) & 1u;
            if (!warp_wait<SLEEP_MMA>(ufull + 8 * ub, uph, abort_flag, wns)) { ok = false; break; }
            const UnitTable *tab = unit_tab(ut_base, ub, UTE).h;
            const int it_u = tab->iter;
            if (it_u < 0) break;
            const UnitInfo ui = tab->ui;
            const bool vf16 = FP8 && tab->vf16 != 0;
            const uint32_t idesc_pv = vf16 ? idesc_pv_h : idesc_pv_b, idesc_l = vf16 ? idesc_l_h : idesc_l_b;
            const uint32_t t_one = tmem + p.t_one + (vf16 ? 8u : 0u);  // the A operand of the row sums
            __syncwarp();
            if (lane == 0) mbar_arrive(ufree + 8 * ub);
            const uint32_t ob = orr.s;
            if (!warp_wait<SLEEP_MMA>(ofree + 8 * ob, orr.ph ^ 1u, abort_flag, wns)) { ok = false; break; }
            tc_fence_after();
            const uint32_t d_o = t_o0 + ob * (uint32_t)((S_::NSUB + 1) * NQ);
            for (int t0 = 0; t0 < ui.T; t0 += p.TPI, ++gp, pr.next(p.NPB)) {
                const uint32_t pb = pr.s;
                const int nt = min(p.TPI, ui.T - t0);
                if (!warp_wait<SLEEP_MMA>(pfull + 8 * pb, pr.ph, abort_flag, wns)) { ok = false; break; }
#pragma unroll 1
                for (int i = 0; i < nt && ok; ++i) {
                    const int t = t0 + i;
                    const uint32_t pa = s_p + pb * PBUF + (uint32_t)i * PTILE;
#pragma unroll
                    for (int h = 0; h < S_::NSUB; ++h) {
                        const uint32_t st = vr.s;
                        if (!warp_wait<SLEEP_MMA>(vfull + 8 * st, vr.ph, abort_flag, wns)) { ok = false; break; }
                        if (!FP8) fence_proxy_async_smem();  // cp.async data -> tensor core reads
                        const uint32_t vb = s_v + st * S_::OP_STAGE, rel = vempty + 8 * st;
                        ++gv;
                        vr.next(p.NV);
                        tc_fence_after();
                        if (lane == 0) {
                            const uint64_t va0 = desc_mnmajor_sw128(vb, v_lbo), pa0 = desc_mnmajor_sw32(pa, TILE_KEYS * 32);
#pragma unroll
                            for (int ks = 0; ks < TILE_KEYS / 16; ++ks)
                                mma_bf16(d_o + h * NQ, desc_advance(va0, ks * 2048), desc_advance(pa0, ks * 512), idesc_pv,
                                         (t > 0 || ks > 0) ? 1u : 0u);
                            mma_commit(rel);
                        }
                        __syncwarp();
                    }
                }
                if (!ok) break;
                if (lane == 0) {
#pragma unroll 1
                    for (int i = 0; i < nt; ++i) {
                        const int t = t0 + i;
                        const uint64_t pa0 = desc_mnmajor_sw32(s_p + pb * PBUF + (uint32_t)i * PTILE, TILE_KEYS * 32);
#pragma unroll
                        for (int ks = 0; ks < TILE_KEYS / 16; ++ks)
                            mma_f16_ta(d_o + S_::NSUB * NQ, t_one, desc_advance(pa0, ks * 512), idesc_l,
                                       (t > 0 || ks > 0) ? 1u : 0u);
                    }
                    mma_commit(pfree + 8 * pb);  // also: this group's O and L are complete
                }
                __syncwarp();
            }
            if (!ok) break;
            ++ua;
            orr.next(p.OB);
        }
        if (!ok) {
            *abort_flag = 1;
            if (lane == 0) raise_error(p.err, SPEC_DEVERR_TIMEOUT);
        }
        if (lane == 0) {
            mma_commit(drain + 8);
            mbar_wait(drain + 8, 0, nullptr, ATT_WAIT_NS);
            // the last phases of the P buffers' "free" barriers and of the P.V completion
            drain_ring(pfree, pr, p.NPB, gp);
            drain_ring(vempty, vr, p.NV, gv);
        }
        __syncwarp();
    } else if (warp < 4) {
        // ================= softmax: one warp per TMEM lane quadrant =================
        const int qd = warp;
        const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
        const int kl = qd * 32 + lane;           // this thread's key within a tile
        float *my_f = sx_f + qd * NQ;
        int *my_msk = sx_msk + qd * NQ;
        const float sl = p.scale_log2;
        const int nch = NQ / 16;                 // 16-column chunks
        {
            // the A operand of the row-sum MMAs, all ones, in this warp's lane quadrant: 8 columns
            // of bf16 pairs, then 8 of f16 pairs (ordered before the first row-sum MMA by this
            // warp's first P hand-off)
            uint32_t one[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) one[j] = j < 8 ? 0x3F803F80u : 0x3C003C00u;
            tmem_st16(tmem + lane_base + p.t_one, one);
            tmem_st_wait();
        }
        uint32_t ua = 0;                  // units
        RingPos sr, pr, pr_last, orr;     // S buffers, P buffers (and the last group's), O buffers
        uint32_t nx = 0;                  // exchanges among the softmax warps (two barriers, alternating)
        bool ok = true;
        // The epilogue of a unit is deferred until the first P of the next unit has been handed
        // off (by then the unit's last P.V has normally completed), so that the softmax warps
        // do not sit idle waiting for it. Pending: its workspace slot, failure, O buffer, the
        // parity of its maxima buffer and its last tile group.
        int pend_u = -1;
        bool pend_failed = false;
        uint32_t pend_ob = 0, pend_mb = 0;
        RingPos pend_pr;
        auto epilogue = [&]() -> bool {
            if (!warp_wait(pfree + 8 * pend_pr.s, pend_pr.ph, abort_flag, wns)) return false;
            tc_fence_after();
            // the unit's partial: O[q][d] (this lane's d) and, from warp 0, (m, l) per column
            // (l = -1 marks a unit whose pages were invalid); the combine pass finishes every row
            const uint32_t orow = t_o0 + lane_base + pend_ob * (uint32_t)((S_::NSUB + 1) * NQ);
            const float *pm = sx_m + (pend_mb * 4 + qd) * NQ;
            float *ml = p.ws_ml + (size_t)pend_u * NQ * 2;
            float *og = p.ws_o + (size_t)pend_u * NQ * D + kl;
#pragma unroll 1
            for (int c = 0; c < nch; ++c) {
#pragma unroll 1
                for (int h = 0; h < S_::NSUB; ++h) {
                    uint32_t r[16];
                    tmem_ld16(orow + h * NQ + c * 16, r);
                    tmem_ld_wait();
                    if (h * 128 + kl < D) {
#pragma unroll
                        for (int j = 0; j < 16; ++j) og[(size_t)(c * 16 + j) * D + h * 128] = __uint_as_float(r[j]);
                    }
                }
                if (qd == 0) {
                    uint32_t lr[16];
                    tmem_ld16(orow + S_::NSUB * NQ + c * 16, lr);  // L: the same on every lane
                    tmem_ld_wait();
                    float l = 0.f;
#pragma unroll
                    for (int j = 0; j < 16; ++j) l = (lane & 15) == j ? __uint_as_float(lr[j]) : l;
                    if (lane < 16) {
                        ml[(c * 16 + lane) * 2] = pm[c * 16 + lane];
                        ml[(c * 16 + lane) * 2 + 1] = pend_failed ? -1.f : l;
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(ofree + 8 * pend_ob);
            pend_u = -1;
            return true;
        };
        while (ok) {
            const uint32_t ub = ua & 1u, uph = (ua >> 1) & 1u;
            if (!warp_wait(ufull + 8 * ub, uph, abort_flag, wns)) { ok = false; break; }
            const UnitTabView tv = unit_tab(ut_base, ub, UTE);
            const UnitTable *tab = tv.h;
            const int it_u = tab->iter;
            if (it_u < 0) break;
            const UnitInfo ui = tab->ui;
            const int u = ui.u;
            (void)u;
            const bool failed = tab->bad != 0;
            const bool pf16 = FP8 && tab->vf16 != 0;  // this unit's P is f16 (its V is too)
            const uint32_t ob = orr.s, mb = ua & 1u;
            float *my_m = sx_m + (mb * 4 + qd) * NQ;
            // the E4M3 query scales of this unit: written by the producer before it published
            // the table, rewritten only for unit ua + 2 (after this warp releases the table)
            const float *qinv = sx_qinv + ub * NQ;
            // per unit: running maxima, and each column's mask over the verify slots: row j of the
            // branch sees every committed position (< pos_b) and the verify slot pos_b + i when
            // bit i of its mask is set (a chain: bits 0..j; a tree: the row's ancestors and itself)
            for (int q = lane; q < NQ; q += 32) {
                my_m[q] = -INFINITY;
                const int j = sx_colj[q];
                my_msk[q] = q < n_q ? (p.anc ? __ldg(p.anc + ui.b * (p.k + 1) + j) : (int)((2u << j) - 1u)) : 0;
            }
            __syncwarp();
            for (int t0 = 0; t0 < ui.T && ok; t0 += p.TPI, sr.next(p.NSB), pr_last = pr, pr.next(p.NPB)) {
                // A group of nt <= TPI tiles shares one P hand-off. After the unit's first group the
                // group is first tried in one pass with the running maxima: P is written and each
                // warp notes whether any of its scores exceeds its column's maximum by more than
                // RESCALE_TAU; only if one does (a flag exchange tells every warp) does the group
                // take the full path: column maxima, their exchange, the lazily raised maxima
                // (with O and L rescaled) and P written again. Each pass exists once in the code
                // (the tiles of a group are selected at run time), to keep the instruction
                // footprint of the softmax warps small.
                const uint32_t sb = sr.s, pb = pr.s;
                const int nt = min(p.TPI, ui.T - t0);
                ok = warp_wait(sfull + 8 * sb, sr.ph, abort_flag, wns);
                if (!ok) break;
                tc_fence_after();
                const uint32_t sgrp = tmem + lane_base + sb * (uint32_t)(p.TPI * NQ);
                // per tile i of the group: this thread's key offset from the split's start, its
                // score factor slk (softmax scale in log2 units; FP8: times the key's K page scale,
                // 0 past the branch's last position) and whether every row sees all 32 keys of
                // the warp (then the per-column masks are skipped; the padding columns hold finite
                // zero scores, their Q rows being 0); bit0/bit1: this key's verify-slot bit (0 past
                // the last slot), all0/all1: the key is a committed one, seen by every row
                const int koff0 = t0 * TILE_KEYS + kl, koff1 = koff0 + TILE_KEYS;
                const int rel0 = koff0 - (ui.pos_b - ui.s0), rel1 = rel0 + TILE_KEYS;
                const bool all0 = rel0 < 0, all1 = rel1 < 0;
                const uint32_t bit0 = (rel0 >= 0 && rel0 < 32) ? 1u << rel0 : 0u;
                const uint32_t bit1 = (rel1 >= 0 && rel1 < 32) ? 1u << rel1 : 0u;
                float slk0 = sl, slk1 = sl;
                if (FP8) {
                    slk0 = ui.s0 + koff0 < ui.kv_end ? sl * tv.ksc[koff0 >> log2P] : 0.f;
                    slk1 = nt > 1 && ui.s0 + koff1 < ui.kv_end ? sl * tv.ksc[koff1 >> log2P] : 0.f;
                }
                const bool vis0 = __all_sync(0xFFFFFFFFu, all0);
                const bool vis1 = __all_sync(0xFFFFFFFFu, all1);
                uint8_t *prow = smem + p.off_p + pb * PBUF + kl * 32;
                const int sw = (kl >> 2) & 1;  // 32-byte swizzle: 16-byte chunk index ^= row bit 2
                // the scores s * slk of chunk c of tile i (both tiles' TMEM loads in flight
                // together, then tile i's registers selected), -inf where the key is not seen by
                // the column's row
                auto scores = [&](int i, int c, const uint32_t (&r0)[16], const uint32_t (&r1)[16], float (&x)[16]) {
                    const float slk = i ? slk1 : slk0;
#pragma unroll
                    for (int j = 0; j < 16; ++j) x[j] = __uint_as_float(i ? r1[j] : r0[j]) * slk;
                    if (!(i ? vis1 : vis0)) {
                        const bool all = i ? all1 : all0;
                        const uint32_t bit = i ? bit1 : bit0;
#pragma unroll
                        for (int j = 0; j < 16; j += 4) {
                            const int4 a = *reinterpret_cast<const int4 *>(my_msk + c * 16 + j);
                            x[j] = (all || ((uint32_t)a.x & bit)) ? x[j] : -INFINITY;
                            x[j + 1] = (all || ((uint32_t)a.y & bit)) ? x[j + 1] : -INFINITY;
                            x[j + 2] = (all || ((uint32_t)a.z & bit)) ? x[j + 2] : -INFINITY;
                            x[j + 3] = (all || ((uint32_t)a.w & bit)) ? x[j + 3] : -INFINITY;
                        }
                    }
                };
                auto issue2 = [&](int c, uint32_t (&r0)[16], uint32_t (&r1)[16]) {
                    tmem_ld16(sgrp + (uint32_t)(c * 16), r0);
                    if (nt > 1) tmem_ld16(sgrp + (uint32_t)(NQ + c * 16), r1);
                };
                auto load2 = [&](int c, uint32_t (&r0)[16], uint32_t (&r1)[16]) {
                    issue2(c, r0, r1);
                    tmem_ld_wait();
                };
                // the flag (and, on the full path, maxima) exchange among the four warps
                auto exchange = [&](bool need_w) -> bool {
                    const uint32_t slot = nx & 1u;
                    if (lane == 0) sx_need[slot * 4 + qd] = need_w ? 1 : 0;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(xbar + 8 * slot);
                    ok = warp_wait(xbar + 8 * slot, (nx >> 1) & 1u, abort_flag, wns);
                    ++nx;
                    if (!ok) return false;
                    const int4 nd = *reinterpret_cast<const int4 *>(sx_need + slot * 4);
                    return (nd.x | nd.y | nd.z | nd.w) != 0;
                };
                bool full = t0 == 0, waited = false;
#pragma unroll 1
                for (int attempt = 0; attempt < 2; ++attempt) {
                    if (full) {
                        // ---- the group's column maxima over this warp's keys: the maximum over the
                        // tiles, then over the warp's 32 keys by one warp reduction per column; lane
                        // l < 16 publishes column c*16 + l. For E4M3 queries the 1/sigma factor is
                        // applied to the maximum (rounding is monotonic, so the result is the maximum
                        // of the scaled scores exactly) ----
                        const uint32_t slot = nx & 1u;
                        float *red = sx_red + slot * 4 * NQ + qd * NQ;
                        bool need = false;
#pragma unroll 1
                        for (int c = 0; c < nch; ++c) {
                            uint32_t r0[16], r1[16];
                            load2(c, r0, r1);
                            float v[16];
#pragma unroll
                            for (int j = 0; j < 16; ++j) v[j] = -INFINITY;
#pragma unroll 1
                            for (int i = 0; i < nt; ++i) {
                                float x[16];
                                scores(i, c, r0, r1, x);
#pragma unroll
                                for (int j = 0; j < 16; ++j) v[j] = fmaxf(v[j], x[j]);
                            }
                            float mine = -INFINITY;
#pragma unroll
                            for (int j = 0; j < 16; ++j) {
                                const float cm = warp_max_f32(v[j]);
                                mine = (lane & 15) == j ? cm : mine;
                            }
                            const int col = c * 16 + (lane & 15);
                            if (FP8) mine *= qinv[col];
                            if (lane < 16) red[col] = mine;
                            need |= mine > my_m[col] + RESCALE_TAU;  // this column's maximum must move
                        }
                        need = __any_sync(0xFFFFFFFFu, need);
                        const bool any_need = exchange(need);
                        if (!ok) break;
                        // ---- the group's maxima over the four warps; lazily raised running maxima
                        // (only when some warp saw a column exceed its maximum by more than
                        // RESCALE_TAU) ----
                        bool resc = false;
                        const float *red_all = sx_red + slot * 4 * NQ;
#pragma unroll 1
                        for (int q = lane; any_need && q < NQ; q += 32) {
                            const float M = fmaxf(fmaxf(red_all[q], red_all[NQ + q]), fmaxf(red_all[2 * NQ + q], red_all[3 * NQ + q]));
                            const float mo = my_m[q];
                            const float mn = (M > mo + RESCALE_TAU) ? M : mo;
                            my_f[q] = mn == mo ? 1.f : (mo == -INFINITY ? 0.f : ex2_approx(mo - mn));
                            resc |= mn != mo && mo != -INFINITY;
                            my_m[q] = mn;
                        }
                        __syncwarp();
                        if (any_need && __any_sync(0xFFFFFFFFu, resc)) {
                            // a running maximum moved: O and L of this unit are rescaled per column,
                            // after the P.V of the previous group (this unit's: t0 > 0 here) has
                            // completed. Its completion is the phase of its P buffer's "free"
                            // barrier that follows the one this warp waited for before writing that
                            // P (a wait is never two phases behind)
                            ok = warp_wait(pfree + 8 * pr_last.s, pr_last.ph, abort_flag, wns);
                            if (!ok) break;
                            tc_fence_after();
                            const uint32_t orow = t_o0 + lane_base + ob * (uint32_t)((S_::NSUB + 1) * NQ);
#pragma unroll 1
                            for (int h = 0; h <= S_::NSUB; ++h) {
#pragma unroll 1
                                for (int c = 0; c < nch; ++c) {
                                    uint32_t r[16];
                                    tmem_ld16(orow + h * NQ + c * 16, r);
                                    tmem_ld_wait();
#pragma unroll
                                    for (int j = 0; j < 16; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * my_f[c * 16 + j]);
                                    tmem_st16(orow + h * NQ + c * 16, r);
                                }
                            }
                            tmem_st_wait();
                        }
                    }
                    // ---- P^T rows of this thread's keys: P = 2^y, y = s * slk (* 1/sigma) - m, the
                    // product and the subtraction fused; ymax: whether some y exceeds RESCALE_TAU.
                    // Each tile's scores of the next chunk start loading from TMEM into its
                    // registers as soon as the tile is computed (the first chunk's while the P
                    // buffer is awaited) ----
                    uint32_t r0[16], r1[16];
                    issue2(0, r0, r1);
                    if (!waited) {
                        ok = warp_wait(pfree + 8 * pb, pr.ph ^ 1u, abort_flag, wns);
                        if (!ok) break;
                        waited = true;
                    }
                    tmem_ld_wait();
                    float ymax = -INFINITY;
#pragma unroll 1
                    for (int c = 0; c < nch; ++c) {
                        float m[16], qs[16];
#pragma unroll
                        for (int j = 0; j < 16; j += 4) {
                            const float4 a = *reinterpret_cast<const float4 *>(my_m + c * 16 + j);
                            m[j] = a.x; m[j + 1] = a.y; m[j + 2] = a.z; m[j + 3] = a.w;
                            if (FP8) {
                                const float4 b4 = *reinterpret_cast<const float4 *>(qinv + c * 16 + j);
                                qs[j] = b4.x; qs[j + 1] = b4.y; qs[j + 2] = b4.z; qs[j + 3] = b4.w;
                            }
                        }
                        // tile i's P from its registers r (never touched while a load into them is
                        // in flight), then that tile's next chunk is requested into the same registers
                        auto ptile = [&](int i, uint32_t (&r)[16]) {
                            const float slk = i ? slk1 : slk0;
                            float y[16];
#pragma unroll
                            for (int j = 0; j < 16; ++j) {
                                const float sj = __uint_as_float(r[j]);
                                y[j] = FP8 ? fmaf(sj * slk, qs[j], -m[j]) : fmaf(sj, slk, -m[j]);
                            }
                            if (!(i ? vis1 : vis0)) {
                                const bool all = i ? all1 : all0;
                                const uint32_t bit = i ? bit1 : bit0;
#pragma unroll
                                for (int j = 0; j < 16; j += 4) {
                                    const int4 a = *reinterpret_cast<const int4 *>(my_msk + c * 16 + j);
                                    y[j] = (all || ((uint32_t)a.x & bit)) ? y[j] : -INFINITY;
                                    y[j + 1] = (all || ((uint32_t)a.y & bit)) ? y[j + 1] : -INFINITY;
                                    y[j + 2] = (all || ((uint32_t)a.z & bit)) ? y[j + 2] : -INFINITY;
                                    y[j + 3] = (all || ((uint32_t)a.w & bit)) ? y[j + 3] : -INFINITY;
                                }
                            }
                            uint32_t pk[8];
#pragma unroll
                            for (int j = 0; j < 16; j += 2) {
                                ymax = fmaxf(ymax, fmaxf(y[j], y[j + 1]));
                                pk[j >> 1] = pack2(ex2_approx(y[j]), ex2_approx(y[j + 1]), pf16);
                            }
                            uint8_t *blk = prow + i * PTILE + c * (TILE_KEYS * 32);
                            *reinterpret_cast<uint4 *>(blk + (sw << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                            *reinterpret_cast<uint4 *>(blk + ((sw ^ 1) << 4)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                            if (c + 1 < nch) tmem_ld16(sgrp + (uint32_t)(i * NQ + (c + 1) * 16), r);
                        };
                        ptile(0, r0);
                        if (nt > 1) ptile(1, r1);
                        if (c + 1 < nch) tmem_ld_wait();
                    }
                    if (attempt == 0 && !full) {
                        // the one-pass try: keep it unless some warp saw a score above its maximum
                        full = exchange(__any_sync(0xFFFFFFFFu, ymax > RESCALE_TAU));
                        if (!ok) break;
                        if (full) continue;
                    }
                    break;
                }
                if (!ok) break;
                tc_fence_before();
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(sfree + 8 * sb);
                    mbar_arrive(pfull + 8 * pb);
                }
                // the previous unit's epilogue, once this unit's first P is on its way
                if (pend_u >= 0) {
                    ok = epilogue();
                    if (!ok) break;
                }
            }
            if (!ok) break;
            // the unit table is no longer read
            __syncwarp();
            if (lane == 0) mbar_arrive(ufree + 8 * ub);
            pend_u = u;
            pend_failed = failed;
            pend_ob = ob;
            pend_mb = mb;
            pend_pr = pr_last;
            ++ua;
            orr.next(p.OB);
        }
        if (ok && pend_u >= 0) ok = epilogue();
        if (!ok) {
            *abort_flag = 1;
            if (qd == 0 && lane == 0) raise_error(p.err, SPEC_DEVERR_TIMEOUT);
        }
    } else if (warp == 11) {
        // ================= FP8: TMA issuers, warp 11: lane 0 K sub-tiles, lane 1 raw V sub-tiles =================
        // (bf16 pools: this warp has no role). The two lanes run independent loops (their waits
        // are per thread, with no warp-wide step), so that the K stream runs ahead of the V
        // stream by the K ring's depth. One box per page-run of rows (min(page size, 128)
        // rows): K boxes land 128- or 64-byte-swizzled, ready for the S MMA; V boxes land
        // unswizzled in a raw stage. Runs past the branch's last position, or of an invalid
        // page, are not loaded.
        if (FP8 && lane < 2) {
            const bool is_v = lane == 1;
            const int depth = is_v ? p.NR : p.NK;
            const uint32_t full0 = is_v ? rfull : kfull, empty0 = is_v ? rempty : kempty;
            const uint32_t ring = is_v ? s_raw : s_k;
            const CUtensorMap *map = is_v ? &map_v : &map_k;
            uint32_t gi = 0, ua = 0;
            RingPos rr;
            bool ok = true;
            const int BR = p.tma_rows, nruns = TILE_KEYS / BR;
            for (;;) {
                const uint32_t ub = ua & 1u, uph = (ua >> 1) & 1u;
                const UnitTabView tv = unit_tab(ut_base, ub, UTE);
                const UnitTable *tab = tv.h;
                if (!lane_poll_wait(ufull + 8 * ub, uph, abort_flag, wns)) { ok = false; break; }
                const int it_u = tab->iter;
                if (it_u < 0) break;
                const UnitInfo ui = tab->ui;
                ++ua;
                for (int t = 0; t < ui.T && ok; ++t) {
                    const int key0 = ui.s0 + t * TILE_KEYS;
                    // the producer may prepare the next unit (see the bf16 loaders)
                    if (!is_v && t == max(0, ui.T - NEXT_UNIT_LEAD)) mbar_arrive(lfin + 8 * ub);
                    for (int h = 0; h < S_::NSUB; ++h, ++gi) {
                        const uint32_t s = rr.s;
                        if (!lane_poll_wait(empty0 + 8 * s, rr.ph ^ 1u, abort_flag, wns)) {
                            ok = false;
                            break;
                        }
                        rr.next(depth);
                        const uint32_t dst_base = ring + s * S_::F8_STAGE;
                        uint32_t bytes = 0;
                        for (int r = 0; r < nruns; ++r) {
                            const int kr = key0 + r * BR;
                            if (kr >= ui.kv_end) break;
                            if (tv.page[(kr - ui.s0) >> log2P] >= 0) bytes += (uint32_t)(BR * S_::SUB);
                        }
                        mbar_arrive_expect_tx(full0 + 8 * s, bytes);
                        for (int r = 0; r < nruns; ++r) {
                            const int kr = key0 + r * BR;
                            if (kr >= ui.kv_end) break;
                            const int pg = tv.page[(kr - ui.s0) >> log2P];
                            if (pg < 0) continue;
                            const int row = (pg * p.kv.n_kv_heads + ui.g) * p.kv.page_size + (kr & (p.kv.page_size - 1));
                            tma_load_2d(dst_base + (uint32_t)(r * BR) * S_::SUB, map, h * S_::SUB, row, full0 + 8 * s);
                        }
                    }
                }
                if (!ok) break;
                mbar_arrive(ufree + 8 * ub);
            }
            // every box lands, and every consumer's release of a stage is delivered, before the
            // CTA may exit
            drain_ring(full0, rr, depth, gi);  // (the stages' releases are plain arrives or drained by their MMA issuer)
            if (!ok) {
                *abort_flag = 1;
                raise_error(p.err, SPEC_DEVERR_TIMEOUT);
            }
        }
        __syncwarp();
    } else if (!FP8) {
        // ================= loaders (bf16): warps 4-5 K, warps 6-7 V, by cp.async =================
        // Each stream has its own ring, so that V stages held until their P.V never hold up
        // the K loads the S MMAs wait for. Each thread copies its own 16-byte pieces of every
        // sub-tile and lets the copies arrive on the stage's barrier by themselves when they
        // land (cp.async.mbarrier.arrive.noinc). Rows past the branch's last position, or of an
        // invalid page, are zero-filled, so every stage is fully written.
        const bool is_v = warp >= 6;
        const int ltid = (warp & 1) * 32 + lane;   // 0..63 within the stream
        constexpr int CH = S_::SUB * 2 / 16;       // 16-byte pieces per row of a sub-tile
        constexpr int RPS = 64 / CH;               // rows per step of the 64 stream threads
        constexpr int NPIECE = TILE_KEYS / RPS;    // pieces per thread per sub-tile
        const int pch = ltid % CH, prow0 = ltid / CH;
        const size_t row_bytes = (size_t)D * 2;
        const uint8_t *pool = reinterpret_cast<const uint8_t *>(is_v ? p.kv.v_pool : p.kv.k_pool);
        const int depth = is_v ? p.NV : p.NK;
        const uint32_t full0 = is_v ? vfull : kfull, empty0 = is_v ? vempty : kempty;
        const uint32_t ring = is_v ? s_v : s_k;
        uint32_t gi = 0, ua = 0;  // sub-tiles issued, units
        RingPos rr;
        bool ok = true;
        for (;;) {
            const uint32_t ub = ua & 1u, uph = (ua >> 1) & 1u;
            const UnitTabView tv = unit_tab(ut_base, ub, UTE);
            const UnitTable *tab = tv.h;
            if (!warp_wait<SLEEP_LOAD>(ufull + 8 * ub, uph, abort_flag, wns)) { ok = false; break; }
            const int it_u = tab->iter;
            if (it_u < 0) break;
            const UnitInfo ui = tab->ui;
            ++ua;
            for (int t = 0; t < ui.T && ok; ++t) {
                const int key0 = ui.s0 + t * TILE_KEYS;
                // NEXT_UNIT_LEAD tiles before the unit's end the K loaders let the producer
                // prepare the next unit, so that its table and Q are there when this unit's last
                // copies have been issued (the K stream runs ahead of the V stream)
                if (!is_v && t == max(0, ui.T - NEXT_UNIT_LEAD)) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(lfin + 8 * ub);
                }
                for (int h = 0; h < S_::NSUB; ++h, ++gi) {
                    const uint32_t s = rr.s;
                    if (!warp_wait<SLEEP_LOAD>(empty0 + 8 * s, rr.ph ^ 1u, abort_flag, wns)) {
                        ok = false;
                        break;
                    }
                    rr.next(depth);
                    const uint32_t dst_base = ring + s * S_::OP_STAGE;
                    const uint8_t *src_col = pool + (size_t)h * S_::SUB * 2 + pch * 16;
                    // pages of >= 8 positions: per group of 8 pieces the table lookups first
                    // (independent loads), then the copies; smaller pages: per-row page-table reads
                    if (!small_pages) {
#pragma unroll 1
                        for (int k0 = 0; k0 < NPIECE; k0 += 8) {
                            int pg[8];
#pragma unroll
                            for (int k = 0; k < 8; ++k) pg[k] = tv.page[(t * TILE_KEYS + (k0 + k) * RPS + prow0) >> log2P];
#pragma unroll
                            for (int k = 0; k < 8; ++k) {
                                const int row = (k0 + k) * RPS + prow0, key = key0 + row;
                                const bool ok_row = key < ui.kv_end && pg[k] >= 0;
                                const uint32_t rowi = ok_row ? (uint32_t)(pg[k] * p.kv.n_kv_heads + ui.g) * (uint32_t)p.kv.page_size +
                                                                   (uint32_t)(key & (p.kv.page_size - 1))
                                                             : 0u;
                                const uint32_t dst = dst_base + (pch >> 3) * (TILE_KEYS * 128) + row * 128 +
                                                     ((((pch & 7) ^ (row & 7)) & 7) << 4);
                                cp_async16_zfill(dst, src_col + (size_t)rowi * row_bytes, ok_row);
                            }
                        }
                    } else {
#pragma unroll 1
                        for (int k = 0; k < NPIECE; ++k) {
                            const int row = k * RPS + prow0, key = key0 + row;
                            const int pg = key < ui.kv_end ? page_of(p.kv, ui.b, key) : -1;
                            const uint32_t rowi = pg < 0 ? 0u
                                                         : (uint32_t)(pg * p.kv.n_kv_heads + ui.g) * (uint32_t)p.kv.page_size +
                                                               (uint32_t)(key & (p.kv.page_size - 1));
                            const uint32_t dst = dst_base + (pch >> 3) * (TILE_KEYS * 128) + row * 128 +
                                                 ((((pch & 7) ^ (row & 7)) & 7) << 4);
                            cp_async16_zfill(dst, src_col + (size_t)rowi * row_bytes, pg >= 0);
                        }
                    }
                    cp_async_arrive(full0 + 8 * s);
                }
            }
            // the unit's table is no longer read by this warp
            __syncwarp();
            if (ok && lane == 0) mbar_arrive(ufree + 8 * ub);
            if (!ok) break;
        }
        // every copy lands before the CTA may exit (the stages' releases, MMA commits, are
        // drained by the MMA issuers)
        cp_async_wait_all();
        __syncwarp();
        if (!ok) {
            *abort_flag = 1;
            if (ltid == 0) raise_error(p.err, SPEC_DEVERR_TIMEOUT);
        }
    } else {
        // ================= FP8 converters, warps 4-7 (one per SM sub-partition) =================
        // Every raw V sub-tile, in ring order, becomes f16(code * page scale) (bf16 for a unit
        // whose V scales leave the f16 range) in the MMA's layout (the V ring), with the rows past
        // the branch's last position written as
        // zeros. Each warp fences its own share and arrives on the stage's barriers (count 4).
        // Their waits do not sleep: the converted V is on the P.V MMAs' critical path.
        const int ctid = (warp - 4) * 32 + lane;  // 0..127
        uint32_t ua = 0;
        RingPos rawr, vr;  // raw V ring, bf16 V ring
        bool ok = true;
        for (;;) {
            const uint32_t ub = ua & 1u, uph = (ua >> 1) & 1u;
            const UnitTabView tv = unit_tab(ut_base, ub, UTE);
            const UnitTable *tab = tv.h;
            if (!warp_wait<SLEEP_LOAD>(ufull + 8 * ub, uph, abort_flag, wns)) { ok = false; break; }
            const int it_u = tab->iter;
            if (it_u < 0) break;
            const UnitInfo ui = tab->ui;
            const bool vf16 = tab->vf16 != 0;
            ++ua;
            for (int t = 0; t < ui.T && ok; ++t) {
                const int nvk = ui.kv_end - (ui.s0 + t * TILE_KEYS);  // valid keys of the tile (>= 1)
#pragma unroll 1
                for (int h = 0; h < S_::NSUB; ++h, rawr.next(p.NR), vr.next(p.NV)) {
                    const uint32_t rs = rawr.s, os = vr.s;
                    if (!warp_wait(rfull + 8 * rs, rawr.ph, abort_flag, wns) ||
                        !warp_wait(vempty + 8 * os, vr.ph ^ 1u, abort_flag, wns)) {
                        ok = false;
                        break;
                    }
                    const uint8_t *raw = smem + p.off_raw + rs * S_::F8_STAGE;
                    uint8_t *op = smem + p.off_v + os * S_::OP_STAGE;
                    // thread ctid converts the 16-byte piece pc of rows row0, row0 + RSTEP, ...: all
                    // its loads first, then the conversions (a warp reads 4 whole rows per load)
                    constexpr int CCH = S_::SUB / 16;        // 16-byte raw pieces per row
                    constexpr int RSTEP = 128 / CCH;         // rows between a thread's pieces
                    constexpr int NIT = TILE_KEYS / RSTEP;   // pieces per thread
                    constexpr int BATCH = NIT < 4 ? NIT : 4; // pieces loaded together
                    int pc = ctid % CCH, row0 = ctid / CCH;
                    if (CCH == 8) {
                        const int g = ctid >> 3, b2 = (ctid >> 2) & 1;
                        pc = (ctid & 3) + 4 * b2;
                        row0 = 2 * (g >> 1) + (b2 ^ (g & 1));
                    }
#pragma unroll 1
                    for (int i0 = 0; i0 < NIT; i0 += BATCH) {
                        uint4 v[BATCH];
                        float vs[BATCH];
#pragma unroll
                        for (int i = 0; i < BATCH; ++i) {
                            const int row = row0 + (i0 + i) * RSTEP;
                            v[i] = *reinterpret_cast<const uint4 *>(raw + row * S_::SUB + pc * 16);
                            vs[i] = tv.vsc[(t * TILE_KEYS + (row < nvk ? row : 0)) >> log2P];
                        }
#pragma unroll
                        for (int i = 0; i < BATCH; ++i) {
                            const int row = row0 + (i0 + i) * RSTEP;
                            const bool live = row < nvk;  // rows past the last position: zeros, never code * 0
                            const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
                            uint32_t hv[8];
                            if (vf16) {
                                // f16(code * scale): the code is exact in f16, one f16 multiply
                                const __half2 s2 = __float2half2_rn(vs[i]);
#pragma unroll
                                for (int e = 0; e < 8; ++e) {
                                    const __half2_raw c2 = __nv_cvt_fp8x2_to_halfraw2(
                                        (__nv_fp8x2_storage_t)((w[e >> 1] >> (16 * (e & 1))) & 0xFFFFu), __NV_E4M3);
                                    const __half2 r2 = __hmul2(*reinterpret_cast<const __half2 *>(&c2), s2);
                                    hv[e] = live ? *reinterpret_cast<const uint32_t *>(&r2) : 0u;
                                }
                            } else {
#pragma unroll
                                for (int e = 0; e < 8; ++e) {
                                    const __half2_raw c2 = __nv_cvt_fp8x2_to_halfraw2(
                                        (__nv_fp8x2_storage_t)((w[e >> 1] >> (16 * (e & 1))) & 0xFFFFu), __NV_E4M3);
                                    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&c2));
                                    hv[e] = live ? pack2(f.x * vs[i], f.y * vs[i], false) : 0u;
                                }
                            }
                            *reinterpret_cast<uint4 *>(op + sw128_off(row, pc * 16, TILE_KEYS * 128)) =
                                make_uint4(hv[0], hv[1], hv[2], hv[3]);
                            *reinterpret_cast<uint4 *>(op + sw128_off(row, pc * 16 + 8, TILE_KEYS * 128)) =
                                make_uint4(hv[4], hv[5], hv[6], hv[7]);
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(vfull + 8 * os);
                        mbar_arrive(rempty + 8 * rs);
                    }
                }
            }
            // the unit's table (its V scales) is no longer read
            __syncwarp();
            if (ok && lane == 0) mbar_arrive(ufree + 8 * ub);
            if (!ok) break;
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

// The split merge. One item = (row r, q head h); W warps share an item (the host picks W
// from the split count; it does not change the arithmetic) and a CTA holds `ipc` items.
// Pass 1: the maximum m over the splits the row reaches (l > 0) and whether any split
// failed (l < 0). Pass 2: warp w sums the groups g = w, w + W, ... of COMBINE_GROUP splits,
// each in ascending split order (the loads of a group issued together), into shared
// memory. Pass 3: the groups are added in ascending order and the row is normalised.
// Within every sum the first term taken is multiplied, the later ones fused-added, so a row
// that one split alone reaches gets that split's O / l bit for bit, however many splits its
// batch had.
__host__ __device__ constexpr int combine_slot_floats(int ng_max, int D, int W) {
    return ng_max * D + ((ng_max + 3) & ~3) + ((2 * W + 3) & ~3);
}

template <int D>
__global__ void __launch_bounds__(512) attn_combine_kernel(AttnParams p, int W, int ipc, int ng_max) {
    // per item (a slot of combine_slot_floats floats, a multiple of 4 so that every slot's
    // float4 rows stay 16-byte aligned): [ng_max][D] group sums, [ng_max] group l, [W]
    // maxima, [W] failure flags
    extern __shared__ float csm[];
    constexpr int E4 = D >= 128 ? D / 128 : 1;  // float4 per lane (d = 64: lanes 16..31 idle)
    grid_dep_wait();  // the split kernel's partial results
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int slot = warp / W, w = warp % W;
    const int item = blockIdx.x * ipc + slot;
    const int R = p.B * (p.k + 1), NQ = p.NQ;
    float *gsum = csm + (size_t)slot * combine_slot_floats(ng_max, D, W);
    float *gl = gsum + (size_t)ng_max * D;
    float *wmax = gl + ((ng_max + 3) & ~3);
    int *wfail = reinterpret_cast<int *>(wmax + W);
    const bool active = D >= 128 || lane < D / 4;
    // the item's splits (none for an item past the end)
    int n_used = 0, q = 0, b = 0, g = 0, r = 0, h = 0;
    size_t u0 = 0;
    if (item < R * p.Hq) {
        r = item / p.Hq;
        h = item % p.Hq;
        b = r / (p.k + 1);
        g = h / p.G;
        q = (r % (p.k + 1)) * p.G + h % p.G;
        const int pos_b = __ldg(p.pos + b);
        if (pos_b >= 0 && pos_b + p.k + 1 <= p.max_pos) {
            n_used = (pos_b + p.k + 1 + p.split_keys - 1) / p.split_keys;
        }
        if (p.anc) {  // a tree row sees itself and only earlier rows: bit j set, none above
            const int j = r % (p.k + 1);
            const uint32_t m = (uint32_t)__ldg(p.anc + r);
            if (!((m >> j) & 1u) || ((m >> j) >> 1) != 0) {
                if (threadIdx.x % (W * 32) == 0) raise_error(p.err, SPEC_DEVERR_TREE);
                n_used = 0;
            }
        }
        u0 = (size_t)(b * p.kv.n_kv_heads + g) * p.n_splits;
    }
    const int ng = (n_used + COMBINE_GROUP - 1) / COMBINE_GROUP;
    // ---- pass 1: maximum over the reached splits; failures ----
    float M = -INFINITY;
    int failed = 0;
    for (int g0 = w * 4 + (lane >> 3); g0 < ng; g0 += 4 * W) {  // 4 groups per warp step
        const int s = g0 * COMBINE_GROUP + (lane & 7);
        if (s < n_used) {
            const float2 v = __ldcg(reinterpret_cast<const float2 *>(p.ws_ml + ((u0 + s) * NQ + q) * 2));
            failed |= v.y < 0.f;
            if (v.y != 0.f) M = fmaxf(M, v.x);  // (a NaN sum from NaN data is reached: it propagates)
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, off));
    failed = __any_sync(0xFFFFFFFFu, failed);
    if (lane == 0) {
        wmax[w] = M;
        wfail[w] = failed;
    }
    __syncthreads();
    M = -INFINITY;
    failed = 0;
    for (int i = 0; i < W; ++i) {
        M = fmaxf(M, wmax[i]);
        failed |= wfail[i];
    }
    const bool skip = n_used == 0 || failed || M == -INFINITY;
    // a tree row whose mask sees no key at all (nothing committed, no slot bit): no output
    if (n_used > 0 && !failed && M == -INFINITY && threadIdx.x % (W * 32) == 0) raise_error(p.err, SPEC_DEVERR_POS);
    // ---- pass 2: group sums ----
    if (!skip) {
        for (int g0 = w; g0 < ng; g0 += W) {
            const int s0 = g0 * COMBINE_GROUP;
            const int nb = min(COMBINE_GROUP, n_used - s0);
            float wl = 0.f, ll = 0.f;  // lane u < nb: weight and l of split s0 + u
            if (lane < nb) {
                const float2 v = __ldcg(reinterpret_cast<const float2 *>(p.ws_ml + ((u0 + s0 + lane) * NQ + q) * 2));
                ll = v.y;
                wl = v.y != 0.f ? merge_weight(v.x, M) : 0.f;
            }
            float4 v[COMBINE_GROUP][E4];
#pragma unroll
            for (int u = 0; u < COMBINE_GROUP; ++u) {
                if (active && u < nb) {
                    const float4 *src = reinterpret_cast<const float4 *>(p.ws_o + ((u0 + s0 + u) * NQ + q) * D) + lane;
#pragma unroll
                    for (int e = 0; e < E4; ++e) v[u][e] = __ldcg(src + 32 * e);
                }
            }
            float L = 0.f;
            float4 acc[E4];
#pragma unroll
            for (int e = 0; e < E4; ++e) acc[e] = make_float4(0.f, 0.f, 0.f, 0.f);
            bool first = true;
#pragma unroll
            for (int u = 0; u < COMBINE_GROUP; ++u) {
                if (u >= nb) break;
                const float wgt = __shfl_sync(0xFFFFFFFFu, wl, u);
                const float l = __shfl_sync(0xFFFFFFFFu, ll, u);
                if (l == 0.f) continue;
                L = first ? wgt * l : fmaf(wgt, l, L);
#pragma unroll
                for (int e = 0; e < E4; ++e) {
                    if (first) {
                        acc[e] = make_float4(wgt * v[u][e].x, wgt * v[u][e].y, wgt * v[u][e].z, wgt * v[u][e].w);
                    } else {
                        acc[e].x = fmaf(wgt, v[u][e].x, acc[e].x);
                        acc[e].y = fmaf(wgt, v[u][e].y, acc[e].y);
                        acc[e].z = fmaf(wgt, v[u][e].z, acc[e].z);
                        acc[e].w = fmaf(wgt, v[u][e].w, acc[e].w);
                    }
                }
                first = false;
            }
            if (active) {
#pragma unroll
                for (int e = 0; e < E4; ++e) reinterpret_cast<float4 *>(gsum + (size_t)g0 * D)[lane + 32 * e] = acc[e];
            }
            if (lane == 0) gl[g0] = L;  // 0: no split of the group reached by the row
        }
    }
    __syncthreads();
    // ---- pass 3: the groups in ascending order, normalised ----
    if (!skip) {
        float L = 0.f;
        bool first = true;
        for (int g0 = 0; g0 < ng; ++g0) {
            const float l = gl[g0];
            if (l == 0.f) continue;
            L = first ? l : L + l;
            first = false;
        }
        uint16_t *dst = p.out + ((size_t)r * p.Hq + h) * D;
        for (int d = w * 32 + lane; d < D; d += W * 32) {
            float acc = 0.f;
            bool f2 = true;
            for (int g0 = 0; g0 < ng; ++g0) {
                if (gl[g0] == 0.f) continue;
                const float x = gsum[(size_t)g0 * D + d];
                acc = f2 ? x : acc + x;
                f2 = false;
            }
            const __nv_bfloat16 ov = __float2bfloat16_rn(__fdiv_rn(acc, L));
            dst[d] = *reinterpret_cast<const uint16_t *>(&ov);
        }
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

// Q [R][Hq][d] viewed as a 3-D tensor (d, Hq, R): a (64, G, k+1) box at (a*64, g*G, b*(k+1))
// holds the n_q query vectors of (branch b, kv head g) in row order j*G + i.
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
// box_rows rows of one sub-tile's width (min(d, 128) bytes) is one page-run of a (page, kv
// head). K boxes land swizzled (the E4M3 MMA operand), V boxes unswizzled (a raw stage).
static bool make_kv_map(CUtensorMap *map, const void *pool, uint64_t rows, int d, int box_rows, bool swizzled) {
    EncodeTiledFnA fn = encode_fn_attn();
    if (!fn) return false;
    const int w = d < 128 ? d : 128;
    cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)d};
    cuuint32_t box[2] = {(cuuint32_t)w, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    const CUtensorMapSwizzle sw =
        !swizzled ? CU_TENSOR_MAP_SWIZZLE_NONE : (w == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(pool), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

// Shared-memory and TMEM plan. In shared memory, in this order (swizzled blocks 1024-aligned):
// bf16 Q buffers, E4M3 Q parts (FP8), P buffers, ring 0 (bf16 K/V or E4M3 K + raw V), ring 1
// (FP8: f16 V), 2 unit tables, softmax scratch, barriers, flags. In TMEM: NSB S buffers of NQ
// columns, then OB sets of (NSUB O blocks + L) of NQ columns each, then the 16 columns of the
// row-sum MMAs' ones operand.
template <int D, bool FP8>
static int plan_attn(AttnParams &p, size_t *smem_bytes) {
    using S_ = AttnShape<D, FP8>;
    const int NQ = p.NQ;
    // unit tables: one entry per page-sized run of a split (pages of >= 8 positions)
    const int ut_entries = p.kv.page_size < 8 ? 0 : (p.split_keys + p.kv.page_size - 1) / p.kv.page_size;
    const uint32_t ut_bytes = 2 * unit_table_stride(ut_entries);
    const uint32_t sx_bytes = (uint32_t)(8 + 8 + 4 + 4 + 2 + 2) * NQ * 4 + 32;
    const uint32_t bars = BAR_BYTES, small = 64;
    // Tile groups of 2 when the ring holds a whole group's K and V (the S of a group's last
    // tile must be able to load while the V of its first tile waits for the softmax), else 1.
    // Then the richest plan whose ring holds 1.5 groups (2 Q buffers first; 2 P buffers for
    // groups of 2, else 3 first), else the deepest ring that holds one group.
    const int qb_opts[2] = {2, 1};
    // (splits of at most two tiles: single tiles, so that a unit's tiles still pipeline)
    for (int TPI = p.split_keys >= 512 ? 2 : 1; TPI >= 1; --TPI) {
        // TMEM: 2 S buffers of a group and 2 O sets preferred, then fewer
        int NSB = 0, OB = 0;
        for (int ob = 2; ob >= 1 && !NSB; --ob)
            for (int nsb = 4 / TPI; nsb >= 2; --nsb)
                if (nsb * TPI * NQ + ob * (S_::NSUB + 1) * NQ + 16 <= 512) {
                    NSB = nsb;
                    OB = ob;
                    break;
                }
        if (!NSB) {
            if (TPI * NQ + (S_::NSUB + 1) * NQ + 16 > 512) continue;
            NSB = 1;
            OB = 1;
        }
        for (int pass = 0; pass < 3; ++pass)
            for (int a = 0; a < 2; ++a)
                for (int c = 0; c < 2; ++c) {
                    const int QB = qb_opts[a], NPB = TPI == 2 ? 2 : 3 - c;
                    if (TPI == 2 && c == 1) continue;
                    const uint32_t q_bytes = FP8 ? 0 : QB * S_::NATOM_Q * NQ * 128;
                    const uint32_t q8_bytes = FP8 ? QB * 2 * S_::NQ8 * NQ * S_::Q8ROW : 0;
                    const uint32_t p_bytes = NPB * TPI * NQ * 256;
                    const uint32_t fixed = align_up(q_bytes + q8_bytes + p_bytes, 1024);
                    const uint32_t tail = ut_bytes + sx_bytes + bars + small + 32;  // + alignment slack
                    if (1024 + fixed + tail > ATT_SMEM_LIMIT) continue;
                    const uint32_t avail = ATT_SMEM_LIMIT - 1024 - fixed - tail;
                    // K ring: at least a group's K sub-tiles (the rich plan: two tiles more); bf16
                    // V ring: a group's V sub-tiles (minimal plan: one tile's); FP8 raw V ring: two
                    // tiles' (minimal: one)
                    const int gsub = S_::NSUB * TPI;
                    int NK, NV, NR = 0;
                    if (!FP8) {
                        if (pass == 2) continue;
                        int n = (int)(avail / S_::OP_STAGE);
                        n = n > 10 ? 10 : n;
                        NV = min(max(pass == 0 ? gsub : S_::NSUB, n - 2 * S_::NSUB), 2 * gsub);
                        NK = n - NV;
                        if (NK < (pass == 0 ? 2 * S_::NSUB : S_::NSUB) || NV < S_::NSUB) continue;
                    } else {
                        // pass 0: converted-V stages for more than a group (the converters then
                        // work on the next group while the P.V of this one is pending), at least
                        // a group and one tile of K; pass 1: one group of V, two of K; pass 2:
                        // one tile of each
                        NR = pass < 2 ? 2 * S_::NSUB : S_::NSUB;
                        const int nv_min = pass == 0 ? gsub + S_::NSUB : (pass == 1 ? gsub : S_::NSUB);
                        const int nk_min = pass == 0 ? gsub + S_::NSUB : (pass == 1 ? 2 * gsub : S_::NSUB);
                        NV = 0;
                        for (int nv = pass == 0 ? 2 * gsub : nv_min; nv >= nv_min; --nv)
                            if (avail >= nv * S_::OP_STAGE + NR * S_::F8_STAGE + nk_min * S_::F8_STAGE) {
                                NV = nv;
                                break;
                            }
                        if (!NV) continue;
                        const uint32_t used = NV * S_::OP_STAGE + NR * S_::F8_STAGE;
                        NK = (int)((avail - used) / S_::F8_STAGE);
                        NK = NK > 8 ? 8 : NK;
                    }
                    if (bar_map(NK, NV, NR, NSB, NPB).end > BAR_BYTES) return SPEC_ERR_UNSUPPORTED;
                    p.TPI = TPI;
                    p.ut_entries = ut_entries;
                    p.NK = NK;
                    p.NV = NV;
                    p.NR = NR;
                    p.NSB = NSB;
                    p.NPB = NPB;
                    p.QB = QB;
                    p.OB = OB;
                    p.off_q = 0;
                    p.off_q8 = p.off_q + q_bytes;
                    p.off_p = p.off_q8 + q8_bytes;
                    p.off_k = align_up(p.off_p + p_bytes, 1024);
                    p.off_v = p.off_k + NK * S_::K_STAGE;
                    p.off_raw = p.off_v + NV * S_::OP_STAGE;
                    p.off_ut = p.off_raw + NR * S_::F8_STAGE;
                    p.off_sx = align_up(p.off_ut + ut_bytes, 16);
                    p.off_bar = align_up(p.off_sx + sx_bytes, 8);
                    p.off_small = p.off_bar + bars;
                    p.t_o = (uint32_t)(NSB * TPI * NQ);
                    p.t_one = p.t_o + (uint32_t)(OB * (S_::NSUB + 1) * NQ);
                    *smem_bytes = 1024 + p.off_small + small;
                    return SPEC_OK;
                }
    }
    return SPEC_ERR_UNSUPPORTED;
}

// FP8 pools: each query vector q (row j*G + i of its (branch, kv head)) becomes two E4M3
// terms, q * sigma = hi + lo with sigma = 2^e chosen so that max|q * sigma| lies in [128, 256)
// (clamped to 2^-126..2^126): exact for every element within 2^10 of the vector's largest.
// Written as [pair][hi, lo][NQ][d] bytes (padding rows zero) with 1/sigma per column, for the
// attention kernel to load by TMA. Grid (branch and kv head, NQ / 4): a warp per query
// vector, so that every vector's load, maximum and conversion run at once.
template <int D>
__global__ void __launch_bounds__(128) attn_qsplit_kernel(const uint16_t *__restrict__ q, int B, int k, int Hq,
                                                          int G, int Hkv, int NQ, uint8_t *q8, float *qinv) {
    grid_dep_wait();  // q may be written by the kernel before this one
    const int pair = blockIdx.x, b = pair / Hkv, g = pair % Hkv;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_q = (k + 1) * G;
    constexpr int EL = D / 32;  // elements per lane
    for (int r = blockIdx.y * 4 + warp; r < NQ; r += 4 * gridDim.y) {
        float x[EL];
        if (r < n_q) {
            const uint16_t *src = q + ((size_t)(b * (k + 1) + r / G) * Hq + g * G + r % G) * D + lane * EL;
#pragma unroll
            for (int e = 0; e < EL; ++e) x[e] = __uint_as_float((uint32_t)src[e] << 16);
        } else {
#pragma unroll
            for (int e = 0; e < EL; ++e) x[e] = 0.f;
        }
        float amax = 0.f;
#pragma unroll
        for (int e = 0; e < EL; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
        int ex = 0;
        if (amax > 0.f) {
            frexpf(amax, &ex);  // amax in [2^(ex-1), 2^ex)
            ex = 8 - ex;        // amax * 2^ex in [128, 256)
            ex = ex > 126 ? 126 : (ex < -126 ? -126 : ex);
        }
        const float sig = ldexpf(1.f, ex);
        if (lane == 0) qinv[(size_t)pair * NQ + r] = ldexpf(1.f, -ex);
        uint8_t *hi_row = q8 + ((size_t)pair * 2 * NQ + r) * D + lane * EL;
        uint8_t *lo_row = hi_row + (size_t)NQ * D;
#pragma unroll
        for (int e = 0; e < EL; e += 2) {
            const float a0 = x[e] * sig, a1 = x[e + 1] * sig;
            const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(make_float2(a0, a1), __NV_SATFINITE, __NV_E4M3);
            const __half2_raw hh = __nv_cvt_fp8x2_to_halfraw2(hi, __NV_E4M3);
            const float2 hf = __half22float2(*reinterpret_cast<const __half2 *>(&hh));
            const __nv_fp8x2_storage_t lo =
                __nv_cvt_float2_to_fp8x2(make_float2(a0 - hf.x, a1 - hf.y), __NV_SATFINITE, __NV_E4M3);
            *reinterpret_cast<__nv_fp8x2_storage_t *>(hi_row + e) = hi;
            *reinterpret_cast<__nv_fp8x2_storage_t *>(lo_row + e) = lo;
        }
    }
}

// The split queries viewed as a 2-D byte tensor (d, pairs * 2 * NQ): a box of one 128-byte
// (d = 64: 64-byte) column block x NQ rows lands in the swizzled K-major layout of the S MMA.
static bool make_q8_map(CUtensorMap *map, const void *q8, uint64_t rows, int d, int NQ) {
    EncodeTiledFnA fn = encode_fn_attn();
    if (!fn) return false;
    const int w = d < 128 ? d : 128;
    cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)d};
    cuuint32_t box[2] = {(cuuint32_t)w, (cuuint32_t)NQ};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(q8), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, w == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, bool FP8>
static int launch_attn(AttnParams &p, cudaStream_t s) {
    size_t smem = 0;
    const int st = plan_attn<D, FP8>(p, &smem);
    if (st) return st;
    CUtensorMap mq, mk, mv;
    if (FP8) {
        // the queries' E4M3 split, written to the workspace by a kernel of its own
        const int pairs = p.B * p.kv.n_kv_heads;
        const int st2 = launch_pdl(attn_qsplit_kernel<D>, dim3(pairs, p.NQ / 4), dim3(128), 0, s, p.q, p.B, p.k, p.Hq, p.G,
                                   p.kv.n_kv_heads, p.NQ, p.q8_g, const_cast<float *>(p.qinv_g));
        if (st2) return st2;
        if (!make_q8_map(&mq, p.q8_g, (uint64_t)pairs * 2 * p.NQ, D, p.NQ)) return SPEC_ERR_CUDA;
    } else if (!make_q_map(&mq, p.q, p.B * (p.k + 1), p.Hq, D, p.G, p.k + 1)) {
        return SPEC_ERR_CUDA;
    }
    mk = mq;
    mv = mq;
    if (FP8) {
        const uint64_t pool_rows = (uint64_t)p.kv.num_pages * p.kv.n_kv_heads * p.kv.page_size;
        if (!make_kv_map(&mk, p.kv.k_pool, pool_rows, D, p.tma_rows, true) ||
            !make_kv_map(&mv, p.kv.v_pool, pool_rows, D, p.tma_rows, false))
            return SPEC_ERR_CUDA;
    }
    // a fixed ceiling (see the skinny GEMM launcher): graphs may mix launch sizes
    if (cudaFuncSetAttribute(attn_kernel<D, FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize, ATT_SMEM_LIMIT) !=
        cudaSuccess)
        return SPEC_ERR_CUDA;
    const int sms = attn_sm_count();
    if (sms < 1) return SPEC_ERR_CUDA;
    const int grid = p.n_units < sms ? p.n_units : sms;
    return launch_pdl(attn_kernel<D, FP8>, dim3(grid), dim3(ATT_THREADS), smem, s, mq, mk, mv, p);
}

// Workspace: a 256-byte header (the unit scheduler's counters: zero before the first call
// and left zero by every call), then the per-unit (m, l) pairs and partial outputs, then
// (FP8 pools) the split queries and their scales.
struct WsLayout {
    size_t ml, o, q8, qinv, total;
};
static WsLayout ws_layout(int B, int Hkv, int n_splits, int NQ, int d, bool fp8) {
    WsLayout w;
    auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
    const size_t pairs = (size_t)B * Hkv, units = pairs * n_splits;
    w.ml = 256;
    w.o = w.ml + up(units * NQ * 2 * 4);
    w.q8 = w.o + up(units * NQ * d * 4);
    w.qinv = w.q8 + (fp8 ? up(pairs * 2 * NQ * d) : 0);
    w.total = w.qinv + (fp8 ? pairs * NQ * 4 : 0);
    return w;
}

// The combine grid: W = warps per (row, head) item, one per group of COMBINE_GROUP splits
// (at most 16; a power of two would leave warps idle and, for long rows, need a second
// wave of CTAs); 8 / W items per CTA when W < 8.
template <int D>
static int launch_combine(const AttnParams &p, cudaStream_t s) {
    const int ng_max = (p.n_splits + COMBINE_GROUP - 1) / COMBINE_GROUP;
    const int W = ng_max < 16 ? ng_max : 16;
    const int ipc = W >= 8 ? 1 : 8 / W;
    const int items = p.B * (p.k + 1) * p.Hq;
    const int grid = (items + ipc - 1) / ipc;
    const size_t smem = (size_t)ipc * combine_slot_floats(ng_max, D, W) * sizeof(float);
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(attn_combine_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) !=
            cudaSuccess)
        return SPEC_ERR_CUDA;
    if (smem > 227 * 1024) return SPEC_ERR_UNSUPPORTED;
    return launch_pdl(attn_combine_kernel<D>, dim3(grid), dim3(ipc * W * 32), smem, s, p, W, ipc, ng_max);
}

// The launch parameters that depend only on the shapes (the caller checks the descriptor
// and fills in the pointers).
static int attn_setup(const spec_kv_desc *kvd, int B, int k, int n_q_heads, int max_pos, AttnParams &p) {
    if (B < 1 || k < 0 || k > SPEC_KMAX || n_q_heads < 1 || max_pos < k + 1) return SPEC_ERR_ARG;
    if (n_q_heads % kvd->n_kv_heads) return SPEC_ERR_ARG;
    const int G = n_q_heads / kvd->n_kv_heads;
    const int n_q = (k + 1) * G;
    const int NQ = ((n_q + 15) / 16) * 16;
    p = AttnParams{};
    p.kv = make_view(kvd);
    p.B = B;
    p.k = k;
    p.Hq = n_q_heads;
    p.G = G;
    p.n_q = n_q;
    p.NQ = NQ;
    p.split_keys = split_keys_for(kvd->n_kv_heads, kvd->kv_dtype == SPEC_KV_FP8_E4M3);
    p.n_splits = (max_pos + p.split_keys - 1) / p.split_keys;
    p.max_pos = max_pos;
    p.n_units = B * kvd->n_kv_heads * p.n_splits;
    p.wait_ns = g_wait_ns;
    p.tma_rows = kvd->kv_dtype == SPEC_KV_FP8_E4M3 ? (kvd->page_size < TILE_KEYS ? kvd->page_size : TILE_KEYS) : 0;
    if (G > 256 || NQ > MAX_NQ) return SPEC_ERR_UNSUPPORTED;
    // FP8 pools are gathered by TMA boxes of one page-run: pages of at least 8 positions (a
    // swizzle atom of rows), row coordinates within 32 bits
    if (kvd->kv_dtype == SPEC_KV_FP8_E4M3 &&
        (kvd->page_size < 8 || (uint64_t)kvd->num_pages * kvd->n_kv_heads * kvd->page_size >= (1ull << 31)))
        return SPEC_ERR_UNSUPPORTED;
    return SPEC_OK;
}

static int plan_dispatch(AttnParams &p, size_t *smem) {
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
    spec::AttnParams p;
    st = spec::attn_setup(kvd, B, k, n_q_heads, max_pos, p);
    if (st) return st;
    size_t smem = 0;
    st = spec::plan_dispatch(p, &smem);
    if (st) return st;
    const int32_t v[SPEC_ATTN_PLAN_FIELDS] = {(int32_t)smem, p.NQ, p.NK, p.NV, p.NR, p.NSB, p.NPB, p.QB, p.OB,
                                              (int32_t)(p.t_one + 16), p.split_keys, p.n_splits,
                                              p.n_units, p.TPI, p.tma_rows,
                                              (int32_t)spec::bar_map(p.NK, p.NV, p.NR, p.NSB, p.NPB).end,
                                              (int32_t)spec::BAR_BYTES};
    for (int i = 0; i < SPEC_ATTN_PLAN_FIELDS; ++i) out[i] = v[i];
    return SPEC_OK;
}

SPEC_API size_t spec_verify_attn_workspace(const spec_kv_desc *kv, int B, int k, int n_q_heads, int max_pos) {
    if (spec::check_kv_desc(kv) || B < 1 || k < 0 || k > SPEC_KMAX || n_q_heads < 1 || max_pos < 1) return 0;
    if (n_q_heads % kv->n_kv_heads) return 0;
    const int G = n_q_heads / kv->n_kv_heads;
    const int NQ = (((k + 1) * G + 15) / 16) * 16;
    const int sk = spec::split_keys_for(kv->n_kv_heads, kv->kv_dtype == SPEC_KV_FP8_E4M3);
    const int n_splits = (max_pos + sk - 1) / sk;
    return spec::ws_layout(B, kv->n_kv_heads, n_splits, NQ, kv->head_dim, kv->kv_dtype == SPEC_KV_FP8_E4M3).total;
}

namespace spec {

// The chain and tree entry points: the same kernels, the tree with per-row slot masks.
static int attn_call(const spec_kv_desc *kvd, const int32_t *pos, int B, int k, int n_q_heads, const void *q,
                     float scale, const int32_t *anc, void *out, void *ws, size_t ws_bytes, int max_pos,
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
    spec::AttnParams p;
    st = spec::attn_setup(kvd, B, k, n_q_heads, max_pos, p);
    if (st) return st;
    p.pos = pos;
    p.anc = anc;
    p.q = (const uint16_t *)q;
    p.out = (uint16_t *)out;
    p.scale_log2 = scale * spec::LOG2E;
    const spec::WsLayout w =
        spec::ws_layout(B, kvd->n_kv_heads, p.n_splits, p.NQ, kvd->head_dim, kvd->kv_dtype == SPEC_KV_FP8_E4M3);
    char *base = (char *)ws;
    p.sched = (unsigned int *)base;
    p.ws_ml = (float *)(base + w.ml);
    p.ws_o = (float *)(base + w.o);
    p.q8_g = (uint8_t *)(base + w.q8);
    p.qinv_g = (const float *)(base + w.qinv);
    p.err = dev_err;
    cudaStream_t s = (cudaStream_t)stream;
    const bool fp8 = kvd->kv_dtype == SPEC_KV_FP8_E4M3;
    switch (kvd->head_dim * 2 + (fp8 ? 1 : 0)) {
        case 128: st = spec::launch_attn<64, false>(p, s); break;
        case 129: st = spec::launch_attn<64, true>(p, s); break;
        case 256: st = spec::launch_attn<128, false>(p, s); break;
        case 257: st = spec::launch_attn<128, true>(p, s); break;
        case 512: st = spec::launch_attn<256, false>(p, s); break;
        default: st = spec::launch_attn<256, true>(p, s); break;
    }
    if (st) return st;
    switch (kvd->head_dim) {
        case 64: return spec::launch_combine<64>(p, s);
        case 128: return spec::launch_combine<128>(p, s);
        default: return spec::launch_combine<256>(p, s);
    }
}

}  // namespace spec

SPEC_API int spec_verify_attn(const spec_kv_desc *kvd, const int32_t *pos, int B, int k, int n_q_heads,
                              const void *q, float scale, void *out, void *ws, size_t ws_bytes, int max_pos,
                              int32_t *dev_err, spec_stream_t stream) {
    return spec::attn_call(kvd, pos, B, k, n_q_heads, q, scale, nullptr, out, ws, ws_bytes, max_pos, dev_err,
                           stream);
}

SPEC_API int spec_verify_attn_tree(const spec_kv_desc *kvd, const int32_t *pos, int B, int k, int n_q_heads,
                                   const void *q, float scale, const int32_t *anc_mask, void *out, void *ws,
                                   size_t ws_bytes, int max_pos, int32_t *dev_err, spec_stream_t stream) {
    if (!anc_mask) return SPEC_ERR_NULL;
    return spec::attn_call(kvd, pos, B, k, n_q_heads, q, scale, anc_mask, out, ws, ws_bytes, max_pos, dev_err,
                           stream);
}

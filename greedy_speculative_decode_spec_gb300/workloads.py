"""Seeded synthetic inputs for the verify step -- the one module that both the CUDA
path's callers (tests, bench) and the CPU oracle's callers use.

It draws random numbers and lays them out; it computes none of the verify step
itself (no append, attention, logits, argmax or acceptance). Planted targets are
built from the inputs' construction (hidden = 8 * W[id] / |W[id]| + noise); that the
planted id really is the argmax with a margin is checked by the oracle in the tests.

Shapes follow the five workloads of the verify step:
  0 tiny          B=1,  k=3, H=256,  4/1 heads,  d=64,  ctx 100,  P=16, V=1024
  1 single stream B=1,  k=4, H=2048, 16/2 heads, d=256, ctx 4096, P=64, V=151936
  2 branches      B=16, k=6, H=4096, 32/8 heads, d=128, ctx~U[512,8192], P=16,
                  16384-page shared pool, acceptance 0.8 -> 0.4 with depth
  3 long context  B=4,  k=3, H=5120, 40/8 heads, d=128, ctx 32K/64K/96K/128K, P=64,
                  FP8 E4M3 pages with per-(page, kv head) scales, + 64 near-tie rows
  4 draft side    M=64 MTP inputs (E[151936,4096], fc [4096,8192]), draft head
                  [32768,4096] with a d2t map, then workload 2's verify with k=4
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass, field

import torch

BF16_NAN_BITS = 0x7FC0   # poison for bf16 pool slots
E4M3_NAN_BITS = 0x7F     # poison for FP8 pool slots


@dataclass(frozen=True)
class VerifyConfig:
    name: str
    B: int
    k: int
    H: int
    Hq: int
    Hkv: int
    d: int
    P: int
    V: int
    ctx: tuple = ()                 # fixed contexts, one per branch
    ctx_range: tuple = ()           # (lo, hi) inclusive uniform draw when ctx is empty
    num_pages: int = 0              # 0 -> pages needed + spare
    kv_dtype: str = "bf16"          # "bf16" | "fp8"
    accept_p: tuple = ()            # acceptance probability per draft depth
    near_tie: int = 0               # extra LM-head rows with an exact top-2 tie
    seed: int = 0
    permute_all_pages: bool = False  # page table row = permutation of the whole pool

    @property
    def R(self) -> int:
        return self.B * (self.k + 1)


def _decay(k, hi, lo):
    if k == 1:
        return (hi,)
    return tuple(hi + (lo - hi) * j / (k - 1) for j in range(k))


CONFIGS: dict[int, VerifyConfig] = {
    0: VerifyConfig("tiny_verify", B=1, k=3, H=256, Hq=4, Hkv=1, d=64, P=16, V=1024, ctx=(100,),
                    num_pages=8, accept_p=(0.7,) * 3, seed=1000, permute_all_pages=True),
    1: VerifyConfig("single_stream_mtp_verify", B=1, k=4, H=2048, Hq=16, Hkv=2, d=256, P=64, V=151936,
                    ctx=(4096,), num_pages=80, accept_p=(0.7,) * 4, seed=1001),
    2: VerifyConfig("batched_branches_shared_pool", B=16, k=6, H=4096, Hq=32, Hkv=8, d=128, P=16, V=151936,
                    ctx_range=(512, 8192), num_pages=16384, accept_p=_decay(6, 0.8, 0.4), seed=1002),
    3: VerifyConfig("long_context_fp8", B=4, k=3, H=5120, Hq=40, Hkv=8, d=128, P=64, V=151936,
                    ctx=(32768, 65536, 98304, 131072), num_pages=5184, kv_dtype="fp8",
                    accept_p=(0.7,) * 3, near_tie=64, seed=1003),
}


# the same workloads by name
WORKLOADS: dict[str, VerifyConfig] = {c.name: c for c in CONFIGS.values()}


@dataclass(frozen=True)
class DraftConfig:
    name: str = "draft_side_batch"
    M: int = 64
    H: int = 4096
    V: int = 151936
    V_draft: int = 32768
    eps: float = 1e-6
    seed: int = 1004
    verify_k: int = 4


DRAFT_CONFIG = DraftConfig()


def config4_verify(dc: DraftConfig = DRAFT_CONFIG) -> VerifyConfig:
    """The verify that follows the draft side: workload 2 with k = verify_k."""
    base = WORKLOADS["batched_branches_shared_pool"]
    B = dc.M // dc.verify_k
    return dataclasses.replace(base, name="draft_side_verify", B=B, k=dc.verify_k,
                               accept_p=_decay(dc.verify_k, 0.8, 0.4), seed=dc.seed + 100)


# ---- helpers ---------------------------------------------------------------------------

def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _randn_bf16(shape, g, device, std=1.0, chunk_rows=8192) -> torch.Tensor:
    """N(0, std^2) rounded to bf16, drawn in row chunks to bound the fp32 temporary."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    if out.numel() == 0:
        return out
    flat = out.view(shape[0], -1)
    for r0 in range(0, shape[0], chunk_rows):
        r1 = min(shape[0], r0 + chunk_rows)
        t = torch.randn((r1 - r0, flat.shape[1]), generator=g, device=device, dtype=torch.float32)
        if std != 1.0:
            t.mul_(std)
        flat[r0:r1] = t.to(torch.bfloat16)
    return out


def _randint(lo, hi, shape, g, device) -> torch.Tensor:
    return torch.randint(lo, hi, shape, generator=g, device=device, dtype=torch.int64)


def _uniform_other(avoid: torch.Tensor, V: int, g, device) -> torch.Tensor:
    """Uniform id in [0, V) different from `avoid` (elementwise)."""
    r = _randint(0, V - 1, avoid.shape, g, device)
    return torch.where(r >= avoid, r + 1, r)


def bits(t: torch.Tensor):
    """bf16 / uint8 tensor -> numpy array of its raw bits (uint16 / uint8)."""
    import numpy as np
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.uint8:
        return t.numpy()
    return t.numpy()


# ---- verify-step inputs ------------------------------------------------------------------

@dataclass
class VerifyInputs:
    cfg: VerifyConfig
    pos: torch.Tensor            # int32 [B]
    page_table: torch.Tensor     # int32 [B][max_pages], -1 = unused
    num_pages: int
    ctx_branch: torch.Tensor     # int32 [N] page-table row of each context row
    ctx_pos: torch.Tensor        # int32 [N] its position
    ctx_k: torch.Tensor          # bf16 [N][Hkv][d]
    ctx_v: torch.Tensor
    k_scale: torch.Tensor | None  # fp32 [num_pages][Hkv] (fp8 only)
    v_scale: torch.Tensor | None
    q: torch.Tensor              # bf16 [R][Hq][d]
    k_new: torch.Tensor          # bf16 [R][Hkv][d]
    v_new: torch.Tensor
    W: torch.Tensor              # bf16 [V][H]
    hidden: torch.Tensor         # bf16 [R][H]
    planted: torch.Tensor        # int32 [R] planted target id of each row
    drafts: torch.Tensor         # int32 [B][k]
    tie_hidden: torch.Tensor | None = None   # bf16 [near_tie][H]
    tie_expect: torch.Tensor | None = None   # int32 [near_tie] (the lower index of the pair)
    tie_pairs: torch.Tensor | None = None    # int32 [near_tie][2]
    extra: dict = field(default_factory=dict)

    @property
    def pool_shape(self):
        c = self.cfg
        return (self.num_pages, c.Hkv, c.P, c.d)

    @property
    def poison_bits(self) -> int:
        return BF16_NAN_BITS if self.cfg.kv_dtype == "bf16" else E4M3_NAN_BITS

    @property
    def max_pos(self) -> int:
        return int(self.pos.max().item()) + self.cfg.k + 1


def planted_hidden(W: torch.Tensor, ids: torch.Tensor, g, device, noise=0.1) -> torch.Tensor:
    """hidden = 8 * W[id] / |W[id]| + N(0, noise^2), rounded to bf16."""
    w = W[ids.to(W.device).long()].to(device=device, dtype=torch.float32)
    w = 8.0 * w / w.norm(dim=1, keepdim=True)
    w += noise * torch.randn(w.shape, generator=g, device=device, dtype=torch.float32)
    return w.to(torch.bfloat16)


def make_lm_head(V: int, H: int, seed: int, device="cpu") -> torch.Tensor:
    return _randn_bf16((V, H), _gen(seed, device), device, std=0.02)


def verify_inputs(cfg: VerifyConfig, device="cpu", W: torch.Tensor | None = None,
                  drafts: torch.Tensor | None = None) -> VerifyInputs:
    """All inputs of one verify step of `cfg`, drawn from cfg.seed on `device`.
    `W` reuses an LM-head weight (tied embeddings). `drafts` [B][k] fixes the draft
    tokens (e.g. a draft head's output): the target of row (b, j < k) is then planted on
    drafts[b][j] with the acceptance probability of depth j, else on another id."""
    planted = None
    g = _gen(cfg.seed, device)
    B, k, P = cfg.B, cfg.k, cfg.P
    if cfg.ctx:
        assert len(cfg.ctx) == B
        ctx = torch.tensor(cfg.ctx, dtype=torch.int64)
    else:
        lo, hi = cfg.ctx_range
        ctx = _randint(lo, hi + 1, (B,), g, device).cpu()
    need = [(int(c) + k + 1 + P - 1) // P for c in ctx]
    num_pages = cfg.num_pages or sum(need) + 8
    assert sum(need) <= num_pages, "pool too small for the contexts"
    max_pages = max(need)
    perm = torch.randperm(num_pages, generator=g, device=device).cpu()
    if cfg.permute_all_pages:
        assert B == 1 and max_pages <= num_pages
        max_pages = num_pages
        page_table = perm.view(1, -1).to(torch.int32)
    else:
        page_table = torch.full((B, max_pages), -1, dtype=torch.int32)
        off = 0
        # pages of all branches interleaved at random in the shared pool
        for b in range(B):
            page_table[b, :need[b]] = perm[off:off + need[b]].to(torch.int32)
            off += need[b]

    # context rows (positions 0..ctx-1 of every branch), values N(0,1) in bf16
    n_ctx = int(ctx.sum())
    ctx_branch = torch.repeat_interleave(torch.arange(B, dtype=torch.int32), ctx)
    ctx_pos = torch.cat([torch.arange(int(c), dtype=torch.int32) for c in ctx])
    ctx_k = _randn_bf16((n_ctx, cfg.Hkv, cfg.d), g, device)
    ctx_v = _randn_bf16((n_ctx, cfg.Hkv, cfg.d), g, device)
    R = cfg.R
    q = _randn_bf16((R, cfg.Hq, cfg.d), g, device)
    k_new = _randn_bf16((R, cfg.Hkv, cfg.d), g, device)
    v_new = _randn_bf16((R, cfg.Hkv, cfg.d), g, device)

    k_scale = v_scale = None
    if cfg.kv_dtype == "fp8":
        # one scale per (page, kv head) = amax / 448 of that block's bf16 values,
        # appended rows included (they are quantised with the same scale)
        k_scale = torch.ones((num_pages, cfg.Hkv), dtype=torch.float32)
        v_scale = torch.ones((num_pages, cfg.Hkv), dtype=torch.float32)
        c0 = 0
        for b in range(B):
            n = int(ctx[b])
            for src_ctx, src_new, sc in ((ctx_k, k_new, k_scale), (ctx_v, v_new, v_scale)):
                rows = torch.cat([src_ctx[c0:c0 + n], src_new[b * (k + 1):(b + 1) * (k + 1)]]).float().cpu()
                npg = need[b]
                padded = torch.zeros((npg * P, cfg.Hkv, cfg.d))
                padded[:rows.shape[0]] = rows
                amax = padded.abs().view(npg, P, cfg.Hkv, cfg.d).amax(dim=(1, 3))
                sc[page_table[b, :npg].long()] = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
            c0 += n

    if W is None:
        W = make_lm_head(cfg.V, cfg.H, cfg.seed + 7, device)
    tie_pairs = None
    if drafts is not None:
        drafts = drafts.to(device=device, dtype=torch.int64).view(B, k)
        p = torch.tensor(cfg.accept_p[:k], dtype=torch.float32, device=device).expand(B, k)
        hit = torch.rand((B, k), generator=g, device=device) < p
        tgt = torch.where(hit, drafts, _uniform_other(drafts, cfg.V, g, device))
        bonus = _randint(0, cfg.V, (B, 1), g, device)
        planted = torch.cat([tgt, bonus], dim=1).reshape(-1)
    if planted is None:
        if cfg.near_tie:
            pairs = torch.randperm(cfg.V, generator=g, device=device)[:2 * cfg.near_tie].view(cfg.near_tie, 2)
            pairs = torch.sort(pairs, dim=1).values
            forbidden = torch.zeros(cfg.V, dtype=torch.bool, device=device)
            forbidden[pairs[:, 1]] = True
            cand = _randint(0, cfg.V, (4 * R,), g, device)
            cand = cand[~forbidden[cand]][:R]
            planted = cand
            tie_pairs = pairs
        else:
            planted = _randint(0, cfg.V, (R,), g, device)
    planted = planted.to(device=device, dtype=torch.int64)
    if tie_pairs is not None:
        # near-tie set: W[j_hi] := W[j_lo], so the two logits are exactly equal
        W = W.clone()
        W[tie_pairs[:, 1]] = W[tie_pairs[:, 0]]
    hidden = planted_hidden(W, planted, g, device)
    # drafts: draft j of branch b is compared with the target of row b*(k+1)+j
    tgt = planted.view(B, k + 1)[:, :k]
    if drafts is not None:
        pass
    elif k > 0:
        p = torch.tensor(cfg.accept_p[:k], dtype=torch.float32, device=device).expand(B, k)
        hit = torch.rand((B, k), generator=g, device=device) < p
        drafts = torch.where(hit, tgt, _uniform_other(tgt, cfg.V, g, device))
    else:
        drafts = torch.zeros((B, 0), dtype=torch.int64, device=device)
    vi = VerifyInputs(cfg=cfg, pos=ctx.to(torch.int32), page_table=page_table, num_pages=num_pages,
                      ctx_branch=ctx_branch, ctx_pos=ctx_pos, ctx_k=ctx_k, ctx_v=ctx_v,
                      k_scale=k_scale, v_scale=v_scale, q=q, k_new=k_new, v_new=v_new, W=W,
                      hidden=hidden, planted=planted.to(torch.int32), drafts=drafts.to(torch.int32))
    if tie_pairs is not None:
        vi.tie_pairs = tie_pairs.to(torch.int32)
        vi.tie_hidden = planted_hidden(W, tie_pairs[:, 0], g, device)
        vi.tie_expect = tie_pairs[:, 0].to(torch.int32)
    return vi


# ---- draft-side inputs --------------------------------------------------------------------

@dataclass
class DraftInputs:
    cfg: DraftConfig
    tok: torch.Tensor       # int32 [M]
    E: torch.Tensor         # bf16 [V][H]  (tied with the verify LM head)
    h: torch.Tensor         # bf16 [M][H]
    g_emb: torch.Tensor     # fp32 [H]
    g_hid: torch.Tensor     # fp32 [H]
    W_fc: torch.Tensor      # bf16 [H][2H]
    W_draft: torch.Tensor   # bf16 [V_draft][H]
    d2t: torch.Tensor       # int32 [V_draft] distinct target ids


def draft_inputs(dc: DraftConfig = DRAFT_CONFIG, device="cpu", E: torch.Tensor | None = None,
                 V: int | None = None, H: int | None = None, V_draft: int | None = None,
                 M: int | None = None) -> DraftInputs:
    V = V or dc.V
    H = H or dc.H
    V_draft = V_draft or dc.V_draft
    M = M or dc.M
    g = _gen(dc.seed, device)
    tok = _randint(0, V, (M,), g, device).to(torch.int32)
    if E is None:
        E = _randn_bf16((V, H), g, device, std=0.02)
    h = _randn_bf16((M, H), g, device)
    g_emb = 0.5 + torch.rand((H,), generator=g, device=device)
    g_hid = 0.5 + torch.rand((H,), generator=g, device=device)
    W_fc = _randn_bf16((H, 2 * H), g, device, std=0.02)
    W_draft = _randn_bf16((V_draft, H), g, device, std=0.02)
    d2t = torch.randperm(V, generator=g, device=device)[:V_draft].to(torch.int32)
    return DraftInputs(dc, tok, E, h, g_emb.float(), g_hid.float(), W_fc, W_draft, d2t)


def scaled(cfg: VerifyConfig, **kw) -> VerifyConfig:
    """A smaller case of the same workload (parity tests that the oracle finishes fast)."""
    return dataclasses.replace(cfg, **kw)


def algorithmic_kv_bytes(cfg: VerifyConfig, pos) -> int:
    """Bytes of K and V one verify step must read: every (page, kv head) block of the
    keys 0..pos[b]+k of every branch, once (elements only; FP8 adds its scales)."""
    esz = 2 if cfg.kv_dtype == "bf16" else 1
    keys = sum(int(p) + cfg.k + 1 for p in pos)
    total = 2 * keys * cfg.Hkv * cfg.d * esz
    if cfg.kv_dtype == "fp8":
        pages = sum(math.ceil((int(p) + cfg.k + 1) / cfg.P) for p in pos)
        total += 2 * pages * cfg.Hkv * 4
    return total

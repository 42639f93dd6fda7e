"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle on the same
seeded inputs. Integers and bytes must match exactly; attention outputs must satisfy
max|gpu - oracle| <= 1e-2 * max|oracle| + 1e-3."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle as orc
from gpu_harness import (DEV, assert_attn_close, assert_pools_equal, gpu_accept, gpu_attention, gpu_lmhead,
                         gpu_pool, lm_ws, oracle_pool)
from greedy_speculative_decode_spec_gb300 import _binding as bnd
from greedy_speculative_decode_spec_gb300.workloads import WORKLOADS, bits, scaled, verify_inputs

pytestmark = pytest.mark.gpu

# Smaller cases of each workload: several tiles and splits, ragged vocab / K / page tails.
SMALL = {
    "tiny": WORKLOADS["tiny_verify"],
    "single_stream": scaled(WORKLOADS["single_stream_mtp_verify"], ctx=(2500,), V=5003, num_pages=48, seed=11),
    "branches": scaled(WORKLOADS["batched_branches_shared_pool"], B=5, ctx_range=(20, 2100), V=3001, H=520, num_pages=1024, seed=12),
    "long_fp8": scaled(WORKLOADS["long_context_fp8"], ctx=(1000, 2500, 60, 3100), V=2050, H=200, num_pages=140, near_tie=16,
                       seed=13),
}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from greedy_speculative_decode_spec_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    bnd.lib()


def _step_parity(vi, full_oracle: bool, n_items=24, n_rows=32):
    c = vi.cfg
    B, k, Hq, d = c.B, c.k, c.Hq, c.d
    okv = oracle_pool(vi)
    gkv = gpu_pool(vi)
    assert_pools_equal(gkv, okv)                      # a1 on the context rows
    pos_d = vi.pos.cuda()
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    bnd.spec_kv_append(gkv.desc, pos_d, B, k, vi.k_new.cuda(), vi.v_new.cuda(), err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert orc.kv_append(okv, vi.pos.numpy(), B, k, bits(vi.k_new), bits(vi.v_new)) == 0
    assert_pools_equal(gkv, okv)                      # a1: the append itself

    # a2
    out, e = gpu_attention(gkv, pos_d, B, k, Hq, vi.q.cuda(), vi.max_pos)
    assert e == 0
    scale = 1.0 / math.sqrt(d)
    if full_oracle:
        ref, oe = orc.verify_attn(okv, vi.pos.numpy(), B, k, Hq, bits(vi.q), scale)
        assert oe == 0
        assert_attn_close(out, ref)
    else:
        # sampled outputs: every branch and every kv head, each at the branch's first and
        # last verify row (a random q head of the group), plus random (row, head) items
        R = B * (k + 1)
        G = Hq // c.Hkv
        rng = np.random.default_rng(c.seed)
        cover = [(b * (k + 1) + j) * Hq + g * G + int(rng.integers(G))
                 for b in range(B) for g in range(c.Hkv) for j in sorted({0, k})]
        items = np.unique(np.concatenate([rng.integers(0, R * Hq, n_items), cover])).astype(np.int32)
        ref, oe = orc.verify_attn_items(okv, vi.pos.numpy(), B, k, Hq, bits(vi.q), scale, items)
        assert oe == 0
        assert_attn_close(out.reshape(R * Hq, d)[torch.from_numpy(items).long().cuda()], ref)
        assert torch.isfinite(out.float()).all()

    # a3
    hid = vi.hidden.cuda()
    W = vi.W.cuda()
    ids, mx, e = gpu_lmhead(hid, W)
    assert e == 0
    np.testing.assert_array_equal(ids, vi.planted.numpy())
    if full_oracle or c.R <= 16:
        rows = np.arange(c.R)
    else:
        # at least 32 rows: every branch's first and last verify row, then random ones
        ends = {b * (k + 1) + j for b in range(B) for j in (0, k)}
        rest = np.setdiff1d(np.arange(c.R), sorted(ends))
        fill = np.random.default_rng(c.seed + 1).choice(rest, max(0, min(len(rest), n_rows - len(ends))),
                                                          replace=False)
        rows = np.sort(np.concatenate([sorted(ends), fill])).astype(np.int64)
    oids, omx, gap, _ = orc.lmhead_argmax(bits(vi.hidden)[rows], bits(vi.W))
    assert gap.min() >= 0.5, "planted margin not met (generator)"   # on every row the oracle sees
    np.testing.assert_array_equal(ids[rows], oids)
    np.testing.assert_allclose(mx[rows], omx, rtol=1e-4, atol=1e-3)

    # a4, on the (verified) target ids
    ids_d = torch.from_numpy(ids).cuda()
    toks, n, a, npos, nxt, h_out = gpu_accept(vi.drafts.cuda(), ids_d, pos_d, B, k, hidden=hid)
    ot, on, oa, onp, onx = orc.accept(vi.drafts.numpy(), ids, vi.pos.numpy(), B, k)
    for g_, o_ in ((toks, ot), (n, on), (a, oa), (npos, onp), (nxt, onx)):
        np.testing.assert_array_equal(g_, o_)
    rows_a = torch.arange(B, device=DEV) * (k + 1) + torch.from_numpy(a).long().cuda()
    assert torch.equal(h_out.view(torch.int16), hid[rows_a].view(torch.int16))

    # near-tie set: the top two logits are exactly equal, the lower index wins
    if vi.tie_hidden is not None:
        tids, _, e = gpu_lmhead(vi.tie_hidden.cuda(), W)
        assert e == 0
        np.testing.assert_array_equal(tids, vi.tie_expect.numpy())
        sel = np.arange(len(tids))
        oti, _, tgap, _ = orc.lmhead_argmax(bits(vi.tie_hidden)[sel], bits(vi.W))
        np.testing.assert_array_equal(tids[sel], oti)
        assert np.all(tgap == 0.0)
    return gkv, okv, out


@pytest.mark.parametrize("name", list(SMALL))
def test_step_parity_small(name):
    _step_parity(verify_inputs(SMALL[name]), full_oracle=True)


@pytest.mark.parametrize("name", ["tiny_verify", "single_stream_mtp_verify", "batched_branches_shared_pool",
                                  "long_context_fp8"])
def test_step_parity_full_size(name):
    """The full workloads, in the launch configuration the benchmark times: pools compared
    byte for byte, attention and logits on sampled outputs, ids on every row."""
    _step_parity(verify_inputs(WORKLOADS[name]), full_oracle=(name == "tiny_verify"))


# ---- row invariance: a row's result does not depend on the batch it is verified in ---------

@pytest.mark.parametrize("name", ["branches", "long_fp8"])
def test_attention_rows_bytewise_equal_one_row_calls(name):
    vi = verify_inputs(SMALL[name])
    c = vi.cfg
    gkv = gpu_pool(vi)
    pos_d = vi.pos.cuda()
    bnd.spec_kv_append(gkv.desc, pos_d, c.B, c.k, vi.k_new.cuda(), vi.v_new.cuda())
    q = vi.q.cuda()
    out, e = gpu_attention(gkv, pos_d, c.B, c.k, c.Hq, q, vi.max_pos + 3000)
    assert e == 0
    for b in range(c.B):
        desc1 = bnd.make_kv_desc(gkv.k, gkv.v, gkv.page_table[b:b + 1].contiguous(), c.P, gkv.k_scale, gkv.v_scale)
        one = type(gkv).__new__(type(gkv))
        one.__dict__.update(gkv.__dict__)
        one.desc = desc1
        for j in (0, c.k // 2, c.k):
            r = b * (c.k + 1) + j
            p = int(vi.pos[b]) + j
            o1, e1 = gpu_attention(one, torch.tensor([p], dtype=torch.int32, device=DEV), 1, 0, c.Hq,
                                   q[r:r + 1].contiguous(), p + 1)
            assert e1 == 0
            assert torch.equal(o1[0].view(torch.int16), out[r].view(torch.int16)), (b, j)


def test_lmhead_logits_bytewise_equal_across_batch_sizes():
    vi = verify_inputs(SMALL["branches"])
    W = vi.W.cuda()
    hid = vi.hidden.cuda()
    M, V = hid.shape[0], W.shape[0]
    logits = torch.empty((M, V), dtype=torch.float32, device=DEV)
    ids = torch.empty(M, dtype=torch.int32, device=DEV)
    bnd.spec_lmhead_logits(hid, W, logits, ids, lm_ws(M, V, W.shape[1]))
    big = hid.repeat(256 // M + 1, 1)[:256].contiguous()      # the same rows first, then others
    lbig = torch.empty((256, V), dtype=torch.float32, device=DEV)
    ibig = torch.empty(256, dtype=torch.int32, device=DEV)
    bnd.spec_lmhead_logits(big, W, lbig, ibig, lm_ws(256, V, W.shape[1]))
    torch.cuda.synchronize()
    assert torch.equal(lbig[:M].view(torch.int32), logits.view(torch.int32))
    for r in (0, 7, M - 1):
        l1 = torch.empty((1, V), dtype=torch.float32, device=DEV)
        i1 = torch.empty(1, dtype=torch.int32, device=DEV)
        bnd.spec_lmhead_logits(hid[r:r + 1].contiguous(), W, l1, i1, lm_ws(1, V, W.shape[1]))
        torch.cuda.synchronize()
        assert torch.equal(l1[0].view(torch.int32), logits[r].view(torch.int32))
        assert int(i1.item()) == int(ids[r].item())
    # the logits agree with the oracle's fp64 logits
    ref = orc.lmhead_logits(bits(vi.hidden)[:4], bits(vi.W))
    np.testing.assert_allclose(logits[:4].cpu().numpy(), ref, rtol=1e-4, atol=2e-3)


# ---- NaN poisoning: unattended slots never reach an output ----------------------------------

@pytest.mark.parametrize("name", ["branches", "long_fp8"])
def test_poisoned_slots_never_reach_outputs(name):
    vi = verify_inputs(SMALL[name])
    c = vi.cfg
    outs = []
    for poison in (True, False):
        gkv = gpu_pool(vi, poison=poison)
        pos_d = vi.pos.cuda()
        bnd.spec_kv_append(gkv.desc, pos_d, c.B, c.k, vi.k_new.cuda(), vi.v_new.cuda())
        out, e = gpu_attention(gkv, pos_d, c.B, c.k, c.Hq, vi.q.cuda(), vi.max_pos)
        assert e == 0 and torch.isfinite(out.float()).all()
        outs.append(out)
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))


# ---- device-side errors: reported, never trapped ---------------------------------------------

def test_bad_page_id_is_reported_not_trapped():
    vi = verify_inputs(SMALL["tiny"])
    c = vi.cfg
    gkv = gpu_pool(vi)
    pt = gkv.page_table.clone()
    pt[0, 6] = c.num_pages + 5          # the page holding positions 96..111
    desc = bnd.make_kv_desc(gkv.k, gkv.v, pt, c.P)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pos_d = vi.pos.cuda()
    before = gkv.k.clone()
    bnd.spec_kv_append(desc, pos_d, c.B, c.k, vi.k_new.cuda(), vi.v_new.cuda(), err)
    torch.cuda.synchronize()
    assert int(err.item()) & bnd.DEVERR_PAGE
    assert torch.equal(gkv.k.view(torch.int16), before.view(torch.int16))   # skipped, nothing written
    err.zero_()
    out = torch.zeros((c.R, c.Hq, c.d), dtype=torch.bfloat16, device=DEV)
    ws = torch.zeros(bnd.spec_verify_attn_workspace(desc, c.B, c.k, c.Hq, vi.max_pos), dtype=torch.uint8, device=DEV)
    bnd.spec_verify_attn(desc, pos_d, c.B, c.k, c.Hq, vi.q.cuda(), 0.125, out, ws, vi.max_pos, err)
    torch.cuda.synchronize()
    assert int(err.item()) & bnd.DEVERR_PAGE
    # a branch whose rows reach beyond max_pos is refused on the device
    err.zero_()
    bnd.spec_verify_attn(gkv.desc, pos_d, c.B, c.k, c.Hq, vi.q.cuda(), 0.125, out, ws, vi.max_pos - 1, err)
    torch.cuda.synchronize()
    assert int(err.item()) & bnd.DEVERR_POS
    # the context is still healthy
    ids, _, e = gpu_lmhead(vi.hidden.cuda(), vi.W.cuda())
    assert e == 0 and np.array_equal(ids, vi.planted.numpy())


def test_position_past_page_table_coverage_is_reported():
    vi = verify_inputs(SMALL["tiny"])
    c = vi.cfg
    gkv = gpu_pool(vi)
    last = (int(vi.pos.max()) + c.k) // c.P     # the page-table column of the last verify row
    pt = gkv.page_table[:, :last].contiguous()  # that column is missing: not covered
    desc = bnd.make_kv_desc(gkv.k, gkv.v, pt, c.P)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pos_d = vi.pos.cuda()
    before = gkv.k.clone()
    bnd.spec_kv_append(desc, pos_d, c.B, c.k, vi.k_new.cuda(), vi.v_new.cuda(), err)
    torch.cuda.synchronize()
    assert int(err.item()) & bnd.DEVERR_COVER
    assert torch.equal(gkv.k.view(torch.int16), before.view(torch.int16))   # skipped, nothing written
    err.zero_()
    out = torch.zeros((c.R, c.Hq, c.d), dtype=torch.bfloat16, device=DEV)
    ws = torch.zeros(bnd.spec_verify_attn_workspace(desc, c.B, c.k, c.Hq, vi.max_pos), dtype=torch.uint8, device=DEV)
    bnd.spec_verify_attn(desc, pos_d, c.B, c.k, c.Hq, vi.q.cuda(), 0.125, out, ws, vi.max_pos, err)
    torch.cuda.synchronize()
    assert int(err.item()) & bnd.DEVERR_COVER


def test_d2t_out_of_range_is_reported():
    vi = verify_inputs(SMALL["tiny"])
    d2t = torch.arange(vi.cfg.V, dtype=torch.int32, device=DEV) * 3
    ids, _, e = gpu_lmhead(vi.hidden.cuda(), vi.W.cuda(), d2t=d2t, d2t_limit=vi.cfg.V)
    assert e & bnd.DEVERR_D2T
    want = np.where(vi.planted.numpy() * 3 < vi.cfg.V, vi.planted.numpy() * 3, -1)
    np.testing.assert_array_equal(ids, want)


# ---- edge shapes -------------------------------------------------------------------------------

@pytest.mark.parametrize("M,V,H", [(1, 1, 8), (1, 777, 64), (3, 129, 72), (256, 1000, 128), (17, 4096, 1032)])
def test_lmhead_edge_shapes(M, V, H):
    g = torch.Generator().manual_seed(M * 7 + V)
    W = (0.02 * torch.randn((V, H), generator=g)).to(torch.bfloat16)
    hid = torch.randn((M, H), generator=g).to(torch.bfloat16)
    ids, mx, e = gpu_lmhead(hid.cuda(), W.cuda())
    oids, omx, gap, _ = orc.lmhead_argmax(bits(hid), bits(W))
    ok = gap > 1e-3 * np.abs(omx) + 1e-4      # clear winners must match exactly
    np.testing.assert_array_equal(ids[ok], oids[ok])
    np.testing.assert_allclose(mx, omx, rtol=1e-4, atol=1e-3)


@pytest.mark.parametrize("P,d,k,B", [(1, 64, 0, 1), (4, 128, 15, 2), (256, 256, 1, 3), (1024, 64, 2, 2)])
def test_attention_edge_shapes(P, d, k, B):
    cfg = scaled(WORKLOADS["tiny_verify"], B=B, k=k, P=P, d=d, Hq=4, Hkv=2, ctx=tuple([0, 1030, 5][:B]), num_pages=0,
                 permute_all_pages=False, accept_p=(0.7,) * k, V=64, H=256, seed=50 + P + k)
    vi = verify_inputs(cfg)
    _step_parity(vi, full_oracle=True)


@pytest.mark.parametrize("P,d,k,B,G", [(8, 64, 3, 2, 2), (64, 256, 1, 2, 4), (16, 128, 15, 2, 2), (8, 128, 0, 1, 5)])
def test_attention_edge_shapes_fp8(P, d, k, B, G):
    """E4M3 pools at every head dimension (the queries' E4M3 split is written straight into
    the 128- or 64-byte-swizzled operand layout), pages down to 8 positions, k = 0 and 15."""
    cfg = scaled(WORKLOADS["tiny_verify"], B=B, k=k, P=P, d=d, Hq=2 * G, Hkv=2, ctx=tuple([3, 1030, 5][:B]),
                 num_pages=0, permute_all_pages=False, accept_p=(0.7,) * k, V=64, H=256, kv_dtype="fp8",
                 seed=70 + P + k + d)
    vi = verify_inputs(cfg)
    _step_parity(vi, full_oracle=True)


def test_accept_random_patterns_max_k():
    rng = np.random.default_rng(9)
    for B, k in ((16, 15), (7, 1), (3, 0), (32, 6)):
        ids = rng.integers(0, 50, B * (k + 1)).astype(np.int32)
        hit = rng.random((B, k)) < 0.8
        drafts = np.where(hit, ids.reshape(B, k + 1)[:, :k], 99).astype(np.int32)
        pos = rng.integers(0, 10 ** 6, B).astype(np.int32)
        got = gpu_accept(torch.from_numpy(drafts).cuda(), torch.from_numpy(ids).cuda(), torch.from_numpy(pos).cuda(),
                         B, k)
        want = orc.accept(drafts, ids, pos, B, k)
        for g_, o_ in zip(got, want):
            np.testing.assert_array_equal(g_, o_)


def _gpu_accept_stop(drafts, ids, pos, B, k, stop, budget, hidden=None):
    i32 = dict(dtype=torch.int32, device=DEV)
    toks = torch.empty((B, k + 1), **i32)
    n, a, npos, nxt, done = (torch.full((B,), -7, **i32) for _ in range(5))
    stop_d = torch.tensor(stop, **i32) if len(stop) else None
    bud_d = None if budget is None else torch.from_numpy(budget).to(DEV)
    h_out = None if hidden is None else torch.zeros((B, hidden.shape[1]), dtype=torch.bfloat16, device=DEV)
    bnd.spec_accept_stop(torch.from_numpy(drafts).to(DEV), torch.from_numpy(ids).to(DEV), torch.from_numpy(pos).to(DEV),
                         B, k, stop_d, bud_d, toks, n, a, npos, nxt, done, hidden=hidden, h_out=h_out)
    torch.cuda.synchronize()
    return [t.cpu().numpy() for t in (toks, n, a, npos, nxt, done)], h_out


def test_accept_stop_matches_oracle():
    rng = np.random.default_rng(21)
    for B, k in ((16, 15), (9, 4), (5, 0), (33, 6)):
        ids = rng.integers(0, 12, B * (k + 1)).astype(np.int32)
        hit = rng.random((B, k)) < 0.85
        drafts = np.where(hit, ids.reshape(B, k + 1)[:, :k], 99).astype(np.int32)
        pos = rng.integers(0, 10 ** 6, B).astype(np.int32)
        for stop, budget in (([], None), ([3, -1, 7], None), ([], rng.integers(-2, k + 3, B).astype(np.int32)),
                             (list(range(0, 12, 2)) + [-1] * 26, rng.integers(0, k + 2, B).astype(np.int32))):
            got, _ = _gpu_accept_stop(drafts, ids, pos, B, k, stop, budget)
            want = orc.accept_stop(drafts, ids, pos, B, k, stop, budget)
            for g_, o_ in zip(got, want):
                np.testing.assert_array_equal(g_, o_)
    # no stop set, no budget: exactly spec_accept
    got, _ = _gpu_accept_stop(drafts, ids, pos, B, k, [], None)
    base = gpu_accept(torch.from_numpy(drafts).cuda(), torch.from_numpy(ids).cuda(), torch.from_numpy(pos).cuda(), B, k)
    for g_, o_ in zip(got[:5], base):
        np.testing.assert_array_equal(g_, o_)


def test_accept_stop_hidden_row_of_last_token():
    rng = np.random.default_rng(22)
    B, k, H = 6, 4, 64
    ids = rng.integers(0, 6, B * (k + 1)).astype(np.int32)
    drafts = ids.reshape(B, k + 1)[:, :k].copy()          # full acceptance everywhere
    pos = np.arange(B, dtype=np.int32) * 10
    hidden = torch.randn((B * (k + 1), H), device=DEV).to(torch.bfloat16)
    budget = np.array([0, 1, 2, 3, 5, 9], np.int32)
    (toks, n, a, npos, nxt, done), h_out = _gpu_accept_stop(drafts, ids, pos, B, k, [], budget, hidden)
    want = orc.accept_stop(drafts, ids, pos, B, k, [], budget)
    np.testing.assert_array_equal(n, want[1])
    for b in range(B):
        if n[b] == 0:
            assert torch.count_nonzero(h_out[b]) == 0     # left unwritten
        else:
            assert torch.equal(h_out[b], hidden[b * (k + 1) + n[b] - 1])


def test_accept_stop_host_errors():
    i32 = dict(dtype=torch.int32, device=DEV)
    t = torch.zeros(8, **i32)
    toks = torch.zeros((1, 2), **i32)
    with pytest.raises(bnd.SpecError):
        bnd.spec_accept_stop(t[:1], t[:2], t[:1], 1, 1, torch.zeros(33, **i32), None, toks, t[:1], t[:1], t[:1], t[:1])


def test_fp8_large_v_scales_take_the_bf16_path():
    """FP8 pools whose V page scales exceed the f16 range of the converted values: those
    units multiply in bf16 (the same codes, every V value and scale times 2^16)."""
    vi = verify_inputs(SMALL["long_fp8"])
    big = 65536.0
    vi.ctx_v = (vi.ctx_v.float() * big).to(torch.bfloat16)
    vi.v_new = (vi.v_new.float() * big).to(torch.bfloat16)
    vi.v_scale = vi.v_scale * big
    _step_parity(vi, full_oracle=True)

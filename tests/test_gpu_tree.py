"""Tree / star verify (f2) on the GPU against the oracle: attention with per-row ancestor
masks over the verify slots, the greedy tree walk, and the KV compaction of the accepted
path (DSSD-dev `_set_rows`, `_star_cycle`)."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle as orc
from gpu_harness import DEV, assert_attn_close, assert_pools_equal, attn_ws, gpu_attention, gpu_pool, oracle_pool
from greedy_speculative_decode_spec_gb300 import _binding as bnd
from greedy_speculative_decode_spec_gb300.workloads import WORKLOADS, bits, scaled, verify_inputs

pytestmark = pytest.mark.gpu

CASES = {
    "bf16": scaled(WORKLOADS["batched_branches_shared_pool"], B=4, ctx_range=(10, 1500), V=3001, H=520, num_pages=512,
                   seed=41),
    "fp8": scaled(WORKLOADS["long_context_fp8"], B=3, ctx=(900, 70, 2100), V=2050, H=200, num_pages=140, seed=42),
    "d256": scaled(WORKLOADS["single_stream_mtp_verify"], ctx=(1300,), V=5003, num_pages=48, seed=43),
}


def random_parents(B, k, rng):
    par = np.zeros((B, k + 1), np.int32)
    for b in range(B):
        for j in range(1, k + 1):
            par[b, j] = rng.integers(0, j)
    return par


def masks_from_parents(par):
    B, kp1 = par.shape
    m = np.zeros((B, kp1), np.int32)
    for b in range(B):
        for j in range(kp1):
            bitset, c = 0, j
            while True:
                bitset |= 1 << c
                if c == 0:
                    break
                c = par[b, c]
            m[b, j] = bitset
    return m


def _appended(vi):
    c = vi.cfg
    gkv, okv = gpu_pool(vi), oracle_pool(vi)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    bnd.spec_kv_append(gkv.desc, vi.pos.cuda(), c.B, c.k, vi.k_new.cuda(), vi.v_new.cuda(), err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert orc.kv_append(okv, vi.pos.numpy(), c.B, c.k, bits(vi.k_new), bits(vi.v_new)) == 0
    return gkv, okv


def _tree_attention(gkv, vi, masks):
    c = vi.cfg
    out = torch.empty((c.B * (c.k + 1), c.Hq, c.d), dtype=torch.bfloat16, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    bnd.spec_verify_attn_tree(gkv.desc, vi.pos.cuda(), c.B, c.k, c.Hq, vi.q.cuda(), 1.0 / math.sqrt(c.d),
                              torch.from_numpy(masks.reshape(-1)).to(DEV), out, attn_ws(gkv, c.B, c.k, c.Hq, vi.max_pos),
                              vi.max_pos, dev_err=err)
    torch.cuda.synchronize()
    return out, int(err.item())


@pytest.mark.parametrize("name", list(CASES))
def test_tree_attention_matches_oracle(name):
    vi = verify_inputs(CASES[name])
    c = vi.cfg
    gkv, okv = _appended(vi)
    rng = np.random.default_rng(7)
    masks = masks_from_parents(random_parents(c.B, c.k, rng))
    out, e = _tree_attention(gkv, vi, masks)
    assert e == 0
    ref, oe = orc.verify_attn_tree(okv, vi.pos.numpy(), c.B, c.k, c.Hq, bits(vi.q), 1.0 / math.sqrt(c.d), masks)
    assert oe == 0
    assert_attn_close(out, ref, "tree attention")


@pytest.mark.parametrize("name", list(CASES))
def test_tree_attention_with_chain_masks_is_the_chain_bit_for_bit(name):
    vi = verify_inputs(CASES[name])
    c = vi.cfg
    gkv, _ = _appended(vi)
    tree_out, e1 = _tree_attention(gkv, vi, orc.chain_masks(c.B, c.k))
    chain_out, e2 = gpu_attention(gkv, vi.pos.cuda(), c.B, c.k, c.Hq, vi.q.cuda(), vi.max_pos)
    assert e1 == 0 and e2 == 0
    assert torch.equal(tree_out.view(torch.int16), chain_out.view(torch.int16))


def test_tree_attention_reports_bad_masks():
    """A row whose mask lacks its own bit, or has a later row's bit, is reported and left
    unwritten; every other row matches the oracle."""
    vi = verify_inputs(CASES["bf16"])
    c = vi.cfg
    gkv, okv = _appended(vi)
    rng = np.random.default_rng(8)
    masks = masks_from_parents(random_parents(c.B, c.k, rng))
    masks[1, 3] &= ~(1 << 3)
    masks[2, 1] |= 1 << 4
    sentinel = torch.full((c.B * (c.k + 1), c.Hq, c.d), 7.0, dtype=torch.bfloat16, device=DEV)
    out = sentinel.clone()
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    bnd.spec_verify_attn_tree(gkv.desc, vi.pos.cuda(), c.B, c.k, c.Hq, vi.q.cuda(), 1.0 / math.sqrt(c.d),
                              torch.from_numpy(masks.reshape(-1)).to(DEV), out,
                              attn_ws(gkv, c.B, c.k, c.Hq, vi.max_pos), vi.max_pos, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == bnd.DEVERR_TREE
    ref, oe = orc.verify_attn_tree(okv, vi.pos.numpy(), c.B, c.k, c.Hq, bits(vi.q), 1.0 / math.sqrt(c.d), masks)
    assert oe == orc.ERR_TREE
    bad = [1 * (c.k + 1) + 3, 2 * (c.k + 1) + 1]
    assert np.isnan(ref[bad]).all()
    assert torch.equal(out[bad], sentinel[bad])
    keep = [r for r in range(c.B * (c.k + 1)) if r not in bad]
    assert_attn_close(out[keep], ref[keep], "tree attention, valid rows")


def _walk_inputs(B, k, rng, V=50):
    par = random_parents(B, k, rng)
    ids = rng.integers(0, V, (B, k + 1)).astype(np.int32)
    drafts = rng.integers(0, V, (B, k)).astype(np.int32)
    # plant walks: along a random root-to-leaf chain of the tree, drafts copy the parent's target
    for b in range(B):
        for j in range(1, k + 1):
            if rng.random() < 0.6:
                drafts[b, j - 1] = ids[b, par[b, j]]
    pos = rng.integers(0, 1000, B).astype(np.int32)
    return par, ids, drafts, pos


def _gpu_walk(drafts, ids, pos, par, B, k):
    i32 = dict(dtype=torch.int32, device=DEV)
    toks, path = torch.empty((B, k + 1), **i32), torch.empty((B, k + 1), **i32)
    n, a, npos, nxt = (torch.empty(B, **i32) for _ in range(4))
    err = torch.zeros(1, **i32)
    bnd.spec_accept_tree(torch.from_numpy(drafts).to(DEV), torch.from_numpy(ids.reshape(-1)).to(DEV),
                         torch.from_numpy(pos).to(DEV), torch.from_numpy(par.reshape(-1)).to(DEV), B, k, toks, n, a,
                         npos, nxt, path, dev_err=err)
    torch.cuda.synchronize()
    return [t.cpu().numpy() for t in (toks, n, a, npos, nxt, path)] + [int(err.item())]


@pytest.mark.parametrize("k", [1, 4, 7, 15])
def test_tree_walk_matches_oracle(k):
    rng = np.random.default_rng(100 + k)
    B = 64
    par, ids, drafts, pos = _walk_inputs(B, k, rng)
    g = _gpu_walk(drafts, ids, pos, par, B, k)
    o = orc.accept_tree(drafts, ids.reshape(-1), pos, par, B, k)
    assert g[6] == 0 and o[6] == 0
    for gi, oi in zip(g[:6], o[:6]):
        assert np.array_equal(gi, oi)
    assert (g[2] > 0).any(), "the planted walks should accept some rows"


def test_tree_walk_reports_bad_parents():
    rng = np.random.default_rng(9)
    B, k = 8, 5
    par, ids, drafts, pos = _walk_inputs(B, k, rng)
    par[3, 4] = 4  # not an earlier row
    g = _gpu_walk(drafts, ids, pos, par, B, k)
    o = orc.accept_tree(drafts, ids.reshape(-1), pos, par, B, k)
    assert g[6] & bnd.DEVERR_TREE and o[6] != 0
    for gi, oi in zip(g[:6], o[:6]):
        assert np.array_equal(gi, oi)


def test_tree_walk_with_chain_parents_is_spec_accept():
    rng = np.random.default_rng(11)
    B, k = 32, 6
    par = np.tile(np.arange(-1, k, dtype=np.int32), (B, 1))
    par[:, 0] = 0
    ids = rng.integers(0, 20, (B, k + 1)).astype(np.int32)
    drafts = np.where(rng.random((B, k)) < 0.7, ids[:, :k], rng.integers(0, 20, (B, k))).astype(np.int32)
    pos = rng.integers(0, 500, B).astype(np.int32)
    g = _gpu_walk(drafts, ids, pos, par, B, k)
    o = orc.accept(drafts, ids.reshape(-1), pos, B, k)
    for gi, oi in zip(g[:5], o[:5]):
        assert np.array_equal(gi, oi)


@pytest.mark.parametrize("name", list(CASES))
def test_kv_compaction_matches_oracle(name):
    vi = verify_inputs(CASES[name])
    c = vi.cfg
    gkv, okv = _appended(vi)
    rng = np.random.default_rng(13)
    par, _, _, _ = _walk_inputs(c.B, c.k, rng)
    # a path per branch: a random walk down the tree, as the walk would produce it
    path = np.full((c.B, c.k + 1), -1, np.int32)
    acc = np.zeros(c.B, np.int32)
    for b in range(c.B):
        path[b, 0], cur, a = 0, 0, 0
        while True:
            kids = [j for j in range(cur + 1, c.k + 1) if par[b, j] == cur]
            if not kids or rng.random() < 0.2:
                break
            cur = kids[rng.integers(len(kids))]
            a += 1
            path[b, a] = cur
        acc[b] = a
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    bnd.spec_kv_compact(gkv.desc, vi.pos.cuda(), torch.from_numpy(path.reshape(-1)).to(DEV),
                        torch.from_numpy(acc).to(DEV), c.B, c.k, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert orc.kv_compact(okv, vi.pos.numpy(), path, acc, c.B, c.k) == 0
    assert_pools_equal(gkv, okv)
    assert acc.sum() > 0


@pytest.mark.parametrize("name", ["batched_branches_shared_pool", "long_context_fp8"])
def test_tree_attention_full_size(name):
    """The full workloads with random trees over their verify slots, in the launch
    configuration the benchmark times: every output against the oracle; chain masks give
    the chain call bit for bit."""
    vi = verify_inputs(WORKLOADS[name])
    c = vi.cfg
    gkv, okv = _appended(vi)
    masks = masks_from_parents(random_parents(c.B, c.k, np.random.default_rng(c.seed)))
    out, e = _tree_attention(gkv, vi, masks)
    assert e == 0
    ref, oe = orc.verify_attn_tree(okv, vi.pos.numpy(), c.B, c.k, c.Hq, bits(vi.q), 1.0 / math.sqrt(c.d), masks)
    assert oe == 0
    assert_attn_close(out, ref, "tree attention, full size")
    tree_out, e1 = _tree_attention(gkv, vi, orc.chain_masks(c.B, c.k))
    chain_out, e2 = gpu_attention(gkv, vi.pos.cuda(), c.B, c.k, c.Hq, vi.q.cuda(), vi.max_pos)
    assert e1 == 0 and e2 == 0
    assert torch.equal(tree_out.view(torch.int16), chain_out.view(torch.int16))

"""The oracle of tree / star verify (a next row of the hot path): tree attention, the greedy
tree walk and KV compaction, pinned against torch's fp64 attention with explicit key lists,
hand-worked examples, the chain special case and invariants over all small trees."""
from __future__ import annotations

import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

from test_oracle_pins import GOLDEN, _attn_case, bits_to_f64


def _ancestor_masks(parent_rows):
    """mask[j] = j and its ancestors (root row 0 included), as bits over the verify slots."""
    masks = []
    for j in range(len(parent_rows)):
        m, c = 0, j
        while c >= 0:
            m |= 1 << c
            c = parent_rows[c] if c > 0 else -1
        masks.append(m)
    return masks


def _random_parents(rng, k):
    return [-1] + [int(rng.integers(0, j)) for j in range(1, k + 1)]


def test_tree_attention_with_chain_masks_is_the_chain(orc):
    torch.manual_seed(3)
    rng = np.random.default_rng(3)
    B, k, Hq, Hkv, d, P = 3, 4, 4, 2, 8, 4
    ctxs = [0, 5, 13]
    kv, q, _, _ = _attn_case(orc, rng, B, k, Hq, Hkv, d, P, ctxs)
    chain, e1 = orc.verify_attn(kv, ctxs, B, k, Hq, q, 0.3)
    tree, e2 = orc.verify_attn_tree(kv, ctxs, B, k, Hq, q, 0.3, orc.chain_masks(B, k))
    assert e1 == e2 == 0
    np.testing.assert_array_equal(chain, tree)


@pytest.mark.parametrize("fp8", [False, True])
def test_tree_attention_matches_sdpa_over_the_row_key_lists(orc, fp8):
    torch.manual_seed(5)
    rng = np.random.default_rng(5)
    B, k, Hq, Hkv, d, P = 3, 5, 4, 2, 8, 4
    ctxs = [2, 9, 0]
    kv, q, dk, dv = _attn_case(orc, rng, B, k, Hq, Hkv, d, P, ctxs, fp8=fp8)
    parents = [_random_parents(rng, k) for _ in range(B)]
    masks = np.array([_ancestor_masks(pr) for pr in parents], np.int32)
    scale = 1 / math.sqrt(d)
    out, err = orc.verify_attn_tree(kv, ctxs, B, k, Hq, q, scale, masks)
    assert err == 0 and np.isfinite(out).all()
    qd = bits_to_f64(q).reshape(B * (k + 1), Hq, d)
    for b in range(B):
        for j in range(k + 1):
            keys = list(range(ctxs[b])) + [ctxs[b] + i for i in range(k + 1) if (masks[b, j] >> i) & 1]
            kk = torch.from_numpy(dk[b, keys]).permute(1, 0, 2)[None]
            vv = torch.from_numpy(dv[b, keys]).permute(1, 0, 2)[None]
            qq = torch.from_numpy(qd[b * (k + 1) + j])[None, :, None, :]
            ref = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, scale=scale, enable_gqa=True)
            np.testing.assert_allclose(out[b * (k + 1) + j], ref[0, :, 0].numpy(), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("bad", ["missing_self", "sees_a_later_row"])
def test_tree_attention_rejects_masks_that_are_not_ancestor_sets(orc, bad):
    """Row j of a tree sees itself and only earlier rows (DSSD-dev `_set_rows`: the row's
    own path): a mask without bit j, or with a bit above j, is reported and its row is NaN;
    the other rows are untouched."""
    rng = np.random.default_rng(21)
    B, k, Hq, Hkv, d, P = 2, 4, 4, 2, 8, 4
    ctxs = [3, 6]
    kv, q, _, _ = _attn_case(orc, rng, B, k, Hq, Hkv, d, P, ctxs)
    masks = np.array([_ancestor_masks(_random_parents(rng, k)) for _ in range(B)], np.int32)
    good, err = orc.verify_attn_tree(kv, ctxs, B, k, Hq, q, 0.3, masks)
    assert err == 0
    bb, j = 1, 2
    masks[bb, j] = (masks[bb, j] & ~(1 << j)) if bad == "missing_self" else (masks[bb, j] | (1 << (j + 1)))
    out, err = orc.verify_attn_tree(kv, ctxs, B, k, Hq, q, 0.3, masks)
    assert err == orc.ERR_TREE
    r = bb * (k + 1) + j
    assert np.isnan(out[r]).all()
    keep = np.arange(B * (k + 1)) != r
    np.testing.assert_array_equal(out[keep], good[keep])


def test_accept_tree_golden(orc):
    with open(os.path.join(GOLDEN, "accept_tree_example.json")) as f:
        fx = json.load(f)
    for c in fx["cases"]:
        k = len(c["drafts"])
        toks, n, a, npos, nxt, path, err = orc.accept_tree(c["drafts"], c["ids"], [c["pos"]], c["parent"], 1, k)
        assert err == 0, c["note"]
        assert toks[0].tolist() == c["tokens"] and path[0].tolist() == c["path"], c["note"]
        assert (n[0], a[0], npos[0], nxt[0]) == (c["n"], c["accepted"], c["new_pos"], c["next"]), c["note"]


@pytest.mark.parametrize("k", [0, 1, 3, 6])
def test_accept_tree_chain_is_the_greedy_chain(orc, k):
    rng = np.random.default_rng(k + 70)
    B = 40
    ids = rng.integers(0, 4, B * (k + 1)).astype(np.int32)
    drafts = rng.integers(0, 4, (B, k)).astype(np.int32)
    pos = rng.integers(0, 100, B).astype(np.int32)
    parent = np.tile(np.arange(-1, k, dtype=np.int32), (B, 1))
    base = orc.accept(drafts, ids, pos, B, k)
    tree = orc.accept_tree(drafts, ids, pos, parent, B, k)
    assert tree[6] == 0
    for x, y in zip(base, tree[:5]):
        np.testing.assert_array_equal(x, y)
    for b in range(B):
        assert tree[5][b, :tree[2][b] + 1].tolist() == list(range(tree[2][b] + 1))


@pytest.mark.parametrize("k", [1, 2, 3, 4])
def test_accept_tree_walk_invariants_over_all_small_trees(orc, k):
    """For every parent array with parent[j] < j and random tokens over a small alphabet:
    the path follows parent links, each accepted token is the previous row's choice, the
    lowest-numbered matching child is taken, and the walk stops only where no child matches."""
    rng = np.random.default_rng(80 + k)
    trees = [[-1] + list(t) for t in itertools.product(*[range(j) for j in range(1, k + 1)])]
    for pr in trees:
        B = 12
        ids = rng.integers(0, 3, B * (k + 1)).astype(np.int32)
        drafts = rng.integers(0, 3, (B, k)).astype(np.int32)
        pos = rng.integers(0, 50, B).astype(np.int32)
        toks, n, a, npos, nxt, path, err = orc.accept_tree(drafts, ids, pos, np.tile(pr, (B, 1)), B, k)
        assert err == 0
        for b in range(B):
            tg = ids[b * (k + 1):(b + 1) * (k + 1)]
            p = path[b, :a[b] + 1].tolist()
            assert p[0] == 0 and np.all(path[b, a[b] + 1:] == -1)
            for i in range(1, len(p)):
                prev, cur = p[i - 1], p[i]
                assert pr[cur] == prev and drafts[b, cur - 1] == tg[prev]
                assert not any(pr[c] == prev and drafts[b, c - 1] == tg[prev] for c in range(1, cur))
            last = p[-1]
            assert not any(pr[c] == last and drafts[b, c - 1] == tg[last] for c in range(1, k + 1))
            assert toks[b, :a[b]].tolist() == [int(drafts[b, c - 1]) for c in p[1:]]
            assert toks[b, a[b]] == tg[last] == nxt[b] and n[b] == a[b] + 1 and npos[b] == pos[b] + a[b] + 1


def test_accept_tree_reports_bad_parents(orc):
    *_, err = orc.accept_tree([1, 2], [1, 2, 3], [0], [-1, 0, 2], 1, 2)     # parent[2] = 2 is not < 2
    assert err == orc.ERR_TREE


def test_compaction_turns_the_path_into_the_chain(orc):
    """After the walk, moving the path's K/V to contiguous slots makes the chain attention of
    the path's rows equal, bit for bit, to their tree attention before the move (bf16)."""
    torch.manual_seed(9)
    rng = np.random.default_rng(9)
    B, k, Hq, Hkv, d, P = 2, 5, 4, 2, 8, 4
    ctxs = [3, 10]
    kv, q, _, _ = _attn_case(orc, rng, B, k, Hq, Hkv, d, P, ctxs, poison=False)
    parents = [[-1, 0, 0, 1, 3, 2], [-1, 0, 1, 0, 3, 4]]
    paths = [[0, 1, 3, 4], [0, 3, 4, 5]]
    masks = np.array([_ancestor_masks(pr) for pr in parents], np.int32)
    tree, err = orc.verify_attn_tree(kv, ctxs, B, k, Hq, q, 0.25, masks)
    assert err == 0
    acc = np.array([len(p) - 1 for p in paths], np.int32)
    path_arr = np.full((B, k + 1), -1, np.int32)
    for b, p in enumerate(paths):
        path_arr[b, :len(p)] = p
    assert orc.kv_compact(kv, ctxs, path_arr, acc, B, k) == 0
    a_max = int(acc.max())
    assert np.all(acc == a_max)
    qr = q.reshape(B, k + 1, Hq, d)
    q_chain = np.stack([qr[b, paths[b]] for b in range(B)]).reshape(B * (a_max + 1), Hq, d)
    chain, err = orc.verify_attn(kv, ctxs, B, a_max, Hq, q_chain, 0.25)
    assert err == 0
    for b in range(B):
        for i, row in enumerate(paths[b]):
            np.testing.assert_array_equal(chain[b * (a_max + 1) + i], tree[b * (k + 1) + row])


def test_compaction_fp8_requantises_with_the_destination_scale(orc):
    torch.manual_seed(13)
    rng = np.random.default_rng(13)
    B, k, Hq, Hkv, d, P = 1, 3, 2, 1, 8, 2
    kv, q, dk, dv = _attn_case(orc, rng, B, k, Hq, Hkv, d, P, [1], fp8=True, poison=False)
    path = np.array([[0, 2, -1, -1]], np.int32)
    before_k = dk[0, 1 + 2].copy()
    assert orc.kv_compact(kv, [1], path, np.array([1], np.int32), B, k) == 0
    page, slot = kv.page_table[0, (1 + 1) // P], (1 + 1) % P
    got_k = np.array([orc.e4m3_decode(c) for c in kv.k_pool[page, 0, slot]]) * kv.k_scale[page, 0]
    want_codes = [orc.e4m3_encode(np.float32(x) / kv.k_scale[page, 0]) for x in before_k[0]]
    np.testing.assert_array_equal(kv.k_pool[page, 0, slot], np.array(want_codes, np.uint8))
    # within one E4M3 step of the source value
    assert np.all(np.abs(got_k - before_k[0]) <= np.abs(before_k[0]) / 8 + kv.k_scale[page, 0] * 2 ** -9)

"""Speculative sampling acceptance (f4) on the GPU against the oracle, with the random
numbers as inputs on both sides (oxinfer `speculative_accept`; DSSD-dev `_sample_verify`).

The kernel takes its probabilities in fp32 and its sums in fp64; the oracle is all fp64.
Decisions must agree except where the oracle's test value lies within 1e-5 (relative) of a
boundary, the only place where both results are correct; the test checks that every
disagreement is such a near-tie, and that there are none on these seeded inputs."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as orc
from gpu_harness import DEV
from greedy_speculative_decode_spec_gb300 import _binding as bnd

pytestmark = pytest.mark.gpu


def _softmax(z, T):
    x = z.astype(np.float64) / T
    e = np.exp(x - x.max())
    return e / e.sum()


def _inputs(B, k, V, T, seed):
    rng = np.random.default_rng(seed)
    logits = (3.0 * rng.standard_normal((B * (k + 1), V))).astype(np.float32)
    q = np.empty((B, k, V), np.float32)
    drafts = np.empty((B, k), np.int32)
    for b in range(B):
        for i in range(k):
            p = _softmax(logits[b * (k + 1) + i], T)
            # the draft distribution: p seen through a perturbed temperature and noise
            qq = _softmax(logits[b * (k + 1) + i] + rng.standard_normal(V).astype(np.float32), T * 1.3)
            q[b, i] = qq.astype(np.float32)
            # a draft drawn from q (likely kept) or a near-argmax of q
            drafts[b, i] = rng.choice(V, p=qq) if rng.random() < 0.7 else int(np.argmax(qq))
    u_acc = rng.random((B, k)).astype(np.float32)
    u_res = rng.random(B).astype(np.float32)
    pos = rng.integers(0, 10000, B).astype(np.int32)
    return logits, q, drafts, u_acc, u_res, pos


def _gpu(logits, q, drafts, u_acc, u_res, pos, B, k, T):
    i32 = dict(dtype=torch.int32, device=DEV)
    toks = torch.empty((B, k + 1), **i32)
    n, a, npos, nxt = (torch.empty(B, **i32) for _ in range(4))
    err = torch.zeros(1, **i32)
    bnd.spec_accept_sample(torch.from_numpy(drafts).to(DEV), torch.from_numpy(logits).to(DEV),
                           torch.from_numpy(q).to(DEV), torch.from_numpy(pos).to(DEV), B, k, T,
                           torch.from_numpy(u_acc).to(DEV), torch.from_numpy(u_res).to(DEV), toks, n, a, npos, nxt,
                           dev_err=err)
    torch.cuda.synchronize()
    return [t.cpu().numpy() for t in (toks, n, a, npos, nxt)] + [int(err.item())]


def _draw_margin(w, u):
    """Distance (relative to the total) of u * sum(w) to the nearest running-sum boundary."""
    c = np.cumsum(w)
    lim = u * c[-1]
    return float(np.min(np.abs(c - lim)) / c[-1])


def _near_tie(b, k, T, logits, q, drafts, u_acc, u_res, a_gpu, a_orc):
    """Whether branch b's disagreement sits within 1e-5 of a decision boundary."""
    for i in range(min(a_gpu, a_orc, k - 1) + 1 if k else 0):
        p = _softmax(logits[b * (k + 1) + i], T)
        d = drafts[b, i]
        r = p[d] / q[b, i, d]
        if abs(float(u_acc[b, i]) - r) <= 1e-5 * max(r, 1e-30) or abs(p[d] - q[b, i, d]) <= 1e-5 * p[d]:
            return True
    a = min(a_gpu, a_orc)
    p = _softmax(logits[b * (k + 1) + a], T)
    w = np.maximum(p - q[b, a].astype(np.float64), 0.0) if a < k else p
    if not (w > 0).any():
        w = p
    return _draw_margin(w, float(u_res[b])) <= 1e-5


# vocabulary chunks of 8192: several with a ragged tail (16-byte vector loads when V % 4 == 0,
# scalar otherwise), one, and the full 151936-entry vocabulary (last: the benchmark's shape)
@pytest.mark.parametrize("B,k,V,T", [(6, 4, 50021, 0.8), (5, 7, 4099, 1.3), (3, 0, 1000, 1.0), (2, 15, 300, 0.5),
                                     (4, 3, 20000, 1.0), (2, 6, 151936, 1.0), (16, 6, 151936, 1.0)])
def test_sample_accept_matches_oracle(B, k, V, T):
    logits, q, drafts, u_acc, u_res, pos = _inputs(B, k, V, T, seed=V + k)
    g_toks, g_n, g_a, g_pos, g_next, err = _gpu(logits, q, drafts, u_acc, u_res, pos, B, k, T)
    assert err == 0
    o_toks, o_n, o_a, o_pos, o_next, o_err = orc.accept_sample(drafts, logits, q, pos, B, k, T, u_acc, u_res)
    assert o_err == 0
    mismatches = [b for b in range(B) if not np.array_equal(g_toks[b], o_toks[b])]
    for b in mismatches:
        assert _near_tie(b, k, T, logits, q, drafts, u_acc, u_res, int(g_a[b]), int(o_a[b])), f"branch {b} differs"
    assert not mismatches, f"near-ties on seeded inputs: {mismatches}"
    assert np.array_equal(g_n, o_n) and np.array_equal(g_a, o_a)
    assert np.array_equal(g_pos, o_pos) and np.array_equal(g_next, o_next)
    assert np.array_equal(g_n, g_a + 1) and np.array_equal(g_pos, pos + g_a + 1)


def test_sample_accept_emits_the_target_distribution():
    """Many branches with the same rows and independent u: the first emitted token follows
    p_0 (the defining property of speculative sampling), whatever q is."""
    B, k, V, T = 4096, 2, 48, 1.0
    rng = np.random.default_rng(5)
    row = (2.0 * rng.standard_normal((k + 1, V))).astype(np.float32)
    logits = np.tile(row, (B, 1)).astype(np.float32)
    qrow = np.stack([_softmax(row[i] + 1.5 * rng.standard_normal(V), T) for i in range(k)]).astype(np.float32)
    q = np.tile(qrow[None], (B, 1, 1)).astype(np.float32)
    drafts = np.stack([[rng.choice(V, p=qrow[i] / qrow[i].sum()) for i in range(k)] for _ in range(B)]).astype(np.int32)
    u_acc = rng.random((B, k)).astype(np.float32)
    u_res = rng.random(B).astype(np.float32)
    pos = np.zeros(B, np.int32)
    toks = _gpu(logits, q, drafts, u_acc, u_res, pos, B, k, T)[0]
    hist = np.bincount(toks[:, 0], minlength=V) / B
    p0 = _softmax(row[0], T)
    tv = 0.5 * np.abs(hist - p0).sum()
    assert tv < 0.05, f"total variation {tv:.3f} from p_0"


def test_sample_accept_host_errors():
    i32 = dict(dtype=torch.int32, device=DEV)
    z = torch.zeros((2, 8), dtype=torch.float32, device=DEV)
    o = [torch.empty(1, **i32) for _ in range(4)]
    with pytest.raises(bnd.SpecError):
        bnd.spec_accept_sample(torch.zeros((1, 1), **i32), z, torch.zeros((1, 1, 8), device=DEV), torch.zeros(1, **i32),
                               1, 1, 0.0, torch.zeros((1, 1), device=DEV), torch.zeros(1, device=DEV),
                               torch.empty((1, 2), **i32), *o)


@pytest.mark.parametrize("bad", ["below", "above", "q_zero"])
def test_invalid_draft_is_rejected_and_reported(bad):
    B, k, V, T = 4, 3, 3001, 1.0
    logits, q, drafts, u_acc, u_res, pos = _inputs(B, k, V, T, seed=77)
    bb, ii = 2, 1
    if bad == "below":
        drafts[bb, ii] = -5
    elif bad == "above":
        drafts[bb, ii] = V
    else:
        q[bb, ii, drafts[bb, ii]] = 0.0
    g = _gpu(logits, q, drafts, u_acc, u_res, pos, B, k, T)
    o = orc.accept_sample(drafts, logits, q, pos, B, k, T, u_acc, u_res)
    assert g[5] == bnd.DEVERR_TOKEN and o[5] == orc.ERR_TOKEN
    assert g[2][bb] <= ii
    for gi, oi in zip(g[:5], o[:5]):
        assert np.array_equal(gi, oi)


def test_sample_accept_reuses_its_workspace():
    """The workspace's per-branch counters are back at zero after a call: a second call on the
    same workspace writes every output again, equal to the first."""
    B, k, V, T = 5, 4, 20000, 0.9
    logits, q, drafts, u_acc, u_res, pos = _inputs(B, k, V, T, seed=123)
    args = [torch.from_numpy(x).to(DEV) for x in (drafts, logits, q, pos)]
    ua, ur = torch.from_numpy(u_acc).to(DEV), torch.from_numpy(u_res).to(DEV)
    ws = torch.zeros(bnd.spec_accept_sample_workspace(B, k, V), dtype=torch.uint8, device=DEV)
    i32 = dict(dtype=torch.int32, device=DEV)
    runs = []
    for _ in range(3):
        toks = torch.full((B, k + 1), -7, **i32)
        outs = [torch.full((B,), -7, **i32) for _ in range(4)]
        err = torch.zeros(1, **i32)
        bnd.spec_accept_sample(*args, B, k, T, ua, ur, toks, *outs, dev_err=err, ws=ws)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        runs.append([toks.cpu()] + [o.cpu() for o in outs])
    for r in runs[1:]:
        for x, y in zip(runs[0], r):
            assert torch.equal(x, y)
    assert int(runs[0][1].min()) >= 1  # every branch's outputs were written

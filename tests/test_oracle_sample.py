"""The oracle of speculative sampling acceptance (a next row of the hot path), pinned by
hand-worked cases, its greedy limit, closed forms and the property that makes it lossless:
the emitted token is distributed exactly as the target p."""
from __future__ import annotations

import json
import os

import numpy as np
import pytest

from test_oracle_pins import GOLDEN


def _softmax(z):
    z = z - z.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=-1, keepdims=True)


def test_accept_sample_golden(orc):
    with open(os.path.join(GOLDEN, "accept_sample_example.json")) as f:
        fx = json.load(f)
    for c in fx["cases"]:
        k = len(c["drafts"])
        logits = np.log(np.array(c["p"], np.float64)).astype(np.float32)
        toks, n, a, npos, nxt, err = orc.accept_sample(c["drafts"], logits, c["q"], [c["pos"]], 1, k, 1.0,
                                                       [c["u_acc"]], [c["u_res"]])
        assert err == 0
        assert toks[0].tolist() == c["tokens"], c["note"]
        assert (n[0], a[0], npos[0], nxt[0]) == (c["n"], c["accepted"], c["new_pos"], c["next"]), c["note"]


@pytest.mark.parametrize("k", [0, 1, 3])
def test_greedy_distributions_give_greedy_acceptance(orc, k):
    """One-hot p (a large logit gap) and one-hot q at each draft: a draft is kept iff it is
    the target argmax, a rejection returns the argmax: the greedy chain, for any u."""
    rng = np.random.default_rng(30 + k)
    B, V = 64, 9
    ids = rng.integers(0, V, B * (k + 1)).astype(np.int32)
    drafts = np.where(rng.random((B, k)) < 0.6, ids.reshape(B, k + 1)[:, :k], rng.integers(0, V, (B, k))).astype(np.int32)
    logits = np.zeros((B * (k + 1), V), np.float32)
    logits[np.arange(B * (k + 1)), ids] = 80.0
    q = np.zeros((B, k, V), np.float32)
    for b in range(B):
        for i in range(k):
            q[b, i, drafts[b, i]] = 1.0
    pos = rng.integers(0, 100, B).astype(np.int32)
    got = orc.accept_sample(drafts, logits, q, pos, B, k, 1.0, rng.random((B, k)), rng.random(B))
    want = orc.accept(drafts, ids, pos, B, k)
    assert got[5] == 0
    for x, y in zip(got[:5], want):
        np.testing.assert_array_equal(x, y)


def test_q_equal_p_keeps_every_draft(orc):
    rng = np.random.default_rng(41)
    B, k, V = 50, 3, 7
    logits = rng.normal(size=(B * (k + 1), V)).astype(np.float32)
    p = _softmax(logits.astype(np.float64) / 0.7).reshape(B, k + 1, V)
    q = p[:, :k].astype(np.float32)
    drafts = rng.integers(0, V, (B, k)).astype(np.int32)
    u_res = rng.random(B).astype(np.float32)
    toks, n, a, npos, nxt, err = orc.accept_sample(drafts, logits, q, np.zeros(B, np.int32), B, k, 0.7,
                                                   rng.random((B, k)) * 0.999, u_res)
    assert err == 0
    # kept when p(d) >= q(d) (float rounding of q may put p a hair below q: then u < ratio ~ 1)
    assert np.all(a == k)
    for b in range(B):
        w = p[b, k]
        bonus = int(np.argmax(np.cumsum(w) > float(u_res[b]) * w.sum()))
        assert toks[b, :k].tolist() == drafts[b].tolist() and toks[b, k] == bonus == nxt[b]


@pytest.mark.parametrize("k", [1, 3])
def test_emitted_token_is_distributed_as_the_target(orc, k):
    """Drafts drawn from q, then accepted or replaced: the first emitted token follows p_0
    (including tokens q never proposes and none that p never produces)."""
    rng = np.random.default_rng(50 + k)
    V, N = 5, 300_000
    p0 = np.array([0.45, 0.25, 0.2, 0.1, 0.0])
    q0 = np.array([0.1, 0.5, 0.0, 0.2, 0.2])
    logits0 = np.log(np.maximum(p0, 1e-300)).astype(np.float32)
    logits0[p0 == 0] = -1e4
    logits = np.tile(rng.normal(size=(k + 1, V)).astype(np.float32), (N, 1))
    logits[0::k + 1] = logits0
    q = np.tile(_softmax(rng.normal(size=(k, V))), (N, 1, 1)).astype(np.float32)
    q[:, 0] = q0
    # drafts drawn from q (inverse CDF, the same rule as the oracle's draws)
    u_d = rng.random((N, k))
    cq = np.cumsum(q.astype(np.float64), axis=-1)
    drafts = (cq <= (u_d[..., None] * cq[..., -1:])).sum(axis=-1).astype(np.int32)
    toks, n, a, npos, nxt, err = orc.accept_sample(drafts, logits, q, np.zeros(N, np.int32), N, k, 1.0,
                                                   rng.random((N, k)), rng.random(N))
    assert err == 0
    hist = np.bincount(toks[:, 0], minlength=V) / N
    np.testing.assert_allclose(hist, p0, atol=4e-3)
    assert hist[4] == 0.0


@pytest.mark.parametrize("bad", ["below", "above", "q_zero"])
def test_invalid_draft_is_rejected_and_reported(orc, bad):
    """A draft is a sample of q, so it lies in [0, V) and has q(d) > 0 (oxinfer
    `speculative_accept`). One that does not is reported and treated as rejected: the row's
    token is drawn from the residual as for any rejection, and the drafts before it stand."""
    rng = np.random.default_rng(61)
    B, k, V = 4, 3, 11
    logits = rng.normal(size=(B * (k + 1), V)).astype(np.float32)
    q = _softmax(rng.normal(size=(B, k, V))).astype(np.float32)
    p = _softmax(logits.astype(np.float64)).reshape(B, k + 1, V)
    drafts = np.argmax(p[:, :k] / q, axis=-1).astype(np.int32)  # ratio > 1: kept for any u
    u_acc, u_res = rng.random((B, k)), rng.random(B)
    bb, ii = 2, 1
    if bad == "below":
        drafts[bb, ii] = -1
    elif bad == "above":
        drafts[bb, ii] = V
    else:
        q[bb, ii, drafts[bb, ii]] = 0.0
    toks, n, a, npos, nxt, err = orc.accept_sample(drafts, logits, q, np.zeros(B, np.int32), B, k, 1.0, u_acc, u_res)
    assert err == orc.ERR_TOKEN
    assert a[bb] == ii and toks[bb, :ii].tolist() == drafts[bb, :ii].tolist()
    w = np.maximum(p[bb, ii] - q[bb, ii].astype(np.float64), 0.0)
    assert toks[bb, ii] == nxt[bb] == int(np.argmax(np.cumsum(w) > u_res[bb] * w.sum()))
    assert all(a[b] == k for b in range(B) if b != bb)

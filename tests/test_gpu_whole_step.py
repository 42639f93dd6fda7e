"""Whole-step exactness on the GPU: the speculative loop driven through the C ABI emits
exactly the one-row greedy stream (span-02 spec.rs, module documentation; oxinfer
qwen_mtp.rs, `OXINFER_CHECK_SPEC`), with every unattended slot poisoned with NaN."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle as orc
from gpu_harness import DEV, lm_ws
from greedy_speculative_decode_spec_gb300 import _binding as bnd
from greedy_speculative_decode_spec_gb300.step import PagedKv
from test_oracle_pins import OracleSide
from toy_lm import ToyLM, run_greedy, run_spec

pytestmark = pytest.mark.gpu


class GpuSide:
    """Drives the toy model through the library: append, attention, LM-head argmax and
    acceptance run on the GPU; only the toy model's q/k/v/hidden rows come from the host."""

    def __init__(self, lm: ToyLM, ctx_tokens, max_len, poison=True):
        self.lm = lm
        P = lm.P
        npg = (max_len + P - 1) // P
        num_pages = npg + 3
        pt = torch.from_numpy(np.random.default_rng(99).permutation(num_pages)[:npg].reshape(1, npg).astype(np.int32))
        self.kv = PagedKv(num_pages, lm.Hkv, P, lm.d, pt.cuda(), poison_bits=None if poison else 0)
        self.max_len = max_len
        rows = [lm.qkv(x, p) for p, x in enumerate(ctx_tokens)]
        k_rows = torch.stack([r[1] for r in rows]).cuda()
        v_rows = torch.stack([r[2] for r in rows]).cuda()
        n = len(ctx_tokens)
        self.kv.write_rows(torch.zeros(n, dtype=torch.int32, device=DEV), torch.arange(n, dtype=torch.int32, device=DEV),
                           k_rows, v_rows)
        self.W = lm.W.cuda()
        self.err = torch.zeros(1, dtype=torch.int32, device=DEV)
        self.attn_log = []

    def step(self, fed, pos, k):
        lm = self.lm
        qs, ks, vs = zip(*[lm.qkv(x, pos + j) for j, x in enumerate(fed)])
        q, kn, vn = torch.stack(qs).cuda(), torch.stack(ks).cuda(), torch.stack(vs).cuda()
        pos_d = torch.tensor([pos], dtype=torch.int32, device=DEV)
        bnd.spec_kv_append(self.kv.desc, pos_d, 1, k, kn, vn, self.err)
        out = torch.empty((k + 1, lm.Hq, lm.d), dtype=torch.bfloat16, device=DEV)
        ws = torch.zeros(bnd.spec_verify_attn_workspace(self.kv.desc, 1, k, lm.Hq, self.max_len), dtype=torch.uint8,
                         device=DEV)
        bnd.spec_verify_attn(self.kv.desc, pos_d, 1, k, lm.Hq, q, 1 / math.sqrt(lm.d), out, ws, self.max_len, self.err)
        o = out.cpu()
        assert torch.isfinite(o.float()).all()
        self.attn_log.append(o)
        hid = torch.stack([lm.hidden(x, pos + j, lm.target(x, pos + j, o[j])) for j, x in enumerate(fed)]).cuda()
        ids = torch.empty(k + 1, dtype=torch.int32, device=DEV)
        bnd.spec_lmhead_argmax(hid, self.W, ids, lm_ws(k + 1, lm.V, lm.H), dev_err=self.err)
        i32 = dict(dtype=torch.int32, device=DEV)
        toks, n, a, npos, nxt = torch.empty((1, k + 1), **i32), *(torch.empty(1, **i32) for _ in range(4))
        drafts = torch.tensor([fed[1:]], dtype=torch.int32, device=DEV)
        bnd.spec_accept(drafts, ids, pos_d, 1, k, toks, n, a, npos, nxt)
        torch.cuda.synchronize()
        assert int(self.err.item()) == 0
        nn = int(n.item())
        assert int(npos.item()) == pos + nn
        return toks[0, :nn].cpu().tolist(), int(a.item())


@pytest.mark.parametrize("k", [1, 4, 7])
def test_gpu_spec_stream_equals_oracle_greedy(k):
    """Cross-check with the oracle: the toy stream ignores attention bits here, so the
    GPU speculative loop must reproduce the oracle's one-row greedy stream exactly."""
    lm = ToyLM(use_attn=False)
    ctx = [int(t) for t in np.random.default_rng(5).integers(0, lm.V, 33)]
    n_tok = 60
    ref = run_greedy(OracleSide(orc, lm, ctx, 33 + n_tok + 20), lm, ctx[-1] + 1, 33, n_tok + k + 1)
    got, acc = run_spec(GpuSide(lm, ctx, 33 + n_tok + 20), lm, ctx[-1] + 1, 33, n_tok, k, ref)
    assert got == ref[:n_tok]
    assert 0 < sum(acc) < k * len(acc)


@pytest.mark.parametrize("k", [2, 6])
def test_gpu_spec_stream_equals_gpu_greedy_through_attention_bits(k):
    """The stream depends on the attention output's bits: the batched verify must give
    each accepted row exactly the bytes of a one-row verify (row invariance), with NaN in
    every unattended slot, and the same bytes again with a zero-filled pool."""
    lm = ToyLM(use_attn=True)
    ctx = [int(t) for t in np.random.default_rng(6).integers(0, lm.V, 1500)]
    n_tok = 50
    L = 1500 + n_tok + 20
    ref = run_greedy(GpuSide(lm, ctx, L), lm, ctx[-1] + 1, 1500, n_tok + k + 1)
    got, acc = run_spec(GpuSide(lm, ctx, L), lm, ctx[-1] + 1, 1500, n_tok, k, ref)
    assert got == ref[:n_tok]
    assert 0 < sum(acc) < k * len(acc)
    s1, s0 = GpuSide(lm, ctx, L), GpuSide(lm, ctx, L, poison=False)
    g1, _ = run_spec(s1, lm, ctx[-1] + 1, 1500, 20, k, ref)
    g0, _ = run_spec(s0, lm, ctx[-1] + 1, 1500, 20, k, ref)
    assert g1 == g0
    for a1, a0 in zip(s1.attn_log, s0.attn_log):
        assert torch.equal(a1.view(torch.int16), a0.view(torch.int16))

"""The timeout path of the bounded pipeline waits, on the GPU, without a fault.

Every wait of the attention and LM-head kernels gives up after a limit (1 s by default).
The test hook spec_test_set_wait_limit shortens it to 1 ns for the next launches, so the
first wait that has to wait at all (the S MMA for its first K tile, which comes from HBM)
gives up: the kernel must raise SPEC_DEVERR_TIMEOUT in dev_err, let what it issued land,
free its TMEM and exit. Then, with the default limit back and the attention workspace
zeroed again (as the header asks after a timeout), the same calls must give the oracle's
results: the context is still usable."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle as orc
from gpu_harness import DEV, assert_attn_close, attn_ws, gpu_pool, lm_ws, oracle_pool
from greedy_speculative_decode_spec_gb300 import _binding as bnd
from greedy_speculative_decode_spec_gb300.workloads import WORKLOADS, bits, scaled, verify_inputs

pytestmark = pytest.mark.gpu

CASES = {
    "bf16": scaled(WORKLOADS["batched_branches_shared_pool"], B=3, ctx_range=(300, 2100), V=3001, H=520, num_pages=512,
                   seed=31),
    "fp8": scaled(WORKLOADS["long_context_fp8"], B=2, ctx=(1500, 700), V=2050, H=200, num_pages=140, seed=32),
}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from greedy_speculative_decode_spec_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    bnd.lib()
    yield
    bnd.spec_test_set_wait_limit(0)


def _attention(gkv, vi, ws, err):
    c = vi.cfg
    out = torch.empty((c.B * (c.k + 1), c.Hq, c.d), dtype=torch.bfloat16, device=DEV)
    bnd.spec_verify_attn(gkv.desc, vi.pos.cuda(), c.B, c.k, c.Hq, vi.q.cuda(), 1.0 / math.sqrt(c.d), out, ws,
                         vi.max_pos, dev_err=err)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("name", list(CASES))
def test_attention_wait_timeout_is_reported_and_the_context_stays_usable(name):
    vi = verify_inputs(CASES[name])
    c = vi.cfg
    gkv = gpu_pool(vi)
    okv = oracle_pool(vi)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    # the verify rows' own K/V, as in a step (the attention reads slots pos .. pos+k)
    bnd.spec_kv_append(gkv.desc, vi.pos.cuda(), c.B, c.k, vi.k_new.cuda(), vi.v_new.cuda(), err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert orc.kv_append(okv, vi.pos.numpy(), c.B, c.k, bits(vi.k_new), bits(vi.v_new)) == 0
    ws = attn_ws(gkv, c.B, c.k, c.Hq, vi.max_pos)
    bnd.spec_test_set_wait_limit(1)
    try:
        _attention(gkv, vi, ws, err)
    finally:
        bnd.spec_test_set_wait_limit(0)
    assert int(err.item()) & bnd.DEVERR_TIMEOUT, f"no timeout reported (dev_err = {int(err.item())})"
    # the context is usable: a CUDA call succeeds, then the same call with the default limit
    # and a re-zeroed workspace matches the oracle
    torch.cuda.synchronize()
    ws.zero_()
    err.zero_()
    out = _attention(gkv, vi, ws, err)
    assert int(err.item()) == 0
    ref, oe = orc.verify_attn(okv, vi.pos.numpy(), c.B, c.k, c.Hq, bits(vi.q), 1.0 / math.sqrt(c.d))
    assert oe == 0
    assert_attn_close(out, ref)


def test_lmhead_wait_timeout_is_reported_and_the_context_stays_usable():
    g = torch.Generator().manual_seed(33)
    M, V, H = 20, 4099, 512
    hidden = (torch.randn(M, H, generator=g) * 0.5).to(torch.bfloat16)
    W = (torch.randn(V, H, generator=g) * 0.05).to(torch.bfloat16)
    hd, Wd = hidden.to(DEV), W.to(DEV)
    ids = torch.empty(M, dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = lm_ws(M, V, H)
    bnd.spec_test_set_wait_limit(1)
    try:
        bnd.spec_lmhead_argmax(hd, Wd, ids, ws, dev_err=err)
        torch.cuda.synchronize()
    finally:
        bnd.spec_test_set_wait_limit(0)
    assert int(err.item()) & bnd.DEVERR_TIMEOUT, f"no timeout reported (dev_err = {int(err.item())})"
    torch.cuda.synchronize()
    ws.zero_()
    err.zero_()
    bnd.spec_lmhead_argmax(hd, Wd, ids, ws, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref_ids, _, _, oe = orc.lmhead_argmax(bits(hidden), bits(W))
    assert oe == 0
    assert np.array_equal(ids.cpu().numpy(), ref_ids)

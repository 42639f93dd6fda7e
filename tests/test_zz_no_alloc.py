"""spec_lmhead_argmax_static (the LM head without a caller workspace) against
spec_lmhead_argmax on the same inputs, two calls in a row. Collected last on purpose: it
must pass both in a fresh process and after everything else has run."""
from __future__ import annotations

import pytest
import torch

from greedy_speculative_decode_spec_gb300 import _binding as bnd
from greedy_speculative_decode_spec_gb300.workloads import make_lm_head, planted_hidden

DEV = "cuda"


def _case(V, H, M, seed):
    W = make_lm_head(V, H, seed, DEV)
    g = torch.Generator(device=DEV)
    g.manual_seed(seed + 1)
    planted = torch.randint(0, V, (M,), generator=g, device=DEV)
    hidden = planted_hidden(W, planted, g, DEV)
    return W, hidden, planted


def _with_workspace(W, hidden, d2t=None, d2t_limit=0):
    M = hidden.shape[0]
    ws = torch.zeros(bnd.spec_lmhead_workspace(M, W.shape[0], W.shape[1]), dtype=torch.uint8, device=DEV)
    ids = torch.empty(M, dtype=torch.int32, device=DEV)
    mx = torch.empty(M, dtype=torch.float32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    bnd.spec_lmhead_argmax(hidden, W, ids, ws, d2t=d2t, d2t_limit=d2t_limit, max_logit=mx, dev_err=err)
    torch.cuda.synchronize()
    return ids, mx, int(err.item())


def _static(W, hidden, d2t=None, d2t_limit=0):
    M = hidden.shape[0]
    ids = torch.full((M,), -7, dtype=torch.int32, device=DEV)
    mx = torch.full((M,), float("nan"), dtype=torch.float32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    bnd.spec_lmhead_argmax_static(hidden, W, ids, d2t=d2t, d2t_limit=d2t_limit, max_logit=mx, dev_err=err)
    torch.cuda.synchronize()
    return ids, mx, int(err.item())


@pytest.mark.gpu
@pytest.mark.parametrize("V,H,M", [(1024, 256, 4), (151936, 2048, 5), (32768, 4096, 64)])
def test_static_scratch_matches_workspace_two_calls(V, H, M):
    W, hidden, planted = _case(V, H, M, seed=2024 + M)
    want_ids, want_mx, e = _with_workspace(W, hidden)
    assert e == 0
    assert torch.equal(want_ids.long(), planted.long())
    ids, mx, e = _static(W, hidden)  # the first call may set the scratch up
    assert e == 0 and torch.equal(ids, want_ids)
    torch.testing.assert_close(mx, want_mx, rtol=0, atol=0)
    # the calls that follow allocate no device memory: neither through torch nor by the driver
    torch.cuda.synchronize()
    before_torch = torch.cuda.memory_allocated()
    before_free = torch.cuda.mem_get_info()[0]
    for _ in range(2):  # each call finds the counter the one before left at zero
        ids, mx, e = _static(W, hidden)
        assert e == 0
        assert torch.equal(ids, want_ids)
        torch.testing.assert_close(mx, want_mx, rtol=0, atol=0)
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == before_torch
    assert torch.cuda.mem_get_info()[0] == before_free


@pytest.mark.gpu
def test_static_scratch_with_d2t():
    V, H, M = 4096, 512, 16
    W, hidden, planted = _case(V, H, M, seed=77)
    d2t = (torch.arange(V, dtype=torch.int32, device=DEV) * 7 + 3) % 100003
    want = _with_workspace(W, hidden, d2t=d2t, d2t_limit=100003)
    for _ in range(2):
        got = _static(W, hidden, d2t=d2t, d2t_limit=100003)
        assert got[2] == 0 and torch.equal(got[0], want[0])
        torch.testing.assert_close(got[1], want[1], rtol=0, atol=0)


@pytest.mark.gpu
def test_static_scratch_rejects_requests_beyond_its_size():
    # M = 256 rows over a vocabulary wide enough for 1024 CTAs needs 2 MB of keys
    V, H, M = 1024 * 128, 64, 256
    assert bnd.spec_lmhead_workspace(M, V, H) > bnd.SPEC_LMHEAD_STATIC_SCRATCH_BYTES
    W = torch.zeros((V, H), dtype=torch.bfloat16, device=DEV)
    hidden = torch.zeros((M, H), dtype=torch.bfloat16, device=DEV)
    ids = torch.empty(M, dtype=torch.int32, device=DEV)
    with pytest.raises(bnd.SpecError) as ex:
        bnd.spec_lmhead_argmax_static(hidden, W, ids)
    assert ex.value.status == bnd.ERR_WORKSPACE

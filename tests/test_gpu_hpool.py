"""The draft head's remembered hidden rows (f1) on the GPU: spec_h_gather / spec_h_scatter
against the oracle bit for bit, invalid slots, and a step-graph cache keyed by (k, B, splits)
whose replays equal eager steps (span-02 engine/crates/model/src/spec.rs, `Spec::body_inner`
and `Spec::step_chunk`)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as orc
from gpu_harness import DEV
from greedy_speculative_decode_spec_gb300 import _binding as bnd
from greedy_speculative_decode_spec_gb300.step import StepGraphCache
from greedy_speculative_decode_spec_gb300.workloads import bits

pytestmark = pytest.mark.gpu


def _bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)


@pytest.mark.parametrize("S,H,B", [(300, 4096, 64), (17, 33, 5), (1, 8, 1)])
def test_gather_scatter_match_oracle(S, H, B):
    rng = np.random.default_rng(S + H)
    hpool = rng.integers(0, 1 << 16, (S, H)).astype(np.uint16)
    hslot = rng.permutation(S)[:B].astype(np.int32)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    g_pool = _bf16(hpool).to(DEV)
    g_slot = torch.from_numpy(hslot).to(DEV)
    h = torch.empty((B, H), dtype=torch.bfloat16, device=DEV)
    bnd.spec_h_gather(h, g_pool, g_slot, dev_err=err)
    torch.cuda.synchronize()
    want, oe = orc.h_gather(hpool, hslot)
    assert int(err.item()) == 0 and oe == 0
    assert np.array_equal(bits(h.cpu()), want)
    h_new = rng.integers(0, 1 << 16, (B, H)).astype(np.uint16)
    bnd.spec_h_scatter(g_pool, _bf16(h_new).to(DEV), g_slot, dev_err=err)
    torch.cuda.synchronize()
    assert orc.h_scatter(hpool, h_new, hslot) == 0
    assert int(err.item()) == 0
    assert np.array_equal(bits(g_pool.cpu()), hpool)


def test_invalid_slots_are_reported_and_skipped():
    rng = np.random.default_rng(3)
    S, H, B = 40, 64, 6
    hpool = rng.integers(0, 1 << 16, (S, H)).astype(np.uint16)
    hslot = np.array([3, -1, 7, S, 0, 39], np.int32)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    sentinel = np.full((B, H), 0x1234, np.uint16)
    h = _bf16(sentinel.copy()).to(DEV)
    bnd.spec_h_gather(h, _bf16(hpool).to(DEV), torch.from_numpy(hslot).to(DEV), dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == bnd.DEVERR_SLOT
    want, oe = orc.h_gather(hpool, hslot)
    assert oe == orc.ERR_SLOT
    got = bits(h.cpu())
    ok = (hslot >= 0) & (hslot < S)
    assert np.array_equal(got[ok], want[ok]) and np.array_equal(got[~ok], sentinel[~ok])


def test_step_graph_cache_replays_equal_eager_steps():
    """A step (gather the branch rows, change them, scatter them back) captured per key
    (k, B, splits) and replayed: the pool after N replays equals N eager steps; a second key
    gets its own graph."""
    S, H = 64, 256
    rng = np.random.default_rng(11)
    base = _bf16(rng.integers(0, 1 << 16, (S, H)).astype(np.uint16) & 0x3FFF).to(DEV)  # finite, < 2
    keys = {(3, 8, 2): torch.arange(0, 16, 2, dtype=torch.int32, device=DEV),
            (4, 5, 1): torch.tensor([63, 1, 30, 7, 12], dtype=torch.int32, device=DEV)}
    err = torch.zeros(1, dtype=torch.int32, device=DEV)

    def make_step(pool, slot, h):
        def step():
            bnd.spec_h_gather(h, pool, slot, dev_err=err)
            h.mul_(0.5).add_(1.0)
            bnd.spec_h_scatter(pool, h, slot, dev_err=err)
        return step

    for key, slot in keys.items():
        B = key[1]
        pool_e, pool_g = base.clone(), base.clone()
        h_e = torch.empty((B, H), dtype=torch.bfloat16, device=DEV)
        h_g = torch.empty((B, H), dtype=torch.bfloat16, device=DEV)
        eager = make_step(pool_e, slot, h_e)
        cache = StepGraphCache()
        for _ in range(6):
            eager()
            cache.run(key, make_step(pool_g, slot, h_g))
        torch.cuda.synchronize()
        assert cache.captured(key), "the step should have been captured"
        assert torch.equal(pool_e.view(torch.int16), pool_g.view(torch.int16))
    assert int(err.item()) == 0

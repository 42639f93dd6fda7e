"""The attention's launch plan (host arithmetic, no GPU): every shape the library accepts
gets a plan that fits the SM's shared memory, TMEM and barrier region, spreads the queries
over the TMEM lane quadrants, and keeps split boundaries independent of the batch."""
from __future__ import annotations

import itertools

import pytest

from greedy_speculative_decode_spec_gb300 import _binding as bnd
from greedy_speculative_decode_spec_gb300.workloads import DRAFT_CONFIG, WORKLOADS, config4_verify

SMEM_LIMIT = 227 * 1024


def _plan(P, d, Hkv, G, B, k, max_pos, fp8=False, num_pages=4096):
    kv = bnd.kv_shape(num_pages, (max_pos + P - 1) // P + 1, P, Hkv, d, fp8)
    return bnd.spec_verify_attn_plan(kv, B, k, G * Hkv, max_pos)


def _check_plan(pl, P, d, Hkv, G, B, k, max_pos, fp8):
    n_q = (k + 1) * G
    assert pl["smem"] <= SMEM_LIMIT
    # four lane quadrants hold the queries, or two when four copies would leave the
    # operand ring too shallow (long head dims)
    assert pl["copies"] * pl["quadrants_per_copy"] == 4 or (pl["copies"], pl["quadrants_per_copy"]) == (2, 1)
    assert pl["quadrants_per_copy"] == (2 if n_q > 32 else 1)
    assert pl["p_rows"] >= min(n_q, 32) and pl["p_rows"] % 16 == 0
    assert pl["q_rows"] == (pl["copies"] - 1) * 32 * pl["quadrants_per_copy"] + pl["p_rows"] <= 128
    # two stages are enough to make progress: S and P.V each free their own stages
    assert pl["ring_stages"] >= 2
    assert (pl["raw_stages"] >= 2) if fp8 else (pl["raw_stages"] == 0)
    assert pl["q_buffers"] in (1, 2) and pl["o_buffers"] in (1, 2)
    assert 256 + pl["o_buffers"] * d <= 512                      # TMEM columns: 2 S buffers + O
    assert pl["barrier_bytes"] <= pl["barrier_bytes_reserved"]
    assert pl["split_keys"] == (256 if Hkv <= 2 else 512 if Hkv <= 4 else 1024)
    assert pl["n_splits"] == -(-max_pos // pl["split_keys"])
    assert pl["n_units"] == B * Hkv * pl["n_splits"]
    assert pl["tma_rows"] == (min(P, 128) if fp8 and P >= 64 else 0)


@pytest.mark.parametrize("d,fp8", [(64, False), (64, True), (128, False), (128, True), (256, False), (256, True)])
def test_plans_fit_for_every_accepted_shape(d, fp8):
    for P, Hkv, G, k in itertools.product((1, 8, 16, 64, 256, 1024), (1, 2, 8), (1, 2, 4, 5, 8, 16), (0, 1, 3, 6, 15)):
        n_q = (k + 1) * G
        if n_q > 64:
            with pytest.raises(bnd.SpecError):
                _plan(P, d, Hkv, G, 3, k, 5000, fp8)
            continue
        pl = _plan(P, d, Hkv, G, 3, k, 5000, fp8)
        _check_plan(pl, P, d, Hkv, G, 3, k, 5000, fp8)


def test_split_geometry_does_not_depend_on_the_batch():
    """Row invariance starts here: a row's split boundaries are the same for any B and k."""
    for Hkv in (1, 2, 4, 8):
        sk = {_plan(16, 128, Hkv, 4, B, k, 9000)["split_keys"] for B in (1, 5, 32) for k in (0, 3, 15 // 4)}
        assert len(sk) == 1


def test_plans_of_the_benchmark_workloads():
    """The plans the measured numbers were taken with (see the ncu summaries)."""
    want = {
        "single_stream_mtp_verify": dict(copies=2, quadrants_per_copy=2, split_layout=1, split_keys=256, n_units=2 * 17, tma_rows=0),
        "batched_branches_shared_pool": dict(copies=4, quadrants_per_copy=1, q_rows=128, ring_stages=5, q_buffers=1, o_buffers=2,
                split_keys=1024, tma_rows=0),
        "long_context_fp8": dict(copies=4, quadrants_per_copy=1, q_rows=128, ring_stages=3, raw_stages=4, q_buffers=1,
                split_keys=1024, tma_rows=64),
    }
    for name, w in want.items():
        c = WORKLOADS[name]
        ctx = max(c.ctx) if c.ctx else c.ctx_range[1]
        max_pos = ctx + c.k + 1 + 4
        kv = bnd.kv_shape(c.num_pages or 4096, -(-max_pos // c.P), c.P, c.Hkv, c.d, c.kv_dtype == "fp8")
        pl = bnd.spec_verify_attn_plan(kv, c.B, c.k, c.Hq, max_pos)
        for key, v in w.items():
            if key == "n_units":
                continue
            assert pl[key] == v, (name, key, pl[key], v)
        assert pl["smem"] <= SMEM_LIMIT
    c4 = config4_verify(DRAFT_CONFIG)
    kv = bnd.kv_shape(c4.num_pages, 600, c4.P, c4.Hkv, c4.d)
    assert bnd.spec_verify_attn_plan(kv, c4.B, c4.k, c4.Hq, 9000)["copies"] == 4


def test_plan_rejects_what_the_call_rejects():
    kv = bnd.kv_shape(64, 16, 16, 2, 128)
    with pytest.raises(bnd.SpecError):
        bnd.spec_verify_attn_plan(kv, 0, 1, 4, 100)        # B < 1
    with pytest.raises(bnd.SpecError):
        bnd.spec_verify_attn_plan(kv, 1, 1, 5, 100)        # q heads not a multiple of kv heads
    with pytest.raises(bnd.SpecError):
        bnd.spec_verify_attn_plan(kv, 1, 16, 4, 100)       # k above the maximum
    with pytest.raises(bnd.SpecError):
        bnd.spec_verify_attn_plan(bnd.kv_shape(64, 16, 16, 2, 96), 1, 1, 4, 100)  # head_dim
    with pytest.raises(bnd.SpecError):
        bnd.spec_verify_attn_plan(bnd.kv_shape(64, 16, 12, 2, 128), 1, 1, 4, 100)  # page size

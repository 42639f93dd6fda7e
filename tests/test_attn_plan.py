"""The attention's launch plan (host arithmetic, no GPU): every shape the library accepts
gets a plan that fits the SM's shared memory, TMEM and barrier region, and keeps split
boundaries independent of the batch."""
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
    nsub = max(1, d // 128)
    assert pl["smem"] <= SMEM_LIMIT
    # the queries of a (branch, kv head) are the MMAs' N side, padded to 16
    assert pl["nq"] == -(-n_q // 16) * 16 <= 128
    # one whole tile of K (every head-dim half) and of V is the least that can make progress:
    # S frees K stages, P.V frees V stages, the converters free raw V stages
    assert pl["k_stages"] >= nsub and pl["v_stages"] >= nsub
    assert (pl["raw_stages"] >= nsub) if fp8 else (pl["raw_stages"] == 0)
    assert pl["s_buffers"] >= 1 and pl["p_buffers"] in (2, 3) and pl["tile_group"] in (1, 2)
    assert pl["q_buffers"] in (1, 2) and pl["o_buffers"] in (1, 2)
    # TMEM: S buffers of a tile group's nq columns per tile, then per O buffer nsub blocks
    # of O and one of row sums, then 16 columns of the row-sum MMAs' ones operand
    assert pl["tmem_cols"] == pl["nq"] * (pl["s_buffers"] * pl["tile_group"] + pl["o_buffers"] * (nsub + 1)) + 16 <= 512
    assert pl["barrier_bytes"] <= pl["barrier_bytes_reserved"]
    assert pl["split_keys"] == (256 if Hkv <= 2 else 512 if Hkv <= 4 else (2048 if fp8 else 1024))
    assert pl["n_splits"] == -(-max_pos // pl["split_keys"])
    assert pl["n_units"] == B * Hkv * pl["n_splits"]
    assert pl["tma_rows"] == (min(P, 128) if fp8 else 0)


@pytest.mark.parametrize("d,fp8", [(64, False), (64, True), (128, False), (128, True), (256, False), (256, True)])
def test_plans_fit_for_every_accepted_shape(d, fp8):
    n_ok = 0
    for P, Hkv, G, k in itertools.product((1, 4, 8, 16, 64, 256, 1024), (1, 2, 8),
                                          (1, 2, 4, 5, 8, 16), (0, 1, 3, 6, 15)):
        n_q = (k + 1) * G
        if n_q > 128 or (fp8 and P < 8):
            with pytest.raises(bnd.SpecError) as ex:
                _plan(P, d, Hkv, G, 3, k, 5000, fp8)
            assert ex.value.status == bnd.ERR_UNSUPPORTED
            continue
        try:
            pl = _plan(P, d, Hkv, G, 3, k, 5000, fp8)
        except bnd.SpecError as ex:
            # only the widest query groups on the longest head dim may lack a plan
            assert ex.status == bnd.ERR_UNSUPPORTED and d == 256 and n_q > 64
            continue
        _check_plan(pl, P, d, Hkv, G, 3, k, 5000, fp8)
        n_ok += 1
    assert n_ok > 0


def test_every_query_group_up_to_64_is_planned():
    """(k+1)*G up to 64 query vectors per kv head is planned for every head dim and dtype."""
    for d, fp8, nq in itertools.product((64, 128, 256), (False, True), (1, 16, 17, 48, 64)):
        pl = _plan(64, d, 8, nq, 4, 0, 4096, fp8)
        _check_plan(pl, 64, d, 8, nq, 4, 0, 4096, fp8)


def test_split_geometry_does_not_depend_on_the_batch():
    """Row invariance starts here: a row's split boundaries are the same for any B and k."""
    for Hkv in (1, 2, 4, 8):
        sk = {_plan(16, 128, Hkv, 4, B, k, 9000)["split_keys"] for B in (1, 5, 32) for k in (0, 3, 15 // 4)}
        assert len(sk) == 1


def test_plans_of_the_benchmark_workloads():
    """The plans the measured numbers were taken with (see the ncu summaries)."""
    want = {
        "single_stream_mtp_verify": dict(nq=48, split_keys=256, tma_rows=0),
        "batched_branches_shared_pool": dict(nq=32, tile_group=2, s_buffers=2, o_buffers=2, split_keys=1024,
                                             tma_rows=0),
        "long_context_fp8": dict(nq=32, tile_group=2, s_buffers=2, split_keys=2048, tma_rows=64),
    }
    for name, w in want.items():
        c = WORKLOADS[name]
        ctx = max(c.ctx) if c.ctx else c.ctx_range[1]
        max_pos = ctx + c.k + 1 + 4
        kv = bnd.kv_shape(c.num_pages or 4096, -(-max_pos // c.P), c.P, c.Hkv, c.d, c.kv_dtype == "fp8")
        pl = bnd.spec_verify_attn_plan(kv, c.B, c.k, c.Hq, max_pos)
        for key, v in w.items():
            assert pl[key] == v, (name, key, pl[key], v)
        assert pl["smem"] <= SMEM_LIMIT
    c4 = config4_verify(DRAFT_CONFIG)
    kv = bnd.kv_shape(c4.num_pages, 600, c4.P, c4.Hkv, c4.d)
    assert bnd.spec_verify_attn_plan(kv, c4.B, c4.k, c4.Hq, 9000)["nq"] == 32


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
    with pytest.raises(bnd.SpecError):
        bnd.spec_verify_attn_plan(bnd.kv_shape(64, 16, 4, 2, 128, True), 1, 1, 4, 100)  # FP8 pages < 8

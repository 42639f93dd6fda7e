"""Several ranks on the CPU (gloo, world size 2): independent verify replicas, and the
merge of a vocabulary-sharded LM-head argmax. Ranks are spawned processes; nothing here
touches a GPU."""
from __future__ import annotations

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

WORLD = 2


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, fn, args):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        fn(rank, world, *args)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def _spawn(fn, *args):
    mp.spawn(_worker, args=(WORLD, _free_port(), fn, args), nprocs=WORLD, join=True)


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


# ---- vocabulary-sharded argmax -----------------------------------------------------------------

def _lm_inputs(V=1001, H=64, M=12, seed=7):
    g = torch.Generator().manual_seed(seed)
    W = (0.02 * torch.randn((V, H), generator=g)).to(torch.bfloat16)
    mid = V // 2
    # duplicated rows: tied maxima across the shard boundary and inside one shard
    W[mid + 10] = W[3]
    W[mid + 40] = W[mid + 20]
    planted = torch.randint(0, V, (M,), generator=g)
    planted[0], planted[1], planted[2] = mid + 10, mid + 40, mid - 1
    Wf = W.float()
    hid = 8 * Wf[planted] / Wf[planted].norm(dim=1, keepdim=True) + 0.1 * torch.randn((M, H), generator=g)
    return W, hid.to(torch.bfloat16)


def _sharded_argmax(rank, world):
    import oracle as orc
    from greedy_speculative_decode_spec_gb300.shard import merge_shard_argmax, shard_bounds
    W, hid = _lm_inputs()
    V = W.shape[0]
    v0, v1 = shard_bounds(V, world, rank)
    ids, mx, _, err = orc.lmhead_argmax(_bits(hid), _bits(W[v0:v1]))
    assert err == 0
    mine = torch.tensor(np.stack([np.asarray(mx, np.float64), np.asarray(ids, np.int64) + v0]), dtype=torch.float64)
    got = [torch.empty_like(mine) for _ in range(world)]
    dist.all_gather(got, mine)
    max_logit = np.stack([g[0].numpy() for g in got]).astype(np.float32)
    gids = np.stack([g[1].numpy() for g in got]).astype(np.int64)
    merged = merge_shard_argmax(max_logit, gids)
    want, _, _, err = orc.lmhead_argmax(_bits(hid), _bits(W))
    assert err == 0
    np.testing.assert_array_equal(merged, np.asarray(want, np.int64))
    assert merged[0] == 3           # tie across the boundary: the lower index (shard 0)
    assert merged[1] == V // 2 + 20  # tie inside shard 1: the lower index


def test_vocab_sharded_argmax_merge_equals_unsharded(orc):
    _spawn(_sharded_argmax)


def test_shard_bounds_cover_the_vocabulary():
    from greedy_speculative_decode_spec_gb300.shard import shard_bounds
    for V in (1, 7, 1001, 151936):
        for world in (1, 2, 3, 8):
            spans = [shard_bounds(V, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == V
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            assert max(b - a for a, b in spans) - min(b - a for a, b in spans) <= 1


def test_merge_marks_failed_rows():
    from greedy_speculative_decode_spec_gb300.shard import merge_shard_argmax
    out = merge_shard_argmax(np.array([[1.0, 2.0], [1.0, 3.0]]), np.array([[5, 1], [-1, 9]]))
    np.testing.assert_array_equal(out, [-1, 9])


# ---- independent replicas ------------------------------------------------------------------------

def _replicas(rank, world):
    """Each rank verifies its own branches (a replica: no exchange inside the step); the
    gathered results equal one process verifying all branches, and the whole-job rate is
    set by the slowest rank."""
    import bench
    import oracle as orc
    from greedy_speculative_decode_spec_gb300.workloads import WORKLOADS, verify_inputs
    vi = verify_inputs(WORKLOADS["tiny_verify"])
    c = vi.cfg
    # rank r takes branch copies r, r + world, ... of a 4-branch batch built from workload 0
    drafts = np.asarray(vi.drafts, np.int32)
    ids_all, _, _, err = orc.lmhead_argmax(_bits(vi.hidden), _bits(vi.W))
    assert err == 0
    B_all = 4
    rng = np.random.default_rng(11)
    pos_all = rng.integers(50, 500, B_all).astype(np.int32)
    ids_b = np.tile(np.asarray(ids_all, np.int32), B_all)
    drafts_b = np.concatenate([np.roll(drafts, s, axis=1) for s in range(B_all)])
    mine = list(range(rank, B_all, world))
    toks, n, a, npos, nxt = orc.accept(drafts_b[mine], ids_b.reshape(B_all, -1)[mine].reshape(-1), pos_all[mine],
                                       len(mine), c.k)
    local = torch.tensor(np.concatenate([np.asarray(n), np.asarray(npos), np.asarray(nxt)]), dtype=torch.int64)
    got = [torch.empty_like(local) for _ in range(world)]
    dist.all_gather(got, local)
    toks1, n1, a1, npos1, nxt1 = orc.accept(drafts_b, ids_b, pos_all, B_all, c.k)
    for r in range(world):
        idx = list(range(r, B_all, world))
        g = got[r].numpy().reshape(3, -1)
        np.testing.assert_array_equal(g[0], np.asarray(n1)[idx])
        np.testing.assert_array_equal(g[1], np.asarray(npos1)[idx])
        np.testing.assert_array_equal(g[2], np.asarray(nxt1)[idx])
    # the bench's whole-job rate: max step time over ranks
    ms_local = 1.0 + rank
    ms_max, value = bench.replica_rate(ms_local, c.B * (c.k + 1), world, "cpu")
    assert ms_max == 1.0 + (world - 1)
    assert value == pytest.approx(world * c.B * (c.k + 1) / (ms_max * 1e-3))


def test_replicas_equal_one_process(orc):
    _spawn(_replicas)

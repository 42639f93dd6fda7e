"""Shared set-up for the GPU parity tests: the same seeded inputs go to the CUDA library
(through its binding) and to the CPU oracle; each side builds its own KV pool with its
own write routine, and the results are compared."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle as orc
from greedy_speculative_decode_spec_gb300 import _binding as bnd
from greedy_speculative_decode_spec_gb300.step import PagedKv
from greedy_speculative_decode_spec_gb300.workloads import BF16_NAN_BITS, E4M3_NAN_BITS, VerifyInputs, bits

DEV = "cuda"


def attn_tolerance(ref: np.ndarray) -> float:
    """max|gpu - oracle| <= 1e-2 * max|oracle| + 1e-3 (the stated float tolerance)."""
    return 1e-2 * float(np.abs(ref).max()) + 1e-3


def assert_attn_close(gpu_bf16: torch.Tensor, ref: np.ndarray, what="attention"):
    g = gpu_bf16.detach().float().cpu().numpy().astype(np.float64).reshape(ref.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite GPU output"
    err = float(np.abs(g - ref).max())
    tol = attn_tolerance(ref)
    assert err <= tol, f"{what}: max abs err {err:.3e} > tolerance {tol:.3e}"
    return err


def oracle_pool(vi: VerifyInputs, poison=True) -> orc.KvPool:
    c = vi.cfg
    shape = vi.pool_shape
    if c.kv_dtype == "bf16":
        fill = BF16_NAN_BITS if poison else 0
        kp, vp = np.full(shape, fill, np.uint16), np.full(shape, fill, np.uint16)
    else:
        fill = E4M3_NAN_BITS if poison else 0
        kp, vp = np.full(shape, fill, np.uint8), np.full(shape, fill, np.uint8)
    kv = orc.KvPool(kp, vp, vi.page_table.numpy(), c.P,
                    None if vi.k_scale is None else vi.k_scale.numpy(),
                    None if vi.v_scale is None else vi.v_scale.numpy())
    err = orc.kv_write_rows(kv, vi.ctx_branch.numpy(), vi.ctx_pos.numpy(), bits(vi.ctx_k), bits(vi.ctx_v))
    assert err == 0
    return kv


def gpu_pool(vi: VerifyInputs, poison=True) -> PagedKv:
    c = vi.cfg
    fp8 = c.kv_dtype == "fp8"
    pb = None if poison else 0
    kv = PagedKv(vi.num_pages, c.Hkv, c.P, c.d, vi.page_table.cuda(), fp8=fp8, poison_bits=pb,
                 k_scale=vi.k_scale, v_scale=vi.v_scale)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    kv.write_rows(vi.ctx_branch.cuda(), vi.ctx_pos.cuda(), vi.ctx_k.cuda(), vi.ctx_v.cuda(), dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return kv


def pool_bits(kv: PagedKv):
    if kv.fp8:
        return kv.k.cpu().numpy(), kv.v.cpu().numpy()
    return bits(kv.k), bits(kv.v)


def assert_pools_equal(gkv: PagedKv, okv: orc.KvPool):
    gk, gv = pool_bits(gkv)
    assert np.array_equal(gk, okv.k_pool), f"K pool differs at {np.argwhere(gk != okv.k_pool)[:5]}"
    assert np.array_equal(gv, okv.v_pool), f"V pool differs at {np.argwhere(gv != okv.v_pool)[:5]}"


def lm_ws(M, V, H):
    return torch.zeros(bnd.spec_lmhead_workspace(M, V, H), dtype=torch.uint8, device=DEV)


def attn_ws(kv: PagedKv, B, k, Hq, max_pos):
    return torch.zeros(max(bnd.spec_verify_attn_workspace(kv.desc, B, k, Hq, max_pos), 256), dtype=torch.uint8,
                       device=DEV)


def gpu_attention(kv: PagedKv, pos, B, k, Hq, q, max_pos, scale=None):
    d = kv.head_dim
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    out = torch.empty((B * (k + 1), Hq, d), dtype=torch.bfloat16, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    bnd.spec_verify_attn(kv.desc, pos, B, k, Hq, q, scale, out, attn_ws(kv, B, k, Hq, max_pos), max_pos,
                         dev_err=err)
    torch.cuda.synchronize()
    return out, int(err.item())


def gpu_lmhead(hidden, W, d2t=None, d2t_limit=0):
    M, H = hidden.shape
    V = W.shape[0]
    ids = torch.empty(M, dtype=torch.int32, device=DEV)
    mx = torch.empty(M, dtype=torch.float32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    bnd.spec_lmhead_argmax(hidden, W, ids, lm_ws(M, V, H), d2t=d2t, d2t_limit=d2t_limit, max_logit=mx, dev_err=err)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), mx.cpu().numpy(), int(err.item())


def gpu_accept(drafts, ids, pos, B, k, hidden=None):
    i32 = dict(dtype=torch.int32, device=DEV)
    toks = torch.empty((B, k + 1), **i32)
    n, a, npos, nxt = (torch.empty(B, **i32) for _ in range(4))
    h_out = None if hidden is None else torch.empty((B, hidden.shape[1]), dtype=torch.bfloat16, device=DEV)
    bnd.spec_accept(drafts, ids, pos, B, k, toks, n, a, npos, nxt, hidden=hidden, h_out=h_out)
    torch.cuda.synchronize()
    res = [t.cpu().numpy() for t in (toks, n, a, npos, nxt)]
    return res + ([h_out] if hidden is not None else [])

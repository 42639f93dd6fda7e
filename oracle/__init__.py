"""CPU oracle of the batched verify step -- test infrastructure only.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
import this package; the product path (the CUDA library and its binding) never does.

The arithmetic lives in ``oracle.c`` (plain C, fp64, straight loops). This module
builds it with gcc and marshals numpy arrays through ctypes; it adds no arithmetic.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "oracle.c"
_LIB = _HERE / "liboracle.so"

ERR_PAGE, ERR_COVER, ERR_TOKEN, ERR_D2T, ERR_POS, ERR_TREE, ERR_SLOT = 1, 2, 4, 8, 16, 32, 64


def build(force: bool = False) -> Path:
    """Compile oracle.c into liboracle.so (OpenMP when the compiler has it)."""
    if _LIB.exists() and not force and _LIB.stat().st_mtime >= _SRC.stat().st_mtime:
        return _LIB
    tmp = _LIB.with_suffix(f".{os.getpid()}.tmp")
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
            "-ffp-contract=off", str(_SRC), "-o", str(tmp), "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB)
    return _LIB


class _Kv(ctypes.Structure):
    _fields_ = [("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p),
                ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
                ("page_table", ctypes.c_void_p),
                ("num_pages", ctypes.c_int32), ("max_pages", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("kv_dtype", ctypes.c_int32)]


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(str(build()))
        _lib.orc_bf16_to_double.restype = ctypes.c_double
        _lib.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
        _lib.orc_double_to_bf16.restype = ctypes.c_uint16
        _lib.orc_double_to_bf16.argtypes = [ctypes.c_double]
        _lib.orc_e4m3_decode.restype = ctypes.c_double
        _lib.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
        _lib.orc_e4m3_encode.restype = ctypes.c_uint8
        _lib.orc_e4m3_encode.argtypes = [ctypes.c_float]
        _lib.orc_threads.restype = ctypes.c_int
        _lib.orc_verify_attn.argtypes = [ctypes.POINTER(_Kv)] + [ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                                                  ctypes.c_int, ctypes.c_void_p, ctypes.c_double,
                                                                  ctypes.c_void_p]
        _lib.orc_verify_attn_items.argtypes = [ctypes.POINTER(_Kv), ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_void_p, ctypes.c_double, ctypes.c_void_p,
                                               ctypes.c_int, ctypes.c_void_p]
        _lib.orc_kv_write_rows.argtypes = [ctypes.POINTER(_Kv), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                           ctypes.c_void_p, ctypes.c_void_p]
        _lib.orc_kv_append.argtypes = [ctypes.POINTER(_Kv), ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_void_p, ctypes.c_void_p]
        _lib.orc_lmhead_argmax.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                                           ctypes.c_void_p, ctypes.c_void_p]
        _lib.orc_lmhead_logits.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_void_p]
        _lib.orc_accept.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int, ctypes.c_int] + [ctypes.c_void_p] * 5
        _lib.orc_verify_attn_tree.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                              ctypes.c_int, ctypes.c_void_p, ctypes.c_double, ctypes.c_void_p,
                                              ctypes.c_void_p]
        _lib.orc_accept_tree.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int, ctypes.c_int] + [ctypes.c_void_p] * 6
        _lib.orc_kv_compact.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int, ctypes.c_int]
        _lib.orc_accept_sample.argtypes = ([ctypes.c_void_p] * 4 + [ctypes.c_int] * 3 + [ctypes.c_double]
                                           + [ctypes.c_void_p] * 7)
        _lib.orc_accept_sample.restype = ctypes.c_int
        _lib.orc_h_gather.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 3
        _lib.orc_h_scatter.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 3
        _lib.orc_accept_stop.argtypes = ([ctypes.c_void_p] * 3 + [ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                          ctypes.c_int] + [ctypes.c_void_p] * 7)
        _lib.orc_mtp_input.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_double, ctypes.c_void_p, ctypes.c_int,
                                                               ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                                               ctypes.c_void_p]
    return _lib


def threads() -> int:
    return int(lib().orc_threads())


def set_threads(n: int) -> None:
    lib().orc_set_threads(int(n))


def _p(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---- number formats -------------------------------------------------------------------

def bf16_to_double(bits: int) -> float:
    return float(lib().orc_bf16_to_double(int(bits) & 0xFFFF))


def double_to_bf16(x: float) -> int:
    return int(lib().orc_double_to_bf16(float(x)))


def e4m3_decode(code: int) -> float:
    return float(lib().orc_e4m3_decode(int(code) & 0xFF))


def e4m3_encode(x: float) -> int:
    return int(lib().orc_e4m3_encode(float(np.float32(x))))


# ---- KV pool ----------------------------------------------------------------------------

class KvPool:
    """Host copy of a paged pool with the library's layout
    [num_pages][Hkv][page_size][d] (uint16 bf16 bits or uint8 E4M3 codes)."""

    def __init__(self, k_pool, v_pool, page_table, page_size, k_scale=None, v_scale=None):
        self.k_pool = np.ascontiguousarray(k_pool)
        self.v_pool = np.ascontiguousarray(v_pool)
        assert self.k_pool.shape == self.v_pool.shape and self.k_pool.ndim == 4
        self.kv_dtype = 0 if self.k_pool.dtype == np.uint16 else 1
        assert self.kv_dtype == 0 or self.k_pool.dtype == np.uint8
        self.page_table = _c(page_table, np.int32)
        self.k_scale = None if k_scale is None else _c(k_scale, np.float32)
        self.v_scale = None if v_scale is None else _c(v_scale, np.float32)
        self.num_pages, self.n_kv_heads, ps, self.head_dim = self.k_pool.shape
        assert ps == page_size
        self.page_size = page_size
        self.max_pages = self.page_table.shape[1]

    def _struct(self) -> _Kv:
        return _Kv(_p(self.k_pool), _p(self.v_pool), _p(self.k_scale), _p(self.v_scale),
                   _p(self.page_table), self.num_pages, self.max_pages, self.page_size,
                   self.n_kv_heads, self.head_dim, self.kv_dtype)


def kv_write_rows(kv: KvPool, row_branch, row_pos, k_rows, v_rows) -> int:
    rb, rp = _c(row_branch, np.int32), _c(row_pos, np.int32)
    kr, vr = _c(k_rows, np.uint16), _c(v_rows, np.uint16)
    s = kv._struct()
    return int(lib().orc_kv_write_rows(ctypes.byref(s), _p(rb), _p(rp), len(rb), _p(kr), _p(vr)))


def kv_append(kv: KvPool, pos, B: int, k: int, k_new, v_new) -> int:
    pos = _c(pos, np.int32)
    kn, vn = _c(k_new, np.uint16), _c(v_new, np.uint16)
    s = kv._struct()
    return int(lib().orc_kv_append(ctypes.byref(s), _p(pos), B, k, _p(kn), _p(vn)))


def verify_attn(kv: KvPool, pos, B: int, k: int, n_q_heads: int, q, scale: float):
    """fp64 outputs [B*(k+1)][Hq][d] and the error bits."""
    pos, q = _c(pos, np.int32), _c(q, np.uint16)
    R = B * (k + 1)
    out = np.empty((R, n_q_heads, kv.head_dim), dtype=np.float64)
    s = kv._struct()
    err = lib().orc_verify_attn(ctypes.byref(s), _p(pos), B, k, n_q_heads, _p(q), float(scale), _p(out))
    return out, int(err)


def chain_masks(B: int, k: int) -> np.ndarray:
    """The ancestor masks of a chain: row j reads verify slots 0..j."""
    return np.tile(((1 << (np.arange(k + 1) + 1)) - 1).astype(np.int32), B).reshape(B, k + 1)


def verify_attn_tree(kv: KvPool, pos, B: int, k: int, n_q_heads: int, q, scale: float, anc_mask):
    """Tree verify attention: row j of branch b reads the committed prefix [0, pos_b) and
    the verify slots pos_b + i with bit i of anc_mask[b][j] set. fp64 [R][Hq][d], errors."""
    pos, q, m = _c(pos, np.int32), _c(q, np.uint16), _c(np.asarray(anc_mask).reshape(-1), np.int32)
    R = B * (k + 1)
    assert m.size == R
    out = np.empty((R, n_q_heads, kv.head_dim), dtype=np.float64)
    s = kv._struct()
    err = lib().orc_verify_attn_tree(ctypes.byref(s), _p(pos), B, k, n_q_heads, _p(q), float(scale), _p(m), _p(out))
    return out, int(err)


def accept_tree(drafts, ids, pos, parent, B: int, k: int):
    """Greedy tree walk: tokens [B][k+1], n, accepted, new_pos, next, path [B][k+1], errors."""
    drafts = _c(np.asarray(drafts).reshape(B, k) if k > 0 else np.zeros((B, 1)), np.int32)
    ids, pos = _c(ids, np.int32), _c(pos, np.int32)
    parent = _c(np.asarray(parent).reshape(B, k + 1), np.int32)
    tokens, path = np.empty((B, k + 1), np.int32), np.empty((B, k + 1), np.int32)
    n, a, npos, nxt = (np.empty(B, np.int32) for _ in range(4))
    err = lib().orc_accept_tree(_p(drafts), _p(ids), _p(pos), _p(parent), B, k, _p(tokens), _p(n), _p(a),
                                _p(npos), _p(nxt), _p(path))
    return tokens, n, a, npos, nxt, path, int(err)


def accept_sample(drafts, logits, q, pos, B: int, k: int, temperature: float, u_acc, u_res):
    """Speculative sampling acceptance with the random numbers given: tokens, n, accepted,
    new_pos, next, error bits (a draft outside [0, V) or with q(d) = 0 is an error and is
    rejected). logits fp32 [B*(k+1)][V]; q fp32 [B][k][V]; u_acc [B][k]; u_res [B]."""
    logits = _c(logits, np.float32)
    V = logits.shape[-1]
    drafts = _c(np.asarray(drafts).reshape(B, k) if k > 0 else np.zeros((B, 1)), np.int32)
    q = _c(np.asarray(q).reshape(B, k, V) if k > 0 else np.zeros((B, 1, V)), np.float32)
    u_acc = _c(np.asarray(u_acc).reshape(B, k) if k > 0 else np.zeros((B, 1)), np.float32)
    pos, u_res = _c(pos, np.int32), _c(u_res, np.float32)
    tokens = np.empty((B, k + 1), np.int32)
    n, a, npos, nxt = (np.empty(B, np.int32) for _ in range(4))
    err = lib().orc_accept_sample(_p(drafts), _p(logits), _p(q), _p(pos), B, k, V, float(temperature), _p(u_acc),
                                  _p(u_res), _p(tokens), _p(n), _p(a), _p(npos), _p(nxt))
    return tokens, n, a, npos, nxt, int(err)


def h_gather(hpool, hslot):
    """(rows [B][H] uint16 with hpool[hslot[b]] (zero where the slot is invalid), error bits)."""
    hpool = _c(hpool, np.uint16)
    hslot = _c(hslot, np.int32)
    n_slots, H = hpool.shape
    out = np.zeros((len(hslot), H), np.uint16)
    err = lib().orc_h_gather(_p(out), _p(hpool), _p(hslot), len(hslot), H, n_slots)
    return out, int(err)


def h_scatter(hpool, h_in, hslot) -> int:
    """hpool[hslot[b]] = h_in[b] in place (uint16 arrays); returns the error bits."""
    assert hpool.dtype == np.uint16 and hpool.flags.c_contiguous
    h_in, hslot = _c(h_in, np.uint16), _c(hslot, np.int32)
    n_slots, H = hpool.shape
    return int(lib().orc_h_scatter(_p(hpool), _p(h_in), _p(hslot), len(hslot), H, n_slots))


def kv_compact(kv: KvPool, pos, path, accepted, B: int, k: int) -> int:
    """Move each accepted row's K/V to the contiguous slot of its rank (in place)."""
    pos, path, acc = _c(pos, np.int32), _c(np.asarray(path).reshape(B, k + 1), np.int32), _c(accepted, np.int32)
    s = kv._struct()
    return int(lib().orc_kv_compact(ctypes.byref(s), _p(pos), _p(path), _p(acc), B, k))


def verify_attn_items(kv: KvPool, pos, B: int, k: int, n_q_heads: int, q, scale: float, items):
    """fp64 outputs [len(items)][d] for items = r * Hq + h."""
    pos, q, items = _c(pos, np.int32), _c(q, np.uint16), _c(items, np.int32)
    out = np.empty((len(items), kv.head_dim), dtype=np.float64)
    s = kv._struct()
    err = lib().orc_verify_attn_items(ctypes.byref(s), _p(pos), B, k, n_q_heads, _p(q), float(scale),
                                      _p(items), len(items), _p(out))
    return out, int(err)


# ---- LM head ----------------------------------------------------------------------------

def lmhead_argmax(hidden, W, d2t=None, d2t_limit: int = 0):
    """ids int32 [M], fp64 max logit [M], fp64 top-2 gap [M], error bits."""
    hidden, W = _c(hidden, np.uint16), _c(W, np.uint16)
    M, H = hidden.shape
    V = W.shape[0]
    assert W.shape[1] == H
    d2t = None if d2t is None else _c(d2t, np.int32)
    ids = np.empty(M, np.int32)
    mx = np.empty(M, np.float64)
    gap = np.empty(M, np.float64)
    err = lib().orc_lmhead_argmax(_p(hidden), _p(W), M, V, H, _p(d2t), int(d2t_limit), _p(ids), _p(mx), _p(gap))
    return ids, mx, gap, int(err)


def lmhead_logits(hidden, W):
    hidden, W = _c(hidden, np.uint16), _c(W, np.uint16)
    M, H = hidden.shape
    V = W.shape[0]
    out = np.empty((M, V), np.float64)
    lib().orc_lmhead_logits(_p(hidden), _p(W), M, V, H, _p(out))
    return out


# ---- accept -----------------------------------------------------------------------------

def accept(drafts, ids, pos, B: int, k: int):
    drafts = _c(np.asarray(drafts).reshape(B, k) if k > 0 else np.zeros((B, 1)), np.int32)
    ids, pos = _c(ids, np.int32), _c(pos, np.int32)
    tokens = np.empty((B, k + 1), np.int32)
    n, a, npos, nxt = (np.empty(B, np.int32) for _ in range(4))
    lib().orc_accept(_p(drafts), _p(ids), _p(pos), B, k, _p(tokens), _p(n), _p(a), _p(npos), _p(nxt))
    return tokens, n, a, npos, nxt


def accept_stop(drafts, ids, pos, B: int, k: int, stop=(), budget=None):
    """Greedy acceptance cut at the first stop token and at the branch's budget:
    tokens [B][k+1], n, accepted, new_pos, next, done."""
    assert k <= 63
    drafts = _c(np.asarray(drafts).reshape(B, k) if k > 0 else np.zeros((B, 1)), np.int32)
    ids, pos = _c(ids, np.int32), _c(pos, np.int32)
    stop_a = _c(np.asarray(stop, np.int32).reshape(-1) if len(stop) else np.full(1, -1), np.int32)
    bud = None if budget is None else _c(budget, np.int32)
    tokens = np.empty((B, k + 1), np.int32)
    n, a, npos, nxt, done = (np.empty(B, np.int32) for _ in range(5))
    lib().orc_accept_stop(_p(drafts), _p(ids), _p(pos), B, k, _p(stop_a), len(stop),
                          None if bud is None else _p(bud), _p(tokens), _p(n), _p(a), _p(npos), _p(nxt), _p(done))
    return tokens, n, a, npos, nxt, done


# ---- MTP input ----------------------------------------------------------------------------

def mtp_input(tok, E, h, g_emb, g_hid, eps: float, W_fc):
    """bf16 concat [M][2H] (uint16 bits), fp64 x [M][H], error bits."""
    tok = _c(tok, np.int32)
    E, h, W_fc = _c(E, np.uint16), _c(h, np.uint16), _c(W_fc, np.uint16)
    g_emb, g_hid = _c(g_emb, np.float32), _c(g_hid, np.float32)
    M, H = h.shape
    V = E.shape[0]
    concat = np.empty((M, 2 * H), np.uint16)
    x = np.empty((M, H), np.float64)
    err = lib().orc_mtp_input(_p(tok), _p(E), _p(h), _p(g_emb), _p(g_hid), float(eps), _p(W_fc),
                              M, H, V, _p(concat), _p(x))
    return concat, x, int(err)

"""Thin ctypes binding of libspecverify (include/spec_verify.h).

Argument marshalling only: every function here passes device pointers, sizes and the
current CUDA stream to the C ABI entry point of the same name and raises `SpecError`
on a non-zero status. There is no fallback: if the library is missing or a tensor is
not on a CUDA device, the call fails loudly.
"""
from __future__ import annotations

import ctypes
import os
from pathlib import Path

import torch

_PKG = Path(__file__).resolve().parent
LIB_PATH = _PKG / "libspecverify.so"

SPEC_OK = 0
STATUS = {-1: "SPEC_ERR_NULL", -2: "SPEC_ERR_ARG", -3: "SPEC_ERR_UNSUPPORTED", -4: "SPEC_ERR_WORKSPACE",
          -5: "SPEC_ERR_CUDA", -6: "SPEC_ERR_ALIGN"}
DEVERR_PAGE, DEVERR_COVER, DEVERR_TOKEN, DEVERR_D2T, DEVERR_POS, DEVERR_TIMEOUT, DEVERR_INTERNAL = 1, 2, 4, 8, 16, 32, 64
DEVERR_TREE = 128
DEVERR_SLOT = 256
KMAX = 15
KV_BF16, KV_FP8_E4M3 = 0, 1

ERR_NULL, ERR_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA, ERR_ALIGN = -1, -2, -3, -4, -5, -6
SPEC_LMHEAD_STATIC_SCRATCH_BYTES = 256 + 1024 * 64 * 8  # as in include/spec_verify.h
SPEC_MAX_STOP = 32                                       # as in include/spec_verify.h
SPEC_ATTN_PLAN_FIELDS = 17                               # as in include/spec_verify.h
ATTN_PLAN_KEYS = ("smem", "nq", "k_stages", "v_stages", "raw_stages", "s_buffers", "p_buffers", "q_buffers", "o_buffers",
                  "tmem_cols", "split_keys", "n_splits", "n_units", "tile_group", "tma_rows", "barrier_bytes",
                  "barrier_bytes_reserved")

EXPORTS = ("spec_strerror", "spec_version", "spec_kv_append", "spec_kv_write_rows",
           "spec_verify_attn_workspace", "spec_verify_attn", "spec_lmhead_workspace",
           "spec_lmhead_argmax", "spec_lmhead_logits", "spec_accept", "spec_mtp_input_workspace",
           "spec_mtp_input", "spec_lmhead_argmax_static", "spec_accept_stop", "spec_verify_attn_plan",
           "spec_test_set_wait_limit", "spec_accept_sample", "spec_accept_sample_workspace",
           "spec_verify_attn_tree", "spec_accept_tree",
           "spec_kv_compact", "spec_h_gather", "spec_h_scatter")


class SpecError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {STATUS.get(status, status)} ({strerror(status)})")


class spec_kv_desc(ctypes.Structure):
    _fields_ = [("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p),
                ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
                ("page_table", ctypes.c_void_p),
                ("num_pages", ctypes.c_int32), ("max_pages", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("kv_dtype", ctypes.c_int32)]


_lib = None
_vp, _i32, _f32, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_KVP = ctypes.POINTER(spec_kv_desc)


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not LIB_PATH.exists():
            raise RuntimeError(f"{LIB_PATH} is not built: run `python -m greedy_speculative_decode_spec_gb300.build` "
                               "(or __graft_entry__.build()) first")
        L = ctypes.CDLL(str(LIB_PATH))
        L.spec_strerror.restype = ctypes.c_char_p
        L.spec_strerror.argtypes = [_i32]
        L.spec_version.restype = _i32
        L.spec_kv_append.argtypes = [_KVP, _vp, _i32, _i32, _vp, _vp, _vp, _vp]
        L.spec_kv_write_rows.argtypes = [_KVP, _vp, _vp, _i32, _vp, _vp, _vp, _vp]
        L.spec_verify_attn_workspace.restype = _sz
        L.spec_verify_attn_workspace.argtypes = [_KVP, _i32, _i32, _i32, _i32]
        L.spec_verify_attn.argtypes = [_KVP, _vp, _i32, _i32, _i32, _vp, _f32, _vp, _vp, _sz, _i32, _vp, _vp]
        L.spec_lmhead_workspace.restype = _sz
        L.spec_lmhead_workspace.argtypes = [_i32, _i32, _i32]
        L.spec_lmhead_argmax.argtypes = [_vp, _vp, _i32, _i32, _i32, _vp, _i32, _vp, _vp, _vp, _sz, _vp, _vp]
        L.spec_lmhead_logits.argtypes = [_vp, _vp, _i32, _i32, _i32, _vp, _vp, _vp, _sz, _vp]
        L.spec_lmhead_argmax_static.argtypes = [_vp, _vp, _i32, _i32, _i32, _vp, _i32, _vp, _vp, _vp, _vp]
        L.spec_accept.argtypes = [_vp, _vp, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _vp]
        L.spec_verify_attn_plan.argtypes = [ctypes.POINTER(spec_kv_desc), _i32, _i32, _i32, _i32, _vp, _i32]
        L.spec_accept_stop.argtypes = [_vp, _vp, _vp, _i32, _i32, _vp, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                       _vp, _i32, _vp, _vp]
        L.spec_accept_sample.argtypes = [_vp, _vp, _vp, _vp, _i32, _i32, _i32, _f32, _vp, _vp, _vp, _vp, _vp, _vp,
                                         _vp, _vp, _sz, _vp, _vp]
        L.spec_accept_sample_workspace.restype = _sz
        L.spec_accept_sample_workspace.argtypes = [_i32, _i32, _i32]
        L.spec_verify_attn_tree.argtypes = [_KVP, _vp, _i32, _i32, _i32, _vp, _f32, _vp, _vp, _vp, _sz, _i32, _vp, _vp]
        L.spec_accept_tree.argtypes = [_vp, _vp, _vp, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]
        L.spec_kv_compact.argtypes = [_KVP, _vp, _vp, _vp, _i32, _i32, _vp, _vp]
        L.spec_h_gather.argtypes = [_vp, _vp, _vp, _i32, _i32, _i32, _vp, _vp]
        L.spec_h_scatter.argtypes = [_vp, _vp, _vp, _i32, _i32, _i32, _vp, _vp]
        L.spec_test_set_wait_limit.argtypes = [ctypes.c_uint64]
        L.spec_test_set_wait_limit.restype = None
        L.spec_mtp_input_workspace.restype = _sz
        L.spec_mtp_input_workspace.argtypes = [_i32, _i32]
        L.spec_mtp_input.argtypes = [_vp, _vp, _vp, _vp, _vp, _f32, _vp, _i32, _i32, _i32, _vp, _vp, _sz, _vp, _vp]
        _lib = L
    return _lib


def strerror(status: int) -> str:
    return lib().spec_strerror(int(status)).decode()


def version() -> int:
    return int(lib().spec_version())


def _ptr(t, name: str, dtype=None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device (no CPU path exists)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


_DEBUG_SYNC = os.environ.get("SPEC_DEBUG_SYNC", "0") == "1"


def _check(fn: str, st: int):
    if st != SPEC_OK:
        raise SpecError(fn, st)
    if _DEBUG_SYNC and not torch.cuda.is_current_stream_capturing():
        # debugging aid: surface an asynchronous fault at the call that caused it
        try:
            torch.cuda.synchronize()
        except Exception as e:  # noqa: BLE001
            raise RuntimeError(f"{fn}: device fault after this call: {e}") from e


def make_kv_desc(k_pool, v_pool, page_table, page_size: int, k_scale=None, v_scale=None) -> spec_kv_desc:
    """Descriptor of a pool [num_pages][Hkv][page_size][d] (bf16, or uint8 E4M3 codes + scales)."""
    num_pages, hkv, ps, d = k_pool.shape
    if ps != page_size or tuple(v_pool.shape) != tuple(k_pool.shape):
        raise ValueError("pool shapes do not match the page size")
    fp8 = k_pool.dtype == torch.uint8
    return spec_kv_desc(_ptr(k_pool, "k_pool"), _ptr(v_pool, "v_pool"),
                        _ptr(k_scale, "k_scale", torch.float32), _ptr(v_scale, "v_scale", torch.float32),
                        _ptr(page_table, "page_table", torch.int32), num_pages, page_table.shape[1], page_size, hkv,
                        d, KV_FP8_E4M3 if fp8 else KV_BF16)


# ---- entry points (same names as the C ABI) -----------------------------------------------

def spec_kv_append(kv: spec_kv_desc, pos, B: int, k: int, k_new, v_new, dev_err=None, stream=None):
    _check("spec_kv_append", lib().spec_kv_append(ctypes.byref(kv), _ptr(pos, "pos", torch.int32), B, k,
                                                  _ptr(k_new, "k_new", torch.bfloat16),
                                                  _ptr(v_new, "v_new", torch.bfloat16),
                                                  _ptr(dev_err, "dev_err", torch.int32), _stream(stream)))


def spec_kv_write_rows(kv: spec_kv_desc, row_branch, row_pos, k_rows, v_rows, dev_err=None, stream=None):
    n = int(row_pos.shape[0])
    _check("spec_kv_write_rows", lib().spec_kv_write_rows(ctypes.byref(kv), _ptr(row_branch, "row_branch", torch.int32),
                                                          _ptr(row_pos, "row_pos", torch.int32), n,
                                                          _ptr(k_rows, "k_rows", torch.bfloat16),
                                                          _ptr(v_rows, "v_rows", torch.bfloat16),
                                                          _ptr(dev_err, "dev_err", torch.int32), _stream(stream)))


def spec_verify_attn_workspace(kv: spec_kv_desc, B: int, k: int, n_q_heads: int, max_pos: int) -> int:
    return int(lib().spec_verify_attn_workspace(ctypes.byref(kv), B, k, n_q_heads, max_pos))


def spec_verify_attn(kv: spec_kv_desc, pos, B: int, k: int, n_q_heads: int, q, scale: float, out, ws,
                     max_pos: int, dev_err=None, stream=None):
    _check("spec_verify_attn", lib().spec_verify_attn(ctypes.byref(kv), _ptr(pos, "pos", torch.int32), B, k, n_q_heads,
                                                      _ptr(q, "q", torch.bfloat16), float(scale),
                                                      _ptr(out, "out", torch.bfloat16), _ptr(ws, "ws"),
                                                      ws.numel() * ws.element_size(), int(max_pos),
                                                      _ptr(dev_err, "dev_err", torch.int32), _stream(stream)))


def spec_lmhead_workspace(M: int, V: int, H: int) -> int:
    return int(lib().spec_lmhead_workspace(M, V, H))


def spec_lmhead_argmax(hidden, W, ids, ws, d2t=None, d2t_limit: int = 0, max_logit=None, dev_err=None,
                       stream=None):
    M, H = hidden.shape
    V = W.shape[0]
    _check("spec_lmhead_argmax", lib().spec_lmhead_argmax(_ptr(hidden, "hidden", torch.bfloat16),
                                                          _ptr(W, "W", torch.bfloat16), M, V, H,
                                                          _ptr(d2t, "d2t", torch.int32), int(d2t_limit),
                                                          _ptr(ids, "ids", torch.int32),
                                                          _ptr(max_logit, "max_logit", torch.float32),
                                                          _ptr(ws, "ws"), ws.numel() * ws.element_size(),
                                                          _ptr(dev_err, "dev_err", torch.int32), _stream(stream)))


def spec_lmhead_argmax_static(hidden, W, ids, d2t=None, d2t_limit: int = 0, max_logit=None, dev_err=None,
                              stream=None):
    """spec_lmhead_argmax without a workspace: the library's own device scratch is used (see
    the header for the size limit, the first-call set-up and the one-call-at-a-time rule)."""
    M, H = hidden.shape
    V = W.shape[0]
    _check("spec_lmhead_argmax_static",
           lib().spec_lmhead_argmax_static(_ptr(hidden, "hidden", torch.bfloat16), _ptr(W, "W", torch.bfloat16), M, V,
                                           H, _ptr(d2t, "d2t", torch.int32), int(d2t_limit),
                                           _ptr(ids, "ids", torch.int32), _ptr(max_logit, "max_logit", torch.float32),
                                           _ptr(dev_err, "dev_err", torch.int32), _stream(stream)))


def spec_lmhead_logits(hidden, W, logits, ids, ws, stream=None):
    M, H = hidden.shape
    V = W.shape[0]
    _check("spec_lmhead_logits", lib().spec_lmhead_logits(_ptr(hidden, "hidden", torch.bfloat16),
                                                          _ptr(W, "W", torch.bfloat16), M, V, H,
                                                          _ptr(logits, "logits", torch.float32),
                                                          _ptr(ids, "ids", torch.int32), _ptr(ws, "ws"),
                                                          ws.numel() * ws.element_size(), _stream(stream)))


def spec_accept(drafts, ids, pos, B: int, k: int, out_tokens, out_n, out_accepted, out_pos, out_next,
                hidden=None, h_out=None, stream=None):
    H = int(hidden.shape[-1]) if hidden is not None else 0
    _check("spec_accept", lib().spec_accept(_ptr(drafts, "drafts", torch.int32) if k > 0 else None,
                                            _ptr(ids, "ids", torch.int32), _ptr(pos, "pos", torch.int32), B, k,
                                            _ptr(out_tokens, "out_tokens", torch.int32),
                                            _ptr(out_n, "out_n", torch.int32),
                                            _ptr(out_accepted, "out_accepted", torch.int32),
                                            _ptr(out_pos, "out_pos", torch.int32),
                                            _ptr(out_next, "out_next", torch.int32),
                                            _ptr(hidden, "hidden", torch.bfloat16), H,
                                            _ptr(h_out, "h_out", torch.bfloat16), _stream(stream)))


def kv_shape(num_pages: int, max_pages: int, page_size: int, n_kv_heads: int, head_dim: int,
             fp8: bool = False) -> spec_kv_desc:
    """A descriptor that carries only shapes (no memory): for spec_verify_attn_plan."""
    return spec_kv_desc(None, None, None, None, None, num_pages, max_pages, page_size, n_kv_heads, head_dim,
                        KV_FP8_E4M3 if fp8 else KV_BF16)


def spec_verify_attn_plan(kv: spec_kv_desc, B: int, k: int, n_q_heads: int, max_pos: int) -> dict:
    """The launch plan spec_verify_attn would use (host arithmetic only, no GPU)."""
    out = (ctypes.c_int32 * SPEC_ATTN_PLAN_FIELDS)()
    _check("spec_verify_attn_plan", lib().spec_verify_attn_plan(ctypes.byref(kv), B, k, n_q_heads, max_pos,
                                                                ctypes.cast(out, ctypes.c_void_p),
                                                                SPEC_ATTN_PLAN_FIELDS))
    return dict(zip(ATTN_PLAN_KEYS, list(out)))


def spec_accept_stop(drafts, ids, pos, B: int, k: int, stop_ids, budget, out_tokens, out_n, out_accepted, out_pos,
                     out_next, out_done=None, hidden=None, h_out=None, stream=None):
    """spec_accept with a stop set (device int32 tensor, entries < 0 unused, or None) and a
    per-branch budget (device int32 [B] or None)."""
    H = int(hidden.shape[-1]) if hidden is not None else 0
    n_stop = 0 if stop_ids is None else int(stop_ids.numel())
    _check("spec_accept_stop", lib().spec_accept_stop(
        _ptr(drafts, "drafts", torch.int32) if k > 0 else None, _ptr(ids, "ids", torch.int32),
        _ptr(pos, "pos", torch.int32), B, k, _ptr(stop_ids, "stop_ids", torch.int32), n_stop,
        _ptr(budget, "budget", torch.int32), _ptr(out_tokens, "out_tokens", torch.int32),
        _ptr(out_n, "out_n", torch.int32), _ptr(out_accepted, "out_accepted", torch.int32),
        _ptr(out_pos, "out_pos", torch.int32), _ptr(out_next, "out_next", torch.int32),
        _ptr(out_done, "out_done", torch.int32), _ptr(hidden, "hidden", torch.bfloat16), H,
        _ptr(h_out, "h_out", torch.bfloat16), _stream(stream)))


def spec_accept_sample_workspace(B: int, k: int, V: int) -> int:
    return int(lib().spec_accept_sample_workspace(B, k, V))


def spec_accept_sample(drafts, logits, q, pos, B: int, k: int, temperature: float, u_acc, u_res, out_tokens, out_n,
                       out_accepted, out_pos, out_next, dev_err=None, ws=None, stream=None):
    """Speculative sampling acceptance; logits fp32 [B*(k+1)][V], q fp32 [B][k][V]; ws: a
    zeroed device byte tensor of spec_accept_sample_workspace(B, k, V) bytes (made here if None)."""
    V = int(logits.shape[-1])
    if ws is None:
        ws = torch.zeros(max(1, spec_accept_sample_workspace(B, k, V)), dtype=torch.uint8, device=logits.device)
    _check("spec_accept_sample", lib().spec_accept_sample(
        _ptr(drafts, "drafts", torch.int32) if k > 0 else None, _ptr(logits, "logits", torch.float32),
        _ptr(q, "q", torch.float32) if k > 0 else None, _ptr(pos, "pos", torch.int32), B, k, V, float(temperature),
        _ptr(u_acc, "u_acc", torch.float32) if k > 0 else None, _ptr(u_res, "u_res", torch.float32),
        _ptr(out_tokens, "out_tokens", torch.int32), _ptr(out_n, "out_n", torch.int32),
        _ptr(out_accepted, "out_accepted", torch.int32), _ptr(out_pos, "out_pos", torch.int32),
        _ptr(out_next, "out_next", torch.int32), _ptr(ws, "ws"), ws.numel() * ws.element_size(),
        _ptr(dev_err, "dev_err", torch.int32), _stream(stream)))


def spec_verify_attn_tree(kv: spec_kv_desc, pos, B: int, k: int, n_q_heads: int, q, scale: float, anc_mask, out, ws,
                          max_pos: int, dev_err=None, stream=None):
    """Tree verify attention: row j reads the committed prefix and the verify slots of its mask."""
    _check("spec_verify_attn_tree", lib().spec_verify_attn_tree(
        ctypes.byref(kv), _ptr(pos, "pos", torch.int32), B, k, n_q_heads, _ptr(q, "q", torch.bfloat16), float(scale),
        _ptr(anc_mask, "anc_mask", torch.int32), _ptr(out, "out", torch.bfloat16), _ptr(ws, "ws"),
        ws.numel() * ws.element_size(), max_pos, _ptr(dev_err, "dev_err", torch.int32), _stream(stream)))


def spec_accept_tree(drafts, ids, pos, parent, B: int, k: int, out_tokens, out_n, out_accepted, out_pos, out_next,
                     out_path, dev_err=None, stream=None):
    _check("spec_accept_tree", lib().spec_accept_tree(
        _ptr(drafts, "drafts", torch.int32) if k > 0 else None, _ptr(ids, "ids", torch.int32),
        _ptr(pos, "pos", torch.int32), _ptr(parent, "parent", torch.int32), B, k,
        _ptr(out_tokens, "out_tokens", torch.int32), _ptr(out_n, "out_n", torch.int32),
        _ptr(out_accepted, "out_accepted", torch.int32), _ptr(out_pos, "out_pos", torch.int32),
        _ptr(out_next, "out_next", torch.int32), _ptr(out_path, "out_path", torch.int32),
        _ptr(dev_err, "dev_err", torch.int32), _stream(stream)))


def spec_kv_compact(kv: spec_kv_desc, pos, path, accepted, B: int, k: int, dev_err=None, stream=None):
    _check("spec_kv_compact", lib().spec_kv_compact(
        ctypes.byref(kv), _ptr(pos, "pos", torch.int32), _ptr(path, "path", torch.int32),
        _ptr(accepted, "accepted", torch.int32), B, k, _ptr(dev_err, "dev_err", torch.int32), _stream(stream)))


def spec_h_gather(h_out, hpool, hslot, dev_err=None, stream=None):
    """h_out[b] = hpool[hslot[b]] (bf16 rows)."""
    B, H = h_out.shape
    _check("spec_h_gather", lib().spec_h_gather(
        _ptr(h_out, "h_out", torch.bfloat16), _ptr(hpool, "hpool", torch.bfloat16), _ptr(hslot, "hslot", torch.int32),
        B, H, int(hpool.shape[0]), _ptr(dev_err, "dev_err", torch.int32), _stream(stream)))


def spec_h_scatter(hpool, h_in, hslot, dev_err=None, stream=None):
    """hpool[hslot[b]] = h_in[b] (bf16 rows; distinct slots)."""
    B, H = h_in.shape
    _check("spec_h_scatter", lib().spec_h_scatter(
        _ptr(hpool, "hpool", torch.bfloat16), _ptr(h_in, "h_in", torch.bfloat16), _ptr(hslot, "hslot", torch.int32),
        B, H, int(hpool.shape[0]), _ptr(dev_err, "dev_err", torch.int32), _stream(stream)))


def spec_test_set_wait_limit(ns: int) -> None:
    """Test hook: limit (ns) of the kernels' pipeline waits for later launches; 0 = default."""
    lib().spec_test_set_wait_limit(int(ns))


def spec_mtp_input_workspace(M: int, H: int) -> int:
    return int(lib().spec_mtp_input_workspace(M, H))


def spec_mtp_input(tok, E, h, g_emb, g_hid, eps: float, W_fc, x_out, ws, dev_err=None, stream=None):
    M, H = h.shape
    V = E.shape[0]
    _check("spec_mtp_input", lib().spec_mtp_input(_ptr(tok, "tok", torch.int32), _ptr(E, "E", torch.bfloat16),
                                                  _ptr(h, "h", torch.bfloat16), _ptr(g_emb, "g_emb", torch.float32),
                                                  _ptr(g_hid, "g_hid", torch.float32), float(eps),
                                                  _ptr(W_fc, "W_fc", torch.bfloat16), M, H, V,
                                                  _ptr(x_out, "x_out", torch.bfloat16), _ptr(ws, "ws"),
                                                  ws.numel() * ws.element_size(),
                                                  _ptr(dev_err, "dev_err", torch.int32), _stream(stream)))

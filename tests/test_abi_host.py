"""The C-ABI library without a GPU: it builds for sm_103a, loads, exports every entry point
include/spec_verify.h declares, and rejects bad arguments on the host before any launch
(so these calls never touch a device)."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

from greedy_speculative_decode_spec_gb300 import _binding as bnd
from greedy_speculative_decode_spec_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spec_verify.h")
FAKE = 0x10000  # a 256-byte aligned non-NULL address: never dereferenced on these paths


@pytest.fixture(scope="module")
def L():
    build.build()
    return bnd.lib()


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(L):
    syms = declared_symbols()
    assert len(syms) >= 12
    for s in syms:
        assert hasattr(L, s), f"{s} declared in the header but not exported"
    assert set(syms) == set(bnd.EXPORTS)


def test_version_and_strerror(L):
    assert bnd.version() >= 100
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert bnd.strerror(code) and bnd.strerror(code) != "unknown status"
    assert bnd.strerror(-99) == "unknown status"


def _desc(**kw):
    d = dict(k_pool=FAKE, v_pool=FAKE, k_scale=None, v_scale=None, page_table=FAKE, num_pages=8, max_pages=8,
             page_size=16, n_kv_heads=1, head_dim=64, kv_dtype=0)
    d.update(kw)
    return bnd.spec_kv_desc(**d)


def test_host_argument_errors(L):
    p = ctypes.c_void_p(FAKE)
    s = None
    d = _desc()
    # descriptor checks
    assert L.spec_kv_append(ctypes.byref(_desc(head_dim=96)), p, 1, 0, p, p, None, s) == -3
    assert L.spec_kv_append(ctypes.byref(_desc(page_size=3)), p, 1, 0, p, p, None, s) == -2
    assert L.spec_kv_append(ctypes.byref(_desc(page_size=2048)), p, 1, 0, p, p, None, s) == -2
    assert L.spec_kv_append(ctypes.byref(_desc(kv_dtype=1)), p, 1, 0, p, p, None, s) == -1   # FP8 without scales
    assert L.spec_kv_append(ctypes.byref(_desc(kv_dtype=7)), p, 1, 0, p, p, None, s) == -3
    assert L.spec_kv_append(ctypes.byref(_desc(k_pool=FAKE + 8)), p, 1, 0, p, p, None, s) == -6
    assert L.spec_kv_append(ctypes.byref(_desc(num_pages=0)), p, 1, 0, p, p, None, s) == -2
    assert L.spec_kv_append(None, p, 1, 0, p, p, None, s) == -1
    # append
    assert L.spec_kv_append(ctypes.byref(d), p, 0, 0, p, p, None, s) == -2
    assert L.spec_kv_append(ctypes.byref(d), p, 1, 16, p, p, None, s) == -2
    assert L.spec_kv_append(ctypes.byref(d), p, 1, -1, p, p, None, s) == -2
    assert L.spec_kv_append(ctypes.byref(d), None, 1, 0, p, p, None, s) == -1
    assert L.spec_kv_append(ctypes.byref(d), p, 1, 0, None, p, None, s) == -1
    assert L.spec_kv_append(ctypes.byref(d), p, 1, 0, ctypes.c_void_p(FAKE + 4), p, None, s) == -6
    assert L.spec_kv_write_rows(ctypes.byref(d), None, p, 3, p, p, None, s) == -1
    assert L.spec_kv_write_rows(ctypes.byref(d), p, p, 0, p, p, None, s) == 0            # no rows: no launch
    # attention
    assert L.spec_verify_attn_workspace(ctypes.byref(d), 1, 3, 4, 104) > 0
    assert L.spec_verify_attn_workspace(ctypes.byref(d), 1, 3, 3, 104) > 0
    assert L.spec_verify_attn_workspace(ctypes.byref(_desc(n_kv_heads=2)), 1, 3, 3, 104) == 0
    ws = L.spec_verify_attn_workspace(ctypes.byref(d), 1, 3, 4, 104)
    assert L.spec_verify_attn(ctypes.byref(d), p, 1, 3, 4, p, ctypes.c_float(0.1), p, p, ws - 1, 104, None, s) == -4
    assert L.spec_verify_attn(ctypes.byref(d), p, 1, 3, 4, p, ctypes.c_float(0.1), p, None, ws, 104, None, s) == -4
    assert L.spec_verify_attn(ctypes.byref(d), p, 1, 3, 4, p, ctypes.c_float(0.1), p, p, ws, 3, None, s) == -2
    assert L.spec_verify_attn(ctypes.byref(_desc(n_kv_heads=3)), p, 1, 3, 4, p, ctypes.c_float(0.1), p, p, ws, 104,
                              None, s) == -2
    assert L.spec_verify_attn(ctypes.byref(d), p, 1, 3, 4, None, ctypes.c_float(0.1), p, p, ws, 104, None, s) == -1
    # LM head
    assert L.spec_lmhead_workspace(0, 100, 64) == 0
    assert L.spec_lmhead_workspace(257, 100, 64) == 0
    w = L.spec_lmhead_workspace(4, 1000, 256)
    assert w > 0
    assert L.spec_lmhead_argmax(p, p, 0, 1000, 256, None, 0, p, None, p, w, None, s) == -2
    assert L.spec_lmhead_argmax(p, p, 4, 1000, 260, None, 0, p, None, p, w, None, s) == -2     # H % 8
    assert L.spec_lmhead_argmax(p, p, 4, 1000, 256, None, 0, p, None, p, w - 1, None, s) == -4
    assert L.spec_lmhead_argmax(p, p, 4, 1000, 256, p, 0, p, None, p, w, None, s) == -2       # d2t without limit
    assert L.spec_lmhead_argmax(None, p, 4, 1000, 256, None, 0, p, None, p, w, None, s) == -1
    assert L.spec_lmhead_argmax(ctypes.c_void_p(FAKE + 2), p, 4, 1000, 256, None, 0, p, None, p, w, None, s) == -6
    assert L.spec_lmhead_logits(p, p, 4, 1000, 256, None, p, p, w, s) == -1
    # accept
    assert L.spec_accept(p, p, p, 0, 3, p, p, p, p, p, None, 0, None, s) == -2
    assert L.spec_accept(p, p, p, 1, 16, p, p, p, p, p, None, 0, None, s) == -2
    assert L.spec_accept(None, p, p, 1, 3, p, p, p, p, p, None, 0, None, s) == -1
    assert L.spec_accept(p, p, p, 1, 3, p, p, p, p, p, p, 64, None, s) == -1                  # hidden without h_out
    # accept with stops and budget: the same checks, plus the stop list
    acs = L.spec_accept_stop
    assert acs(p, p, p, 0, 3, None, 0, None, p, p, p, p, p, None, None, 0, None, s) == -2
    assert acs(p, p, p, 1, 16, None, 0, None, p, p, p, p, p, None, None, 0, None, s) == -2
    assert acs(None, p, p, 1, 3, None, 0, None, p, p, p, p, p, None, None, 0, None, s) == -1
    assert acs(p, p, p, 1, 3, p, 33, None, p, p, p, p, p, None, None, 0, None, s) == -2      # too many stop ids
    assert acs(p, p, p, 1, 3, p, -1, None, p, p, p, p, p, None, None, 0, None, s) == -2
    assert acs(p, p, p, 1, 3, None, 2, None, p, p, p, p, p, None, None, 0, None, s) == -1    # stop ids missing
    assert acs(p, p, p, 1, 3, None, 0, None, p, p, p, p, p, None, p, 64, None, s) == -1      # hidden without h_out
    # MTP input
    assert L.spec_mtp_input_workspace(64, 100) == 0
    mw = L.spec_mtp_input_workspace(64, 256)
    assert mw > 0
    assert L.spec_mtp_input(p, p, p, p, p, ctypes.c_float(1e-6), p, 64, 100, 1000, p, p, mw, None, s) == -2
    assert L.spec_mtp_input(p, p, p, p, p, ctypes.c_float(1e-6), p, 0, 256, 1000, p, p, mw, None, s) == -2
    assert L.spec_mtp_input(p, p, p, p, p, ctypes.c_float(1e-6), p, 64, 256, 1000, p, p, mw - 1, None, s) == -4
    assert L.spec_mtp_input(p, p, p, p, p, ctypes.c_float(-1.0), p, 64, 256, 1000, p, p, mw, None, s) == -2
    assert L.spec_mtp_input(p, None, p, p, p, ctypes.c_float(1e-6), p, 64, 256, 1000, p, p, mw, None, s) == -1
    # speculative sampling acceptance: workspace query, then the host checks (nothing launches)
    f = ctypes.c_float
    assert L.spec_accept_sample_workspace(0, 3, 1000) == 0
    assert L.spec_accept_sample_workspace(1, 16, 1000) == 0
    sw = L.spec_accept_sample_workspace(16, 6, 151936)
    assert sw >= 12 * 16 * 7 * 19   # per (verify row, vocabulary chunk of 8192): fp32 max, fp64 sum
    sa = L.spec_accept_sample
    assert sa(p, p, p, p, 16, 6, 151936, f(1.0), p, p, p, p, p, p, p, p, sw - 1, None, s) == -4
    assert sa(p, p, p, p, 16, 6, 151936, f(1.0), p, p, p, p, p, p, p, None, sw, None, s) == -4
    assert sa(p, p, p, p, 16, 6, 151936, f(1.0), p, p, p, p, p, p, p, ctypes.c_void_p(FAKE + 8), sw, None, s) == -6
    assert sa(p, p, p, p, 16, 6, 151936, f(0.0), p, p, p, p, p, p, p, p, sw, None, s) == -2
    assert sa(p, p, p, p, 16, 16, 151936, f(1.0), p, p, p, p, p, p, p, p, sw, None, s) == -2
    assert sa(p, p, p, p, 16, 6, 1 << 24, f(1.0), p, p, p, p, p, p, p, p, sw, None, s) == -2
    assert sa(p, p, None, p, 16, 6, 151936, f(1.0), p, p, p, p, p, p, p, p, sw, None, s) == -1   # q missing


def test_binding_refuses_cpu_tensors(L):
    import torch
    x = torch.zeros(4, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA"):
        bnd._ptr(x, "x")

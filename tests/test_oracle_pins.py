"""Pins of the CPU oracle against things other than itself: library routines, closed
forms, brute force on tiny inputs, the pages' worked examples and invariants.
No GPU is needed."""
from __future__ import annotations

import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

from toy_lm import ToyLM, run_greedy, run_spec

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(b: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).double().numpy()


# ---- number formats --------------------------------------------------------------------------

def test_bf16_decode_matches_torch(orc):
    for b in [0x0000, 0x8000, 0x3F80, 0xBF80, 0x7F7F, 0x0001, 0x0080, 0x4049, 0xC2F7]:
        want = torch.tensor([b], dtype=torch.int32).to(torch.int16).view(torch.bfloat16).double().item()
        assert orc.bf16_to_double(b) == want


def test_bf16_rounding_matches_torch(orc):
    rng = np.random.default_rng(0)
    xs = np.concatenate([rng.standard_normal(3000) * 10.0 ** rng.integers(-30, 30, 3000),
                         [1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 2 ** -130, 3.0e38, -3.0e38]])
    xs = xs.astype(np.float32)  # exactly representable in both
    want = bf16_bits(torch.from_numpy(xs).to(torch.bfloat16))
    got = np.array([orc.double_to_bf16(float(x)) for x in xs], dtype=np.uint16)
    np.testing.assert_array_equal(got, want)
    # closed forms: ties go to the even mantissa
    assert orc.double_to_bf16(1 + 2 ** -8) == 0x3F80
    assert orc.double_to_bf16(1 + 3 * 2 ** -8) == 0x3F82
    assert orc.double_to_bf16(float("nan")) == 0x7FC0
    assert orc.double_to_bf16(-0.0) == 0x8000


def test_e4m3_decode_all_codes_match_torch(orc):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    lib = codes.view(torch.float8_e4m3fn).double().numpy()
    for c in range(256):
        got = orc.e4m3_decode(c)
        if math.isnan(lib[c]):
            assert math.isnan(got), c
        else:
            assert got == lib[c] and math.copysign(1, got) == math.copysign(1, lib[c]), c
    # closed forms of the OCP E4M3 format
    assert orc.e4m3_decode(0x7E) == 448.0
    assert orc.e4m3_decode(0x01) == 2.0 ** -9
    assert orc.e4m3_decode(0x08) == 2.0 ** -6
    assert orc.e4m3_decode(0x38) == 1.0
    assert math.isnan(orc.e4m3_decode(0x7F)) and math.isnan(orc.e4m3_decode(0xFF))


def test_e4m3_encode_roundtrip_and_ties(orc):
    for c in range(256):
        if c & 0x7F == 0x7F:
            continue
        assert orc.e4m3_encode(orc.e4m3_decode(c)) == c, hex(c)
    # every midpoint between neighbours rounds to the code with an even mantissa
    for c in range(0, 0x7E):
        lo, hi = orc.e4m3_decode(c), orc.e4m3_decode(c + 1)
        mid = (lo + hi) / 2
        assert float(np.float32(mid)) == mid
        want = c if c % 2 == 0 else c + 1
        assert orc.e4m3_encode(mid) == want, hex(c)
        assert orc.e4m3_encode(-mid) == 0x80 | want
    # satfinite: at and beyond the largest finite magnitude
    for x in [448.0, 449.0, 463.9, 464.0, 1e6, float("inf")]:
        assert orc.e4m3_encode(x) == 0x7E
        assert orc.e4m3_encode(-x) == 0xFE
    assert orc.e4m3_encode(float("nan")) == 0x7F


def test_e4m3_encode_matches_torch_in_range(orc):
    rng = np.random.default_rng(1)
    xs = np.concatenate([rng.standard_normal(4000) * 60, rng.standard_normal(2000) * 0.01,
                         rng.uniform(-463.9, 463.9, 2000)]).astype(np.float32)
    want = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([orc.e4m3_encode(float(x)) for x in xs], dtype=np.uint8)
    np.testing.assert_array_equal(got, want)


# ---- KV write ------------------------------------------------------------------------------------

def _tiny_pool(rng, num_pages, Hkv, P, d, dtype="bf16"):
    if dtype == "bf16":
        return np.full((num_pages, Hkv, P, d), 0x7FC0, np.uint16), np.full((num_pages, Hkv, P, d), 0x7FC0, np.uint16)
    return np.full((num_pages, Hkv, P, d), 0x7F, np.uint8), np.full((num_pages, Hkv, P, d), 0x7F, np.uint8)


def test_kv_write_rows_bf16_places_bits(orc):
    rng = np.random.default_rng(2)
    num_pages, Hkv, P, d, B = 12, 2, 4, 8, 2
    kp, vp = _tiny_pool(rng, num_pages, Hkv, P, d)
    pt = rng.permutation(num_pages)[:10].reshape(B, 5).astype(np.int32)
    kv = orc.KvPool(kp, vp, pt, P)
    rows = [(0, 3), (0, 4), (1, 19), (1, 0), (0, 17)]
    krows = rng.integers(0, 0x7F00, (len(rows), Hkv, d)).astype(np.uint16)
    vrows = rng.integers(0, 0x7F00, (len(rows), Hkv, d)).astype(np.uint16)
    err = orc.kv_write_rows(kv, [r[0] for r in rows], [r[1] for r in rows], krows, vrows)
    assert err == 0
    touched = np.zeros((num_pages, Hkv, P), bool)
    for i, (b, p) in enumerate(rows):
        page, slot = pt[b, p // P], p % P
        np.testing.assert_array_equal(kv.k_pool[page, :, slot], krows[i])
        np.testing.assert_array_equal(kv.v_pool[page, :, slot], vrows[i])
        touched[page, :, slot] = True
    assert np.all(kv.k_pool[~touched] == 0x7FC0) and np.all(kv.v_pool[~touched] == 0x7FC0)


def test_kv_write_rows_errors(orc):
    num_pages, Hkv, P, d = 4, 1, 4, 8
    kp, vp = _tiny_pool(None, num_pages, Hkv, P, d)
    pt = np.array([[0, 1, -1], [2, 7, 3]], np.int32)
    kv = orc.KvPool(kp, vp, pt, P)
    z = np.zeros((1, Hkv, d), np.uint16)
    assert orc.kv_write_rows(kv, [0], [9], z, z) == orc.ERR_PAGE      # entry -1
    assert orc.kv_write_rows(kv, [1], [5], z, z) == orc.ERR_PAGE      # entry 7 >= num_pages
    assert orc.kv_write_rows(kv, [0], [12], z, z) == orc.ERR_COVER    # beyond the table width
    assert orc.kv_write_rows(kv, [0], [-1], z, z) == orc.ERR_POS
    assert np.all(kv.k_pool == 0x7FC0)


def test_kv_write_rows_fp8_matches_library_quantiser(orc):
    rng = np.random.default_rng(3)
    num_pages, Hkv, P, d, n = 6, 2, 8, 16, 20
    kp, vp = _tiny_pool(rng, num_pages, Hkv, P, d, "fp8")
    pt = rng.permutation(num_pages)[:3].reshape(1, 3).astype(np.int32)
    ks = rng.uniform(0.001, 0.05, (num_pages, Hkv)).astype(np.float32)
    vs = rng.uniform(0.001, 0.05, (num_pages, Hkv)).astype(np.float32)
    kv = orc.KvPool(kp, vp, pt, P, ks, vs)
    kf = torch.randn((n, Hkv, d), generator=torch.Generator().manual_seed(4)).to(torch.bfloat16)
    vf = torch.randn((n, Hkv, d), generator=torch.Generator().manual_seed(5)).to(torch.bfloat16)
    assert orc.kv_write_rows(kv, np.zeros(n, np.int32), np.arange(n, dtype=np.int32), bf16_bits(kf), bf16_bits(vf)) == 0
    for p in range(n):
        page, slot = pt[0, p // P], p % P
        for g in range(Hkv):
            for pool, src, sc in ((kv.k_pool, kf, ks), (kv.v_pool, vf, vs)):
                q = src[p, g].float() / torch.tensor(sc[page, g])     # IEEE fp32 division
                want = q.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
                # the library conversion does not saturate; the format's satfinite value does
                sat = (q.abs() >= 464).numpy()
                want = np.where(sat, np.where(q.numpy() < 0, 0xFE, 0x7E), want).astype(np.uint8)
                np.testing.assert_array_equal(pool[page, g, slot], want)


# ---- attention ----------------------------------------------------------------------------------

def _attn_case(orc, rng, B, k, Hq, Hkv, d, P, ctxs, poison=True, fp8=False):
    """Random pool + dense copies of every branch's keys, written by the test itself."""
    maxp = max(ctxs) + k + 1
    npb = (maxp + P - 1) // P
    num_pages = B * npb + 3
    perm = rng.permutation(num_pages)[:B * npb].reshape(B, npb).astype(np.int32)
    kp, vp = _tiny_pool(rng, num_pages, Hkv, P, d, "fp8" if fp8 else "bf16")
    if not poison:
        kp[:] = 0
        vp[:] = 0
    dense_k = np.zeros((B, maxp, Hkv, d))
    dense_v = np.zeros((B, maxp, Hkv, d))
    ksc = vsc = None
    if fp8:
        ksc = rng.uniform(0.01, 0.02, (num_pages, Hkv)).astype(np.float32)
        vsc = rng.uniform(0.01, 0.02, (num_pages, Hkv)).astype(np.float32)
    for b in range(B):
        for p in range(ctxs[b] + k + 1):
            page, slot = perm[b, p // P], p % P
            if fp8:
                codes_k = rng.integers(0, 0x7E, (Hkv, d)).astype(np.uint8) | (rng.integers(0, 2, (Hkv, d)) * 0x80).astype(np.uint8)
                codes_v = rng.integers(0, 0x7E, (Hkv, d)).astype(np.uint8) | (rng.integers(0, 2, (Hkv, d)) * 0x80).astype(np.uint8)
                kp[page, :, slot] = codes_k
                vp[page, :, slot] = codes_v
                lib_k = torch.from_numpy(codes_k).view(torch.float8_e4m3fn).double().numpy()
                lib_v = torch.from_numpy(codes_v).view(torch.float8_e4m3fn).double().numpy()
                dense_k[b, p] = lib_k * ksc[page][:, None]
                dense_v[b, p] = lib_v * vsc[page][:, None]
            else:
                kb = bf16_bits(torch.randn((Hkv, d), dtype=torch.float64).to(torch.bfloat16))
                vb = bf16_bits(torch.randn((Hkv, d), dtype=torch.float64).to(torch.bfloat16))
                kp[page, :, slot] = kb
                vp[page, :, slot] = vb
                dense_k[b, p] = bits_to_f64(kb)
                dense_v[b, p] = bits_to_f64(vb)
    kv = orc.KvPool(kp, vp, perm, P, ksc, vsc)
    R = B * (k + 1)
    q = bf16_bits(torch.randn((R, Hq, d), dtype=torch.float64).to(torch.bfloat16))
    return kv, q, dense_k, dense_v


@pytest.mark.parametrize("fp8", [False, True])
def test_attention_matches_sdpa_fp64(orc, fp8):
    torch.manual_seed(11)
    rng = np.random.default_rng(11)
    B, k, Hq, Hkv, d, P = 3, 2, 4, 2, 8, 4
    ctxs = [1, 7, 12]
    kv, q, dk, dv = _attn_case(orc, rng, B, k, Hq, Hkv, d, P, ctxs, fp8=fp8)
    scale = 1 / math.sqrt(d)
    out, err = orc.verify_attn(kv, ctxs, B, k, Hq, q, scale)
    assert err == 0 and np.isfinite(out).all()
    qd = bits_to_f64(q).reshape(B * (k + 1), Hq, d)
    for b in range(B):
        for j in range(k + 1):
            p = ctxs[b] + j
            r = b * (k + 1) + j
            # library routine: SDPA over the row's exact key list, GQA by consecutive grouping
            kk = torch.from_numpy(dk[b, :p + 1]).permute(1, 0, 2)[None]    # [1, Hkv, T, d]
            vv = torch.from_numpy(dv[b, :p + 1]).permute(1, 0, 2)[None]
            qq = torch.from_numpy(qd[r])[None, :, None, :]                   # [1, Hq, 1, d]
            ref = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, scale=scale, enable_gqa=True)
            np.testing.assert_allclose(out[r], ref[0, :, 0].numpy(), rtol=1e-12, atol=1e-12)


def test_attention_closed_forms(orc):
    rng = np.random.default_rng(12)
    B, k, Hq, Hkv, d, P = 1, 0, 2, 1, 8, 4
    # one key: the output is V_0
    kv, q, dk, dv = _attn_case(orc, rng, B, k, Hq, Hkv, d, P, [0])
    out, _ = orc.verify_attn(kv, [0], B, k, Hq, q, 0.3)
    np.testing.assert_array_equal(out[0, 0], dv[0, 0, 0])
    # identical keys: the output is the mean of V
    kv, q, dk, dv = _attn_case(orc, rng, B, k, Hq, Hkv, d, P, [9])
    for p in range(10):
        page, slot = kv.page_table[0, p // P], p % P
        kv.k_pool[page, :, slot] = kv.k_pool[kv.page_table[0, 0], :, 0]
    out, _ = orc.verify_attn(kv, [9], B, k, Hq, q, 0.3)
    np.testing.assert_allclose(out[0, 1], dv[0, :10, 0].mean(axis=0), rtol=1e-13, atol=1e-13)
    # a score gap >= 50: the output is V of the best key
    kv, q, dk, dv = _attn_case(orc, rng, B, k, Hq, Hkv, d, P, [5])
    qv = bits_to_f64(q)[0, 0]
    best = 3
    page, slot = kv.page_table[0, best // P], best % P
    kv.k_pool[page, 0, slot] = bf16_bits(torch.from_numpy(np.sign(qv) * 64.0).to(torch.bfloat16))
    out, _ = orc.verify_attn(kv, [5], B, k, Hq, q, 1.0)
    np.testing.assert_allclose(out[0, 0], dv[0, best, 0], rtol=0, atol=1e-15)


def test_attention_page_permutation_and_poison_invariance(orc):
    rng = np.random.default_rng(13)
    B, k, Hq, Hkv, d, P = 2, 3, 4, 2, 8, 4
    ctxs = [5, 10]
    kv, q, dk, dv = _attn_case(orc, rng, B, k, Hq, Hkv, d, P, ctxs, poison=True)
    out1, err = orc.verify_attn(kv, ctxs, B, k, Hq, q, 0.35)
    assert err == 0 and np.isfinite(out1).all()
    # replace every unattended slot by zeros: bitwise the same outputs
    kp2, vp2 = kv.k_pool.copy(), kv.v_pool.copy()
    kp2[kp2 == 0x7FC0] = 0
    vp2[vp2 == 0x7FC0] = 0
    out2, _ = orc.verify_attn(orc.KvPool(kp2, vp2, kv.page_table, P), ctxs, B, k, Hq, q, 0.35)
    np.testing.assert_array_equal(out1, out2)
    # move every page elsewhere in a bigger pool: bitwise the same outputs
    num2 = kv.num_pages + 5
    perm = rng.permutation(num2)[:kv.num_pages]
    kp3 = np.full((num2,) + kv.k_pool.shape[1:], 0x7FC0, np.uint16)
    vp3 = kp3.copy()
    kp3[perm] = kv.k_pool
    vp3[perm] = kv.v_pool
    pt3 = perm[kv.page_table].astype(np.int32)
    out3, _ = orc.verify_attn(orc.KvPool(kp3, vp3, pt3, P), ctxs, B, k, Hq, q, 0.35)
    np.testing.assert_array_equal(out1, out3)


def test_attention_rows_equal_one_row_calls(orc):
    rng = np.random.default_rng(14)
    B, k, Hq, Hkv, d, P = 2, 3, 4, 1, 8, 4
    ctxs = [6, 3]
    kv, q, dk, dv = _attn_case(orc, rng, B, k, Hq, Hkv, d, P, ctxs)
    out, _ = orc.verify_attn(kv, ctxs, B, k, Hq, q, 0.35)
    qr = q.reshape(B * (k + 1), Hq, d)
    for b in range(B):
        for j in range(k + 1):
            one, _ = orc.verify_attn(orc.KvPool(kv.k_pool, kv.v_pool, kv.page_table[b:b + 1], P),
                                     [ctxs[b] + j], 1, 0, Hq, qr[b * (k + 1) + j][None], 0.35)
            np.testing.assert_array_equal(one[0], out[b * (k + 1) + j])
    items = np.array([3, 9, 30, 31], np.int32)
    sub, _ = orc.verify_attn_items(kv, ctxs, B, k, Hq, q, 0.35, items)
    np.testing.assert_array_equal(sub, out.reshape(-1, d)[items])


# ---- LM head -------------------------------------------------------------------------------------

def _lm_case(seed, M, V, H, planted=True):
    g = torch.Generator().manual_seed(seed)
    W = (0.02 * torch.randn((V, H), generator=g)).to(torch.bfloat16)
    ids = torch.randint(0, V, (M,), generator=g)
    if planted:
        w = W[ids].float()
        hid = (8.0 * w / w.norm(dim=1, keepdim=True) + 0.1 * torch.randn((M, H), generator=g)).to(torch.bfloat16)
    else:
        hid = torch.randn((M, H), generator=g).to(torch.bfloat16)
    return W, hid, ids


def test_lmhead_matches_library_matmul(orc):
    W, hid, _ = _lm_case(20, 9, 1500, 96, planted=False)
    ids, mx, gap, err = orc.lmhead_argmax(bf16_bits(hid), bf16_bits(W))
    logits = hid.double() @ W.double().T                 # library matmul, fp64
    want = torch.argmax(logits.float(), dim=1)           # decision on fp32 logits, first max
    assert err == 0
    np.testing.assert_array_equal(ids, want.numpy())
    np.testing.assert_allclose(mx, logits.max(dim=1).values.numpy(), rtol=1e-12)
    full = orc.lmhead_logits(bf16_bits(hid), bf16_bits(W))
    np.testing.assert_allclose(full, logits.numpy(), rtol=1e-12, atol=1e-12)


def test_lmhead_planted_margin_and_ties(orc):
    W, hid, planted = _lm_case(21, 16, 2048, 256)
    ids, mx, gap, _ = orc.lmhead_argmax(bf16_bits(hid), bf16_bits(W))
    np.testing.assert_array_equal(ids, planted.numpy())
    assert gap.min() >= 0.5
    # duplicate the winner into a higher and a lower index: the lowest index wins
    W2 = W.clone()
    lo = [int(v) - 1 for v in planted[:4]]
    for r in range(4):
        W2[lo[r]] = W2[planted[r]]
    W2[2047] = W2[planted[5]]
    ids2, _, gap2, _ = orc.lmhead_argmax(bf16_bits(hid), bf16_bits(W2))
    for r in range(4):
        assert ids2[r] == min(lo[r], int(planted[r])) and gap2[r] == 0.0
    assert ids2[5] == min(int(planted[5]), 2047)


def test_lmhead_d2t(orc):
    W, hid, planted = _lm_case(22, 6, 512, 64)
    d2t = np.random.default_rng(0).permutation(100000)[:512].astype(np.int32)
    ids, _, _, err = orc.lmhead_argmax(bf16_bits(hid), bf16_bits(W), d2t, 100000)
    assert err == 0
    np.testing.assert_array_equal(ids, d2t[planted.numpy()])
    ids, _, _, err = orc.lmhead_argmax(bf16_bits(hid), bf16_bits(W), d2t, 10)
    assert err == orc.ERR_D2T and np.all((ids == -1) | (ids < 10))


# ---- accept ----------------------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["greedy_accept_example.json", "accept_loop_example.json"])
def test_accept_golden(orc, name):
    with open(os.path.join(GOLDEN, name)) as f:
        fx = json.load(f)
    for c in fx["cases"]:
        k = len(c["drafts"])
        toks, n, a, npos, nxt = orc.accept(c["drafts"], c["ids"], [c["pos"]], 1, k)
        assert toks[0].tolist() == c["tokens"]
        assert (n[0], a[0], npos[0], nxt[0]) == (c["n"], c["accepted"], c["new_pos"], c["next"])


@pytest.mark.parametrize("k", range(0, 9))
def test_accept_exhaustive_patterns(orc, k):
    rng = np.random.default_rng(k)
    pats = list(itertools.product([True, False], repeat=k))
    B = len(pats)
    ids = rng.integers(0, 1000, (B, k + 1)).astype(np.int32)
    drafts = np.where(np.array(pats, bool).reshape(B, k), ids[:, :k], ids[:, :k] + 1000).astype(np.int32)
    pos = rng.integers(0, 5000, B).astype(np.int32)
    toks, n, a, npos, nxt = orc.accept(drafts, ids.reshape(-1), pos, B, k)
    for b, pat in enumerate(pats):
        want_a = next((i for i, m in enumerate(pat) if not m), k)
        assert a[b] == want_a and n[b] == want_a + 1 and npos[b] == pos[b] + want_a + 1
        assert toks[b, :want_a].tolist() == drafts[b, :want_a].tolist()
        assert toks[b, want_a] == ids[b, want_a] == nxt[b]
        assert np.all(toks[b, want_a + 1:] == -1)


def test_accept_stop_golden(orc):
    with open(os.path.join(GOLDEN, "accept_stop_example.json")) as f:
        fx = json.load(f)
    for c in fx["cases"]:
        k = len(c["drafts"])
        bud = None if c["budget"] is None else [c["budget"]]
        toks, n, a, npos, nxt, done = orc.accept_stop(c["drafts"], c["ids"], [c["pos"]], 1, k, c["stop"], bud)
        assert toks[0].tolist() == c["tokens"], c["note"]
        assert (n[0], a[0], npos[0], nxt[0], done[0]) == (c["n"], c["accepted"], c["new_pos"], c["next"], c["done"]), c["note"]


@pytest.mark.parametrize("k", [0, 1, 3, 6])
def test_accept_stop_reduces_to_greedy_and_is_a_prefix(orc, k):
    """No stop set and no budget gives the plain greedy result; with them, the kept tokens
    are a prefix of it, ending on the first stop token of the run or at the budget."""
    rng = np.random.default_rng(40 + k)
    pats = list(itertools.product([True, False], repeat=k))
    B = len(pats)
    ids = rng.integers(0, 8, (B, k + 1)).astype(np.int32)
    drafts = np.where(np.array(pats, bool).reshape(B, k), ids[:, :k], ids[:, :k] + 8).astype(np.int32)
    pos = rng.integers(0, 5000, B).astype(np.int32)
    base = orc.accept(drafts, ids.reshape(-1), pos, B, k)
    same = orc.accept_stop(drafts, ids.reshape(-1), pos, B, k)
    for x, y in zip(base, same[:5]):
        np.testing.assert_array_equal(x, y)
    assert not same[5].any()
    stop = [3, -1, 6]
    budget = rng.integers(-1, k + 3, B).astype(np.int32)
    toks, n, a, npos, nxt, done = orc.accept_stop(drafts, ids.reshape(-1), pos, B, k, stop, budget)
    btoks, bn = base[0], base[1]
    for b in range(B):
        run = btoks[b, :bn[b]].tolist()
        first = next((i for i, t in enumerate(run) if t in (3, 6)), None)
        want = len(run) if first is None else first + 1
        want = min(want, max(int(budget[b]), 0))
        assert n[b] == want and toks[b, :want].tolist() == run[:want] and np.all(toks[b, want:] == -1)
        assert npos[b] == pos[b] + want and a[b] == min(base[2][b], want)
        assert nxt[b] == (run[want - 1] if want else -1)
        ends_on_stop = want > 0 and run[want - 1] in (3, 6)
        assert done[b] == int(ends_on_stop or want == max(int(budget[b]), 0))


# ---- MTP input -----------------------------------------------------------------------------------

def test_mtp_input_closed_form(orc):
    H, V, M, eps = 64, 10, 3, 1e-6
    c = 0.375
    E = bf16_bits(torch.full((V, H), c).to(torch.bfloat16))
    hid = bf16_bits(torch.full((M, H), -2.0).to(torch.bfloat16))
    g_e = np.linspace(0.5, 1.5, H).astype(np.float32)
    g_h = np.linspace(1.5, 0.5, H).astype(np.float32)
    # fc = [I | 0] selects the embedding half, [0 | I] the hidden half
    for half in (0, 1):
        Wfc = np.zeros((H, 2 * H), np.float32)
        Wfc[np.arange(H), half * H + np.arange(H)] = 1.0
        concat, x, err = orc.mtp_input([1, 4, 9], E, hid, g_e, g_h, eps, bf16_bits(torch.from_numpy(Wfc).to(torch.bfloat16)))
        assert err == 0
        if half == 0:
            want = c / math.sqrt(c * c + eps) * g_e.astype(np.float64)
        else:
            want = -2.0 / math.sqrt(4.0 + eps) * g_h.astype(np.float64)
        want_bf = bits_to_f64(bf16_bits(torch.from_numpy(want).to(torch.bfloat16)))
        for m in range(M):
            np.testing.assert_array_equal(x[m], want_bf)


def test_mtp_input_matches_library_ops(orc):
    g = torch.Generator().manual_seed(30)
    H, V, M, eps = 128, 50, 5, 1e-6
    E = (0.02 * torch.randn((V, H), generator=g)).to(torch.bfloat16)
    hid = torch.randn((M, H), generator=g).to(torch.bfloat16)
    g_e = (0.5 + torch.rand(H, generator=g)).float()
    g_h = (0.5 + torch.rand(H, generator=g)).float()
    Wfc = (0.02 * torch.randn((H, 2 * H), generator=g)).to(torch.bfloat16)
    tok = torch.tensor([0, 49, 7, 7, 23])
    concat, x, err = orc.mtp_input(tok.numpy(), bf16_bits(E), bf16_bits(hid), g_e.numpy(), g_h.numpy(), eps,
                                   bf16_bits(Wfc))
    assert err == 0
    rms = lambda y, gg: y / torch.sqrt((y * y).mean(dim=-1, keepdim=True) + eps) * gg.double()
    e_half = rms(E[tok].double(), g_e).to(torch.bfloat16)
    h_half = rms(hid.double(), g_h).to(torch.bfloat16)
    ref_c = torch.cat([e_half, h_half], dim=1)
    # the fp64 norm can land on the other side of a bf16 rounding boundary only by 1 ulp
    diff = np.abs(bits_to_f64(concat) - ref_c.double().numpy())
    assert (diff <= np.abs(ref_c.double().numpy()) * 2 ** -8 + 1e-30).all()
    np.testing.assert_array_equal(concat, bf16_bits(ref_c))
    ref_x = bits_to_f64(concat) @ Wfc.double().numpy().T
    np.testing.assert_allclose(x, ref_x, rtol=1e-12, atol=1e-12)
    _, _, err = orc.mtp_input([50, 0, 0, 0, 0], bf16_bits(E), bf16_bits(hid), g_e.numpy(), g_h.numpy(), eps,
                              bf16_bits(Wfc))
    assert err == orc.ERR_TOKEN


# ---- whole step: the emitted stream equals one-row greedy decoding ------------------------------

class OracleSide:
    """Drives the toy model through the oracle (pool, page table and positions on the host)."""

    def __init__(self, orc, lm: ToyLM, ctx_tokens, max_len, poison=True):
        self.orc, self.lm = orc, lm
        P = lm.P
        npg = (max_len + P - 1) // P
        self.num_pages = npg + 3
        rng = np.random.default_rng(99)
        pt = rng.permutation(self.num_pages)[:npg].reshape(1, npg).astype(np.int32)
        fill = 0x7FC0 if poison else 0
        shape = (self.num_pages, lm.Hkv, P, lm.d)
        self.kv = orc.KvPool(np.full(shape, fill, np.uint16), np.full(shape, fill, np.uint16), pt, P)
        for p, x in enumerate(ctx_tokens):
            _, kk, vv = lm.qkv(x, p)
            assert orc.kv_write_rows(self.kv, [0], [p], bf16_bits(kk)[None], bf16_bits(vv)[None]) == 0
        self.attn_log = []

    def step(self, fed, pos, k):
        lm, orc = self.lm, self.orc
        qs, ks, vs = zip(*[lm.qkv(x, pos + j) for j, x in enumerate(fed)])
        q, kn, vn = torch.stack(qs), torch.stack(ks), torch.stack(vs)
        assert orc.kv_append(self.kv, [pos], 1, k, bf16_bits(kn), bf16_bits(vn)) == 0
        out, err = orc.verify_attn(self.kv, [pos], 1, k, lm.Hq, bf16_bits(q), 1 / math.sqrt(lm.d))
        assert err == 0 and np.isfinite(out).all()
        o_bf = torch.from_numpy(out).to(torch.bfloat16)
        self.attn_log.append(out)
        hid = torch.stack([lm.hidden(x, pos + j, lm.target(x, pos + j, o_bf[j])) for j, x in enumerate(fed)])
        ids, _, gap, _ = orc.lmhead_argmax(bf16_bits(hid), bf16_bits(lm.W))
        assert gap.min() > 0.5
        toks, n, a, npos, nxt = orc.accept(np.array(fed[1:], np.int32), ids, [pos], 1, k)
        assert npos[0] == pos + n[0]
        return toks[0, :n[0]].tolist(), int(a[0])


@pytest.mark.parametrize("k", [1, 3, 6])
def test_spec_stream_equals_one_row_greedy(orc, k):
    lm = ToyLM()
    ctx = [int(t) for t in np.random.default_rng(5).integers(0, lm.V, 21)]
    n_tok = 40
    ref_side = OracleSide(orc, lm, ctx, 21 + n_tok + 20)
    ref = run_greedy(ref_side, lm, x0=ctx[-1] + 1, pos0=21, n_tokens=n_tok + k + 1)
    side = OracleSide(orc, lm, ctx, 21 + n_tok + 20)
    got, acc = run_spec(side, lm, x0=ctx[-1] + 1, pos0=21, n_tokens=n_tok, k=k, ref=ref)
    assert got == ref[:n_tok]
    assert 0 < sum(acc) < k * len(acc)      # both accepted and rejected drafts occurred
    # poison-free pool: the same stream and bitwise the same attention outputs
    side0 = OracleSide(orc, lm, ctx, 21 + n_tok + 20, poison=False)
    got0, _ = run_spec(side0, lm, x0=ctx[-1] + 1, pos0=21, n_tokens=n_tok, k=k, ref=ref)
    assert got0 == got
    for a1, a0 in zip(side.attn_log, side0.attn_log):
        np.testing.assert_array_equal(a1, a0)


def test_hidden_pool_gather_scatter_are_fancy_indexing(orc):
    """h_gather is numpy's row indexing hpool[hslot]; h_scatter is hpool[hslot] = h (distinct
    slots); an invalid slot is reported and its row skipped; scatter then gather returns the
    scattered rows (span-02 `Spec::body_inner`: gather at a step's start, scatter at its end)."""
    rng = np.random.default_rng(77)
    S, H, B = 37, 33, 9
    hpool = rng.integers(0, 1 << 16, (S, H)).astype(np.uint16)
    hslot = rng.permutation(S)[:B].astype(np.int32)
    got, err = orc.h_gather(hpool, hslot)
    assert err == 0 and np.array_equal(got, hpool[hslot])
    h_new = rng.integers(0, 1 << 16, (B, H)).astype(np.uint16)
    pool2 = hpool.copy()
    assert orc.h_scatter(pool2, h_new, hslot) == 0
    want = hpool.copy()
    want[hslot] = h_new
    assert np.array_equal(pool2, want)
    back, err = orc.h_gather(pool2, hslot)
    assert err == 0 and np.array_equal(back, h_new)
    bad = hslot.copy()
    bad[2], bad[5] = -1, S
    got, err = orc.h_gather(hpool, bad)
    assert err == orc.ERR_SLOT
    ok = np.ones(B, bool)
    ok[[2, 5]] = False
    assert np.array_equal(got[ok], hpool[bad[ok]]) and not got[~ok].any()
    pool3 = hpool.copy()
    assert orc.h_scatter(pool3, h_new, bad) == orc.ERR_SLOT
    want = hpool.copy()
    want[bad[ok]] = h_new[ok]
    assert np.array_equal(pool3, want)

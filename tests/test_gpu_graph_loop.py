"""Device-resident step state: a speculative decode loop captured once in a CUDA graph and
replayed step after step, with no host upload of positions or tokens between steps.

The step (append, verify attention, LM-head argmax, acceptance) runs through the C ABI;
spec_accept advances the branch positions in place (out_pos = pos) and writes the next
fed token (out_next) and the draft head's hidden row (h_out) on the device (span-02
spec.rs, module documentation; flashrt-structures decode_loop/whole_step.py,
`generate_speculative`: state stays on the device, pos advances by accepted + 1). The
toy model around it is a table model whose rows are gathers, so that it can sit inside
the graph. Checked against the oracle: the emitted stream of every branch equals one-row
greedy decoding of the same toy model, the positions equal the context length plus the
tokens emitted, and the KV pool's committed slots equal an oracle pool written from the
emitted stream.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle as orc
from gpu_harness import DEV, lm_ws
from greedy_speculative_decode_spec_gb300 import _binding as bnd
from greedy_speculative_decode_spec_gb300.step import PagedKv
from greedy_speculative_decode_spec_gb300.workloads import bits

pytestmark = pytest.mark.gpu


class TableToy:
    """Toy target model made of gathers: token x at position p has
    q = bf16(Eq[x] + Pq[p]) (k and v likewise), target id (x * 1000003 + p * 7919 + seed) mod V,
    and a hidden row planted on the target: bf16(8 W[t] / |W[t]| + 0.1 N[(31 x + p) mod 97])."""

    def __init__(self, V=2048, H=256, Hq=8, Hkv=2, d=64, L=4096, seed=5):
        g = torch.Generator().manual_seed(seed)
        self.V, self.H, self.Hq, self.Hkv, self.d, self.seed = V, H, Hq, Hkv, d, seed
        self.Eq, self.Ek, self.Ev = (torch.randn(V, h, d, generator=g) for h in (Hq, Hkv, Hkv))
        self.Pq, self.Pk, self.Pv = (0.5 * torch.randn(L, h, d, generator=g) for h in (Hq, Hkv, Hkv))
        self.W = (0.02 * torch.randn(V, H, generator=g)).to(torch.bfloat16)
        self.N = torch.randn(97, H, generator=g)

    def to(self, dev):
        t = TableToy.__new__(TableToy)
        t.__dict__.update({k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in self.__dict__.items()})
        return t

    def qkv(self, x, p):
        x, p = x.long(), p.long()
        return ((self.Eq[x] + self.Pq[p]).to(torch.bfloat16), (self.Ek[x] + self.Pk[p]).to(torch.bfloat16),
                (self.Ev[x] + self.Pv[p]).to(torch.bfloat16))

    def target(self, x, p):
        return (x.long() * 1000003 + p.long() * 7919 + self.seed) % self.V

    def hidden(self, x, p, tgt):
        w = self.W[tgt].float()
        h = 8.0 * w / w.norm(dim=-1, keepdim=True) + 0.1 * self.N[(31 * x.long() + p.long()) % 97]
        return h.to(torch.bfloat16)


def oracle_greedy(toy: TableToy, x0: int, pos0: int, n: int):
    """One-row greedy decoding of the toy on the oracle: the LM-head argmax of each row."""
    out, x, p = [], x0, pos0
    while len(out) < n:
        xt, pt = torch.tensor([x]), torch.tensor([p])
        hid = toy.hidden(xt, pt, toy.target(xt, pt))
        ids, _, _, e = orc.lmhead_argmax(bits(hid), bits(toy.W))
        assert e == 0
        out.append(int(ids[0]))
        x, p = out[-1], p + 1
    return out


def _mix(a: torch.Tensor) -> torch.Tensor:
    """A counter-based hash to [0, 2^31) (drafter randomness on the device)."""
    a = (a * 0x9E3779B1 + 0x7F4A7C15) & 0xFFFFFFFF
    a = ((a ^ (a >> 15)) * 0x2C1B3C6D) & 0xFFFFFFFF
    a = ((a ^ (a >> 12)) * 0x297A2D39) & 0xFFFFFFFF
    return (a ^ (a >> 15)) & 0x7FFFFFFF


@pytest.mark.parametrize("k", [3, 6])
def test_graph_replayed_loop_emits_the_greedy_stream(k):
    B, P, STEPS, p_hit = 3, 16, 64, 0.75
    toy_c = TableToy()
    toy = toy_c.to(DEV)
    ctx_len = [37, 150, 90]
    x0_host = [11, 401, 1999]
    n_ref = STEPS * (k + 1) + k + 1
    refs = [oracle_greedy(toy_c, x0_host[b], ctx_len[b], n_ref) for b in range(B)]

    # paged pool holding each branch's context (context tokens: a fixed pseudo-random stream)
    max_pos = max(ctx_len) + n_ref + k + 2
    npg = (max_pos + P - 1) // P
    num_pages = B * npg + 5
    pt = torch.from_numpy(np.random.default_rng(17).permutation(num_pages)[:B * npg].reshape(B, npg).astype(np.int32))
    kv = PagedKv(num_pages, toy_c.Hkv, P, toy_c.d, pt.to(DEV))
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ctx_tok = [torch.from_numpy(np.random.default_rng(100 + b).integers(0, toy_c.V, ctx_len[b])) for b in range(B)]
    rb = torch.cat([torch.full((ctx_len[b],), b, dtype=torch.int32) for b in range(B)])
    rp = torch.cat([torch.arange(ctx_len[b], dtype=torch.int32) for b in range(B)])
    _, kr, vr = toy_c.qkv(torch.cat(ctx_tok), rp)
    kv.write_rows(rb.to(DEV), rp.to(DEV), kr.to(DEV), vr.to(DEV), dev_err=err)

    # device-resident state
    i32 = dict(dtype=torch.int32, device=DEV)
    pos = torch.tensor(ctx_len, **i32)
    x0 = torch.tensor(x0_host, **i32)
    cnt = torch.zeros(B, dtype=torch.int64, device=DEV)
    step_ctr = torch.zeros(1, dtype=torch.int64, device=DEV)
    ref_d = torch.tensor(refs, dtype=torch.int64, device=DEV)
    LOG = n_ref + k + 2
    log = torch.full((B, LOG + 1), -1, dtype=torch.int64, device=DEV)  # last column: scratch
    drafts = torch.zeros((B, k), **i32)
    R = B * (k + 1)
    attn_out = torch.empty((R, toy_c.Hq, toy_c.d), dtype=torch.bfloat16, device=DEV)
    aws = torch.zeros(max(bnd.spec_verify_attn_workspace(kv.desc, B, k, toy_c.Hq, max_pos), 256), dtype=torch.uint8,
                      device=DEV)
    lws = lm_ws(R, toy_c.V, toy_c.H)
    ids = torch.empty(R, **i32)
    toks = torch.empty((B, k + 1), **i32)
    n_out, a_out = torch.empty(B, **i32), torch.empty(B, **i32)
    h_next = torch.empty((B, toy_c.H), dtype=torch.bfloat16, device=DEV)
    jj = torch.arange(k + 1, device=DEV)
    bb = torch.arange(B, device=DEV)

    def make_drafts():
        # draft j copies the reference stream with probability p_hit, else a different token
        want = ref_d.gather(1, cnt[:, None] + jj[None, :k])
        r = _mix(step_ctr * 7919 + bb[:, None] * 131 + jj[None, :k])
        wrong = (want + 1 + (r >> 8) % (toy_c.V - 1)) % toy_c.V
        drafts.copy_(torch.where((r & 0xFF) < int(p_hit * 256), want, wrong).to(torch.int32))

    def step():
        fed = torch.cat([x0[:, None], drafts], dim=1)                 # [B][k+1]
        p = pos[:, None].long() + jj[None, :]
        q, kn, vn = toy.qkv(fed.reshape(-1), p.reshape(-1))
        bnd.spec_kv_append(kv.desc, pos, B, k, kn, vn, err)
        bnd.spec_verify_attn(kv.desc, pos, B, k, toy_c.Hq, q, 1.0 / math.sqrt(toy_c.d), attn_out, aws, max_pos, err)
        hid = toy.hidden(fed.reshape(-1), p.reshape(-1), toy.target(fed.reshape(-1), p.reshape(-1)))
        bnd.spec_lmhead_argmax(hid, toy.W, ids, lws, dev_err=err)
        bnd.spec_accept(drafts, ids, pos, B, k, toks, n_out, a_out, pos, x0, hidden=hid, h_out=h_next)
        keep = jj[None, :] < n_out[:, None].long()
        col = torch.where(keep, cnt[:, None] + jj[None, :], torch.full_like(cnt[:, None], LOG))
        log.scatter_(1, col, toks.long())
        cnt.add_(n_out.long())
        step_ctr.add_(1)
        make_drafts()

    make_drafts()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # one eager step warms up the libraries before capture
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(STEPS - 1):
        g.replay()
    torch.cuda.synchronize()
    assert int(err.item()) == 0

    emitted = cnt.cpu().numpy()
    L = log.cpu().numpy()
    for b in range(B):
        n = int(emitted[b])
        assert STEPS <= n <= STEPS * (k + 1)
        assert list(L[b, :n]) == refs[b][:n], f"branch {b}: stream differs from one-row greedy"
    assert np.array_equal(pos.cpu().numpy(), np.array(ctx_len) + emitted)
    assert np.array_equal(x0.cpu().numpy(), [refs[b][int(emitted[b]) - 1] for b in range(B)])
    assert emitted.sum() > B * STEPS * 1.5, "the drafter should get tokens accepted"

    # the committed KV slots hold exactly the rows of context + emitted stream (fed tokens:
    # x0, then the emitted tokens except the last, at positions ctx_len .. pos-1)
    okv = orc.KvPool(np.zeros(kv.k.shape, np.uint16), np.zeros(kv.v.shape, np.uint16), pt.numpy(), P)
    fed_rows, fed_pos, fed_b = [], [], []
    for b in range(B):
        n = int(emitted[b])
        stream = list(ctx_tok[b].numpy()) + [x0_host[b]] + refs[b][:n - 1]
        fed_rows += stream
        fed_pos += list(range(len(stream)))
        fed_b += [b] * len(stream)
    _, ko, vo = toy_c.qkv(torch.tensor(fed_rows), torch.tensor(fed_pos))
    assert orc.kv_write_rows(okv, np.array(fed_b, np.int32), np.array(fed_pos, np.int32), bits(ko), bits(vo)) == 0
    gk, gv = bits(kv.k), bits(kv.v)
    for b in range(B):
        for p in range(int(ctx_len[b] + emitted[b])):
            pg, sl = int(pt[b, p // P]), p % P
            assert np.array_equal(gk[pg, :, sl], okv.k_pool[pg, :, sl]), (b, p)
            assert np.array_equal(gv[pg, :, sl], okv.v_pool[pg, :, sl]), (b, p)

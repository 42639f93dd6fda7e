"""Draft side: the MTP input stage x = fc([rmsnorm(E[tok]), rmsnorm(h)]) and the trimmed
draft head with its d2t map, then the verify of the drafts it produced."""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

import oracle as orc
from gpu_harness import DEV, assert_attn_close, gpu_lmhead
from greedy_speculative_decode_spec_gb300 import _binding as bnd
from greedy_speculative_decode_spec_gb300.workloads import (DRAFT_CONFIG, bits, config4_verify, draft_inputs, scaled,
                                                            verify_inputs)
from test_gpu_parity import _step_parity

pytestmark = pytest.mark.gpu

SMALL_DRAFT = dataclasses.replace(DRAFT_CONFIG, M=16, H=256, V=3001, V_draft=1000, seed=77)


def _gpu_mtp(di):
    M, H = di.h.shape
    x = torch.empty((M, H), dtype=torch.bfloat16, device=DEV)
    ws = torch.zeros(bnd.spec_mtp_input_workspace(M, H), dtype=torch.uint8, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    bnd.spec_mtp_input(di.tok.cuda(), di.E.cuda(), di.h.cuda(), di.g_emb.cuda(), di.g_hid.cuda(), di.cfg.eps,
                       di.W_fc.cuda(), x, ws, err)
    torch.cuda.synchronize()
    return x, int(err.item())


def _near_tie_ok(gpu_ids, x_bits, W_draft, d2t, tau):
    """ids must match the oracle where its top-2 gap exceeds tau; elsewhere the GPU's choice
    must be within tau of the oracle's maximum logit."""
    oids, omx, gap, err = orc.lmhead_argmax(x_bits, bits(W_draft), d2t.numpy(), 1 << 30)
    assert err == 0
    clear = gap > tau
    np.testing.assert_array_equal(gpu_ids[clear], oids[clear])
    if (~clear).any():
        inv = {int(t): i for i, t in enumerate(d2t.numpy())}
        rows = np.nonzero(~clear)[0]
        lg = orc.lmhead_logits(x_bits[rows], bits(W_draft))
        for j, r in enumerate(rows):
            assert lg[j, inv[int(gpu_ids[r])]] >= omx[r] - tau[r]
    return oids


def _draft_side(dc, W_verify=None):
    di = draft_inputs(dc, E=W_verify, V=dc.V, H=dc.H, V_draft=dc.V_draft, M=dc.M)
    x, e = _gpu_mtp(di)
    assert e == 0
    concat, x_ref, oe = orc.mtp_input(di.tok.numpy(), bits(di.E), bits(di.h), di.g_emb.numpy(), di.g_hid.numpy(),
                                      dc.eps, bits(di.W_fc))
    assert oe == 0
    assert_attn_close(x, x_ref, "MTP x")
    # draft head on the same bf16 x for both sides: only fp32-vs-fp64 accumulation differs
    x_ref_bf = torch.from_numpy(x_ref).to(torch.bfloat16)
    d2t = di.d2t
    ids_same, _, e = gpu_lmhead(x_ref_bf.cuda(), di.W_draft.cuda(), d2t=d2t.cuda(), d2t_limit=dc.V)
    assert e == 0
    xb = bits(x_ref_bf)
    absx = np.abs(x_ref_bf.double().numpy())
    tau_same = 1e-4 * absx.sum(axis=1) * float(di.W_draft.float().abs().max()) + 1e-4
    oracle_drafts = _near_tie_ok(ids_same, xb, di.W_draft, d2t, tau_same)
    # the GPU's own chain: x from the GPU, then the draft head
    ids_chain, _, e = gpu_lmhead(x, di.W_draft.cuda(), d2t=d2t.cuda(), d2t_limit=dc.V)
    assert e == 0
    rms_w = float(di.W_draft.float().pow(2).mean().sqrt())
    tau_chain = 20 * 2.0 ** -9 * np.sqrt((absx ** 2).sum(axis=1)) * rms_w + tau_same
    _near_tie_ok(ids_chain, xb, di.W_draft, d2t, tau_chain)
    return di, oracle_drafts


def test_mtp_input_and_draft_head_small():
    _draft_side(SMALL_DRAFT)


def test_draft_then_verify_small():
    dc = SMALL_DRAFT
    vcfg = scaled(config4_verify(dc), V=dc.V, H=dc.H, ctx_range=(30, 1500), num_pages=1024)
    di, drafts = _draft_side(dc)
    vi = verify_inputs(vcfg, drafts=torch.from_numpy(drafts).view(vcfg.B, vcfg.k), W=di.E)
    _step_parity(vi, full_oracle=True)


def test_draft_then_verify_full_size():
    dc = DRAFT_CONFIG
    vcfg = config4_verify(dc)
    from greedy_speculative_decode_spec_gb300.workloads import make_lm_head
    W = make_lm_head(dc.V, dc.H, vcfg.seed + 7)
    di, drafts = _draft_side(dc, W_verify=W)
    vi = verify_inputs(vcfg, drafts=torch.from_numpy(drafts).view(vcfg.B, vcfg.k), W=W)
    _step_parity(vi, full_oracle=False)


def test_mtp_bad_token_is_reported():
    di = draft_inputs(SMALL_DRAFT, V=SMALL_DRAFT.V, H=SMALL_DRAFT.H, V_draft=SMALL_DRAFT.V_draft, M=SMALL_DRAFT.M)
    di.tok[3] = SMALL_DRAFT.V + 1
    x, e = _gpu_mtp(di)
    assert e & bnd.DEVERR_TOKEN


def test_graph_replay_mixes_launch_sizes_of_one_kernel():
    """One CUDA graph holding launches of the same kernel with different shared-memory
    sizes (a 64-row and a 16-row MTP input, a 64-row and an 80-row LM head), replayed
    twice: the replays must reproduce the eager results bit for bit."""
    dc = SMALL_DRAFT
    big = draft_inputs(dc, V=dc.V, H=dc.H, V_draft=dc.V_draft, M=64)
    small = draft_inputs(dataclasses.replace(dc, seed=78), V=dc.V, H=dc.H, V_draft=dc.V_draft, M=16)
    hid80 = torch.randn((80, dc.H), generator=torch.Generator().manual_seed(5)).to(torch.bfloat16).cuda()
    W = small.W_draft.cuda()
    bufs = []
    for di in (big, small):
        M, H = di.h.shape
        bufs.append(dict(di=di, dev={k: getattr(di, k).cuda() for k in ("tok", "E", "h", "g_emb", "g_hid", "W_fc")},
                         x=torch.empty((M, H), dtype=torch.bfloat16, device=DEV),
                         ws=torch.zeros(bnd.spec_mtp_input_workspace(M, H), dtype=torch.uint8, device=DEV)))
    ids64 = torch.empty(64, dtype=torch.int32, device=DEV)
    ids80 = torch.empty(80, dtype=torch.int32, device=DEV)
    ws64 = torch.zeros(bnd.spec_lmhead_workspace(64, W.shape[0], dc.H), dtype=torch.uint8, device=DEV)
    ws80 = torch.zeros(bnd.spec_lmhead_workspace(80, W.shape[0], dc.H), dtype=torch.uint8, device=DEV)

    def step():
        for b in bufs:
            d = b["dev"]
            bnd.spec_mtp_input(d["tok"], d["E"], d["h"], d["g_emb"], d["g_hid"], dc.eps, d["W_fc"], b["x"], b["ws"])
        bnd.spec_lmhead_argmax(bufs[0]["x"], W, ids64, ws64)
        bnd.spec_lmhead_argmax(hid80, W, ids80, ws80)

    step()
    torch.cuda.synchronize()
    want = [b["x"].clone() for b in bufs] + [ids64.clone(), ids80.clone()]
    for t in [b["x"] for b in bufs] + [ids64, ids80]:
        t.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    got = [b["x"] for b in bufs] + [ids64, ids80]
    for w_, g_ in zip(want, got):
        assert torch.equal(w_.view(torch.int16) if w_.dtype == torch.bfloat16 else w_,
                           g_.view(torch.int16) if g_.dtype == torch.bfloat16 else g_)

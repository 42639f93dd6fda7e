"""One batched verify step on the device: the calls of the C ABI in the order of
span-02 engine/crates/model/src/spec.rs, `Spec::body_inner` (KV append inside the
verify forward, attention, LM-head argmax, acceptance), plus the next draft step's
MTP input from the accepted rows (oxinfer src/qwen_mtp.rs, module documentation).

This module only allocates device buffers (through PyTorch) and issues the library
calls on one stream; every step of the path runs in the library's kernels.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import _binding as bnd


class PagedKv:
    """A shared paged KV pool on the device: K and V [num_pages][Hkv][P][d] (bf16, or
    uint8 E4M3 codes with fp32 scales [num_pages][Hkv]) and an int32 page table."""

    def __init__(self, num_pages: int, n_kv_heads: int, page_size: int, head_dim: int, page_table: torch.Tensor,
                 fp8: bool = False, poison_bits: int | None = None, k_scale=None, v_scale=None, device="cuda"):
        shape = (num_pages, n_kv_heads, page_size, head_dim)
        if fp8:
            fill = 0x7F if poison_bits is None else poison_bits
            self.k = torch.full(shape, fill, dtype=torch.uint8, device=device)
            self.v = torch.full(shape, fill, dtype=torch.uint8, device=device)
        else:
            fill = 0x7FC0 if poison_bits is None else poison_bits
            self.k = torch.full(shape, fill, dtype=torch.int16, device=device).view(torch.bfloat16)
            self.v = torch.full(shape, fill, dtype=torch.int16, device=device).view(torch.bfloat16)
        self.fp8 = fp8
        self.page_table = page_table.to(device=device, dtype=torch.int32).contiguous()
        self.k_scale = None if k_scale is None else k_scale.to(device=device, dtype=torch.float32).contiguous()
        self.v_scale = None if v_scale is None else v_scale.to(device=device, dtype=torch.float32).contiguous()
        self.page_size, self.head_dim, self.n_kv_heads, self.num_pages = page_size, head_dim, n_kv_heads, num_pages
        self.desc = bnd.make_kv_desc(self.k, self.v, self.page_table, page_size, self.k_scale, self.v_scale)

    def write_rows(self, row_branch, row_pos, k_rows, v_rows, dev_err=None, stream=None):
        bnd.spec_kv_write_rows(self.desc, row_branch, row_pos, k_rows, v_rows, dev_err, stream)


@dataclass
class StepOutputs:
    attn: torch.Tensor        # bf16 [R][Hq][d]
    ids: torch.Tensor         # int32 [R]
    max_logit: torch.Tensor   # fp32 [R]
    tokens: torch.Tensor      # int32 [B][k+1]
    n: torch.Tensor           # int32 [B]
    accepted: torch.Tensor    # int32 [B]
    new_pos: torch.Tensor     # int32 [B]
    next_tok: torch.Tensor    # int32 [B]
    h_next: torch.Tensor      # bf16 [B][H]
    mtp_x: torch.Tensor | None  # bf16 [B][H]
    dev_err: torch.Tensor     # int32 [1]


class VerifyStep:
    """Buffers and calls of one verify step for fixed (B, k, heads, H, V, max_pos)."""

    def __init__(self, kv: PagedKv, B: int, k: int, n_q_heads: int, W: torch.Tensor, max_pos: int,
                 mtp: dict | None = None, device="cuda"):
        self.kv, self.B, self.k, self.Hq, self.W, self.max_pos = kv, B, k, n_q_heads, W, max_pos
        self.V, self.H = W.shape
        R = B * (k + 1)
        self.R = R
        d = kv.head_dim
        self.scale = 1.0 / (d ** 0.5)
        i32 = dict(dtype=torch.int32, device=device)
        self.attn_ws = torch.zeros(max(bnd.spec_verify_attn_workspace(kv.desc, B, k, n_q_heads, max_pos), 256),
                                   dtype=torch.uint8, device=device)
        self.head_ws = torch.zeros(bnd.spec_lmhead_workspace(R, self.V, self.H), dtype=torch.uint8, device=device)
        self.out = StepOutputs(
            attn=torch.empty((R, n_q_heads, d), dtype=torch.bfloat16, device=device),
            ids=torch.empty(R, **i32), max_logit=torch.empty(R, dtype=torch.float32, device=device),
            tokens=torch.empty((B, k + 1), **i32), n=torch.empty(B, **i32), accepted=torch.empty(B, **i32),
            new_pos=torch.empty(B, **i32), next_tok=torch.empty(B, **i32),
            h_next=torch.empty((B, self.H), dtype=torch.bfloat16, device=device), mtp_x=None,
            dev_err=torch.zeros(1, **i32))
        self.mtp = mtp
        if mtp is not None:
            self.mtp_ws = torch.zeros(bnd.spec_mtp_input_workspace(B, self.H), dtype=torch.uint8, device=device)
            self.out.mtp_x = torch.empty((B, self.H), dtype=torch.bfloat16, device=device)
        # append 1, attention 2 (FP8 pools 3: the query split first), LM head 1, accept 1;
        # the MTP input adds 3
        self.launches_verify = 5 + (1 if kv.fp8 else 0)
        self.launches_mtp = 3 if mtp is not None else 0

    def run(self, pos, q, k_new, v_new, hidden, drafts, stream=None, with_mtp: bool = True) -> StepOutputs:
        """The verify step's calls on `stream`; with_mtp adds the next draft step's MTP input
        (when the step was built with one)."""
        o, kv = self.out, self.kv
        bnd.spec_kv_append(kv.desc, pos, self.B, self.k, k_new, v_new, o.dev_err, stream)
        bnd.spec_verify_attn(kv.desc, pos, self.B, self.k, self.Hq, q, self.scale, o.attn, self.attn_ws,
                             self.max_pos, o.dev_err, stream)
        bnd.spec_lmhead_argmax(hidden, self.W, o.ids, self.head_ws, max_logit=o.max_logit, dev_err=o.dev_err,
                               stream=stream)
        bnd.spec_accept(drafts, o.ids, pos, self.B, self.k, o.tokens, o.n, o.accepted, o.new_pos, o.next_tok,
                        hidden=hidden, h_out=o.h_next, stream=stream)
        if self.mtp is not None and with_mtp:
            m = self.mtp
            bnd.spec_mtp_input(o.next_tok, m["E"], o.h_next, m["g_emb"], m["g_hid"], m["eps"], m["W_fc"], o.mtp_x,
                               self.mtp_ws, o.dev_err, stream)
        return o


class StepGraphCache:
    """CUDA graphs of a step, one per key, e.g. (k, B, splits) (span-02
    engine/crates/model/src/spec.rs, `Spec::step_chunk`: a graph cache keyed by the step's
    shape, eager execution when capture fails).

    run(key, step) executes the step once per call: the first call for a key runs it
    eagerly (which also warms the libraries up), the second captures it and replays the
    graph, later calls replay it. The step must use the same device buffers on every call
    (its state, such as positions advanced in place by spec_accept, lives in them); a key
    whose capture raised runs eagerly from then on."""

    def __init__(self):
        self._graphs: dict = {}
        self._seen: set = set()
        self._eager: set = set()

    def run(self, key, step) -> None:
        g = self._graphs.get(key)
        if g is not None:
            g.replay()
            return
        if key in self._eager or key not in self._seen:
            self._seen.add(key)
            step()
            return
        g = torch.cuda.CUDAGraph()
        try:
            with torch.cuda.graph(g):
                step()
        except RuntimeError:
            self._eager.add(key)
            step()
            return
        self._graphs[key] = g
        g.replay()

    def captured(self, key) -> bool:
        return key in self._graphs

"""A toy deterministic target model for whole-step exactness checks.

The pages' exactness claim (span-02 spec.rs, module documentation; oxinfer
qwen_mtp.rs, `OXINFER_CHECK_SPEC` re-run of each verify token as a one-token
forward): a speculative loop emits exactly the tokens of one-row greedy decoding.

The toy model: token x at position p has seeded q/k/v rows (a function of x and p
only) and a hidden row planted on the id
    f(x, p, o) = (hash(x, p) + t(o)) mod V
where o is the row's attention output, so that the emitted stream depends on the
attention (reading a stale, rejected or poisoned slot changes it). Both the spec
loop and the one-row loop are driven by a `Side`: the oracle or the CUDA library.
"""
from __future__ import annotations

import numpy as np
import torch


class ToyLM:
    def __init__(self, V=512, H=256, Hq=4, Hkv=2, d=64, P=16, seed=7, use_attn=True):
        self.V, self.H, self.Hq, self.Hkv, self.d, self.P, self.seed = V, H, Hq, Hkv, d, P, seed
        self.use_attn = use_attn  # False: the stream ignores attention bits (cross-precision checks)
        g = torch.Generator().manual_seed(seed)
        self.W = (0.02 * torch.randn((V, H), generator=g)).to(torch.bfloat16)

    def _rng(self, x: int, p: int, salt: int):
        return np.random.default_rng([self.seed, salt, int(x), int(p)])

    def qkv(self, x: int, p: int):
        r = self._rng(x, p, 1)
        q = torch.from_numpy(r.standard_normal((self.Hq, self.d)).astype(np.float32)).to(torch.bfloat16)
        k = torch.from_numpy(r.standard_normal((self.Hkv, self.d)).astype(np.float32)).to(torch.bfloat16)
        v = torch.from_numpy(r.standard_normal((self.Hkv, self.d)).astype(np.float32)).to(torch.bfloat16)
        return q, k, v

    @staticmethod
    def attn_tag(o_bf16: torch.Tensor) -> int:
        """t(o): a small integer read from the bf16 bits of the row's attention output."""
        b = o_bf16.reshape(-1)[:8].view(torch.int16).to(torch.int64)
        return int((b & 0x7).sum().item())

    def target(self, x: int, p: int, o_bf16: torch.Tensor) -> int:
        h = (int(x) * 1000003 + int(p) * 7919 + self.seed) % self.V
        return (h + (self.attn_tag(o_bf16) if self.use_attn else 0)) % self.V

    def hidden(self, x: int, p: int, tgt: int) -> torch.Tensor:
        r = self._rng(x, p, 2)
        w = self.W[tgt].float()
        h = 8.0 * w / w.norm() + 0.1 * torch.from_numpy(r.standard_normal(self.H).astype(np.float32))
        return h.to(torch.bfloat16)


def run_greedy(side, lm: ToyLM, x0: int, pos0: int, n_tokens: int):
    """One-row greedy: each step feeds one token (k = 0) and emits the argmax."""
    out, x, pos = [], x0, pos0
    while len(out) < n_tokens:
        toks, _ = side.step([x], pos, 0)
        out += toks
        x, pos = toks[-1], pos + 1
    return out[:n_tokens]


def run_spec(side, lm: ToyLM, x0: int, pos0: int, n_tokens: int, k: int, ref: list, p_hit=0.7, seed=3):
    """Speculative loop; draft j copies the reference stream with probability p_hit."""
    rng = np.random.default_rng(seed)
    out, x, pos = [], x0, pos0
    accepted_hist = []
    while len(out) < n_tokens:
        drafts = []
        for j in range(k):
            want = ref[len(out) + j] if len(out) + j < len(ref) else 0
            if rng.random() < p_hit:
                drafts.append(int(want))
            else:
                drafts.append(int((want + 1 + rng.integers(lm.V - 1)) % lm.V))
        toks, a = side.step([x] + drafts, pos, k)
        accepted_hist.append(a)
        out += toks
        x, pos = toks[-1], pos + len(toks)
    return out[:n_tokens], accepted_hist

#!/usr/bin/env python3
"""Benchmark of the batched verify step (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--no-all]

A step = one pass of the verify hot path on one batch of synthetic input:
KV append -> verify attention -> LM head + argmax -> chain acceptance, on one stream
(captured in a CUDA graph). The draft-side workload (4) adds the MTP input and the trimmed
draft head in front of its verify. The same step followed by the next draft step's MTP
input is reported separately ("us_per_step_with_mtp_input").
The headline workload is the long-context FP8 verify (B=4, k=3, contexts 32K..128K, 40/8
heads, d=128, E4M3 pages of 64, H=5120, V=151936): the largest single-GPU workload, with
the most bytes per step. The other workloads are reported under "all_configs".

--only attn|lmhead runs just that call of the workload (W + K plain launches, no graph):
the command the ncu summaries under profiles/ are taken with.

--next times the calls beyond the chain step (hidden-row pool, graph replay against eager
launches, tree verify, stop-aware and sampling acceptance) on the batched-branches workload
and prints their own JSON line; --next --only sample runs just the sampling call (W + K plain
launches), the command its launch list is taken with.

--impl reference times the CPU oracle (the plain fp64 reference) on the same workload,
one bounded sample per step, on this host's cores.
Under torchrun (N > 1) every rank runs an independent replica (weak scaling; the path
has no exchange step), and the time is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_HBM_GBS = 6800.0

METRIC = "verified rows/s (B*(k+1) rows per verify step); us per verify step; HBM GB/s of the bandwidth kernels"

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of the kernel as it
# stands, from one ncu capture on that workload (profiles/); absent where none was taken.
LMHEAD_TRAFFIC: dict = {
    "long_context_fp8": 1_556_650_000 + 3_300_608,               # profiles/lmhead_argmax_long_context_fp8.md
    "batched_branches_shared_pool": 1_248_504_000 + 3_307_776,   # profiles/lmhead_argmax_batched_branches_shared_pool.md
    "single_stream_mtp_verify": 622_523_392 + 3_362_048,         # profiles/lmhead_argmax_single_stream_mtp_verify.md
}
ATTN_TRAFFIC: dict = {
    "long_context_fp8": 673_155_328 + 19_923_456,    # profiles/verify_attn_long_context_fp8.md
    "single_stream_mtp_verify": 8_535_552 + 0,       # profiles/verify_attn_single_stream_mtp_verify.md
    "batched_branches_shared_pool": 272_015_360 + 6_432_000,  # profiles/verify_attn_batched_branches_shared_pool.md
}


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines: list[str] = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                smax.append(float(f[1]))
            except ValueError:
                continue
            for nm, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------------------------

def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _setup_workload(cid: int, dev: str):
    """Inputs of workload `cid` drawn on the device, KV context written by the library."""
    import torch
    from greedy_speculative_decode_spec_gb300.step import PagedKv, VerifyStep
    from greedy_speculative_decode_spec_gb300.workloads import (CONFIGS, DRAFT_CONFIG, algorithmic_kv_bytes,
                                                                config4_verify, draft_inputs, make_lm_head,
                                                                verify_inputs)
    draft = None
    if cid == 4:
        # the draft side (MTP input for 64 rows, draft head + d2t), then the verify of
        # workload 2 with k = 4; the LM head weight doubles as the tied embedding table
        dc = DRAFT_CONFIG
        cfg = config4_verify(dc)
        W = make_lm_head(cfg.V, cfg.H, cfg.seed + 7, dev)
        draft = draft_inputs(dc, device=dev, E=W)
        vi = verify_inputs(cfg, device=dev, W=W)
    else:
        cfg = CONFIGS[cid]
        vi = verify_inputs(cfg, device=dev)
    c = vi.cfg
    kv = PagedKv(vi.num_pages, c.Hkv, c.P, c.d, vi.page_table.to(dev), fp8=c.kv_dtype == "fp8",
                 k_scale=vi.k_scale, v_scale=vi.v_scale, device=dev)
    kv.write_rows(vi.ctx_branch.to(dev), vi.ctx_pos.to(dev), vi.ctx_k.to(dev), vi.ctx_v.to(dev))
    del vi.ctx_k, vi.ctx_v
    # the next draft step's MTP input (tied embedding table = LM head weight)
    g = torch.Generator(device=dev)
    g.manual_seed(c.seed + 11)
    mtp = dict(E=vi.W, g_emb=(0.5 + torch.rand(c.H, generator=g, device=dev)).float(),
               g_hid=(0.5 + torch.rand(c.H, generator=g, device=dev)).float(), eps=1e-6,
               W_fc=(0.02 * torch.randn((c.H, 2 * c.H), generator=g, device=dev)).to(torch.bfloat16))
    step = VerifyStep(kv, c.B, c.k, c.Hq, vi.W, vi.max_pos, mtp=mtp, device=dev)
    inputs = dict(pos=vi.pos.to(dev), q=vi.q, k_new=vi.k_new, v_new=vi.v_new, hidden=vi.hidden, drafts=vi.drafts.to(dev))
    # the verify rows' K/V in their slots, so that a call timed alone (--only) reads the same pool a step does
    from greedy_speculative_decode_spec_gb300 import _binding as bnd
    bnd.spec_kv_append(kv.desc, inputs["pos"], c.B, c.k, vi.k_new, vi.v_new)
    kv_bytes = algorithmic_kv_bytes(c, vi.pos.tolist())
    w_bytes = c.V * c.H * 2
    return dict(cfg=c, vi=vi, kv=kv, step=step, inputs=inputs, draft=draft, kv_bytes=kv_bytes, w_bytes=w_bytes)


class DraftStage:
    """Workload 4's draft side: MTP input for M rows, then the trimmed draft head + d2t."""

    def __init__(self, draft, dev):
        import torch
        from greedy_speculative_decode_spec_gb300 import _binding as bnd
        self.bnd, self.d = bnd, draft
        M, H = draft.h.shape
        self.x = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
        self.ids = torch.empty(M, dtype=torch.int32, device=dev)
        self.mtp_ws = torch.zeros(bnd.spec_mtp_input_workspace(M, H), dtype=torch.uint8, device=dev)
        self.head_ws = torch.zeros(bnd.spec_lmhead_workspace(M, draft.W_draft.shape[0], H), dtype=torch.uint8,
                                   device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)

    def run(self):
        d, b = self.d, self.bnd
        b.spec_mtp_input(d.tok, d.E, d.h, d.g_emb, d.g_hid, d.cfg.eps, d.W_fc, self.x, self.mtp_ws, self.err)
        b.spec_lmhead_argmax(self.x, d.W_draft, self.ids, self.head_ws, d2t=d.d2t, d2t_limit=d.E.shape[0],
                             dev_err=self.err)


def replica_rate(ms_local: float, rows: int, world: int, device) -> tuple[float, float]:
    """Whole-job rate of `world` independent replicas, each verifying `rows` rows per step:
    the slowest rank's step time sets the pace (max over ranks)."""
    import torch
    import torch.distributed as dist
    ms_max = ms_local
    if world > 1:
        t = torch.tensor([ms_local], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_max = float(t.item())
    return ms_max, world * rows / (ms_max * 1e-3)


def _graph_of(fn):
    """A CUDA graph holding one call of fn (so that timing sees device work only, not the
    host cost of the call)."""
    import torch
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def _time_region(fn, steps, flush, stream):
    """CUDA-event time of each call of fn (L2 flushed before each, outside the events)."""
    import torch
    evs = []
    for _ in range(steps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        evs.append((a, b))
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def _time_in_graph(fn, steps, flush):
    """Device time of one call of fn: CUDA events recorded inside its graph, on the launching
    stream, right before and after the call's kernels (so the graph launch itself is not
    counted); the L2 flushed before every replay. Falls back to events around the replay where
    this PyTorch cannot record events as graph nodes."""
    import torch
    try:
        a = torch.cuda.Event(enable_timing=True, external=True)
        b = torch.cuda.Event(enable_timing=True, external=True)
    except TypeError:
        g = _graph_of(fn)
        return _time_region(g.replay, steps, flush, torch.cuda.current_stream())
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        a.record()
        fn()
        b.record()
    torch.cuda.synchronize()
    ts = []
    for _ in range(steps):
        flush()
        g.replay()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    del g
    return ts


def run_ours(args):
    import torch
    import torch.distributed as dist
    from greedy_speculative_decode_spec_gb300 import _binding as bnd
    from greedy_speculative_decode_spec_gb300 import build as pkg_build

    world, rank, local = _dist()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    pkg_build.build()
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    hbm_peak, peak_kind = _peaks()
    stream = torch.cuda.current_stream()
    # 512 MiB: longer on the GPU than the host needs to prepare the next launch, so the
    # per-kernel event timings below see only device time
    flush_buf = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    flush_sink = torch.zeros((), dtype=torch.int64, device=dev)

    def flush():
        # write 512 MiB (evicts the step's data from the 126 MB L2), then read 256 MiB of it:
        # the read evicts the dirty lines, so their write-back happens here, not inside the
        # next timed step
        flush_buf.fill_(1)
        flush_sink.copy_(flush_buf[: 256 << 20].view(torch.int64).sum())

    def log(msg):
        print(f"[bench] {msg}", file=sys.stderr, flush=True)

    def calls(w):
        """The step's calls of workload w: (verify step, attention alone, LM head alone)."""
        step, inp, c = w["step"], w["inputs"], w["cfg"]
        ds = w["ds"]
        o, kv = step.out, step.kv

        def one(with_mtp=False):
            if ds is not None:
                ds.run()
            step.run(inp["pos"], inp["q"], inp["k_new"], inp["v_new"], inp["hidden"], inp["drafts"],
                     with_mtp=with_mtp)

        def attn():
            bnd.spec_verify_attn(kv.desc, inp["pos"], c.B, c.k, c.Hq, inp["q"], step.scale, o.attn, step.attn_ws,
                                 step.max_pos, o.dev_err)

        def head():
            bnd.spec_lmhead_argmax(inp["hidden"], step.W, o.ids, step.head_ws, max_logit=o.max_logit,
                                   dev_err=o.dev_err)
        return one, attn, head

    def setup(cid):
        log(f"workload {cid}: set-up")
        w = _setup_workload(cid, dev)
        w["ds"] = DraftStage(w["draft"], dev) if w["draft"] is not None else None
        return w

    def measure(cid, steps, warmup, with_e2e=False, with_clocks=False):
        w = setup(cid)
        step, inp, c = w["step"], w["inputs"], w["cfg"]
        one, attn, head = calls(w)
        log(f"workload {cid}: eager steps")
        for _ in range(2):
            one()
        torch.cuda.synchronize()
        assert int(step.out.dev_err.item()) == 0, "device error during the step"
        log(f"workload {cid}: graph")
        graph = _graph_of(one)
        for _ in range(warmup):
            graph.replay()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        sampler = ClockSampler(local) if with_clocks else None
        if sampler:
            sampler.start()
        t_steps = _time_region(graph.replay, steps, flush, stream)
        torch.cuda.synchronize()
        clocks = sampler.stop() if sampler else None
        if world > 1:
            dist.barrier()
        del graph
        log(f"workload {cid}: per-kernel timing")
        # per-call times of the two bandwidth calls (events inside each call's graph, same
        # stream, same flush)
        t_attn = _time_in_graph(attn, steps, flush)
        t_head = _time_in_graph(head, steps, flush)
        # the same step followed by the next draft step's MTP input
        g_mtp = _graph_of(lambda: one(with_mtp=True))
        for _ in range(warmup):
            g_mtp.replay()
        t_mtp = _time_region(g_mtp.replay, steps, flush, stream)
        del g_mtp
        res = dict(cfg=c, ms=statistics.median(t_steps), t_attn=statistics.median(t_attn),
                   t_head=statistics.median(t_head), ms_mtp=statistics.median(t_mtp), kv_bytes=w["kv_bytes"],
                   w_bytes=w["w_bytes"], clocks=clocks,
                   launches=step.launches_verify + (4 if w["ds"] is not None else 0))
        if with_e2e:
            log(f"workload {cid}: end to end")
            res["e2e"] = measure_e2e(step, inp, steps, flush)
        log(f"workload {cid}: done")
        del w, step
        torch.cuda.empty_cache()
        return res

    def measure_e2e(step, inp, steps, flush):
        """Host buffers in, host results out, copies inside the timed region."""
        names_in = ["pos", "q", "k_new", "v_new", "hidden", "drafts"]
        host = {n: inp[n].cpu().pin_memory() for n in names_in}
        dev_in = {n: torch.empty_like(inp[n]) for n in names_in}
        o = step.out
        outs = [o.tokens, o.n, o.accepted, o.new_pos, o.next_tok]
        host_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in outs]
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = sum(t.numel() * t.element_size() for t in host_out)

        def one():
            for n in names_in:
                dev_in[n].copy_(host[n], non_blocking=True)
            step.run(dev_in["pos"], dev_in["q"], dev_in["k_new"], dev_in["v_new"], dev_in["hidden"], dev_in["drafts"],
                     with_mtp=False)
            for h, t in zip(host_out, outs):
                h.copy_(t, non_blocking=True)

        for _ in range(3):
            one()
        torch.cuda.synchronize()
        ts = _time_region(one, steps, flush, stream)
        return dict(ms=statistics.median(ts), h2d=h2d, d2h=d2h)

    if args.only:
        # one call of the workload, W + K plain launches (the command ncu captures use)
        w = setup(args.config)
        _, attn, head = calls(w)
        fn = attn if args.only == "attn" else head
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        ts = _time_region(fn, args.steps, flush, stream)
        assert int(w["step"].out.dev_err.item()) == 0, "device error"
        print(json.dumps({"only": args.only, "workload": w["cfg"].name, "us": round(statistics.median(ts) * 1e3, 2),
                          "calls": args.warmup + args.steps}), flush=True)
        return

    def kernel_entry(name, bytes_, ms, workload, traffic):
        gbs = bytes_ / (ms * 1e-3) / 1e9
        return {"bound": "hbm", "kernel": name, "achieved": round(gbs, 1), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(gbs / hbm_peak, 4), "peak_kind": peak_kind, "algorithmic_bytes": bytes_,
                "kernel_us": round(ms * 1e3, 2), "traffic": traffic.get(workload)}

    main = measure(args.config, args.steps, args.warmup, with_e2e=True, with_clocks=True)
    c = main["cfg"]
    rows = c.B * (c.k + 1)
    ms_max, value = replica_rate(main["ms"], rows, world, dev)
    others = {}
    if args.all and rank == 0:
        for cid in (0, 1, 2, 3, 4):
            if cid == args.config:
                continue
            r = measure(cid, max(5, min(args.steps, 20)), max(3, args.warmup))
            rc = r["cfg"]
            R = rc.B * (rc.k + 1)
            a = kernel_entry("spec_verify_attn", r["kv_bytes"], r["t_attn"], rc.name, ATTN_TRAFFIC)
            h = kernel_entry("spec_lmhead_argmax", r["w_bytes"], r["t_head"], rc.name, LMHEAD_TRAFFIC)
            others[str(cid)] = {
                "workload": rc.name, "us_per_step": round(r["ms"] * 1e3, 2), "rows_per_s": round(R / (r["ms"] * 1e-3), 1),
                "us_per_step_with_mtp_input": round(r["ms_mtp"] * 1e3, 2),
                "attn_us": a["kernel_us"], "attn_gbs": a["achieved"], "attn_frac": a["frac"], "attn_traffic": a["traffic"],
                "lmhead_us": h["kernel_us"], "lmhead_gbs": h["achieved"], "lmhead_frac": h["frac"],
                "lmhead_traffic": h["traffic"], "kv_bytes": r["kv_bytes"], "w_bytes": r["w_bytes"]}
    if rank != 0:
        return
    e2e = main["e2e"]
    attn_e = kernel_entry("spec_verify_attn", main["kv_bytes"], main["t_attn"], c.name, ATTN_TRAFFIC)
    head_e = kernel_entry("spec_lmhead_argmax", main["w_bytes"], main["t_head"], c.name, LMHEAD_TRAFFIC)
    # the dominant kernel (the larger share of the step) is the line's roofline
    dom, sec = (head_e, attn_e) if main["t_head"] >= main["t_attn"] else (attn_e, head_e)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "rows/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_max, 4), "us_per_step": round(ms_max * 1e3, 2),
        "us_per_step_with_mtp_input": round(main["ms_mtp"] * 1e3, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": c.kv_dtype if c.kv_dtype == "bf16" else "bf16+e4m3",
        "data": "synthetic (seeded; random-init weights)",
        "config": {"workload": c.name, "B": c.B, "k": c.k, "rows": rows, "H": c.H, "q_heads": c.Hq, "kv_heads": c.Hkv,
                   "head_dim": c.d, "context": list(c.ctx) or list(c.ctx_range), "page_size": c.P, "vocab": c.V,
                   "kv_dtype": c.kv_dtype, "step": "kv append + verify attention + LM head argmax + accept",
                   "parallelism": f"replicas x{world}", "graph": "CUDA graph per step",
                   "l2": "flushed before every timed step (512 MiB write, then 256 MiB read so that the dirty lines are written back before the timed region)"},
        "roofline": dom,
        "roofline_other": sec,
        "e2e": {"value": round(rows / (e2e["ms"] * 1e-3), 1), "unit": "rows/s", "ms_per_step": round(e2e["ms"], 4),
                "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"]},
        "gpu_launches": main["launches"] * args.steps,
        "clocks": main["clocks"],
        "all_configs": others,
    }
    if world == 1 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(args.config, budget_s=args.cpu_budget)
    print(json.dumps(line), flush=True)


# ---- the oracle on the host cores ------------------------------------------------------------

def _sample_call(B, k, V, g, dev, toks, n, a, npos, nxt, err):
    """Sampling acceptance inputs on the device (logits 3·N(0,1); q = softmax of the logits plus
    N(0,1) noise at temperature 1.3; drafts drawn from q; uniform random numbers) and the call."""
    import torch
    from greedy_speculative_decode_spec_gb300 import _binding as bnd
    logits = 3.0 * torch.randn((B * (k + 1), V), generator=g, device=dev)
    qd = torch.softmax((logits.view(B, k + 1, V)[:, :k] + torch.randn((B, k, V), generator=g, device=dev)) / 1.3,
                       dim=-1).contiguous()
    sdrafts = torch.multinomial(qd.view(B * k, V), 1, generator=g).view(B, k).to(torch.int32)
    u_acc = torch.rand((B, k), generator=g, device=dev)
    u_res = torch.rand(B, generator=g, device=dev)
    spos = torch.randint(0, 8000, (B,), generator=g, device=dev, dtype=torch.int32)
    sws = torch.zeros(bnd.spec_accept_sample_workspace(B, k, V), dtype=torch.uint8, device=dev)
    return lambda: bnd.spec_accept_sample(sdrafts, logits, qd, spos, B, k, 1.0, u_acc, u_res, toks, n, a, npos, nxt,
                                          err, ws=sws)


def run_next_sample_only(args):
    """--next --only sample: W + K plain launches of the sampling call at the batched-branches
    shape (B=16, k=6, V=151936), the command its launch list is taken with."""
    import torch
    from greedy_speculative_decode_spec_gb300 import build as pkg_build
    pkg_build.build()
    dev = "cuda:0"
    torch.cuda.set_device(0)
    g = torch.Generator(device=dev)
    g.manual_seed(2024)
    B, k, V = 16, 6, 151936
    i32 = dict(dtype=torch.int32, device=dev)
    toks = torch.empty((B, k + 1), **i32)
    n, a, npos, nxt = (torch.empty(B, **i32) for _ in range(4))
    err = torch.zeros(1, **i32)
    call = _sample_call(B, k, V, g, dev, toks, n, a, npos, nxt, err)
    for _ in range(args.warmup + args.steps):
        call()
    torch.cuda.synchronize()
    assert int(err.item()) == 0, "device error in the sampling call"
    print(json.dumps({"mode": "next_rows", "only": "sample", "calls": args.warmup + args.steps,
                      "accepted": a.cpu().tolist()}), flush=True)


def run_next(args):
    """The calls beyond the chain step, on the batched-branches workload (B=16, k=6, 32/8
    heads, d=128, bf16 pages of 16; V=151936, H=4096), each timed alone from a CUDA graph with
    the L2 flushed before every replay: the hidden-row pool gather and scatter, eager launches
    against one graph replay of the whole step (also on the single-stream workload), tree
    attention over a binary tree of the 7 verify slots, the tree walk and the compaction of its
    path, acceptance with stop ids and budgets, and speculative sampling acceptance. One JSON
    line; bytes are the algorithmic bytes of each call."""
    import torch
    from greedy_speculative_decode_spec_gb300 import _binding as bnd
    from greedy_speculative_decode_spec_gb300 import build as pkg_build

    pkg_build.build()
    dev = "cuda:0"
    torch.cuda.set_device(0)
    hbm_peak, peak_kind = _peaks()
    stream = torch.cuda.current_stream()
    flush_buf = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    flush_sink = torch.zeros((), dtype=torch.int64, device=dev)

    def flush():
        # as in the step timing: write 512 MiB, then read 256 MiB of it, so that the dirty
        # lines are written back here and not inside the timed call
        flush_buf.fill_(1)
        flush_sink.copy_(flush_buf[: 256 << 20].view(torch.int64).sum())

    def timed(fn, steps, reps=1):
        def body():
            for _ in range(reps):
                fn()
        for _ in range(3):
            body()
        ts = _time_in_graph(body, steps, flush)
        return statistics.median(ts) * 1e3 / reps  # us per call

    def small(e, fn):
        # a latency-bound call: also its time per call in a graph of 20 back-to-back calls
        e["us_each_of_20"] = round(timed(fn, steps, reps=20), 2)
        return e

    def entry(us, nbytes=None):
        e = {"us": round(us, 2)}
        if nbytes is not None:
            gbs = nbytes / (us * 1e-6) / 1e9
            e.update(bytes=int(nbytes), gbs=round(gbs, 1), frac=round(gbs / hbm_peak, 4))
        return e

    steps = args.steps
    rows = {}
    i32 = dict(dtype=torch.int32, device=dev)
    g = torch.Generator(device=dev)
    g.manual_seed(2024)

    # ---- f1: eager launches against one graph replay of the whole step; back to back (no
    # flush, events around 20 steps) the host's launch cost shows where the step is short ----
    def b2b(fn, n=20):
        import torch as _t
        for _ in range(3):
            fn()
        _t.cuda.synchronize()
        a_, b_ = _t.cuda.Event(enable_timing=True), _t.cuda.Event(enable_timing=True)
        a_.record(stream)
        for _ in range(n):
            fn()
        b_.record(stream)
        _t.cuda.synchronize()
        return a_.elapsed_time(b_) * 1e3 / n

    for cid in (0, 1, 2):
        w = _setup_workload(cid, dev)
        step, inp = w["step"], w["inputs"]

        def one():
            step.run(inp["pos"], inp["q"], inp["k_new"], inp["v_new"], inp["hidden"], inp["drafts"], with_mtp=False)
        for _ in range(3):
            one()
        torch.cuda.synchronize()
        eager = statistics.median(_time_region(one, steps, flush, stream)) * 1e3
        rows[f"step_eager_{w['cfg'].name}"] = entry(eager)
        rows[f"step_graph_{w['cfg'].name}"] = entry(timed(one, steps))
        gstep = _graph_of(one)
        rows[f"step_eager_{w['cfg'].name}"]["back_to_back_us"] = round(b2b(one), 2)
        rows[f"step_graph_{w['cfg'].name}"]["back_to_back_us"] = round(b2b(gstep.replay), 2)
        del gstep
        if cid == 2:
            kept = w
        else:
            del w, step, inp
            torch.cuda.empty_cache()
    w = kept
    c, step, inp, kv = w["cfg"], w["step"], w["inputs"], w["kv"]
    B, k, H, V, R = c.B, c.k, c.H, c.V, c.B * (c.k + 1)
    err = torch.zeros(1, **i32)

    # ---- f1: hidden-row pool (64 slots of H bf16), gather then scatter of B rows ----
    hpool = torch.randn((64, H), generator=g, device=dev).to(torch.bfloat16)
    hslot = torch.randperm(64, generator=g, device=dev)[:B].to(torch.int32)
    h = torch.empty((B, H), dtype=torch.bfloat16, device=dev)
    row_bytes = 2 * B * H * 2  # each row read once and written once
    gat = lambda: bnd.spec_h_gather(h, hpool, hslot, err)  # noqa: E731
    sca = lambda: bnd.spec_h_scatter(hpool, h, hslot, err)  # noqa: E731
    rows["h_gather"] = small(entry(timed(gat, steps), row_bytes), gat)
    rows["h_scatter"] = small(entry(timed(sca, steps), row_bytes), sca)

    # ---- f2: tree attention (binary tree over the 7 slots), tree walk, path compaction ----
    parent = [-1, 0, 0, 1, 1, 2, 2][: k + 1]
    masks = []
    for j in range(k + 1):
        m, x = 0, j
        while x >= 0:
            m |= 1 << x
            x = parent[x]
        masks.append(m)
    anc = torch.tensor(masks * B, **i32)
    out = torch.empty((R, c.Hq, c.d), dtype=torch.bfloat16, device=dev)

    def tree_attn():
        bnd.spec_verify_attn_tree(kv.desc, inp["pos"], B, k, c.Hq, inp["q"], step.scale, anc, out, step.attn_ws,
                                  step.max_pos, err)
    rows["verify_attn_tree"] = entry(timed(tree_attn, steps), w["kv_bytes"])
    par = torch.tensor([max(p, 0) for p in parent] * B, **i32)
    ids = torch.randint(0, V, (B, k + 1), generator=g, device=dev, dtype=torch.int32)
    drafts = torch.randint(0, V, (B, k), generator=g, device=dev, dtype=torch.int32)
    drafts[:, 0] = ids[:, 0]  # every walk takes its first step
    drafts[:, 2] = ids[:, 1]
    toks, path = torch.empty((B, k + 1), **i32), torch.empty((B, k + 1), **i32)
    n, a, npos, nxt = (torch.empty(B, **i32) for _ in range(4))
    walk = lambda: bnd.spec_accept_tree(drafts, ids, inp["pos"], par, B, k, toks, n, a, npos, nxt, path, err)  # noqa: E731
    rows["accept_tree"] = small(entry(timed(walk, steps)), walk)
    torch.cuda.synchronize()
    moved = int(a.sum().item())  # rows moved by the compaction: K and V of every kv head
    kv_row = 2 * c.Hkv * c.d * (2 if c.kv_dtype == "bf16" else 1)
    comp = lambda: bnd.spec_kv_compact(kv.desc, inp["pos"], path, a, B, k, err)  # noqa: E731
    rows["kv_compact"] = small(entry(timed(comp, steps), 2 * moved * kv_row), comp)

    # ---- f3: acceptance with stop ids and per-branch budgets ----
    stop = torch.tensor([151643, 151645, -1, -1], **i32)
    budget = torch.randint(1, 2 * (k + 1), (B,), generator=g, device=dev, dtype=torch.int32)
    stp = lambda: bnd.spec_accept_stop(inp["drafts"], step.out.ids, inp["pos"], B, k, stop, budget, toks, n, a,  # noqa: E731
                                       npos, nxt)
    rows["accept_stop"] = small(entry(timed(stp, steps)), stp)

    # ---- f4: speculative sampling acceptance, fp32 logits [R][V] and draft probabilities [B][k][V] ----
    del w, kept, step
    torch.cuda.empty_cache()
    call = _sample_call(B, k, V, g, dev, toks, n, a, npos, nxt, err)
    us = timed(call, steps)
    torch.cuda.synchronize()
    # bytes: every verify row's logits once (all rows' softmax statistics are computed) and
    # the q row of each rejected draft; "needed_bytes": only the rows up to the decisive one
    acc = a.cpu().tolist()
    nb = R * V * 4 + sum(V * 4 for x in acc if x < k)
    rows["accept_sample"] = entry(us, nb)
    rows["accept_sample"]["needed_bytes"] = sum((min(x, k) + 1) * V * 4 + (V * 4 if x < k else 0) for x in acc)
    rows["accept_sample"]["accepted"] = acc
    assert int(err.item()) == 0, "device error in the next-row calls"
    line = {"mode": "next_rows", "workload": c.name, "steps": steps, "hbm_peak_gbs": hbm_peak, "peak": peak_kind,
            "timing": "CUDA-event median over graph replays (events recorded inside the graph around the call), "
                      "L2 flushed before each; eager: plain launches, events around them",
            "rows": rows}
    print(json.dumps(line), flush=True)


def _oracle_sample(cid: int):
    """A bounded sample of workload `cid` for the oracle: one verify row (b=0, j=k) through
    append, attention over all q heads, the full-vocabulary LM head and acceptance."""
    import numpy as np
    import oracle as orc
    from greedy_speculative_decode_spec_gb300.workloads import CONFIGS, bits, scaled, verify_inputs
    cfg = CONFIGS[cid]
    # one branch only (the oracle's input is the same workload restricted to branch 0)
    one = scaled(cfg, B=1, ctx=(cfg.ctx[0],) if cfg.ctx else (cfg.ctx_range[1],), ctx_range=(), num_pages=0,
                 near_tie=0)
    vi = verify_inputs(one)
    c = vi.cfg
    fp8 = c.kv_dtype == "fp8"
    shape = vi.pool_shape
    kp = np.full(shape, 0x7F if fp8 else 0x7FC0, np.uint8 if fp8 else np.uint16)
    okv = orc.KvPool(kp, kp.copy(), vi.page_table.numpy(), c.P,
                     None if vi.k_scale is None else vi.k_scale.numpy(), None if vi.v_scale is None else vi.v_scale.numpy())
    assert orc.kv_write_rows(okv, vi.ctx_branch.numpy(), vi.ctx_pos.numpy(), bits(vi.ctx_k), bits(vi.ctx_v)) == 0
    hid = bits(vi.hidden)
    W = bits(vi.W)
    q = bits(vi.q)
    kn, vn = bits(vi.k_new), bits(vi.v_new)
    items = np.arange(c.k * c.Hq, (c.k + 1) * c.Hq, dtype=np.int32)   # row k, every head

    def run():
        orc.kv_append(okv, vi.pos.numpy(), 1, c.k, kn, vn)
        orc.verify_attn_items(okv, vi.pos.numpy(), 1, c.k, c.Hq, q, 1.0 / math.sqrt(c.d), items)
        ids, _, _, _ = orc.lmhead_argmax(hid[c.k:c.k + 1], W)
        orc.accept(vi.drafts.numpy(), np.concatenate([vi.planted.numpy()[:c.k], ids]), vi.pos.numpy(), 1, c.k)
    desc = (f"1 verify row of {c.name} (b=0, j=k): KV append, attention over {c.Hq} q heads and "
            f"{int(vi.pos[0]) + c.k + 1} keys, LM head over V={c.V} x H={c.H}, acceptance")
    return run, desc


def cpu_baseline(cid: int, budget_s: float = 20.0):
    import oracle as orc
    orc.build()
    run, desc = _oracle_sample(cid)
    n, t0 = 0, time.perf_counter()
    while True:
        run()
        n += 1
        dt = time.perf_counter() - t0
        if dt >= budget_s or n >= 50:
            break
    return {"value": round(n / dt, 4), "unit": "rows/s", "cores": orc.threads(), "kind": "oracle",
            "sample": f"{n} x {desc}", "seconds": round(dt, 2)}


def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return
    import oracle as orc
    from greedy_speculative_decode_spec_gb300.workloads import CONFIGS
    orc.build()
    c = CONFIGS[args.config]
    run, desc = _oracle_sample(args.config)
    for _ in range(args.warmup):
        run()
    ts = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        run()
        ts.append(time.perf_counter() - t0)
    sec = statistics.median(ts)
    value = 1.0 / sec  # one verify row per sample
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "rows/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(sec * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": {"workload": c.name, "B": c.B, "k": c.k, "rows_per_sample": 1},
            "cpu_baseline": {"value": round(value, 4), "unit": "rows/s", "cores": orc.threads(), "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": round(value, 4), "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=3, choices=[0, 1, 2, 3, 4])
    ap.add_argument("--only", choices=["attn", "lmhead", "sample"], default=None)
    ap.add_argument("--no-all", dest="all", action="store_false")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--next", action="store_true")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.only == "sample" and not args.next:
        ap.error("--only sample goes with --next")
    if args.next:
        run_next_sample_only(args) if args.only == "sample" else run_next(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

"""Benchmark: EAGLE-3 tree verify step at B = 64, Llama-3-8B shape, on one GB300.

One step = the whole hot path over one batch of 64 sequences:
  EAGLE-2 expansion, 8 levels (draft LM-head GEMM 4096 -> 128256 on the tcgen05
  tensor cores for 1 + 7 x 10 frontier rows per sequence, softmax + top-10 per
  row, per-level select), rerank to 60 nodes, tree attention for one layer
  (32 q / 8 kv heads, d = 128, committed KV length 4096), verify-and-accept
  (V = 128256, T = 1), and KV compaction over 32 layers.
Metric: tree-verify steps/s (value) and accepted tokens/s; the dominant kernel's
roofline fraction against the measured peaks.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Multi-GPU: the path shards by sequence with no exchange, so N ranks run N
independent batches (weak scaling); rank 0 prints the line.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "tree-verify steps/sec & accepted tokens/s at B=64; HBM GB/s vs roofline"
# DRAM bytes (read + write) of one 640 x 4096 -> 128256 LM-head GEMM launch with its
# per-tile partials (the step's form), from an ncu capture of the current kernel:
# 1.0795e9 read + 0.3035e9 written.
GEMM_LAUNCH_DRAM_BYTES = 1.3830e9
CFG = W.CONFIGS["eagle3_b64"]
SEED = 0


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm_gbs=d["hbm_gbs"], bf16_tflops=d["bf16_tflops"],
                    bf16_tflops_sustained=d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of the SM clock and throttle reasons, each stamped on arrival;
    stop(t0, t1) keeps the samples that arrived inside the timed region [t0, t1]."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = 20):
        self.idx = gpu_index
        self.interval = interval_ms
        self.proc = None
        self.lines = []

    def start(self, wait_first_s: float = 3.0):
        """Start sampling; return once the first sample has arrived (or after wait_first_s)."""
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.interval)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
            return
        t_end = time.perf_counter() + wait_first_s
        while not self.lines and time.perf_counter() < t_end:
            time.sleep(0.01)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def stop(self, t0=None, t1=None):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(2 * self.interval / 1000.0)          # the sample that covers t1
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        slack = self.interval / 1000.0
        inside = [ln for ts, ln in self.lines
                  if t0 is None or (t0 <= ts <= t1 + slack)]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in inside:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for nm, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "interval_ms": self.interval,
                "window": "samples that arrived inside the timed region",
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------- our arm
class Step:
    """Resident inputs and the call sequence of one verify step (all library calls)."""

    def __init__(self, dev, seed=SEED):
        import torch

        import eagle_tree_speculative_gb300 as E
        self.E, self.torch, self.dev = E, torch, dev
        c = CFG
        B, k, D, n, V, H = c.B, c.top_k, c.depth, c.n, c.V, c.H
        self.B, self.k, self.D, self.n, self.V, self.H, self.R = B, k, D, n, V, H, c.R
        # draft LM head, hidden states per level (host-generated, uploaded once)
        self.w = W.lm_head(V, H, c.w_std, seed).to(dev)
        self.hidden = [W.hidden_states(B, 1 if l == 1 else k, H, l, seed).to(dev)
                       for l in range(1, D + 1)]
        self.logits = torch.empty(B, c.R, V, device=dev)          # draft-logit storage
        self.state = torch.empty(E.tree_state_size(B, k, D), dtype=torch.uint8, device=dev)
        # per-tile softmax statistics and top-k from the GEMM epilogue (fused top-k)
        self.partials = torch.empty(E.expand_scratch_size(B, V, k) // 4, device=dev)
        self.tokens = torch.empty(B, n, dtype=torch.int32, device=dev)
        self.parent = torch.empty_like(self.tokens)
        self.draft_row = torch.empty_like(self.tokens)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        # attention inputs: queries of the tree nodes, one layer of the 32-layer cache
        g = torch.Generator(device=dev).manual_seed(seed + 1)
        self.q = torch.randn(B, n, c.Hq, c.head_dim, device=dev, generator=g).to(torch.bfloat16)
        shape = (c.n_layers, B, c.Hkv, c.Lmax, c.head_dim)
        self.kc = torch.randn(shape, device=dev, generator=g, dtype=torch.bfloat16)
        self.vc = torch.randn(shape, device=dev, generator=g, dtype=torch.bfloat16)
        self.kv_len0 = torch.full((B,), c.L, dtype=torch.int32, device=dev)
        self.kv_len = self.kv_len0.clone()
        self.attn_out = torch.empty_like(self.q)
        ws = E.tree_attn_workspace_size(B, n, c.Hq, c.Hkv, c.head_dim, c.Lmax)
        self.attn_ws = torch.empty(max(ws, 1), dtype=torch.uint8, device=dev)
        self.accept_len = torch.empty(B, dtype=torch.int32, device=dev)
        self.path = torch.empty(B, D + 1, dtype=torch.int32, device=dev)
        self.emit = torch.empty(B, D + 1, dtype=torch.int32, device=dev)
        # one expansion to fix the tree, then the synthetic target logits: the draft row of
        # each expanded node plus N(0, sigma^2) noise, a fresh N(0, s^2) row for leaves
        self.expand()
        torch.cuda.synchronize()
        self.gemm_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                        for _ in range(D)]
        self.target = synth_target(torch, self.logits, self.draft_row, c.sigma,
                                   float(c.w_std * np.sqrt(H)), g)
        torch.cuda.synchronize()
        self.gemm_ms = 0.0          # accumulated in-kernel GEMM time of timed steps
        self.gemm_rows = 0
        self.gemm_full_ms = 0.0     # the same for the full-width levels (B x top_k rows)
        self.gemm_full_launches = 0

    def expand(self, time_gemm=False):
        E = self.E
        for lvl in range(1, self.D + 1):
            k_in = 1 if lvl == 1 else self.k
            off = 0 if lvl == 1 else 1 + (lvl - 2) * self.k
            if time_gemm:
                self.gemm_ev[lvl - 1][0].record()
            E.eagle_lmhead_gemm(self.hidden[lvl - 1].view(self.B * k_in, self.H), self.w,
                                out=self.logits, ldo=self.V, rows_per_group=k_in,
                                group_stride=self.R, row_offset=off, dev_status=self.status,
                                partials=self.partials)
            if time_gemm:
                self.gemm_ev[lvl - 1][1].record()
            E.eagle2_expand(lvl, lvl == self.D, self.logits, self.k, self.D, self.n, self.state,
                            out_tokens=self.tokens, out_parent=self.parent,
                            out_draft_row=self.draft_row, dev_status=self.status,
                            partials=self.partials)

    def collect_gemm_times(self):
        """Add the GEMM launch times recorded by the last time_gemm step (events are reused)."""
        for lvl in range(1, self.D + 1):
            e0, e1 = self.gemm_ev[lvl - 1]
            t = e0.elapsed_time(e1)
            self.gemm_ms += t
            self.gemm_rows += self.B * (1 if lvl == 1 else self.k)
            if lvl > 1:
                self.gemm_full_ms += t
                self.gemm_full_launches += 1

    def run(self, seed, time_gemm=False):
        E = self.E
        self.expand(time_gemm)
        E.eagle_tree_attn(self.q, self.kc[0], self.vc[0], self.kv_len, self.parent,
                          out=self.attn_out, workspace=self.attn_ws, dev_status=self.status)
        E.eagle_verify_accept(self.target, self.logits, self.tokens, self.parent, self.D, 1.0, seed,
                              draft_row=self.draft_row, accept_len=self.accept_len, path=self.path,
                              emit=self.emit, dev_status=self.status)
        E.eagle_kv_compact(self.kc, self.vc, self.kv_len, self.path, self.accept_len, self.D,
                           dev_status=self.status)
        self.kv_len.copy_(self.kv_len0)      # keep the committed length fixed across steps

    # kernels launched per step: per level GEMM + top-k + select (+ rerank at the last),
    # attention (+ combine when split), verify, compaction
    def launches_per_step(self):
        c = CFG
        ws = self.E.tree_attn_workspace_size(self.B, self.n, c.Hq, c.Hkv, c.head_dim, c.Lmax)
        return self.D * 3 + 1 + (2 if ws else 1) + 1 + 1


def synth_target(torch, logits, draft_row, sigma, leaf_std, g):
    """Target logits per tree node: the node's draft row plus N(0, sigma^2) noise where
    the node was expanded, a fresh N(0, leaf_std^2) row for a leaf."""
    B, n = draft_row.shape
    V = logits.shape[-1]
    rows = draft_row.long()
    target = torch.empty(B, n, V, device=logits.device)
    for b in range(B):
        r = rows[b]
        noise = torch.randn(n, V, device=logits.device, generator=g) * sigma
        target[b] = torch.where((r >= 0)[:, None], logits[b, r.clamp(min=0)] + noise,
                                torch.randn(n, V, device=logits.device, generator=g) * leaf_std)
    return target


def reduce_over_ranks(x, dist, device, op):
    """Max ("max") or sum ("sum") of a per-rank figure over all ranks; no-op alone.

    Ranks run independent batches, so this is the only exchange: the slowest rank's
    timed region and the total accepted tokens."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


def step_throughput(world, ms_per_step):
    """Whole-job steps/s: every rank completes one step of its own batch per
    ms_per_step (the max over ranks)."""
    return world * 1000.0 / ms_per_step


def time_region_steps(fn, steps, torch):
    """Total device time of `steps` calls of fn and each call's own time (ms): one event
    before every step and one after the last, all on the launching stream."""
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    ev[0].record()
    for i in range(steps):
        fn(i)
        ev[i + 1].record()
    torch.cuda.synchronize()
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
    return ev[0].elapsed_time(ev[-1]), per


def time_region(fn, steps, torch):
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(steps):
        fn(i)
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)


def run_ours(args, rank, world, dist):
    import torch
    local = int(os.environ.get("LOCAL_RANK", 0))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks = measured_peaks()
    st = Step(dev)
    for i in range(args.warmup):
        st.run(1000 + i)
    torch.cuda.synchronize()
    if int(st.status.item()) != 0:
        raise RuntimeError(f"device status {int(st.status.item())} during warm-up")

    # -------- device-resident timed region: the captured step, replayed --------
    graph = None
    try:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, capture_error_mode="relaxed"):
            st.run(77)
        graph.replay()
        torch.cuda.synchronize()
    except Exception as exc:  # capture unsupported: time the eager calls instead
        graph = None
        print(f"graph capture failed ({exc}); timing eager launches", file=sys.stderr)
    clocks = ClockSampler(local)
    clocks.start()
    if dist:
        dist.barrier()
    step_fn = (lambda i: graph.replay()) if graph is not None else (lambda i: st.run(i))
    t0 = time.perf_counter()
    ms, per_step = time_region_steps(step_fn, args.steps, torch)
    t1 = time.perf_counter()
    clk = clocks.stop(t0, t1)
    ms = reduce_over_ranks(ms, dist, dev, "max")
    ms_per_step = ms / args.steps
    step_median = reduce_over_ranks(float(np.median(per_step)), dist, dev, "max")
    acc_graph = float(st.accept_len.sum().item() + st.B)   # the replayed step's accepted tokens

    # -------- eager timed region: per-launch GEMM times (CUDA events on the stream) --------
    accepted = torch.zeros((), dtype=torch.int64, device=dev)
    eager_steps = max(10, min(args.steps, 50))
    torch.cuda.synchronize()
    t_eager = 0.0
    for i in range(eager_steps):
        e0 = time.perf_counter()
        st.run(i, time_gemm=True)
        accepted.add_(st.accept_len.sum() + st.B)
        torch.cuda.synchronize()
        t_eager += time.perf_counter() - e0
        st.collect_gemm_times()
    tok_per_step = float(accepted.item()) / eager_steps
    tok_all_ranks = reduce_over_ranks(tok_per_step, dist, dev, "sum")
    gemm_ms, gemm_rows = st.gemm_ms, st.gemm_rows
    gemm_flops = 2.0 * gemm_rows * st.H * st.V
    # roofline of the dominant kernel: the full-width GEMM launches (640 x 4096 -> 128256)
    full_ms = st.gemm_full_ms / st.gemm_full_launches
    full_flops = 2.0 * st.B * st.k * st.H * st.V
    gemm_tflops = full_flops / (full_ms * 1e-3) / 1e12
    peak = peaks["bf16_tflops_sustained"]

    # -------- per-call breakdown (separate short timing) --------
    br = breakdown(st, torch)
    ttt = ttt_attn_figures(torch, dev, peaks)
    other = {"chain_b1_b1000": chain_config(torch, dev),
             "eagle2_b1_vicuna13b": eagle2_b1_config(torch, dev, peaks)}

    # -------- end to end through the public API with host buffers --------
    e2e = run_e2e(st, torch, max(5, min(args.steps, 20)), graph)
    e2e_in_place = run_e2e(st, torch, max(5, min(args.steps, 20)), graph, target_in_place=True)
    if int(st.status.item()) != 0:
        raise RuntimeError(f"device status {int(st.status.item())}")

    out = {
        "metric": METRIC,
        "value": round(step_throughput(world, ms_per_step), 3),
        "unit": "steps/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "ms_per_step_median": round(step_median, 4),
        "ms_per_step_p10_p90": [round(float(np.percentile(per_step, 10)), 4),
                                round(float(np.percentile(per_step, 90)), 4)],
        "timing": ("CUDA graph of one step replayed; value from the whole timed region, median "
                   "from one event pair per step") if graph is not None else "eager launches",
        "eager_ms_per_step_wall": round(1e3 * t_eager / eager_steps, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16 GEMM/attention (fp32 accumulate), f32 logits",
        "data": "synthetic (seeded normals; random-init LM head; no datasets or trained weights)",
        "config": workload_config(world),
        "accepted_tokens_per_s": round(tok_all_ranks * 1000.0 / ms_per_step, 1),
        "mean_accept_len_plus_1": round(tok_all_ranks / (world * st.B), 4),
        "graph_step_accepted_tokens": acc_graph,
        "roofline": {"kernel": "lmhead_gemm_kernel (tcgen05), 640 x 4096 -> 128256 launches",
                     "bound": "tensor",
                     "achieved": round(gemm_tflops, 1), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(gemm_tflops / peak, 4), "traffic": GEMM_LAUNCH_DRAM_BYTES,
                     "traffic_note": "dram__bytes_read.sum + dram__bytes_write.sum of one "
                                     "640-row launch with per-tile partials (ncu); "
                                     "algorithmic 1.384e9",
                     "peak_source": f"{peaks['source']} bf16_tflops_sustained",
                     "flops_per_launch": full_flops,
                     "ms_per_launch": round(full_ms, 4),
                     "gemm_ms_per_step_all_levels": round(gemm_ms / eager_steps, 4),
                     "gemm_flops_per_step_all_levels": gemm_flops / eager_steps,
                     "timed": f"{eager_steps} eager steps, events around each launch"},
        "breakdown_ms": br,
        "verify_step": {
            "calls": "tree attention (1 layer) + verify-and-accept (T = 1) + KV compaction "
                     "(32 layers), one after another; the draft expansion excluded",
            "ms_median": br["verify_step"],
            "steps_per_s": round(world * 1e3 / br["verify_step"], 1),
            "accepted_tokens_per_s": round(world * st.B * br["verify_step_mean_accept_len_plus_1"]
                                           * 1e3 / br["verify_step"], 1),
            "timing": "median of 200 calls after 20 warm-up, one event pair per call"},
        "roofline_hbm": hbm_rooflines(br, peaks),
        "other_configs": other,
        "ttt_attn": ttt,
        "e2e": e2e,
        "e2e_target_in_place": e2e_in_place,
        "gpu_launches": st.launches_per_step() * args.steps,
        "gpu_launches_note": "library kernels per step x timed steps",
        "clocks": clk,
    }
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(budget_s=args.cpu_budget)
    return out


TTT_SHAPE = dict(B=8, S=2048, Hq=32, Hkv=8, R1=8, r=7)


def ttt_inputs(torch, dev, B, S, Hq, Hkv, R1, g):
    d = 128
    q = torch.empty(B, S, Hq, d, dtype=torch.bfloat16, device=dev).normal_(generator=g)
    k = torch.empty(B, Hkv, R1, S, d, dtype=torch.bfloat16, device=dev).normal_(generator=g)
    v = torch.empty_like(k).normal_(generator=g)
    return q, k, v


def ttt_attn_figures(torch, dev, peaks, reps=20):
    """Training-time-test attention of one layer, timed alone: Llama-3-8B heads (32 q /
    8 kv), 8 sequences of 2048 positions, the queries of round 7 of 8 and of round 0.
    FLOPs count the visible keys only (causal part + r diagonal keys per row)."""
    import eagle_tree_speculative_gb300 as E
    c = TTT_SHAPE
    B, S, Hq, Hkv, R1, d = c["B"], c["S"], c["Hq"], c["Hkv"], c["R1"], 128
    g = torch.Generator(device=dev).manual_seed(SEED + 23)
    q, k, v = ttt_inputs(torch, dev, B, S, Hq, Hkv, R1, g)
    out = torch.empty_like(q)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    res = {"shape": "B=8, S=2048, 32 q / 8 kv heads, d=128, 8 rounds stored",
           "l2": "inputs larger than L2 (q 134 MB, K and V 268 MB each)"}
    peak = peaks["bf16_tflops"]
    for r in (c["r"], 0):
        fn = lambda: E.eagle_ttt_attn(q, k, v, r, out=out, dev_status=st)  # noqa: E731
        for _ in range(3):
            fn()
        ms = time_region(lambda i: fn(), reps, torch) / reps
        flops = 4.0 * d * Hq * B * S * (S + 1) / 2 + 4.0 * d * Hq * B * S * r
        hbm = 2 * (2 * B * S * Hq * d) + 2 * (2 * B * Hkv * (1 + r) * S * d)
        tf = flops / (ms * 1e-3) / 1e12
        res[f"round{r}"] = {"ms": round(ms, 4), "TFLOPs": round(tf, 1),
                            "frac_of_bf16_peak": round(tf / peak, 4),
                            "GBps_algorithmic": round(hbm / (ms * 1e-3) / 1e9, 1),
                            "flops": flops, "hbm_bytes": hbm}
    res["peak_source"] = f"{peaks['source']} bf16_tflops (burst: the kernel is timed alone)"
    if int(st.item()) != 0:
        raise RuntimeError(f"ttt attention device status {int(st.item())}")
    del q, k, v, out
    torch.cuda.empty_cache()
    return res


def timed_ms(fn, torch, reps=20, warm=3):
    """Median per-call device time (ms) of fn over reps calls, one event pair per call."""
    for _ in range(warm):
        fn()
    _, per = time_region_steps(lambda i: fn(), reps, torch)
    return float(np.median(per))


def chain_config(torch, dev, reps=200):
    """Chain verify (config 0): root + 5 drafts, V = 32000, target ~ N(0, 2^2), draft =
    target + N(0, 0.5^2), drafts sampled from p (T = 1) or its argmax (T = 0); no
    attention.  Latency of one B = 1 call, and throughput of 1000 independent steps as
    one B = 1000 call."""
    import eagle_tree_speculative_gb300 as E
    c = W.CONFIGS["chain"]
    n, V, D = c.n, c.V, c.depth
    g = torch.Generator(device=dev).manual_seed(SEED + 31)
    res = {"workload": "chain verify, 5 drafts, V=32000, sigma=0.5; B=1 latency and one B=1000 "
                       "launch (1000 independent steps); no attention"}
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    for B in (1, 1000):
        tgt = torch.randn(B, n, V, device=dev, generator=g) * c.target_std
        drf = tgt + torch.randn(B, n, V, device=dev, generator=g) * c.sigma
        par = torch.arange(-1, n - 1, dtype=torch.int32, device=dev).repeat(B, 1).contiguous()
        for T in (1.0, 0.0):
            tok = torch.full((B, n), -1, dtype=torch.int32, device=dev)
            if T > 0:
                pr = torch.softmax(drf[:, :n - 1] / T, -1).reshape(-1, V)
                tok[:, 1:] = torch.multinomial(pr, 1, generator=g).view(B, n - 1).int()
            else:
                tok[:, 1:] = drf[:, :n - 1].argmax(-1).int()
            acc = torch.empty(B, dtype=torch.int32, device=dev)
            path = torch.empty(B, D + 1, dtype=torch.int32, device=dev)
            emit = torch.empty_like(path)
            fn = lambda: E.eagle_verify_accept(tgt, drf, tok, par, D, T, 5, accept_len=acc,  # noqa
                                               path=path, emit=emit, dev_status=st)
            ms = timed_ms(fn, torch, reps=reps if B == 1 else 50)
            key = f"T{int(T)}"
            if B == 1:
                res[f"B1_{key}_us_per_step"] = round(ms * 1e3, 2)
            else:
                res[f"B1000_{key}_steps_per_s"] = round(1000.0 / (ms * 1e-3), 1)
                res[f"B1000_{key}_ms_per_launch"] = round(ms, 4)
                res[f"B1000_{key}_mean_accept_len_plus_1"] = round(float(acc.float().mean()) + 1, 4)
    if int(st.item()) != 0:
        raise RuntimeError(f"chain device status {int(st.item())}")
    return res


def eagle2_b1_config(torch, dev, peaks, reps=100):
    """EAGLE-2 tree at B = 1, Vicuna-13B shape (config 1): expansion of a 60-node depth-6
    top-10 tree from given draft logits (V = 32000), tree attention of one layer (40 / 40
    heads, d = 128, KV 2048: the split-KV path), verify at T = 0 and T = 1, and KV
    compaction over 40 layers.  Latency of each call and of the whole step as one graph."""
    import eagle_tree_speculative_gb300 as E
    c = W.CONFIGS["eagle2_b1"]
    B, n, D, k, V = 1, c.n, c.depth, c.top_k, c.V
    layers = 40
    g = torch.Generator(device=dev).manual_seed(SEED + 41)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    trow = torch.randn(B, c.R, V, device=dev, generator=g) * c.target_std
    drows = trow + torch.randn(B, c.R, V, device=dev, generator=g) * c.sigma
    state = torch.empty(E.tree_state_size(B, k, D), dtype=torch.uint8, device=dev)
    tok = torch.empty(B, n, dtype=torch.int32, device=dev)
    par, row = torch.empty_like(tok), torch.empty_like(tok)

    def expand():
        for lvl in range(1, D + 1):
            E.eagle2_expand(lvl, lvl == D, drows, k, D, n, state, out_tokens=tok, out_parent=par,
                            out_draft_row=row, dev_status=st)
    expand()
    torch.cuda.synchronize()
    r = row.long()[0]
    tgt = torch.where((r >= 0)[:, None], trow[0, r.clamp(min=0)],
                      torch.randn(n, V, device=dev, generator=g) * c.target_std)[None].contiguous()
    q = torch.randn(B, n, c.Hq, c.head_dim, device=dev, generator=g).to(torch.bfloat16)
    kc = torch.randn(layers, B, c.Hkv, c.Lmax, c.head_dim, device=dev, generator=g,
                     dtype=torch.bfloat16)
    vc = torch.randn_like(kc)
    kv0 = torch.full((B,), c.L, dtype=torch.int32, device=dev)
    kv = kv0.clone()
    out = torch.empty_like(q)
    ws_n = E.tree_attn_workspace_size(B, n, c.Hq, c.Hkv, c.head_dim, c.Lmax)
    ws = torch.empty(max(ws_n, 1), dtype=torch.uint8, device=dev)
    acc = torch.empty(B, dtype=torch.int32, device=dev)
    path = torch.empty(B, D + 1, dtype=torch.int32, device=dev)
    emit = torch.empty_like(path)
    attn = lambda: E.eagle_tree_attn(q, kc[0], vc[0], kv0, par, out=out, workspace=ws,  # noqa
                                     dev_status=st)
    res = {"workload": "EAGLE-2 tree, B=1, Vicuna-13B shape: 60 nodes, depth 6, top-10, "
                       "V=32000 (expansion from given logits), attention 40/40 heads d=128 "
                       "KV 2048 (split KV), compaction 40 layers",
           "split_kv_workspace_bytes": int(ws_n)}
    res["expand_6_levels_us"] = round(timed_ms(expand, torch, reps) * 1e3, 2)
    a = timed_ms(attn, torch, reps)
    kv_bytes = 2 * B * c.Hkv * (c.L + n) * c.head_dim * 2
    res["tree_attn_us"] = round(a * 1e3, 2)
    res["tree_attn_GBps"] = round(kv_bytes / (a * 1e-3) / 1e9, 1)
    res["tree_attn_frac_hbm"] = round(kv_bytes / (a * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)

    def comp():
        E.eagle_kv_compact(kc, vc, kv, path, acc, D, dev_status=st)
        kv.copy_(kv0)
    for T in (0.0, 1.0):
        ver = lambda: E.eagle_verify_accept(tgt, drows, tok, par, D, T, 3, draft_row=row,  # noqa
                                            accept_len=acc, path=path, emit=emit, dev_status=st)
        v = timed_ms(ver, torch, reps)
        res[f"verify_T{int(T)}_us"] = round(v * 1e3, 2)
        res[f"accept_len_T{int(T)}"] = int(acc.item())

        def step():
            expand()
            attn()
            ver()
            comp()
        gr = torch.cuda.CUDAGraph()
        step()
        torch.cuda.synchronize()
        with torch.cuda.graph(gr, capture_error_mode="relaxed"):
            step()
        res[f"step_T{int(T)}_us_graph"] = round(timed_ms(gr.replay, torch, reps) * 1e3, 2)
    res["kv_compact_40_layers_us"] = round(timed_ms(comp, torch, reps) * 1e3, 2)
    if int(st.item()) != 0:
        raise RuntimeError(f"eagle2_b1 device status {int(st.item())}")
    return res


def sweep_70b(torch, dev, peaks, reps=20):
    """The Llama-70B sweep (config 4): 64 q / 8 kv heads, d = 128, 48-node depth-6 top-10
    trees.  Each call is timed alone (median of `reps`):
      attention   one layer over B x L (B in 1/8/32/64, L in 512 .. 32768); its binding
                  roof is the larger of bytes / HBM peak and FLOPs / bf16 peak (burst: the
                  kernel is timed alone);
      verify      B x V x T x sigma (V in 32000/128256, T in 0/1, sigma in 0.1/0.5/1.0),
                  trees expanded on the GPU from synthetic draft rows (target = draft -
                  noise on expanded nodes, fresh rows at leaves); reports the accepted
                  length histogram, tau = mean(accept_len + 1), alpha1 = P(accept_len >= 1)
                  and GB/s over the visited rows (each visited node's target and draft row
                  once; T = 0 reads target rows only);
      softmax     the eager statistics of every target row, per B x V;
      compaction  80 layers (Llama-70B) per B.
    The step grid adds attention(B, L) + verify(B, V, T, sigma) + compaction(B)."""
    import eagle_tree_speculative_gb300 as E
    c = W.CONFIGS["sweep_70b"]
    ex = c.extra
    n, D, k, Hq, Hkv, d = c.n, c.depth, c.top_k, c.Hq, c.Hkv, c.head_dim
    R = c.R
    layers = 80
    hbm, tc = peaks["hbm_gbs"], peaks["bf16_tflops"]
    g = torch.Generator(device=dev).manual_seed(SEED + 51)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    res = {"attn": [], "verify": [], "softmax": [], "compact": [],
           "peaks": {"hbm_gbs": hbm, "bf16_tflops": tc, "source": peaks["source"]}}
    Bmax = max(ex["B"])

    def tree_for(V, sigma):
        trow = torch.randn(Bmax, R, V, device=dev, generator=g) * c.target_std
        drows = trow + torch.randn(Bmax, R, V, device=dev, generator=g) * sigma
        state = torch.empty(E.tree_state_size(Bmax, k, D), dtype=torch.uint8, device=dev)
        tok = torch.empty(Bmax, n, dtype=torch.int32, device=dev)
        par, row = torch.empty_like(tok), torch.empty_like(tok)
        for lvl in range(1, D + 1):
            E.eagle2_expand(lvl, lvl == D, drows, k, D, n, state, out_tokens=tok,
                            out_parent=par, out_draft_row=row, dev_status=st)
        rows = row.long()
        tgt = torch.empty(Bmax, n, V, device=dev)
        for b in range(Bmax):
            r = rows[b]
            tgt[b] = torch.where((r >= 0)[:, None], trow[b, r.clamp(min=0)],
                                 torch.randn(n, V, device=dev, generator=g) * c.target_std)
        del trow, state
        return tgt, drows, tok, par, row

    # ---- attention over B x L (trees of the V = 32000, sigma = 0.5 case) ----
    _, _, _, par_a, _ = tree_for(32000, 0.5)
    for B in ex["B"]:
        parent = par_a[:B].contiguous()
        for L in ex["L"]:
            Lmax = L + n
            q = torch.randn(B, n, Hq, d, device=dev, generator=g).to(torch.bfloat16)
            kc = torch.randn(B, Hkv, Lmax, d, device=dev, generator=g, dtype=torch.bfloat16)
            vc = torch.randn_like(kc)
            kv = torch.full((B,), L, dtype=torch.int32, device=dev)
            out = torch.empty_like(q)
            wsn = E.tree_attn_workspace_size(B, n, Hq, Hkv, d, Lmax)
            ws = torch.empty(max(wsn, 1), dtype=torch.uint8, device=dev)
            ms = timed_ms(lambda: E.eagle_tree_attn(q, kc, vc, kv, parent, out=out, workspace=ws,
                                                    dev_status=st), torch, reps)
            nbytes = 2 * B * Hkv * Lmax * d * 2 + 2 * B * n * Hq * d * 2
            flops = 4.0 * B * n * Hq * d * Lmax
            t_h, t_t = nbytes / (hbm * 1e9), flops / (tc * 1e12)
            res["attn"].append({"B": B, "L": L, "ms": round(ms, 4),
                                "GBps": round(nbytes / (ms * 1e-3) / 1e9, 1),
                                "TFLOPs": round(flops / (ms * 1e-3) / 1e12, 1),
                                "bound": "hbm" if t_h >= t_t else "tensor",
                                "frac": round(max(t_h, t_t) / (ms * 1e-3), 4),
                                "split_kv": bool(wsn)})
            del q, kc, vc, out, ws
    torch.cuda.empty_cache()
    # ---- verify and softmax statistics over B x V x T x sigma ----
    for V in ex["V"]:
        for sigma in ex["sigma"]:
            tgt, drows, tok, par, row = tree_for(V, sigma)
            for B in ex["B"]:
                t_, d_, k_, p_, r_ = (x[:B].contiguous() for x in (tgt, drows, tok, par, row))
                acc = torch.empty(B, dtype=torch.int32, device=dev)
                path = torch.empty(B, D + 1, dtype=torch.int32, device=dev)
                emit = torch.empty_like(path)
                for T in (0.0, 1.0):
                    ms = timed_ms(lambda: E.eagle_verify_accept(
                        t_, d_, k_, p_, D, T, 11, draft_row=r_, accept_len=acc, path=path,
                        emit=emit, dev_status=st), torch, reps)
                    a = acc.cpu().numpy()
                    nbytes = float((a + 1).sum()) * V * 4 * (2 if T > 0 else 1)
                    res["verify"].append({
                        "B": B, "V": V, "T": T, "sigma": sigma, "us": round(ms * 1e3, 2),
                        "GBps_visited": round(nbytes / (ms * 1e-3) / 1e9, 1),
                        "frac_visited": round(nbytes / (ms * 1e-3) / 1e9 / hbm, 4),
                        "tau": round(float(a.mean()) + 1, 4),
                        "alpha1": round(float((a >= 1).mean()), 4),
                        "accept_len_hist": np.bincount(a, minlength=D + 1).tolist()})
                if sigma == ex["sigma"][0]:
                    ms = timed_ms(lambda: E.eagle_softmax_stats(t_, 1.0, dev_status=st,
                                                                argmax=False), torch, reps)
                    nbytes = B * n * V * 4
                    res["softmax"].append({"B": B, "V": V, "ms": round(ms, 4),
                                           "GBps": round(nbytes / (ms * 1e-3) / 1e9, 1),
                                           "frac": round(nbytes / (ms * 1e-3) / 1e9 / hbm, 4)})
            del tgt, drows, tok, par, row
            torch.cuda.empty_cache()
    # ---- compaction, 80 layers ----
    for B in ex["B"]:
        Lmax = 512 + n
        kc = torch.randn(layers, B, Hkv, Lmax, d, device=dev, generator=g, dtype=torch.bfloat16)
        vc = torch.randn_like(kc)
        kv0 = torch.full((B,), 512, dtype=torch.int32, device=dev)
        kv = kv0.clone()
        path = torch.full((B, D + 1), -1, dtype=torch.int32, device=dev)
        path[:, :5] = torch.tensor([0, 3, 14, 25, 36], dtype=torch.int32)
        acc = torch.full((B,), 4, dtype=torch.int32, device=dev)

        def comp():
            E.eagle_kv_compact(kc, vc, kv, path, acc, D, dev_status=st)
            kv.copy_(kv0)
        ms = timed_ms(comp, torch, reps)
        res["compact"].append({"B": B, "layers": layers, "accepted": 4, "us": round(ms * 1e3, 2)})
        del kc, vc
        torch.cuda.empty_cache()
    if int(st.item()) != 0:
        raise RuntimeError(f"sweep device status {int(st.item())}")
    # ---- the step grid ----
    attn = {(r["B"], r["L"]): r["ms"] for r in res["attn"]}
    comp = {r["B"]: r["us"] * 1e-3 for r in res["compact"]}
    grid = []
    for r in res["verify"]:
        for L in ex["L"]:
            ms = attn[(r["B"], L)] + r["us"] * 1e-3 + comp[r["B"]]
            grid.append({"B": r["B"], "L": L, "V": r["V"], "T": r["T"], "sigma": r["sigma"],
                         "ms": round(ms, 4), "steps_per_s": round(1e3 / ms, 1),
                         "accepted_tokens_per_s": round(r["B"] * r["tau"] * 1e3 / ms, 1)})
    res["step_grid"] = grid
    return res


def breakdown(st, torch, reps=20):
    """Per-call device time (ms) with its HBM figure, each call timed alone."""
    E = st.E
    c = CFG
    res = {}

    def t(fn):
        return timed_ms(fn, torch, reps)

    res["expand_8_levels"] = round(t(lambda: st.expand()), 4)
    a = t(lambda: E.eagle_tree_attn(st.q, st.kc[0], st.vc[0], st.kv_len0, st.parent,
                                    out=st.attn_out, workspace=st.attn_ws))
    kv_bytes = 2 * c.B * c.Hkv * (c.L + c.n) * c.head_dim * 2
    flops = 4.0 * c.B * c.n * c.Hq * c.head_dim * (c.L + c.n)
    qo_bytes = 2 * c.B * c.n * c.Hq * c.head_dim * 2
    res["tree_attn_1_layer"] = round(a, 4)
    res["tree_attn_GBps"] = round((kv_bytes + qo_bytes) / (a * 1e-3) / 1e9, 1)
    res["tree_attn_TFLOPs"] = round(flops / (a * 1e-3) / 1e12, 1)
    res["tree_attn_bytes"] = kv_bytes + qo_bytes
    v = t(lambda: E.eagle_verify_accept(st.target, st.logits, st.tokens, st.parent, st.D, 1.0, 7,
                                        draft_row=st.draft_row, accept_len=st.accept_len,
                                        path=st.path, emit=st.emit))
    res["verify_accept"] = round(v, 4)
    rows_visited = float(st.accept_len.sum().item() + st.B)
    res["verify_visited_row_bytes"] = 2 * rows_visited * c.V * 4
    res["verify_visited_row_GBps"] = round(2 * rows_visited * c.V * 4 / (v * 1e-3) / 1e9, 1)

    def comp():
        E.eagle_kv_compact(st.kc, st.vc, st.kv_len, st.path, st.accept_len, st.D)
        st.kv_len.copy_(st.kv_len0)
    res["kv_compact_32_layers"] = round(t(comp), 4)

    # the verify step alone, the draft expansion excluded: attention (1 layer), the walk
    # and the compaction (32 layers) one after another, 200 calls after 20 warm-up
    def vstep():
        E.eagle_tree_attn(st.q, st.kc[0], st.vc[0], st.kv_len0, st.parent, out=st.attn_out,
                          workspace=st.attn_ws)
        E.eagle_verify_accept(st.target, st.logits, st.tokens, st.parent, st.D, 1.0, 7,
                              draft_row=st.draft_row, accept_len=st.accept_len, path=st.path,
                              emit=st.emit)
        comp()
    res["verify_step"] = round(timed_ms(vstep, torch, reps=200, warm=20), 4)
    res["verify_step_mean_accept_len_plus_1"] = round(float(st.accept_len.float().mean()) + 1, 4)
    # T = 1: the row statistics (max, sum) the walk needs; the argmax is the T = 0 output
    s = t(lambda: E.eagle_softmax_stats(st.target, 1.0, argmax=False))
    res["softmax_stats_all_rows_standalone"] = round(s, 4)
    res["softmax_stats_bytes"] = st.target.numel() * 4
    res["softmax_stats_GBps"] = round(st.target.numel() * 4 / (s * 1e-3) / 1e9, 1)
    return res


def hbm_rooflines(br, peaks):
    """HBM roofline fractions of the step's memory-bound calls, each timed alone (median):
    algorithmic bytes per launch / time, against the measured copy bandwidth."""
    hbm = peaks["hbm_gbs"]
    out = {}
    for name, key_ms, key_b, what in (
            ("tree_attn", "tree_attn_1_layer", "tree_attn_bytes",
             "K and V of the committed cache plus the tree rows, Q and O, one layer"),
            ("verify_accept", "verify_accept", "verify_visited_row_bytes",
             "target and draft rows of the visited nodes, once each (re-reads not counted)"),
            ("softmax_stats", "softmax_stats_all_rows_standalone", "softmax_stats_bytes",
             "every target row once (the eager statistics pass)")):
        gbs = br[key_b] / (br[key_ms] * 1e-3) / 1e9
        out[name] = {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(gbs / hbm, 4), "bytes_per_launch": br[key_b],
                     "ms_per_launch": br[key_ms], "bytes": what}
    out["peak_source"] = f"{peaks['source']} hbm_gbs (copy bandwidth)"
    return out


def run_e2e(st, torch, steps, graph=None, copy_streams=4, target_chunks=8, target_in_place=False):
    """The same step with the step's inputs in pinned host memory: every step copies its
    hidden states, queries and target logits host -> device, runs the step (the captured
    graph of library calls when available, else the eager calls) and reads the emitted
    tokens back.  Pipelined: two sets of input buffers, each with its own captured graph;
    while step i runs on one set, the inputs of step i+1 are copied into the other on
    `copy_streams` streams (the target logits split into `target_chunks` pieces), and a
    set is refilled only after the step that read it is done.  The timed region holds
    every step's copies and reads, the first step's copies included.

    target_in_place: the target logits stay in pinned host memory and the verify walk
    reads the rows it visits there (unified addressing over the CPU-GPU link); the
    hidden states and queries are copied as above."""
    host_hidden = [h.cpu().pin_memory() for h in st.hidden]
    host_target = st.target.cpu().pin_memory()
    host_q = st.q.cpu().pin_memory()
    out_acc = torch.empty(st.B, dtype=torch.int32).pin_memory()
    out_emit = torch.empty(st.B, st.D + 1, dtype=torch.int32).pin_memory()
    h2d = sum(h.numel() * h.element_size() for h in host_hidden) + \
        (0 if target_in_place else host_target.numel() * 4) + host_q.numel() * 2
    d2h = out_acc.numel() * 4 + out_emit.numel() * 4

    dev_target = st.target
    if target_in_place:
        sets = [(st.hidden, host_target, st.q),
                ([torch.empty_like(h) for h in st.hidden], host_target, torch.empty_like(st.q))]
    else:
        sets = [(st.hidden, st.target, st.q),
                ([torch.empty_like(h) for h in st.hidden], torch.empty_like(st.target),
                 torch.empty_like(st.q))]
    saved = (st.hidden, st.target, st.q)

    def use(k):
        st.hidden, st.target, st.q = sets[k]

    graphs = [graph, None]
    if target_in_place and graph is not None:
        graphs = [None, None]             # the given graph reads the device target
    if graph is not None:
        for k in (0, 1):
            if graphs[k] is not None:
                continue
            use(k)
            try:
                gk = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gk, capture_error_mode="relaxed"):
                    st.run(77)
                graphs[k] = gk
            except Exception:
                graphs = [None, None]
                break
        st.hidden, st.target, st.q = saved
        torch.cuda.synchronize()

    # the copies of one step, spread over the copy streams
    def pieces(k):
        hid, tgt, q = sets[k]
        out = [(d, s_) for d, s_ in zip(hid, host_hidden)] + [(q, host_q)]
        if not target_in_place:
            step = (st.B + target_chunks - 1) // target_chunks
            for b0 in range(0, st.B, step):
                out.append((tgt[b0:b0 + step], host_target[b0:b0 + step]))
        return out

    compute = torch.cuda.current_stream()
    cstreams = [torch.cuda.Stream() for _ in range(copy_streams)]
    free = [torch.cuda.Event(), torch.cuda.Event()]        # the step that read set k is done
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)

    def issue_copies(i):
        k = i % 2
        done = []
        for c, cs in enumerate(cstreams):
            cs.wait_event(free[k] if i >= 2 else start)
            with torch.cuda.stream(cs):
                for j, (dst, src) in enumerate(pieces(k)):
                    if j % copy_streams == c:
                        dst.copy_(src, non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(cs)
            done.append(ev)
        return done

    def issue_step(i, copied):
        k = i % 2
        for ev in copied:
            compute.wait_event(ev)
        if graphs[k] is not None:
            graphs[k].replay()
        else:
            use(k)
            st.run(5000 + i)
            st.hidden, st.target, st.q = saved
        free[k].record(compute)
        out_acc.copy_(st.accept_len, non_blocking=True)
        out_emit.copy_(st.emit, non_blocking=True)

    def run(n):
        start.record(compute)
        copied = issue_copies(0)
        for i in range(n):
            nxt = issue_copies(i + 1) if i + 1 < n else None
            issue_step(i, copied)
            copied = nxt
        end.record(compute)

    run(2)                                                 # warm-up of both graphs
    torch.cuda.synchronize()
    run(steps)
    torch.cuda.synchronize()
    ms = start.elapsed_time(end)
    assert st.target is dev_target
    res = {"value": round(1000.0 * steps / ms, 3), "unit": "steps/s",
           "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
           "pipelined": f"2 input buffer sets, {copy_streams} copy streams"}
    if target_in_place:
        res["target_logits"] = ("pinned host memory read in place by the verify walk "
                                f"({host_target.numel() * 4} bytes resident; only the visited "
                                "rows cross the link, not counted in h2d_bytes_per_step)")
    return res


# ---------------------------------------------------------------- oracle (CPU) arm
class OracleSample:
    """A bounded sample of one step, run by the CPU oracle as it stands.

    Per sample: one sequence's expansion from its 71 draft-logit rows (top-10 /
    select / rerank), its verify walk, its 32-layer compaction, its tree attention
    restricted to one of the 8 kv heads (4 query heads), and ONE row of the LM-head
    GEMM.  The step estimate scales each part to the full step: attention x8 heads
    x64 sequences, GEMM x4544 rows, the rest x64 sequences.
    """

    def __init__(self, seed=SEED):
        import oracle
        self.o = oracle
        c = CFG
        self.c = c
        trow, drows = W.tree_draft_rows(c, seed, B=1)
        self.drows = drows
        self.tree = oracle.eagle2_from_logits(drows, c.top_k, c.depth, c.n)
        self.tgt = W.assemble_target(trow, self.tree["draft_row"], self.tree["cand"],
                                     c.target_std, seed)
        G = c.Hq // c.Hkv
        self.q, self.k, self.v, self.kv_len = W.attn_inputs(1, c.n, G, 1, c.head_dim, c.L, c.Lmax, seed)
        self.h = W.to_bf16(W.normal((1, c.H), 1.0, seed, 99))
        self.w = W.lm_head(c.V, c.H, c.w_std, seed)
        kc, vc = W.kv_cache(1, 1, c.Hkv, c.Lmax, c.head_dim, seed)
        import torch
        self.kb = kc.view(torch.int16).numpy().view(np.uint16)
        self.vb = vc.view(torch.int16).numpy().view(np.uint16)
        self.gemm_rows = c.B * c.R - c.B * (c.top_k - 1)    # 64 + 7 * 640 = 4544

    def run(self):
        o, c = self.o, self.c
        t = {}
        t0 = time.perf_counter()
        o.eagle2_from_logits(self.drows, c.top_k, c.depth, c.n)
        t["expand"] = time.perf_counter() - t0
        t0 = time.perf_counter()
        r = o.verify_accept(self.tgt, self.drows, self.tree["tokens"], self.tree["parent"], c.depth,
                            1.0, 0, draft_row=self.tree["draft_row"])
        t["verify"] = time.perf_counter() - t0
        t0 = time.perf_counter()
        o.tree_attn(self.q, self.k, self.v, self.kv_len, self.tree["parent"], c.head_dim ** -0.5)
        t["attn_1head"] = time.perf_counter() - t0
        t0 = time.perf_counter()
        o.lmhead_rows(self.h, self.w, np.zeros(1, np.int32))
        t["gemm_1row"] = time.perf_counter() - t0
        t0 = time.perf_counter()
        kl = np.full(1, c.L, np.int32)
        for _ in range(c.n_layers):
            kl[0] = c.L
            o.kv_compact(self.kb, self.vb, kl, r["path"], r["accept_len"], c.depth)
        t["compact"] = time.perf_counter() - t0
        est = (c.B * (t["expand"] + t["verify"] + t["compact"] + c.Hkv * t["attn_1head"])
               + self.gemm_rows * t["gemm_1row"])
        return est, t


def cpu_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def set_oracle_threads(n):
    """Thread count of the oracle's OpenMP loops (its libgomp ICV on this thread)."""
    import ctypes

    import oracle
    oracle.lib()
    ctypes.CDLL("libgomp.so.1").omp_set_num_threads(int(n))


SAMPLE_DESC = ("one sequence per sample: expansion from 71 draft-logit rows, verify walk, "
               "32-layer compaction, tree attention for 1 of 8 kv heads, 1 of 4544 LM-head "
               "rows; scaled to the full B=64 step (x64 sequences, x8 heads, x4544 rows)")


def oracle_rate(s, budget_s, threads):
    """Median sampled step estimate of the oracle at `threads` OpenMP threads."""
    set_oracle_threads(threads)
    ests, secs = [], []
    t_start = time.perf_counter()
    while not ests or time.perf_counter() - t_start < budget_s:
        t0 = time.perf_counter()
        est, _ = s.run()
        secs.append(time.perf_counter() - t0)
        ests.append(est)
    return float(np.median(ests)), float(np.median(secs)), len(ests)


def cpu_baseline(budget_s=15.0):
    """The oracle as it stands on the host cores, at all threads (the contract figure) and
    at one thread."""
    s = OracleSample()
    allc = cpu_threads()
    est, sec, n = oracle_rate(s, budget_s, allc)
    est1, sec1, n1 = oracle_rate(s, budget_s / 2, 1)
    set_oracle_threads(allc)
    return {"value": round(1.0 / est, 6), "unit": "steps/s", "cores": allc,
            "kind": "oracle", "sample": SAMPLE_DESC + f"; {n} samples of {sec:.2f} s",
            "one_thread": {"value": round(1.0 / est1, 6), "unit": "steps/s", "cores": 1,
                           "sample": f"the same sample; {n1} samples of {sec1:.2f} s"}}


def workload_config(world):
    return {"workload": "EAGLE-3 tree verify step, B=64, Llama-3-8B shape: EAGLE-2 "
                        "expansion 8 levels x top-10 (LM head 4096->128256), rerank to 60 "
                        "nodes, tree attention 1 layer (32q/8kv heads, d=128, KV 4096), "
                        "verify V=128256 T=1 sigma=0.3, KV compaction 32 layers",
            "B": CFG.B, "nodes": CFG.n, "depth": CFG.depth, "top_k": CFG.top_k,
            "vocab": CFG.V, "hidden": CFG.H, "kv_len": CFG.L, "attn_layers": 1,
            "compact_layers": CFG.n_layers, "temperature": 1.0,
            "l2": "inputs larger than L2 (LM head 1.05 GB, logits 2.3 GB, KV 1.1 GB/layer)",
            "parallelism": f"replicas x{world} (sequence-sharded, no collective)"}


def run_reference(args, rank, world):
    """The oracle arm: each step is one bounded sample of the workload (one sequence's
    expansion, walk and compaction, one kv head's attention, one LM-head row), timed on
    the host cores; `value` extrapolates it to the full B=64 step."""
    if rank != 0:
        return None
    s = OracleSample()
    allc = cpu_threads()
    set_oracle_threads(allc)
    for _ in range(args.warmup):
        s.run()
    ests, secs = [], []
    t_start = time.perf_counter()
    for _ in range(args.steps):
        t0 = time.perf_counter()
        ests.append(s.run()[0])
        secs.append(time.perf_counter() - t0)
    wall = time.perf_counter() - t_start
    est = float(np.median(ests))
    value = 1.0 / est
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "steps/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * wall / args.steps, 1),
            "ms_per_step_note": "wall time of one bounded sample (what was timed); value is "
                                "extrapolated from it to the full step",
            "ms_per_full_step_extrapolated": round(est * 1e3, 1),
            "sample_seconds_median": round(float(np.median(secs)), 3),
            "extrapolated": True,
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64 (CPU oracle)", "data": "synthetic",
            "config": workload_config(world),
            "cpu_baseline": {"value": round(value, 6), "unit": "steps/s", "cores": allc,
                             "kind": "oracle", "sample": SAMPLE_DESC},
            "e2e": {"value": round(value, 6), "unit": "steps/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


KERNEL_CASES = ("gemm", "topk", "fused", "attn", "verify", "verify_filtered", "compact",
                "softmax", "ttt")


def kernel_case(name, reps):
    """Launch one library call `reps` times on a single-kernel workload of the step's
    shapes (inputs larger than L2, a few GB on the device), for profiler captures.

      gemm     LM-head GEMM of one full level: 640 x 4096 -> 128256
      topk     expansion levels 1-2 over [64, 71, 128256] draft logits: the level-2
               launch is the full 640-row top-10
      fused    expansion levels 1-2 from hidden states, as the step runs them: GEMM
               with per-tile (max, sum) partials, then the top-k merge that rescans
               only the tiles able to hold a row's top-10
      attn     tree attention, one layer, B=64, 32/8 heads, KV 4096, 60 nodes
      verify   verify-and-accept, B=32, 60 nodes, V=128256, T=1
      verify_filtered  the same with top-k 50 and top-p 0.9 (row filters, then the walk)
      compact  KV compaction, 32 layers, B=4 (8 kv heads, Lmax 4156)
      softmax  softmax statistics of [32, 60, 128256] target logits
      ttt      training-time-test attention, B=8, S=2048, 32/8 heads, round 7 of 8
    """
    import torch

    import eagle_tree_speculative_gb300 as E
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    c = CFG
    g = torch.Generator(device=dev).manual_seed(SEED + 11)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    leaf_std = float(c.w_std * np.sqrt(c.H))

    def normal(shape, std, dtype=torch.float32):      # generated in place: no f32 temporaries
        return torch.empty(shape, dtype=dtype, device=dev).normal_(0.0, std, generator=g)

    def expanded(B):
        logits = normal((B, c.R, c.V), leaf_std)
        state = torch.empty(E.tree_state_size(B, c.top_k, c.depth), dtype=torch.uint8, device=dev)
        tok = torch.empty(B, c.n, dtype=torch.int32, device=dev)
        par, row = torch.empty_like(tok), torch.empty_like(tok)
        for lvl in range(1, c.depth + 1):
            E.eagle2_expand(lvl, lvl == c.depth, logits, c.top_k, c.depth, c.n, state,
                            out_tokens=tok, out_parent=par, out_draft_row=row, dev_status=st)
        return logits, state, tok, par, row

    if name == "gemm":
        M = c.B * c.top_k
        h = normal((M, c.H), 1.0, torch.bfloat16)
        w = normal((c.V, c.H), c.w_std, torch.bfloat16)
        out = torch.empty(M, c.V, device=dev)
        fn = lambda: E.eagle_lmhead_gemm(h, w, out=out, dev_status=st)  # noqa: E731
    elif name == "topk":
        logits = normal((c.B, c.R, c.V), leaf_std)
        state = torch.empty(E.tree_state_size(c.B, c.top_k, c.depth), dtype=torch.uint8,
                            device=dev)

        def fn():
            for lvl in (1, 2):
                E.eagle2_expand(lvl, 0, logits, c.top_k, c.depth, c.n, state, dev_status=st)
    elif name == "fused":
        B, k = c.B, c.top_k
        w = normal((c.V, c.H), c.w_std, torch.bfloat16)
        hid = [normal((B, 1 if lvl == 1 else k, c.H), 1.0, torch.bfloat16) for lvl in (1, 2)]
        logits = torch.empty(B, c.R, c.V, device=dev)
        state = torch.empty(E.tree_state_size(B, k, c.depth), dtype=torch.uint8, device=dev)
        part = torch.empty(E.expand_scratch_size(B, c.V, k) // 4, device=dev)

        def fn():
            for lvl in (1, 2):
                E.eagle2_expand(lvl, 0, logits, k, c.depth, c.n, state, hidden=hid[lvl - 1],
                                lm_head_w=w, partials=part, dev_status=st)
    elif name == "attn":
        B = c.B
        _, _, _, par, _ = expanded(8)
        parent = par.repeat(B // 8, 1).contiguous()
        q = normal((B, c.n, c.Hq, c.head_dim), 1.0, torch.bfloat16)
        kc = normal((B, c.Hkv, c.Lmax, c.head_dim), 1.0, torch.bfloat16)
        vc = normal((B, c.Hkv, c.Lmax, c.head_dim), 1.0, torch.bfloat16)
        kv_len = torch.full((B,), c.L, dtype=torch.int32, device=dev)
        out = torch.empty_like(q)
        ws = E.tree_attn_workspace_size(B, c.n, c.Hq, c.Hkv, c.head_dim, c.Lmax)
        wsb = torch.empty(max(ws, 1), dtype=torch.uint8, device=dev)
        fn = lambda: E.eagle_tree_attn(q, kc, vc, kv_len, parent, out=out,  # noqa: E731
                                       workspace=wsb, dev_status=st)
    elif name in ("verify", "verify_filtered", "softmax"):
        B = 32
        logits, _, tok, par, row = expanded(B)
        target = synth_target(torch, logits, row, c.sigma, leaf_std, g)
        if name == "verify":
            fn = lambda: E.eagle_verify_accept(target, logits, tok, par, c.depth, 1.0, 7,  # noqa
                                               draft_row=row, dev_status=st)
        elif name == "verify_filtered":
            ws = torch.empty(E.verify_filter_workspace_size(B, c.n, c.R), dtype=torch.uint8,
                             device=dev)
            fn = lambda: E.eagle_verify_accept(target, logits, tok, par, c.depth, 1.0, 7,  # noqa
                                               draft_row=row, dev_status=st, top_k=50, top_p=0.9,
                                               workspace=ws)
        else:
            fn = lambda: E.eagle_softmax_stats(target, 1.0, dev_status=st,  # noqa: E731
                                               argmax=False)
    elif name == "compact":
        B = 4
        shape = (c.n_layers, B, c.Hkv, c.Lmax, c.head_dim)
        kc = normal(shape, 1.0, torch.bfloat16)
        vc = normal(shape, 1.0, torch.bfloat16)
        kv_len0 = torch.full((B,), c.L, dtype=torch.int32, device=dev)
        kv_len = kv_len0.clone()
        # every sequence accepts a path of depth 6 through nodes 0, 2, 5, 9, 14, 20, 27
        path = torch.full((B, c.depth + 1), -1, dtype=torch.int32, device=dev)
        path[:, :7] = torch.tensor([0, 2, 5, 9, 14, 20, 27], dtype=torch.int32)
        acc = torch.full((B,), 6, dtype=torch.int32, device=dev)

        def fn():
            E.eagle_kv_compact(kc, vc, kv_len, path, acc, c.depth, dev_status=st)
            kv_len.copy_(kv_len0)
    elif name == "ttt":
        t = TTT_SHAPE
        q, k, v = ttt_inputs(torch, dev, t["B"], t["S"], t["Hq"], t["Hkv"], t["R1"], g)
        out = torch.empty_like(q)
        fn = lambda: E.eagle_ttt_attn(q, k, v, t["r"], out=out, dev_status=st)  # noqa: E731
    else:
        raise ValueError(name)
    fn()                                   # warm-up (first-call set-up stays untimed)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    status = int(st.item())
    print(json.dumps({"kernel_case": name, "reps": reps,
                      "ms_per_call": round(e0.elapsed_time(e1) / reps, 4), "dev_status": status}))
    if status != 0:
        raise RuntimeError(f"device status {status}")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--config", choices=["eagle3_b64", "sweep_70b"], default="eagle3_b64",
                    help="eagle3_b64: the B=64 step (the benchmark line, with the chain and "
                         "B=1 Vicuna configs under other_configs); sweep_70b: the Llama-70B "
                         "grid, one JSON line")
    ap.add_argument("--kernel-case", choices=KERNEL_CASES, default=None,
                    help="profile helper: launch one call on its own workload and exit")
    ap.add_argument("--reps", type=int, default=3)
    args = ap.parse_args()
    if args.kernel_case:
        kernel_case(args.kernel_case, args.reps)
        return
    if args.config == "sweep_70b":
        import torch
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        print(json.dumps({"sweep_70b": sweep_70b(torch, dev, measured_peaks())}), flush=True)
        return
    args.warmup = max(args.warmup, 3)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if args.impl == "reference":
        out = run_reference(args, rank, world)
        if out is not None:
            print(json.dumps(out), flush=True)
        return
    if world > 1:
        import torch.distributed as dist
        import torch
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group("nccl")
    out = run_ours(args, rank, world, dist)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

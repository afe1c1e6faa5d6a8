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
# DRAM bytes (read + write) of one 640 x 4096 -> 128256 LM-head GEMM launch, from an
# ncu capture of the current kernel: 1.0965e9 read + 0.3010e9 written.
GEMM_LAUNCH_DRAM_BYTES = 1.3976e9
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
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
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
                "samples": len(sm), "reasons": sorted(reasons)}


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
    if dist:
        dist.barrier()
    clocks = ClockSampler(local)
    clocks.start()
    if graph is not None:
        ms = time_region(lambda i: graph.replay(), args.steps, torch)
    else:
        ms = time_region(lambda i: st.run(i), args.steps, torch)
    clk = clocks.stop()
    ms = reduce_over_ranks(ms, dist, dev, "max")
    ms_per_step = ms / args.steps
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
        "timing": "CUDA graph of one step replayed" if graph is not None else "eager launches",
        "eager_ms_per_step_wall": round(1e3 * t_eager / eager_steps, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16 GEMM/attention (fp32 accumulate), f32 logits",
        "data": "synthetic (seeded normals; random-init LM head; no datasets or trained weights)",
        "config": {"workload": "EAGLE-3 tree verify step, B=64, Llama-3-8B shape: EAGLE-2 "
                               "expansion 8 levels x top-10 (LM head 4096->128256), rerank to 60 "
                               "nodes, tree attention 1 layer (32q/8kv heads, d=128, KV 4096), "
                               "verify V=128256 T=1 sigma=0.3, KV compaction 32 layers",
                   "B": CFG.B, "nodes": CFG.n, "depth": CFG.depth, "top_k": CFG.top_k,
                   "vocab": CFG.V, "hidden": CFG.H, "kv_len": CFG.L, "attn_layers": 1,
                   "compact_layers": CFG.n_layers, "temperature": 1.0,
                   "l2": "inputs larger than L2 (LM head 1.05 GB, logits 2.3 GB, KV 1.1 GB/layer)",
                   "parallelism": f"replicas x{world} (sequence-sharded, no collective)"},
        "accepted_tokens_per_s": round(tok_all_ranks * 1000.0 / ms_per_step, 1),
        "mean_accept_len_plus_1": round(tok_all_ranks / (world * st.B), 4),
        "graph_step_accepted_tokens": acc_graph,
        "roofline": {"kernel": "lmhead_gemm_kernel (tcgen05), 640 x 4096 -> 128256 launches",
                     "bound": "tensor",
                     "achieved": round(gemm_tflops, 1), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(gemm_tflops / peak, 4), "traffic": GEMM_LAUNCH_DRAM_BYTES,
                     "traffic_note": "dram__bytes_read.sum + dram__bytes_write.sum of one "
                                     "640-row launch (ncu); algorithmic 1.384e9",
                     "peak_source": f"{peaks['source']} bf16_tflops_sustained",
                     "flops_per_launch": full_flops,
                     "ms_per_launch": round(full_ms, 4),
                     "gemm_ms_per_step_all_levels": round(gemm_ms / eager_steps, 4),
                     "gemm_flops_per_step_all_levels": gemm_flops / eager_steps,
                     "timed": f"{eager_steps} eager steps, events around each launch"},
        "breakdown_ms": br,
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


def breakdown(st, torch, reps=20):
    """Per-call device time (ms) with its HBM figure, each call timed alone."""
    E = st.E
    c = CFG
    res = {}

    def t(fn):
        for _ in range(3):
            fn()
        return time_region(lambda i: fn(), reps, torch) / reps

    res["expand_8_levels"] = round(t(lambda: st.expand()), 4)
    a = t(lambda: E.eagle_tree_attn(st.q, st.kc[0], st.vc[0], st.kv_len0, st.parent,
                                    out=st.attn_out, workspace=st.attn_ws))
    kv_bytes = 2 * c.B * c.Hkv * (c.L + c.n) * c.head_dim * 2
    flops = 4.0 * c.B * c.n * c.Hq * c.head_dim * (c.L + c.n)
    res["tree_attn_1_layer"] = round(a, 4)
    res["tree_attn_GBps"] = round(kv_bytes / (a * 1e-3) / 1e9, 1)
    res["tree_attn_TFLOPs"] = round(flops / (a * 1e-3) / 1e12, 1)
    v = t(lambda: E.eagle_verify_accept(st.target, st.logits, st.tokens, st.parent, st.D, 1.0, 7,
                                        draft_row=st.draft_row, accept_len=st.accept_len,
                                        path=st.path, emit=st.emit))
    res["verify_accept"] = round(v, 4)
    rows_visited = float(st.accept_len.sum().item() + st.B)
    res["verify_visited_row_GBps"] = round(2 * rows_visited * c.V * 4 / (v * 1e-3) / 1e9, 1)

    def comp():
        E.eagle_kv_compact(st.kc, st.vc, st.kv_len, st.path, st.accept_len, st.D)
        st.kv_len.copy_(st.kv_len0)
    res["kv_compact_32_layers"] = round(t(comp), 4)
    s = t(lambda: E.eagle_softmax_stats(st.target, 1.0))
    res["softmax_stats_all_rows_standalone"] = round(s, 4)
    res["softmax_stats_GBps"] = round(st.target.numel() * 4 / (s * 1e-3) / 1e9, 1)
    return res


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


SAMPLE_DESC = ("one sequence per sample: expansion from 71 draft-logit rows, verify walk, "
               "32-layer compaction, tree attention for 1 of 8 kv heads, 1 of 4544 LM-head "
               "rows; scaled to the full B=64 step (x64 sequences, x8 heads, x4544 rows)")


def cpu_baseline(budget_s=15.0):
    s = OracleSample()
    ests = []
    t_start = time.perf_counter()
    while not ests or time.perf_counter() - t_start < budget_s:
        est, _ = s.run()
        ests.append(est)
    est = float(np.median(ests))
    return {"value": round(1.0 / est, 6), "unit": "steps/s", "cores": cpu_threads(),
            "kind": "oracle", "sample": SAMPLE_DESC + f"; {len(ests)} samples"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    s = OracleSample()
    for _ in range(args.warmup):
        s.run()
    ests = [s.run()[0] for _ in range(args.steps)]
    est = float(np.median(ests))
    value = 1.0 / est
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "steps/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(est * 1e3, 1), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64 (CPU oracle)", "data": "synthetic",
            "config": {"workload": "EAGLE-3 tree verify step, B=64, Llama-3-8B shape "
                                   "(same workload as the GPU arm; bounded CPU sample, scaled)"},
            "cpu_baseline": {"value": round(value, 6), "unit": "steps/s", "cores": cpu_threads(),
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
            fn = lambda: E.eagle_softmax_stats(target, 1.0, dev_status=st)  # noqa: E731
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
    ap.add_argument("--kernel-case", choices=KERNEL_CASES, default=None,
                    help="profile helper: launch one call on its own workload and exit")
    ap.add_argument("--reps", type=int, default=3)
    args = ap.parse_args()
    if args.kernel_case:
        kernel_case(args.kernel_case, args.reps)
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

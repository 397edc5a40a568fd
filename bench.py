#!/usr/bin/env python
"""Benchmark of the DFlash speculate-and-verify step on GB300.

Metric: verified (emitted) tokens/s per GB300 and draft+verify step time, on
a Qwen3-8B-shaped random-init bf16 target with a 5-layer block-diffusion
drafter (B = 16, batch 1, 2048-token random prompt).  One step = one block
draft pass + one target verify pass + accept/commit + KV injection.

Timing: W untimed warm-up steps, then K steps between CUDA events on the
launching stream, bracketed by a barrier and a device synchronize; max over
ranks.  Every step streams ~19 GB of weights, far above the 129 MB L2, so no
explicit L2 flush is needed between steps.  SM clocks are sampled with
nvidia-smi during the timed region.

Also reported: the end-to-end rate through the C ABI with host buffers
(H2D of each step's anchors from pinned memory, D2H of its emitted tokens),
the GEMM kernel class against the measured HBM peak (live CUDA-event timing
from the library's profiler over a second pass of the same steps), the AR
step cost and the projected speedup S = C_AR * E[L] / C_DF with E[L] from
the pages, and the CPU oracle timed on a bounded sample on the host cores.

--impl reference times that oracle alone (the reference arm: the pages ship
no code, so the plain CPU restatement is the baseline program).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
E2E_WARMUP = 2  # untimed end-to-end steps before the timed ones
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as wl  # noqa: E402

PAGES_ACCEPT_LEN = 7.84  # mean acceptance length on MATH-500 (Deep Research Report)
METRIC = "verified tokens/s per GB300 and draft+verify step µs (Qwen3-8B shape, B=16)"


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def sustained_tflops():
    """bf16 tensor peak for a kernel timed inside a long step (the power-capped
    figure), and where it comes from."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        if "bf16_tflops_sustained" in p:
            return float(p["bf16_tflops_sustained"]), "measured"
    return 1700.0, "fallback"


def gemm_roofline(nbytes: float, flops: float, ms: float, hbm_gbs: float, tflops: float):
    """(bound, achieved, peak, unit) of a kernel class from its algorithmic bytes
    and flops and its time: HBM while its arithmetic intensity is below the
    machine balance (peak flop/s over peak bytes/s), the tensor pipe above it."""
    secs = ms / 1e3
    if secs <= 0:
        return "hbm", 0.0, hbm_gbs, "GB/s"
    if flops / max(nbytes, 1.0) < (tflops * 1e12) / (hbm_gbs * 1e9):
        return "hbm", nbytes / secs / 1e9, hbm_gbs, "GB/s"
    return "tensor", flops / secs / 1e12, tflops, "TFLOP/s"


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU oracle sample (the reported CPU baseline and the reference arm)
# ---------------------------------------------------------------------------
class OracleSample:
    """Times the oracle on a bounded sample of one step and extrapolates.

    Sample: one target layer and one draft layer over 2 block rows (with the
    real P-row context in attention), 1/16 of the lm_head rows for 1 token
    row, and the fused injection projection for 1 row -- all with the
    oracle's own fp64 functions.  Extrapolated to one step of the workload:
    B rows x L target layers, B rows x L_d draft layers, 2B-1 lm_head rows,
    B injected rows at most (a+1 with random weights: 1).
    """

    def __init__(self, w: wl.Workload):
        from oracle import numerics as nm
        from oracle.models import Weights
        s = w.shape
        self.w, self.s, self.nm = w, s, nm
        self.W = Weights(wl.SyntheticWeights(s, w.seed))
        P = (w.prompt_len[0] + w.prompt_len[1]) // 2
        rng = np.random.default_rng(5)
        self.P = P
        self.ck = nm.round_bf16(rng.standard_normal((P, s.n_kv_heads, s.head_dim)))
        self.cv = nm.round_bf16(rng.standard_normal((P, s.n_kv_heads, s.head_dim)))
        self.x = rng.standard_normal((2, s.d_model)) * 0.1
        self.hcat = rng.standard_normal((1, s.n_inject * s.d_model)) * 0.1
        keys = ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate", "w_up", "w_down")
        for pre in ("layers.0", "draft.layers.0"):
            for k in keys:
                self.W[f"{pre}.{k}"]
        sw = self.W.source
        rows = sw.offsets("lm_head")[: s.vocab // 16]
        self.lm_part = wl.pool_rows(sw.pool(), rows, s.d_model).astype(np.float64)
        self.W["final_norm"], self.W["draft.fuse"]

    def step_seconds(self):
        from oracle.models import _layer
        nm, s, W, P = self.nm, self.s, self.W, self.P
        B = self.w.block_size
        prec = nm.Precision("bf16emu")
        pos = P + np.arange(2)

        def causal(q, k, v):
            kk, vv = np.concatenate([self.ck, k]), np.concatenate([self.cv, v])
            return np.stack([nm.attend(q[i], kk[: P + i + 1], vv[: P + i + 1]) for i in range(2)])

        def full(q, k, v):
            kk, vv = np.concatenate([self.ck, k]), np.concatenate([self.cv, v])
            return np.stack([nm.attend(q[i], kk, vv) for i in range(2)])

        t = time.perf_counter()
        _layer(W, s, prec, "layers.0", self.x, pos, causal)
        t_tl = (time.perf_counter() - t) / 2
        t = time.perf_counter()
        _layer(W, s, prec, "draft.layers.0", self.x, pos, full)
        t_dl = (time.perf_counter() - t) / 2
        t = time.perf_counter()
        nm.linear(nm.rmsnorm(self.x[:1], W["final_norm"], s.rms_eps), self.lm_part)
        t_lm = (time.perf_counter() - t) * 16
        t = time.perf_counter()
        nm.linear(self.hcat, W["draft.fuse"])
        t_inj = time.perf_counter() - t
        rows_v = self.w.tree_budget + 1 if self.w.tree_budget else B
        per_seq = (rows_v * s.n_layers * t_tl + B * s.n_draft_layers * t_dl
                   + (rows_v + B - 1) * t_lm + t_inj)
        sampled = 2 * t_tl + 2 * t_dl + t_lm / 16 + t_inj
        return per_seq * self.w.batch, sampled

    def describe(self, sampled):
        s, B, b = self.s, self.w.block_size, self.w.batch
        rows_v = self.w.tree_budget + 1 if self.w.tree_budget else B
        return (f"oracle (fp64 numpy) on 2 rows of 1 target layer and 1 draft layer at context "
                f"{self.P}, 1/16 of the lm_head for 1 row, the fuse projection for 1 row; "
                f"extrapolated per sequence to {rows_v} verify rows x {s.n_layers} target layers, "
                f"{B} draft rows x {s.n_draft_layers} draft layers and {rows_v + B - 1} lm_head "
                f"rows, times {b} sequence(s) per step; {sampled:.2f}s of CPU work per sample")


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def reduce_over_ranks(ms: float, emitted: int, world: int):
    """Whole-job timing of N independent replicas: the slowest rank's timed
    region and the tokens all ranks emitted (rank-local values when N = 1)."""
    if world <= 1:
        return ms, emitted
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    n = torch.tensor([emitted], dtype=torch.float64)
    dist.all_reduce(n, op=dist.ReduceOp.SUM)
    return float(t.item()), int(n.item())


def run_reference(args, w: wl.Workload) -> None:
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    smp = OracleSample(w)
    for _ in range(args.warmup):
        smp.step_seconds()
    times, sampled = [], []
    for _ in range(args.steps):
        sec, cpu_s = smp.step_seconds()
        times.append(sec)
        sampled.append(cpu_s)
    per_step = statistics.median(times)
    sample_s = statistics.median(sampled)
    info = smp.describe(sample_s) + f"; {args.steps} samples, median"
    value = w.batch * 1.0 / per_step  # random-init weights: one verified token per sequence and step
    # steps / ms_per_step describe what was timed: one bounded sample per
    # step; the metric is extrapolated from it to a whole step of the workload
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": sample_s * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "extrapolated": True, "extrapolated_ms_per_workload_step": per_step * 1e3,
        "config": {"workload": w.name, "batch": w.batch, "prompt_len": w.prompt_len[0],
                   "block": w.block_size},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": info},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def run_ours(args, w: wl.Workload) -> None:
    import torch
    import torch.distributed as dist

    from block_diffusion_speculative_injection_gb300 import capi
    from block_diffusion_speculative_injection_gb300.engine import DFlashEngine, capture_step_graph

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("gloo")

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()

    B = w.block_size
    b = w.batch
    lens = wl.prompt_lengths(w)
    prompts = wl.prompts(w)
    total_steps = args.warmup + args.steps + args.prof_steps + args.e2e_steps + E2E_WARMUP + 4
    max_ctx = max(lens) + B * (total_steps + 2) + args.ar_steps + 64
    tree = w.tree_budget > 0
    nmax = w.tree_budget + 1 if tree else 0
    max_ctx += nmax
    eng = DFlashEngine(w.shape, B, b, max_ctx, max_rows=max(max(lens), b * max(B, nmax)),
                       max_tree_nodes=nmax, seed=w.seed)

    def one_step(anchor_buf):
        if tree:
            r = eng.tree_step(sid, anchor_buf, w.topk, w.tree_budget)
            return r["emitted"], r["accept_len"], r["next_anchor"]
        o = eng.step(sid, anchor_buf)
        return o.emitted, o.accept_len, o.next_anchor

    ctx = eng.ctx
    sid = eng.seq_ids(b)
    stream = torch.cuda.current_stream()

    anchors = eng.prefill(prompts)
    for _ in range(args.warmup):
        one_step(anchors)
        anchors = eng.next_anchor[:b].clone()
    graph = ar_graph = None
    per_step_launches = None
    if not args.no_graph:
        l_cap = capi.dflash_launch_count(ctx)
        graph = capture_step_graph(eng, sid, tree=tree, topk=w.topk, budget=w.tree_budget)
        per_step_launches = capi.dflash_launch_count(ctx) - l_cap
        for _ in range(2):
            graph.replay()
    gen = eng.gen_counts()
    sampler = ClockSampler(local)
    sampler.start()
    barrier()
    g0 = gen.clone()
    l0 = capi.dflash_launch_count(ctx)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    if graph is not None:
        for _ in range(args.steps):
            graph.replay()
    else:
        for _ in range(args.steps):
            one_step(eng.next_anchor[:b])
    ev1.record(stream)
    barrier()
    clocks = sampler.stop()
    launches = (per_step_launches * args.steps if graph is not None
                else capi.dflash_launch_count(ctx) - l0)
    ms = ev0.elapsed_time(ev1)
    anchors = eng.next_anchor[:b].clone()
    emitted = int((gen - g0)[:b].sum().item())
    ms, emitted_all = reduce_over_ranks(ms, emitted, world)
    value = emitted_all / (ms / 1e3)
    step_ms = ms / args.steps
    tau = emitted / (args.steps * b)

    # live per-kernel timing over a second pass of the same steps
    capi.dflash_profile(ctx, True)
    for _ in range(args.prof_steps):
        one_step(anchors)
        anchors = eng.next_anchor[:b].clone()
    capi.dflash_profile(ctx, False)
    prof = {}
    names = {capi.PROF_GEMM: "gemm_tc_kernel", capi.PROF_ATTN: "attention", capi.PROF_ROW: "row_ops",
             capi.PROF_VOCAB: "vocab_reduce", capi.PROF_SPEC: "accept_tree"}
    for k, name in names.items():
        n, kms, kbytes, kflops = capi.dflash_profile_read(ctx, k)
        prof[name] = {"launches_per_step": n / max(args.prof_steps, 1),
                      "ms_per_step": kms / max(args.prof_steps, 1),
                      "bytes": kbytes, "flops": kflops, "ms": kms, "n": n}
    hbm, tflops, src = peaks()
    t_sus, t_src = sustained_tflops()
    g = prof["gemm_tc_kernel"]
    gemm_step_bytes = g["bytes"] / max(args.prof_steps, 1)
    # one launch: algorithmic bytes / flops per launch over the mean launch time
    bound, achieved, peak, unit = gemm_roofline(g["bytes"] / max(g["n"], 1), g["flops"] / max(g["n"], 1),
                                                g["ms"] / max(g["n"], 1), hbm, t_sus)
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "gemm_traffic.json")
    if os.path.exists(tpath):
        with open(tpath) as f:
            tj = json.load(f)
        if tj.get("workload") == w.name and tj.get("kernel_rev") == KERNEL_REV:
            traffic = tj.get("dram_bytes_per_launch")

    # AR step cost (the B = 1 path: verify the anchor alone, commit it)
    for _ in range(3):
        eng.ar_step(sid, anchors)
        anchors = eng.next_anchor[:b].clone()
    if not args.no_graph:
        ar_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(ar_graph):
            eng.ar_step(sid, eng.next_anchor[:b])
        ar_graph.replay()
    barrier()
    ev0.record(stream)
    for _ in range(args.ar_steps):
        if ar_graph is not None:
            ar_graph.replay()
        else:
            eng.ar_step(sid, eng.next_anchor[:b])
    ev1.record(stream)
    barrier()
    ar_ms = ev0.elapsed_time(ev1) / args.ar_steps
    anchors = eng.next_anchor[:b].clone()

    # end to end through the C ABI with host buffers
    h_anchor = torch.empty(b, dtype=torch.int32, pin_memory=True)
    h_anchor.copy_(anchors.cpu())
    h_emit = torch.empty(b, max(B, nmax), dtype=torch.int32, pin_memory=True)
    h_acc = torch.empty(b, dtype=torch.int32, pin_memory=True)
    d_anchor = torch.empty(b, dtype=torch.int32, device="cuda")
    q_rows = nmax if tree else B

    def e2e_step():
        if graph is not None:
            # the captured step reads its anchors from the engine's next-anchor
            # buffer and leaves its results in the engine's step buffers
            eng.next_anchor[:b].copy_(h_anchor, non_blocking=True)
            graph.replay()
            em = eng.emitted[: b * q_rows].view(b, q_rows)
            acc, nxt = eng.accept_len[:b], eng.next_anchor[:b]
        else:
            d_anchor.copy_(h_anchor, non_blocking=True)
            em, acc, nxt = one_step(d_anchor)
        h_emit[:, :q_rows].copy_(em.view(b, q_rows), non_blocking=True)
        h_acc.copy_(acc, non_blocking=True)
        h_anchor.copy_(nxt, non_blocking=True)
        stream.synchronize()
        return int(h_acc.sum().item()) + b

    for _ in range(E2E_WARMUP):  # first pinned copies and host ops, untimed
        e2e_step()
    barrier()
    t0 = time.perf_counter()
    e2e_tokens = 0
    for _ in range(args.e2e_steps):
        e2e_tokens += e2e_step()
    e2e_s = time.perf_counter() - t0
    barrier()
    e2e_value = e2e_tokens * world / e2e_s

    if rank != 0:
        eng.close()
        return
    weights = eng.weights
    eng.close()
    del eng
    torch.cuda.empty_cache()
    # the other bars of the step, measured in the same run (one GPU only: at
    # N > 1 the replicas would repeat them)
    extras = None
    if world == 1 and not args.no_extras and w.name == "qwen3_8b_b1":
        sx, wx = max(5, min(args.steps, 20)), 3
        extras = {}
        pts, clk = attn_op_points(min(args.steps, 10), wx, local)
        head = next(pt for pt in pts if pt["ctx"] == 16384 and pt["batch"] == 32)
        extras["attn_op"] = {
            "kernel": ATTN_KERNELS, "headline": {"ctx": 16384, "batch": 32, "us": head["us"],
                                                 "gbs": head["gbs"], "frac": head["frac"]},
            "points": [{k: pt[k] for k in ("ctx", "batch", "us", "gbs", "frac")} for pt in pts],
            "peak_gbs": hbm, "peak_source": src,
            "l2": "256 MB buffer written before every timed call", "clocks": clk}
        extras["b32"] = workload_steps(wl.WORKLOADS["qwen3_8b_b32"], sx, wx, 3, local,
                                       weights=weights)[0]
        del weights  # the Qwen-shaped weights are not needed past this point
        torch.cuda.empty_cache()
        extras["ddtree_b4"] = workload_steps(wl.WORKLOADS["llama31_8b_ddtree_b4"], sx, wx, 3,
                                             local)[0]
    else:
        del weights
    cpu = None
    if not args.no_cpu_baseline:
        smp = OracleSample(w)
        smp.step_seconds()
        secs, cpu_s, t_end = [], [], time.perf_counter() + 10.0
        while time.perf_counter() < t_end or len(secs) < 3:
            a, c = smp.step_seconds()
            secs.append(a)
            cpu_s.append(c)
        sec = statistics.median(secs)
        cpu = {"value": b / sec, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
               "sample": smp.describe(statistics.median(cpu_s)) + f"; {len(secs)} samples, median"}
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded random-init weights, uniform random prompt tokens)",
        "config": {"workload": w.name, "batch": b, "prompt_len": lens[0],
                   "block": B, "draft_layers": w.shape.n_draft_layers,
                   "inject_layers": list(w.shape.inject_layers), "parallelism": "replicas",
                   "l2": "no flush: every step streams ~19 GB of weights (> 129 MB L2)"},
        "step_us": step_ms * 1e3,
        "graph": graph is not None,
        "tau": tau,
        "ar_step_us": ar_ms * 1e3,
        "projected_speedup": ar_ms * PAGES_ACCEPT_LEN / step_ms,
        "gpu_launches": launches,
        "roofline": {"bound": bound, "kernel": "gemm_tc_kernel", "achieved": achieved,
                     "peak": peak, "unit": unit, "frac": achieved / peak, "traffic": traffic,
                     "peak_source": src if bound == "hbm" else t_src + " (sustained bf16)",
                     "bytes_per_launch": g["bytes"] / g["n"] if g["n"] else None,
                     "launches_per_step": g["launches_per_step"],
                     "ms_per_step": g["ms_per_step"],
                     # the graph-replayed step: every GEMM byte of a step over the
                     # whole step time (a lower bound on the GEMMs' own rate)
                     "achieved_over_step": gemm_step_bytes / (step_ms / 1e3) / 1e9,
                     "frac_over_step": gemm_step_bytes / (step_ms / 1e3) / 1e9 / hbm},
        "kernel_ms_per_step": {k: v["ms_per_step"] for k, v in prof.items()},
        "clocks": clocks,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": 4 * b,
                "d2h_bytes_per_step": 4 * b * (nmax if tree else B) + 8 * b,
                "how": ("replay of the captured step" if graph is not None else "eager C-ABI calls")
                       + "; anchors in from pinned host memory, emitted tokens, accept lengths and "
                         "next anchors out, a stream synchronize, every step"},
        "cpu_baseline": cpu,
    }
    if extras is not None:
        line.update(extras)
        line["bars"] = {
            "attention_hbm_frac": {f"ctx{pt['ctx']}_b{pt['batch']}": round(pt["frac"], 3)
                                   for pt in extras["attn_op"]["points"] if pt["ctx"] >= 8192},
            "b32_gemm_frac_sustained_live": extras["b32"]["gemm"]["frac_live"],
            "b32_gemm_frac_sustained_over_step": extras["b32"]["gemm"]["frac_over_step"]}
    print(json.dumps(line))


KERNEL_REV = "gemm-v11"  # vocabulary epilogue, token-tile-first grid, persistent form (12 epilogue warps, top-2 lm_head, stream-K remainder), batched cluster epilogue, 12 warps above 128 rows, split-chunk pair epilogues
ATTN_KERNELS = "attn_tc_kernel (+ attn_combine_kernel)"


def attn_op_points(steps: int, warmup: int, local: int, only=None):
    """Block attention op (dflash_block_attention) over the grid of context
    lengths x batches: Q [b,16,32,128], K/V [b,8,ctx+16,128] bf16, block
    visible without mask.  Each point: `warmup` calls, then `steps` calls
    timed one by one with CUDA events on the launching stream, a 256 MB
    buffer written and another 256 MB read between calls so that every call
    starts with a cold L2 that holds no dirty lines (a write alone leaves the
    L2 full of the flush buffer's lines, whose write-back then lands inside
    the timed call), and the GPU kept busy (a timed sleep) while the host
    prepares the call, so that the events bracket the GPU's work and not the
    host's argument marshalling; the median against the measured HBM peak.
    Returns (points, clocks)."""
    import torch

    from block_diffusion_speculative_injection_gb300 import capi
    from block_diffusion_speculative_injection_gb300.engine import device_operand

    H, HKV, HD = wl.ATTN_OP_HEADS
    BLK = 16
    hbm, _, _ = peaks()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    flush_rd = torch.ones(256 << 20, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    sampler = ClockSampler(local)
    points = []
    sampler.start()
    grid = [only] if only else [(c, b) for c in wl.ATTN_OP_CTX for b in wl.ATTN_OP_BATCH]
    for ctx, b in grid:
        q = device_operand("q", b * BLK * H).view(b, BLK, H, HD)
        k = device_operand("k", b * HKV * (ctx + BLK)).view(b, HKV, ctx + BLK, HD)
        v = device_operand("v", b * HKV * (ctx + BLK)).view(b, HKV, ctx + BLK, HD)
        out = torch.empty_like(q)
        need = capi.dflash_block_attention_workspace(b, H, HKV, ctx, BLK)
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
        for _ in range(warmup):
            capi.dflash_block_attention(b, H, HKV, ctx, BLK, 0, q, k, v, out, ws)
        times = []
        for _ in range(steps):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            flush.fill_(1)
            flush_rd.sum(dtype=torch.int32)  # evicts the fill's dirty lines before e0
            torch.cuda._sleep(200000)  # ~0.1 ms: covers the host side of the call
            e0.record(stream)
            capi.dflash_block_attention(b, H, HKV, ctx, BLK, 0, q, k, v, out, ws)
            e1.record(stream)
            e1.synchronize()
            times.append(e0.elapsed_time(e1) * 1e3)
        us = statistics.median(times)
        nbytes = b * (4096 * ctx + 327680)  # ctx + block K/V, Q and O per sequence
        gbs = nbytes / (us * 1e-6) / 1e9
        points.append({"ctx": ctx, "batch": b, "us": us, "bytes": nbytes, "gbs": gbs,
                       "frac": gbs / hbm, "roofline_us": nbytes / (hbm * 1e9) * 1e6})
        del q, k, v, out, ws
    clocks = sampler.stop()
    del flush
    torch.cuda.empty_cache()
    return points, clocks


def run_attn_op(args) -> None:
    """The block attention op grid as its own benchmark line (headline point:
    the largest context and batch)."""
    import torch

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    hbm, _, src = peaks()
    only = None
    if args.attn_point:  # one point of the grid, e.g. for a profiler capture
        c, b = args.attn_point.lower().split("x")
        only = (int(c), int(b))
    points, clocks = attn_op_points(args.steps, args.warmup, local, only)
    head = points[0] if only else next(
        pt for pt in points if pt["ctx"] == max(wl.ATTN_OP_CTX) and pt["batch"] == max(wl.ATTN_OP_BATCH))
    line = {
        "metric": "block attention op: achieved HBM bandwidth (Q [b,16,32,128] over ctx+16 keys, GQA 4:1)",
        "value": head["gbs"], "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": head["us"] / 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) operands)",
        "config": {"workload": "attn_op", "points": f"ctx {list(wl.ATTN_OP_CTX)} x batch {list(wl.ATTN_OP_BATCH)}",
                   "headline_point": {"ctx": head["ctx"], "batch": head["batch"]},
                   "l2": "256 MB buffer written before every timed call",
                   "host": "GPU kept busy while the host prepares each timed call"},
        "roofline": {"bound": "hbm", "kernel": ATTN_KERNELS, "achieved": head["gbs"],
                     "peak": hbm, "unit": "GB/s", "frac": head["gbs"] / hbm, "traffic": None,
                     "peak_source": src},
        "points": points,
        "clocks": clocks,
    }
    print(json.dumps(line))


def workload_steps(w: wl.Workload, steps: int, warmup: int, prof_steps: int, local: int,
                   weights=None):
    """Graph-replayed steps of one workload on this GPU (the same step the
    headline times: draft, verify, accept, injection; the tree step for a
    DDTree workload).  Returns (summary, weights) so that a later workload of
    the same model can reuse the uploaded weights."""
    import torch

    from block_diffusion_speculative_injection_gb300 import capi
    from block_diffusion_speculative_injection_gb300.engine import DFlashEngine, capture_step_graph

    B, b = w.block_size, w.batch
    lens = wl.prompt_lengths(w)
    tree = w.tree_budget > 0
    nmax = w.tree_budget + 1 if tree else 0
    total = warmup + steps + prof_steps + 6
    max_ctx = max(lens) + B * (total + 2) + nmax + 64
    eng = DFlashEngine(w.shape, B, b, max_ctx, max_rows=max(max(lens), b * max(B, nmax)),
                       max_tree_nodes=nmax, seed=w.seed, weights=weights)
    sid = eng.seq_ids(b)
    eng.prefill(wl.prompts(w))

    def one():
        if tree:
            eng.tree_step(sid, eng.next_anchor[:b], w.topk, w.tree_budget)
        else:
            eng.step(sid, eng.next_anchor[:b])

    for _ in range(warmup):
        one()
    graph = capture_step_graph(eng, sid, tree=tree, topk=w.topk, budget=w.tree_budget)
    for _ in range(2):
        graph.replay()
    stream = torch.cuda.current_stream()
    gen = eng.gen_counts()
    sampler = ClockSampler(local)
    sampler.start()
    torch.cuda.synchronize()
    g0 = gen.clone()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(steps):
        graph.replay()
    ev1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    ms = ev0.elapsed_time(ev1)
    emitted = int((gen - g0)[:b].sum().item())
    step_ms = ms / steps
    capi.dflash_profile(eng.ctx, True)
    for _ in range(prof_steps):
        one()
    capi.dflash_profile(eng.ctx, False)
    n, gms, gbytes, gflops = capi.dflash_profile_read(eng.ctx, capi.PROF_GEMM)
    na, ams, _, _ = capi.dflash_profile_read(eng.ctx, capi.PROF_ATTN)
    t_sus, t_src = sustained_tflops()
    flops_step = gflops / max(prof_steps, 1)
    gemm_ms_live = gms / max(prof_steps, 1)
    # GEMM launches grouped by their work (one group per projection shape)
    by_shape = {}
    for lms, lfl in capi.dflash_profile_list(eng.ctx, capi.PROF_GEMM):
        g = by_shape.setdefault(round(lfl / 1e9, 3), [0, 0.0])
        g[0] += 1
        g[1] += lms
    shapes = [{"gflop": k, "launches_per_step": v[0] / max(prof_steps, 1),
               "ms_per_step": v[1] / max(prof_steps, 1),
               "tflops": k * v[0] / v[1] if v[1] else None}
              for k, v in sorted(by_shape.items(), key=lambda kv: -kv[1][1])]
    out = {
        "workload": w.name, "batch": b, "block": B, "steps": steps, "warmup": warmup,
        "prompt_len": [min(lens), max(lens)], "tree_nodes": nmax or None,
        "step_ms": step_ms, "tokens_per_s": emitted / (ms / 1e3), "tau": emitted / (steps * b),
        "gemm": {"launches_per_step": n / max(prof_steps, 1), "tflop_per_step": flops_step / 1e12,
                 "ms_per_step_live": gemm_ms_live,
                 "tflops_live": flops_step / (gemm_ms_live / 1e3) / 1e12 if gemm_ms_live else None,
                 "frac_live": (flops_step / (gemm_ms_live / 1e3) / 1e12 / t_sus) if gemm_ms_live else None,
                 "tflops_over_step": flops_step / (step_ms / 1e3) / 1e12,
                 "frac_over_step": flops_step / (step_ms / 1e3) / 1e12 / t_sus,
                 "peak_tflops": t_sus, "peak_source": t_src + " (sustained bf16)",
                 "by_shape_live": shapes},
        "attention_ms_per_step_live": ams / max(prof_steps, 1),
        "clocks": clocks,
        "timing": "CUDA-graph replays, CUDA events on the launching stream; live per-launch "
                  "classes from an eager pass with an event pair around every launch",
    }
    weights = eng.weights
    eng.close()
    del eng, graph
    torch.cuda.empty_cache()
    return out, weights


def run_spec_sample_op(args) -> None:
    """Temperature-1 acceptance op (dflash_spec_accept_sampled) and the draft
    draws (dflash_sample_rows) on seeded fp32 logits of the Qwen3-8B
    vocabulary, block 16, batch 1 and 32.  Each timed call reads both
    [batch, 16, V] logit arrays once (per-chunk stats) and the two rows of
    each sequence's final draw once more; the inputs exceed L2 at batch 32,
    and a 256 MB buffer is written before every timed call."""
    import torch

    from block_diffusion_speculative_injection_gb300 import capi

    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    V, B = wl.QWEN3_8B.vocab, 16
    hbm, _, src = peaks()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    sampler = ClockSampler(int(os.environ.get("LOCAL_RANK", "0")))
    sampler.start()
    points = []

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        ts = []
        for _ in range(args.steps):
            flush.fill_(1)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            e1.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3)
        return statistics.median(ts)

    for batch in (1, 32):
        dl, tl, ud, ua, ur = wl.sampling_inputs(batch, B, V)
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
        dlg, tlg, uag, urg = t(dl[:, 1:]), t(tl), t(ua), t(ur)  # drafter slots 1..B-1
        tokens = torch.zeros(batch, B, dtype=torch.int32, device="cuda")
        acc = torch.zeros(batch, dtype=torch.int32, device="cuda")
        em = torch.zeros(batch, dtype=torch.int32, device="cuda")
        ws = torch.empty(capi.dflash_spec_accept_workspace(batch, B, V), dtype=torch.uint8,
                         device="cuda")
        rows = batch * (B - 1)
        uds = t(ud[:, 1:].reshape(-1))
        wsd = torch.empty(capi.dflash_sample_workspace(rows, V), dtype=torch.uint8, device="cuda")
        us_draw = timed(lambda: capi.dflash_sample_rows(rows, V, dlg, uds, tokens, wsd))
        us_acc = timed(lambda: capi.dflash_spec_accept_sampled(batch, B, V, dlg, tlg, tokens, uag, urg,
                                                               acc, em, ws))
        b_draw = rows * V * 4 + rows * 4096 * 4           # one pass + one chunk re-read per row
        b_acc = (rows + batch * B) * V * 4 + 2 * batch * V * 4  # both arrays + the final draw's rows
        points.append({"batch": batch, "op": "sample_rows", "us": us_draw, "bytes": b_draw,
                       "gbs": b_draw / us_draw / 1e3, "frac": b_draw / us_draw / 1e3 / hbm})
        points.append({"batch": batch, "op": "spec_accept_sampled", "us": us_acc, "bytes": b_acc,
                       "gbs": b_acc / us_acc / 1e3, "frac": b_acc / us_acc / 1e3 / hbm})
        del dlg, tlg, ws, wsd
    clocks = sampler.stop()
    head = next(p for p in points if p["batch"] == 32 and p["op"] == "spec_accept_sampled")
    print(json.dumps({
        "metric": "temperature-1 acceptance op: achieved HBM bandwidth (block 16, vocab 151936)",
        "value": head["gbs"], "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": head["us"] / 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded logits and uniforms)",
        "config": {"workload": "spec_sample", "batch": [1, 32], "block": B, "vocab": V,
                   "l2": "256 MB buffer written before every timed call",
                   "host": "GPU kept busy while the host prepares each timed call"},
        "roofline": {"bound": "hbm", "kernel": "samp_stats_kernel (+ accept, final draw)",
                     "achieved": head["gbs"], "peak": hbm, "unit": "GB/s", "frac": head["frac"],
                     "traffic": None, "peak_source": src},
        "points": points, "clocks": clocks}))


def run_concurrency(args) -> None:
    """Concurrency sweep of the DFlash step on the Qwen3-8B shape (block 16,
    2048-token random prompts): for b = 1, 2, 4, 8, 16, 32 sequences, the
    step time and the plain AR step time (both CUDA-graph replays, CUDA
    events on the launching stream), verified tokens/s, and the projected
    speedup S = C_AR * E[L] / C_DF with E[L] from the pages -- the quantity
    whose decay with concurrency the pages report."""
    import torch

    from block_diffusion_speculative_injection_gb300 import capi
    from block_diffusion_speculative_injection_gb300.engine import DFlashEngine, capture_step_graph

    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    w = wl.WORKLOADS["qwen3_8b_b1"]
    B, P = w.block_size, wl.prompt_lengths(w)[0]
    batches = (1, 2, 4, 8, 16, 32)
    nb = max(batches)
    prompts = [wl.prompt_tokens(w, s, P) for s in range(nb)]
    steps_total = len(batches) * (args.warmup + args.steps) * 2 + 8
    used = P + B * steps_total + 64  # cache slots a sequence reaches in this sweep
    s_ = w.shape
    page_bytes = (s_.n_layers + s_.n_draft_layers) * 2 * s_.n_kv_heads * capi.PAGE_SLOTS * s_.head_dim * 2
    if args.kv_pages:
        # serving configuration: slots admit requests of up to 32K tokens, and
        # pages come from one pool sized for what the sequences use
        max_ctx = max(32768, used)
        pages = nb * -(-used // capi.PAGE_SLOTS)
    else:
        max_ctx, pages = used, 0
    eng = DFlashEngine(w.shape, B, nb, max_ctx, max_rows=max(P, nb * B), seed=w.seed, kv_pages=pages)
    if args.kv_pages:
        for q in range(nb):  # the graph replays below map nothing
            eng.reserve(q, used)
    kv = {"mode": "paged" if args.kv_pages else "fixed regions", "max_ctx": max_ctx,
          "pages": pages if args.kv_pages else nb * -(-max_ctx // capi.PAGE_SLOTS),
          "bytes": (pages if args.kv_pages else nb * -(-max_ctx // capi.PAGE_SLOTS)) * page_bytes,
          "fixed_regions_bytes_at_max_ctx": nb * -(-max_ctx // capi.PAGE_SLOTS) * page_bytes}
    eng.prefill(prompts)
    stream = torch.cuda.current_stream()
    sampler = ClockSampler(int(os.environ.get("LOCAL_RANK", "0")))
    sampler.start()
    points = []
    for b in batches:
        sid = eng.seq_ids(b)
        for _ in range(2):
            eng.step(sid, eng.next_anchor[:b].clone())
        g = capture_step_graph(eng, sid)
        ag = torch.cuda.CUDAGraph()
        with torch.cuda.graph(ag):
            eng.ar_step(sid, eng.next_anchor[:b])

        def timed(graph):
            for _ in range(args.warmup):
                graph.replay()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record(stream)
            for _ in range(args.steps):
                graph.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) / args.steps

        step_ms = timed(g)
        ar_ms = timed(ag)
        points.append({"batch": b, "step_ms": step_ms, "ar_step_ms": ar_ms,
                       "tokens_per_s_tau1": b / (step_ms / 1e3),
                       "ar_tokens_per_s": b / (ar_ms / 1e3),
                       "projected_speedup": ar_ms * PAGES_ACCEPT_LEN / step_ms})
        del g, ag
    clocks = sampler.stop()
    eng.close()
    head = points[-1]
    print(json.dumps({
        "metric": "DFlash step over concurrency (Qwen3-8B shape, B=16, prompt 2048): projected speedup at b=32",
        "value": head["projected_speedup"], "unit": "x", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["step_ms"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded random-init weights, uniform random prompt tokens)",
        "config": {"workload": "concurrency", "batches": list(batches), "block": B, "prompt_len": P,
                   "expected_accept_len": PAGES_ACCEPT_LEN, "kv_cache": kv,
                   "l2": "no flush: every step streams ~19 GB of weights"},
        "points": points, "clocks": clocks}))


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="qwen3_8b_b1",
                    choices=["qwen3_8b_b1", "qwen3_8b_b32", "llama31_8b_ddtree_b4", "qwen3_8b_slice_b1",
                             "qwen3_8b_slice_b32", "attn_op", "spec_sample", "concurrency",
                             "tiny_f32_e2e",
                             "mini_bf16_e2e"])
    ap.add_argument("--prof-steps", type=int, default=10)
    ap.add_argument("--ar-steps", type=int, default=50)
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--attn-point", default="",
                    help="attn_op workload: only the point CTXxBATCH (e.g. 8192x8)")
    ap.add_argument("--kv-pages", action="store_true",
                    help="concurrency workload: paged KV cache (32K-slot sequences, shared page pool)")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the attention-op grid, batch-32 and DDTree measurements that the "
                         "default single-GPU run adds to its line")
    ap.add_argument("--no-graph", action="store_true",
                    help="time eager C-ABI calls instead of a CUDA-graph replay of the step")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.workload in ("attn_op", "spec_sample", "concurrency"):
        if args.impl == "reference":
            raise SystemExit("op and sweep workloads have no reference arm; their oracle checks are in tests/")
        {"attn_op": run_attn_op, "spec_sample": run_spec_sample_op,
         "concurrency": run_concurrency}[args.workload](args)
        return
    w = wl.WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()

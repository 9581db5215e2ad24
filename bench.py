#!/usr/bin/env python
"""Benchmark of the greedy draft-and-verify round on one GB300.

One step = one round: dflash_draft_block (context append of the previous
round's accepted rows, the drafter's single parallel pass over the block, the
shared head with row argmax) then dflash_verify (the target's causal pass over
the block, head + argmax, greedy acceptance and rollback).

A random-init drafter accepts almost nothing, so the acceptance length is
controlled by the proposal passed to dflash_verify: the target's own greedy
stream (found first on the same GPU, one token per round) is planted so that
each round accepts tau-1 drafts and then hits a wrong token; every kernel of
the round still runs in full.  tau = 6.5 alternates 6 and 7.

Reported (one JSON line on rank 0):
  value        effective tokens/s = batch * tau / (t_draft + t_verify) at tau = 6.5
               (device-resident inputs, CUDA events on the session stream)
  per_tau      the same at tau in {1, 4, 6.5}, with t_draft and t_verify medians
  e2e          the same metric through the C ABI with host buffers: proposals
               from pinned host memory, drafts / accepted / bonus copied back
               every round, wall-clock timed
  roofline     the dominant kernel class (CUDA-event profile of the round)
               against the measured HBM copy bandwidth
  cpu_baseline the CPU oracle on a bounded sample, extrapolated per round
  secondary    (default workload only) the concurrency-32 ragged workload at tau = 6.5:
               t_draft, t_verify, tokens/s, and its layer + head GEMMs' flops over
               their time against the sustained bf16 tensor peak

--impl reference times the CPU oracle alone on the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "draft+verify round latency (ms) and effective tokens/s at block 16, one GB300"
DEFAULT_WORKLOAD = "qwen3_8b_b1_p512"
TAU_PLANS = {"1": [1], "4": [4], "6.5": [6, 7]}


# ------------------------------------------------------------------ helpers
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu = gpu
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def job_throughput(tokens_local: float, seconds_local: float, world: int):
    """Whole-job throughput of independent replicas: the tokens all ranks produced over
    the slowest rank's time (sum and max over the process group; none when world == 1).
    Returns (tokens per second, slowest time in seconds)."""
    if world == 1:
        return tokens_local / seconds_local, seconds_local
    import torch
    dist = torch.distributed
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([seconds_local], dtype=torch.float64, device=dev)
    n = torch.tensor([tokens_local], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(n, op=dist.ReduceOp.SUM)
    return float(n.item()) / float(t.item()), float(t.item())


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs"), d.get("bf16_tflops"), d.get("bf16_tflops_sustained"), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def kernel_source_hash(files=None) -> str:
    """Hash of the kernel sources (the listed csrc files, or all of them)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "block_diffusion_speculative_ctx_gb300", "csrc")
    for f in sorted(files if files else os.listdir(csrc)):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_class: str, workload: str):
    """DRAM bytes per launch of a kernel class from a committed ncu summary,
    only if the kernels are unchanged since the counters were taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload, {}).get(kernel_class)
    if not e or e.get("source_hash") != kernel_source_hash(e.get("sources")):
        return None
    return e.get("dram_bytes_per_launch")


# --------------------------------------------------------------- our arm
def stream_for(sess, prompts, need: int, B: int):
    """The target's greedy continuation of each prompt (first token first),
    found with the library itself: rounds whose proposals are all wrong emit
    exactly the target's next token."""
    import numpy as np
    first = sess.prefill(prompts)
    b = len(prompts)
    out = [[int(t)] for t in first]
    wrong = np.zeros((b, max(B - 1, 1)), np.int32)
    while min(len(o) for o in out) < need:
        drafts = sess.draft_block()
        for s in range(b):
            wrong[s, :] = (np.int64(drafts[s, 0]) + 1) % sess.w.vocab if B > 1 else 0
        acc, bon = sess.verify(wrong)
        for s in range(b):
            out[s] += [int(x) for x in wrong[s, : acc[s]]] + [int(bon[s])]
    return [np.array(o, dtype=np.int64) for o in out]


def plan_proposals(streams, taus, rounds: int, B: int, vocab: int):
    """Proposals [rounds, b, B-1] and intended accepts [rounds, b]."""
    import numpy as np
    b = len(streams)
    props = np.zeros((rounds, b, max(B - 1, 1)), np.int32)
    accs = np.zeros((rounds, b), np.int32)
    for s in range(b):
        g = 1
        st = streams[s]
        for r in range(rounds):
            a = max(0, min(taus[r % len(taus)] - 1, B - 1))
            for j in range(B - 1):
                idx = g + j
                true = int(st[idx]) if idx < len(st) else 0
                props[r, s, j] = true if j < a else (true + 1) % vocab
            accs[r, s] = a
            g += a + 1
    return props, accs


def timed_rounds(sess, props_dev, acc_dev, bon_dev, drafts_dev, first: int, count: int):
    """Run rounds [first, first+count) with device-resident buffers; returns
    per-round (t_draft, t_verify) in ms and the total elapsed ms."""
    import torch
    stream = torch.cuda.current_stream()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(count)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(count):
        r = first + i
        ev[i][0].record(stream)
        sess.draft_block(drafts_dev)
        ev[i][1].record(stream)
        sess.verify(props_dev[r], acc_dev[r], bon_dev[r])
        ev[i][2].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    per = [(e[0].elapsed_time(e[1]), e[1].elapsed_time(e[2])) for e in ev]
    return per, start.elapsed_time(end)


def workload_of(args):
    """The named workload, with the block size overridden by --block."""
    from synth import configs
    w = configs.get(args.workload)
    return w.with_(block_size=args.block) if args.block else w


def run_ncu_target(args, local):
    """Short run for profiler launch lists: prefill, then W + K rounds with the
    drafter's own proposals (no stream discovery, no timing output)."""
    import numpy as np
    import torch

    import synth
    from synth import configs
    from block_diffusion_speculative_ctx_gb300 import Session, build as dbuild

    torch.cuda.set_device(local)
    dbuild.build()
    w = workload_of(args)
    B, b = w.block_size, w.batch
    prompts = synth.prompts(w)
    if args.ncu_prompt_len:
        # shorter prompts: the prefill's GEMMs stay at or under 256 rows (the per-tile kernel),
        # so a kernel filter on the persistent GEMM counts the round's launches only
        prompts = [p[: args.ncu_prompt_len] for p in prompts]
        w = w.with_(prompt_lens=tuple(len(p) for p in prompts))
    sess = Session(w, max_seq_len=max(w.prompt_lens) + (args.warmup + args.steps + 4) * B)
    sess.prefill(prompts)
    drafts = torch.zeros((b, max(B - 1, 1)), dtype=torch.int32, device="cuda")
    acc = torch.zeros((b,), dtype=torch.int32, device="cuda")
    bon = torch.zeros((b,), dtype=torch.int32, device="cuda")
    l0 = sess.stats().kernel_launches
    for _ in range(args.warmup + args.steps):
        sess.draft_block(drafts)
        sess.verify(drafts, acc, bon)
    torch.cuda.synchronize()
    n = sess.stats().kernel_launches - l0
    print(json.dumps({"ncu_target": w.name, "rounds": args.warmup + args.steps, "launches": n,
                      "launches_per_round": n / (args.warmup + args.steps)}))
    sess.close()


def run_sampled(args, local):
    """Rounds at temperature T > 0 (speculative rejection sampling) with the drafter's own
    sampled proposals; uniforms are drawn on the device beforehand.  Acceptance is whatever
    the random-init models give, so the line reports the measured tau beside the latency."""
    import numpy as np
    import torch

    import synth
    from block_diffusion_speculative_ctx_gb300 import Session, build as dbuild

    torch.cuda.set_device(local)
    dbuild.build()
    w = workload_of(args)
    B, b, T = w.block_size, w.batch, args.temperature
    K, W = args.steps, args.warmup
    sess = Session(w, max_seq_len=max(w.prompt_lens) + (K + W + 8) * B)
    sess.set_sampling_filter(args.top_k, args.top_p)
    sess.prefill(synth.prompts(w))
    g = torch.Generator(device="cuda")
    g.manual_seed(1234)
    ud = torch.rand((K + W + 3, b, max(B - 1, 1)), generator=g, device="cuda")
    uv = torch.rand((K + W + 3, b, B), generator=g, device="cuda")
    drafts = torch.zeros((b, max(B - 1, 1)), dtype=torch.int32, device="cuda")
    acc = torch.zeros((K + W, b), dtype=torch.int32, device="cuda")
    emit = torch.zeros((b,), dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    for r in range(W):
        sess.draft_block_sampled(T, ud[r], drafts)
        sess.verify_sampled(T, drafts, uv[r], acc[r], emit)
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    for i in range(K):
        r = W + i
        ev[i][0].record(stream)
        sess.draft_block_sampled(T, ud[r], drafts)
        ev[i][1].record(stream)
        sess.verify_sampled(T, drafts, uv[r], acc[r], emit)
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    td = float(np.median([e[0].elapsed_time(e[1]) for e in ev]))
    tv = float(np.median([e[1].elapsed_time(e[2]) for e in ev]))
    tau = float((acc[W:].float() + 1).mean().item())
    # the sampling kernels' own share of a round (their launch-level CUDA-event times)
    sess.set_profiling(True)
    for r in range(K + W, K + W + 3):
        sess.draft_block_sampled(T, ud[r], drafts)
        sess.verify_sampled(T, drafts, uv[r], acc[0], emit)
    torch.cuda.synchronize()
    sess.set_profiling(False)
    prof = sess.profile()["sampling"]
    sess.close()
    print(json.dumps({
        "metric": "sampled draft+verify round latency (ms) and effective tokens/s, one GB300", "value": b * tau / (td + tv) * 1e3,
        "unit": "tokens/s", "n_gpus": 1, "steps": K, "warmup": W, "ms_per_step": td + tv, "higher_is_better": True,
        "t_draft_ms": td, "t_verify_ms": tv, "tau_measured": tau, "dtype": w.dtype, "data": "synthetic",
        "sampling_kernels": {"ms_per_round": prof["ms"] / 3, "launches_per_round": prof["launches"] / 3,
                             "gbs": prof["bytes"] / max(prof["ms"], 1e-9) / 1e6},
        "config": {"workload": w.name, "batch": b, "block": B, "temperature": T, "top_k": args.top_k,
                   "top_p": args.top_p,
                   "proposals": "the drafter's own, drawn at T; uniforms from a seeded device generator"}}))


def run_train(args, local):
    """The drafter's training forward (dflash_train_forward): one causal target pass over
    the workload's first prompt as the clean sequence, then one drafter pass over M anchor
    blocks (evenly spaced) and the position-weighted loss; CUDA-event time per call."""
    import numpy as np
    import torch

    import synth
    from block_diffusion_speculative_ctx_gb300 import Session, build as dbuild

    torch.cuda.set_device(local)
    dbuild.build()
    w = workload_of(args)
    B, M = w.block_size, args.train_forward
    x = np.asarray(synth.prompts(w)[0], dtype=np.int64)
    anchors = np.linspace(1, len(x) - B, M).astype(np.int64)
    lam = 7.0 if B == 16 else 5.0 if B == 10 else 4.0
    sess = Session(w, max_batch=M + 1, max_seq_len=len(x) + 2 * B)
    for _ in range(args.warmup):
        loss = sess.train_forward(x, anchors, lam)
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        loss = sess.train_forward(x, anchors, lam)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    sess.close()
    print(json.dumps({
        "metric": "drafter training forward (loss value) latency and predicted tokens/s, one GB300",
        "value": M * (B - 1) / (ms * 1e-3), "unit": "tokens/s", "ms_per_step": ms, "steps": args.steps,
        "warmup": args.warmup, "higher_is_better": True, "dtype": w.dtype, "data": "synthetic", "loss": loss,
        "config": {"workload": w.name, "sequence": len(x), "anchors": M, "block": B, "lambda": lam}}))


def run_ours(args, rank, world, local):
    import numpy as np
    import torch

    import synth
    from synth import configs
    from block_diffusion_speculative_ctx_gb300 import Session, build as dbuild

    torch.cuda.set_device(local)
    dbuild.build()
    w = workload_of(args)
    B, b = w.block_size, w.batch
    K, W = args.steps, args.warmup
    rounds = W + K
    need = rounds * 7 + B + 2
    # room for the host's length bound (+B per round without a sync) so that no
    # capacity refresh lands inside a timed region
    max_seq = max(w.prompt_lens) + rounds * B + 4 * B
    t0 = time.time()
    sess = Session(w, max_seq_len=max_seq)
    if args.runtime_block:
        # rounds at a smaller block than the drafter's configured one (same weights and caches)
        sess.set_block_size(args.runtime_block)
        B = args.runtime_block
    t_init = time.time() - t0
    prompts = synth.prompts(w)
    # clocks are sampled from the start of the stream discovery (the GPU is busy from here on)
    # to the end of the last timed region: the three tau regions and the e2e region lie inside
    sampler = ClockSampler(local)
    sampler.__enter__()
    t0 = time.time()
    streams = stream_for(sess, prompts, need, B)
    t_stream = time.time() - t0

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    drafts_dev = torch.zeros((b, max(B - 1, 1)), dtype=torch.int32, device="cuda")
    per_tau = {}
    launches_per_round = None
    clocks = None
    for tau_name in ("1", "4", "6.5"):
        props, accs = plan_proposals(streams, TAU_PLANS[tau_name], rounds, B, w.vocab)
        props_dev = torch.from_numpy(props).cuda()
        acc_dev = torch.zeros((rounds, b), dtype=torch.int32, device="cuda")
        bon_dev = torch.zeros((rounds, b), dtype=torch.int32, device="cuda")
        sess.prefill(prompts)
        timed_rounds(sess, props_dev, acc_dev, bon_dev, drafts_dev, 0, W)       # warm-up rounds
        l0 = sess.stats().kernel_launches
        barrier()
        torch.cuda.synchronize()
        headline = tau_name == "6.5"
        per, total_ms = timed_rounds(sess, props_dev, acc_dev, bon_dev, drafts_dev, W, K)
        torch.cuda.synchronize()
        barrier()
        launches = sess.stats().kernel_launches - l0
        got = acc_dev.cpu().numpy()[W:]
        tau = float(np.mean(got + 1))
        job_tps, job_s = job_throughput(float((got + 1).sum()), total_ms * 1e-3, world)
        ms_step = job_s * 1e3 / K
        td = statistics.median(p[0] for p in per)
        tv = statistics.median(p[1] for p in per)
        per_tau[tau_name] = {
            "tau_planned": float(np.mean(accs[W:] + 1)), "tau": tau, "ms_per_step": ms_step,
            "t_draft_ms": td, "t_verify_ms": tv,
            "tokens_per_s": job_tps,
        }
        if headline:
            launches_per_round = launches / K
            head_launches = launches

    # ---- end to end through the C ABI with host buffers
    props, accs = plan_proposals(streams, TAU_PLANS["6.5"], rounds, B, w.vocab)
    pinned = torch.from_numpy(props).pin_memory()
    host_props = pinned.numpy()
    acc_h = torch.zeros((b,), dtype=torch.int32).pin_memory().numpy()
    bon_h = torch.zeros((b,), dtype=torch.int32).pin_memory().numpy()
    drafts_h = torch.zeros((b, max(B - 1, 1)), dtype=torch.int32).pin_memory().numpy()
    sess.prefill(prompts)
    emitted = 0
    for r in range(W):
        sess.draft_block(drafts_h)
        sess.verify(host_props[r], acc_h, bon_h)
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for r in range(W, W + K):
        sess.draft_block(drafts_h)
        sess.verify(host_props[r], acc_h, bon_h)
        emitted += int(acc_h.sum()) + b
    e2e_s_local = time.perf_counter() - t0
    sampler.__exit__()
    clocks = sampler.summary()
    clocks["window"] = "stream discovery through the last timed region (tau 1, 4, 6.5 and e2e)"
    e2e_tps, e2e_s = job_throughput(float(emitted), e2e_s_local, world)
    e2e = {"value": e2e_tps, "unit": "tokens/s",
           "h2d_bytes_per_step": int(b * max(B - 1, 0) * 4),
           "d2h_bytes_per_step": int(b * max(B - 1, 0) * 4 + 2 * b * 4),
           "ms_per_step": 1e3 * e2e_s / K}

    # ---- kernel-class profile of the headline round (separate pass, events between launches)
    props_dev = torch.from_numpy(props).cuda()
    acc_dev = torch.zeros((rounds, b), dtype=torch.int32, device="cuda")
    bon_dev = torch.zeros((rounds, b), dtype=torch.int32, device="cuda")
    sess.prefill(prompts)
    timed_rounds(sess, props_dev, acc_dev, bon_dev, drafts_dev, 0, W)
    sess.profile_reset()
    sess.set_profiling(True)
    timed_rounds(sess, props_dev, acc_dev, bon_dev, drafts_dev, W, K)
    sess.set_profiling(False)
    prof = sess.profile()
    # one warm prefill of the same prompts (time to first token, CUDA events inside the library)
    p0 = sess.stats().prefill_ms
    sess.prefill(prompts)
    prefill_ms = sess.stats().prefill_ms - p0
    sess.close()

    hbm, tf, tf_sus, peak_src = measured_peaks()
    total_ms = sum(v["ms"] for v in prof.values()) or 1.0
    dom = max(prof, key=lambda k: prof[k]["ms"])
    dv = prof[dom]
    achieved = dv["bytes"] / (dv["ms"] * 1e-3) / 1e9 if dv["ms"] > 0 else 0.0
    traffic = ncu_traffic(dom, args.workload)
    roofline = {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm, "traffic": traffic, "peak_source": peak_src,
                "bytes_per_launch": dv["bytes"] / max(dv["launches"], 1),
                "ms_per_launch": dv["ms"] / max(dv["launches"], 1), "share": dv["ms"] / total_ms}
    kernels = {k: {"ms_per_round": v["ms"] / K, "launches_per_round": v["launches"] / K,
                   "GBps": (v["bytes"] / (v["ms"] * 1e-3) / 1e9) if v["ms"] > 0 else 0.0,
                   "share": v["ms"] / total_ms} for k, v in prof.items() if v["launches"]}
    # whole-round HBM roofline: algorithmic bytes of a round over its time
    round_bytes = sum(v["bytes"] for v in prof.values()) / K

    h = per_tau["6.5"]
    line = {
        "metric": METRIC, "value": h["tokens_per_s"], "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": h["ms_per_step"], "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic (seeded random-init weights N(0,0.02), uniform prompt ids)",
        "config": {"workload": w.name, "batch": b, "prompt_len": list(w.prompt_lens)[:4], "block": B,
                   "configured_block": w.block_size, "tau": 6.5, "draft_layers": w.draft_layers, "target_layers": w.target_layers,
                   "l2": "inputs larger than L2: every round streams all weights (~19.7 GB)",
                   "parallelism": f"replicas x{world}"},
        "t_draft_ms": h["t_draft_ms"], "t_verify_ms": h["t_verify_ms"], "tau": h["tau"],
        "per_tau": per_tau, "e2e": e2e, "roofline": roofline,
        "round_hbm": {"bytes_per_round": round_bytes, "GBps": round_bytes / (h["ms_per_step"] * 1e-3) / 1e9,
                      "frac": round_bytes / (h["ms_per_step"] * 1e-3) / 1e9 / hbm},
        "kernels": kernels, "gpu_launches": int(head_launches), "launches_per_round": launches_per_round,
        "clocks": clocks, "setup_s": {"init": t_init, "stream": t_stream},
        "prefill": {"ms": prefill_ms, "tokens": int(sum(w.prompt_lens)),
                    "tokens_per_s": sum(w.prompt_lens) / (prefill_ms * 1e-3) if prefill_ms > 0 else None},
    }
    if world == 1 and not args.no_secondary and args.workload == DEFAULT_WORKLOAD and not args.block \
            and not args.runtime_block:
        line["secondary"] = run_secondary(SECONDARY_WORKLOAD, min(K, 20), W)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, budget_s=args.cpu_budget)
    if rank == 0:
        print(json.dumps(line), flush=True)


SECONDARY_WORKLOAD = "qwen3_8b_c32_ragged"
GEMM_CLASSES = ("gemm_qkv", "gemm_o", "gemm_gate_up", "gemm_down", "gemm_head", "gemm_fc", "gemm_ctx_kv")


def run_secondary(name: str, K: int, W: int):
    """The concurrency-32 workload at tau = 6.5, measured the same way as the headline
    (planted proposals, K timed rounds after W warm-up rounds, CUDA events on the session
    stream), plus a kernel-class profile pass whose GEMM flops over GEMM time are set
    against the sustained bf16 peak (these GEMMs are compute-bound at 512 rows)."""
    import numpy as np
    import torch

    import synth
    from synth import configs
    from block_diffusion_speculative_ctx_gb300 import Session

    w = configs.get(name)
    B, b = w.block_size, w.batch
    rounds = W + K
    need = rounds * 7 + B + 2
    t0 = time.time()
    sess = Session(w, max_seq_len=max(w.prompt_lens) + rounds * B + 4 * B)
    prompts = synth.prompts(w)
    streams = stream_for(sess, prompts, need, B)
    props, accs = plan_proposals(streams, TAU_PLANS["6.5"], rounds, B, w.vocab)
    props_dev = torch.from_numpy(props).cuda()
    acc_dev = torch.zeros((rounds, b), dtype=torch.int32, device="cuda")
    bon_dev = torch.zeros((rounds, b), dtype=torch.int32, device="cuda")
    drafts_dev = torch.zeros((b, max(B - 1, 1)), dtype=torch.int32, device="cuda")
    sess.prefill(prompts)
    timed_rounds(sess, props_dev, acc_dev, bon_dev, drafts_dev, 0, W)
    torch.cuda.synchronize()
    per, total_ms = timed_rounds(sess, props_dev, acc_dev, bon_dev, drafts_dev, W, K)
    got = acc_dev.cpu().numpy()[W:]
    tokens = float((got + 1).sum())
    td = statistics.median(p[0] for p in per)
    tv = statistics.median(p[1] for p in per)
    # kernel-class profile of the same rounds (events between launches: not the headline timing)
    sess.prefill(prompts)
    timed_rounds(sess, props_dev, acc_dev, bon_dev, drafts_dev, 0, W)
    sess.profile_reset()
    sess.set_profiling(True)
    timed_rounds(sess, props_dev, acc_dev, bon_dev, drafts_dev, W, K)
    sess.set_profiling(False)
    prof = sess.profile()
    p0 = sess.stats().prefill_ms
    sess.prefill(prompts)
    prefill_ms = sess.stats().prefill_ms - p0
    sess.close()
    _, _, tf_sus, peak_src = measured_peaks()
    g_ms = sum(prof[k]["ms"] for k in GEMM_CLASSES if k in prof)
    g_fl = sum(prof[k]["flops"] for k in GEMM_CLASSES if k in prof)
    achieved = g_fl / (g_ms * 1e-3) / 1e12 if g_ms > 0 else 0.0
    per_class = {k: {"ms_per_round": prof[k]["ms"] / K,
                     "TFLOPs": prof[k]["flops"] / (prof[k]["ms"] * 1e-3) / 1e12 if prof[k]["ms"] > 0 else 0.0}
                 for k in GEMM_CLASSES if k in prof and prof[k]["launches"]}
    return {
        "workload": w.name, "batch": b, "block": B, "tau": float(np.mean(got + 1)), "steps": K, "warmup": W,
        "t_draft_ms": td, "t_verify_ms": tv, "ms_per_step": total_ms / K,
        "tokens_per_s": tokens / (total_ms * 1e-3),
        "roofline": {"kernel": "layer and head GEMMs of the round (all classes)", "bound": "tensor",
                     "achieved": achieved, "peak": tf_sus, "unit": "TFLOP/s", "frac": achieved / tf_sus,
                     "peak_source": peak_src + " (sustained bf16)", "gemm_ms_per_round": g_ms / K,
                     "gemm_tflop_per_round": g_fl / K / 1e12, "traffic": None},
        "gemms": per_class,
        "prefill": {"ms": prefill_ms, "tokens": int(sum(w.prompt_lens))},
        "setup_s": time.time() - t0,
    }


# --------------------------------------------------------- CPU oracle arm
def cpu_sample_round_s(w, ctx_len: int, state=None):
    """Seconds for one round of the oracle on the workload, from a bounded
    sample: one target layer and one draft layer at full width (plus the
    shared head), timed, then scaled to the workload's layer counts."""
    import numpy as np
    from oracle import model as om

    if state is None:
        w1 = w.with_(target_layers=1, draft_layers=1, ctx_layer_ids=(0,))
        m = om.Model(w1)
        rng = np.random.default_rng(0)
        B = w.block_size
        # caches with ctx_len committed rows (values do not matter for timing)
        tc = m.new_target_cache()
        dc = m.new_draft_cache()
        kv = lambda: rng.standard_normal((ctx_len, w.n_kv_heads, w.head_dim)) * 0.1
        tc.append(0, kv(), kv())
        dc.append(0, kv(), kv())
        for name in ("embed", "head", "final_norm", "draft_norm", "fc", "fc_norm", "t0.wq", "t0.wk", "t0.wv",
                     "t0.wo", "t0.w_gate", "t0.w_up", "t0.w_down", "d0.wq", "d0.wk", "d0.wv", "d0.wo",
                     "d0.w_gate", "d0.w_up", "d0.w_down"):
            m.w(name)                                   # materialise weights outside the timed region
        state = (m, tc, dc, B, [0.0, 0.0])
    m, tc, dc, B, state_times = state
    block = np.arange(B) % w.vocab
    t = time.perf_counter()
    m.draft_forward(int(block[0]), dc)                    # 1 draft layer + head (B rows)
    t_draft1 = time.perf_counter() - t
    t = time.perf_counter()
    tcc = tc.copy()
    lg, _ = m.target_forward(block, tcc)                  # 1 target layer + head (B rows)
    t_verify1 = time.perf_counter() - t
    t = time.perf_counter()
    m.logits(np.zeros((B, w.d_model)), "final_norm")      # the head alone
    t_head = time.perf_counter() - t
    t_draft = w.draft_layers * max(t_draft1 - t_head, 0.0) + t_head
    t_verify = w.target_layers * max(t_verify1 - t_head, 0.0) + t_head
    state_times[0], state_times[1] = t_draft, t_verify
    return t_draft + t_verify, state


def oracle_tokens_per_s(tau: float, s_per_sequence_round: float) -> float:
    """Throughput of the CPU oracle, which handles the sequences of a batch one after
    another: b sequences take b rounds of one sequence and emit b * tau tokens."""
    return tau / s_per_sequence_round


def cpu_baseline(w, budget_s: float = 20.0):
    import numpy as np
    try:
        cores = len(os.sched_getaffinity(0))
    except Exception:
        cores = os.cpu_count() or 1
    t0 = time.time()
    ctx = max(w.prompt_lens)
    s, st = cpu_sample_round_s(w, ctx)
    samples = [(s, st[4][0], st[4][1])]
    while time.time() - t0 < budget_s and len(samples) < 5:
        s, st = cpu_sample_round_s(w, ctx, st)
        samples.append((s, st[4][0], st[4][1]))
    per_round, td, tv = sorted(samples)[(len(samples) - 1) // 2]   # the median sample (lower middle)
    tau = 6.5
    # the oracle runs the batch's sequences one after another: a round of b sequences takes
    # b * per_round and emits b * tau tokens
    return {"value": oracle_tokens_per_s(tau, per_round), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "s_per_round": per_round, "t_draft_ms": 1e3 * td, "t_verify_ms": 1e3 * tv,
            "sample": (f"fp64 numpy oracle: 1 target layer + 1 draft layer + shared head over one "
                       f"block of {w.block_size} rows at context {ctx}, timed {len(samples)}x, scaled to "
                       f"{w.target_layers}+{w.draft_layers} layers; tau=6.5; the oracle handles the batch one "
                       f"sequence at a time")}


def run_reference(args, rank, world):
    if rank != 0:
        return
    from synth import configs
    w = workload_of(args)
    ctx = max(w.prompt_lens)
    try:
        cores = len(os.sched_getaffinity(0))
    except Exception:
        cores = os.cpu_count() or 1
    _, st = cpu_sample_round_s(w, ctx)
    n_warm = 0
    for _ in range(args.warmup):
        cpu_sample_round_s(w, ctx, st)
        n_warm += 1
        if time.time() - args._t0 > 60:
            break
    per = []
    t0 = time.time()
    for i in range(args.steps):
        t1 = time.perf_counter()
        s, _ = cpu_sample_round_s(w, ctx, st)
        per.append((s, st[4][0], st[4][1], time.perf_counter() - t1))
        if time.time() - t0 > 150:                       # keep the whole run within a few minutes
            break
    per_round, td, tv, wall = sorted(per)[(len(per) - 1) // 2]   # the median sample (lower middle)
    tau = 6.5
    value = oracle_tokens_per_s(tau, per_round)
    # a step is one timed sample (one target layer + one draft layer + the head, at full width);
    # ms_per_step is its measured wall time, and the full round is extrapolated from it
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": len(per), "warmup": n_warm, "ms_per_step": wall * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "block": w.block_size, "tau": tau},
        "step": "one sample: 1 target layer + 1 draft layer + the shared head over one block, fp64 oracle",
        "extrapolated_round_ms": per_round * 1e3, "layers_sampled": {"target": 1, "draft": 1},
        "layers_extrapolated": {"target": w.target_layers, "draft": w.draft_layers},
        "t_draft_ms": 1e3 * td, "t_verify_ms": 1e3 * tv,
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": "fp64 numpy oracle, 1 target + 1 draft layer + head per step, scaled to the "
                                   "workload's layer counts, one sequence of the batch at a time"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--block", type=int, default=0, help="block size B (default: the workload's, 16)")
    ap.add_argument("--runtime-block", type=int, default=0, metavar="B",
                    help="run the rounds at block B below the configured one (dflash_set_block_size)")
    ap.add_argument("--temperature", type=float, default=0.0,
                    help="T > 0: time sampled rounds (speculative rejection sampling) instead of greedy ones")
    ap.add_argument("--top-k", type=int, default=0, help="with --temperature: top-k filter of both laws (0: off)")
    ap.add_argument("--top-p", type=float, default=1.0, help="with --temperature: top-p filter of both laws (1: off)")
    ap.add_argument("--train-forward", type=int, default=0, metavar="M",
                    help="time the drafter's training forward with M anchor blocks instead of rounds")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the concurrency-32 line that the default run adds (secondary)")
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    ap.add_argument("--ncu-target", action="store_true",
                    help="short fixed run for profiler launch lists (prints no benchmark line)")
    ap.add_argument("--ncu-prompt-len", type=int, default=0, metavar="N",
                    help="with --ncu-target: cut every prompt to its first N tokens")
    args = ap.parse_args()
    args._t0 = time.time()
    if args.warmup < 3:
        args.warmup = 3
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.ncu_target:
        run_ncu_target(args, local)
        return
    if args.temperature > 0:
        run_sampled(args, local)
        return
    if args.train_forward > 0:
        run_train(args, local)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
    try:
        run_ours(args, rank, world, local)
    finally:
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()

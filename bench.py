#!/usr/bin/env python3
"""Benchmark of one pass of the shared-prefix classifier path on GB300.

A step is one whole pass over one batch of synthetic input: host planning
(token trie, staged rounds, KV pages, launch lists) and descriptor upload,
the prefix and branch attention of every staged round (cascade attention
that also writes the shared segments into the paged pool, split merges), the
fused LM-head readout and the label softmax.  The default workload is the yes/no configuration: Hq 32 / Hkv 4 /
d 128, a 2000-token shared prefix with 5 branches of 48 tokens, H 2048,
V 151936, two labels per branch.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                       [--config NAME]
Prints one JSON line (rank 0).
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
sys.path.insert(0, ROOT)

METRIC = "branch-prefill tokens/s & label decisions/s at 1 GB300; % of roofline"
DEFAULT_CONFIG = "batch64"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="libsp", choices=["libsp", "reference"])
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--schedule", default="tree", choices=["tree", "all", "rounds"],
                    help="attention calls of a step: one tree call for the whole trie, one "
                         "prefix and one branch call covering every staged round, or one "
                         "pair of calls per round (same work and results)")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the oracle timing (short profiling runs)")
    ap.add_argument("--only", default="all", choices=["all", "attention", "readout"],
                    help="profiling runs: time one phase of the step alone (only its inputs "
                         "on the device) and print its timing line instead of the bench line")
    return ap.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def job_time(local_ms, ws, device=None):
    """Whole-job time of a replica run: the slowest rank's time (max over
    ranks; the value every rank returns).  `device` holds the reduction
    tensor (a CUDA device with NCCL, the CPU with gloo)."""
    if ws <= 1:
        return float(local_ms)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(local_ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(units_per_rank, ws, ms_per_step):
    """Aggregate throughput: the units all ranks processed per second."""
    return units_per_rank * ws / (ms_per_step / 1e3)


# --------------------------------------------------------------------------
# clocks sampled during the timed region
class ClockSampler:
    """nvidia-smi samples every 100 ms on a reader thread, each stamped with
    the host time it arrived; the summary keeps the samples between mark()
    (the start of the timed region, after the warm-up) and stop()."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t_mark = 0.0

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def mark(self):
        self.t_mark = time.time()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        t_stop = time.time()
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, pw, mx, reasons = [], [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        window = [ln for t, ln in self.lines if self.t_mark <= t <= t_stop + 0.15]
        if not window:  # a timed region shorter than one sample: the nearest sample
            after = [ln for t, ln in self.lines if t >= self.t_mark]
            window = after[:1] or [ln for _, ln in self.lines[-1:]]
        for ln in window:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            try:
                pw.append(float(parts[3]))
            except ValueError:
                pass
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_median": statistics.median(pw) if pw else None}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def kernel_traffic(kernel_file: str, config: str):
    """DRAM bytes per launch from the committed ncu summary
    (profiles/traffic_<kernel file>_<config>.txt), if the kernel source is
    unchanged since it was captured; else None."""
    src = os.path.join(ROOT, "prefill_only_shared_gb300", "csrc", kernel_file)
    summ = os.path.join(ROOT, "profiles", f"traffic_{os.path.splitext(kernel_file)[0]}_{config}.txt")
    if not (os.path.exists(src) and os.path.exists(summ)):
        return None
    fields = {}
    for line in open(summ):
        if ":" in line and not line.startswith(("#", "|", " ")):
            k, v = line.split(":", 1)
            fields[k.strip()] = v.strip()
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
    if fields.get("source_sha256") != sha or "dram_bytes_per_launch" not in fields:
        return None
    return int(fields["dram_bytes_per_launch"])


# --------------------------------------------------------------------------
def attention_flops(plan_segments, wl):
    """Algorithmic attention FLOPs of one pass: 4 * d * Hq per (query, visible
    key) pair (2 for q.k, 2 for p.v), over every computed row."""
    import numpy as np
    sh = wl.shape
    seg = plan_segments
    n = len(seg["len"])
    ctx_before = np.zeros(n, dtype=np.int64)
    for s in range(n):
        p = seg["parent"][s]
        ctx_before[s] = 0 if p < 0 else ctx_before[p] + seg["len"][p]
    prefix, branch = 0, 0
    for s in range(n):
        L = int(seg["len"][s])
        pairs = L * int(ctx_before[s]) + L * (L + 1) // 2
        if seg["shared"][s]:
            prefix += pairs
        else:
            branch += pairs
    f = 4 * sh.head_dim * sh.n_q_heads
    return prefix * f, branch * f


def run_libsp(args, ws, rank, local):
    import numpy as np
    import torch
    from prefill_only_shared_gb300 import build as B
    B.ensure_built()
    from prefill_only_shared_gb300 import sp
    from prefill_only_shared_gb300.pipeline import SharedPrefixClassifier
    from prefill_only_shared_gb300.workloads import make_workload

    torch.cuda.set_device(local)
    dev = torch.device(f"cuda:{local}")
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    wl = make_workload(args.config, seed=0)
    sh = wl.shape
    clf = SharedPrefixClassifier(sh.n_q_heads, sh.n_kv_heads, sh.head_dim, sh.hidden, sh.vocab,
                                 device=dev)
    if args.only != "all":
        return run_phase(args, wl, clf, dev) if rank == 0 else None
    q, k, v = wl.q.to(dev), wl.k.to(dev), wl.v.to(dev)
    h, W = wl.h.to(dev), wl.W.to(dev)
    off = torch.from_numpy(wl.label_off).to(dev)
    ids = torch.from_numpy(wl.label_ids).to(dev)
    n_labels = int(wl.label_ids.shape[0])
    N = wl.n_branches
    stream = torch.cuda.current_stream(dev)

    # events around the readout call of every timed step (dominant kernel)
    def step(ev=None, schedule=args.schedule):
        plan = clf.plan(wl.req_of_branch, wl.tok_offsets, wl.tokens)
        if ev is not None:
            ev[0].record(stream)
        clf.attention(plan, q, k, v, stream, schedule)
        if ev is not None:
            ev[1].record(stream)
        logprobs, lse = clf.logprobs(h, W, off, ids, n_labels, stream)
        if ev is not None:
            ev[2].record(stream)
        clf.softmax(logprobs, off, stream)
        if ev is not None:
            ev[3].record(stream)
        return plan

    plan = step()
    torch.cuda.synchronize()
    sp.sp_check_device_error()
    stats = plan.stats()
    segs = plan.segments()
    attn_launches = clf.last_attention_launches
    launches_per_step = clf.last_attention_launches + clf.last_logprob_launches + \
        clf.last_softmax_launches
    branch_tokens = int(sum(segs["len"][i] for i in range(len(segs["len"])) if not segs["shared"][i]))
    branch_tokens += int(plan.branches()["recompute"].sum())
    f_prefix, f_branch = attention_flops(segs, wl)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # phase events inside the timed region
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_stop = torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler.mark()
    t_start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t_stop.record(stream)
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    total_ms = job_time(t_start.elapsed_time(t_stop), ws, dev)
    attn_ms = [e[0].elapsed_time(e[1]) for e in evs]
    lm_ms = [e[1].elapsed_time(e[2]) for e in evs]
    sm_ms = [e[2].elapsed_time(e[3]) for e in evs]
    sp.sp_check_device_error()

    # the other attention schedules, same steps, for comparison
    others = {}
    for other in ("tree", "all", "rounds"):
        if other == args.schedule:
            continue
        for _ in range(args.warmup):
            step(schedule=other)
        torch.cuda.synchronize()
        o0 = torch.cuda.Event(enable_timing=True)
        o1 = torch.cuda.Event(enable_timing=True)
        o0.record(stream)
        for i in range(args.steps):
            step(schedule=other)
        o1.record(stream)
        torch.cuda.synchronize()
        others[other] = job_time(o0.elapsed_time(o1), ws, dev) / args.steps
        sp.sp_check_device_error()

    # ---- prefix cache: the same request again, its shared segments cached ------
    # (a hot request: only the remainders -- each branch's own suffix -- are
    # computed, the state's K/V are read from the pool the cold call wrote)
    cclf = SharedPrefixClassifier(sh.n_q_heads, sh.n_kv_heads, sh.head_dim, sh.hidden, sh.vocab,
                                  device=dev, prefix_cache_pages=int(stats["pages_used"]) + 64)
    cold = cclf.plan(wl.req_of_branch, wl.tok_offsets, wl.tokens)
    cclf.attention(cold, q, k, v, stream, args.schedule)
    del cold
    warm_plan = cclf.plan(wl.req_of_branch, wl.tok_offsets, wl.tokens)
    warm_stats = warm_plan.stats()
    del warm_plan
    Tw = warm_stats["node_tokens"]
    qw, kw, vw = q[:Tw], k[:Tw], v[:Tw]  # timing inputs: the rows' values do not matter

    def warm_step(ev=None):
        p = cclf.plan(wl.req_of_branch, wl.tok_offsets, wl.tokens)
        if ev is not None:
            ev[0].record(stream)
        cclf.attention(p, qw, kw, vw, stream, args.schedule)
        if ev is not None:
            ev[1].record(stream)
        lp, _ = cclf.logprobs(h, W, off, ids, n_labels, stream)
        cclf.softmax(lp, off, stream)
        return p

    for _ in range(args.warmup):
        warm_step()
    torch.cuda.synchronize()
    wev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    w0 = torch.cuda.Event(enable_timing=True)
    w1 = torch.cuda.Event(enable_timing=True)
    w0.record(stream)
    for i in range(args.steps):
        warm_step(wev[i])
    w1.record(stream)
    torch.cuda.synchronize()
    sp.sp_check_device_error()
    warm_ms = job_time(w0.elapsed_time(w1), ws, dev) / args.steps
    warm_attn = statistics.mean(e[0].elapsed_time(e[1]) for e in wev)
    warm_launches = cclf.last_launches
    del cclf

    # ---- multi-token options with a calibration prior ---------------------------
    # (the readout at every option token -- one label per row -- then the option
    # scores and their calibrated softmax per question; the LM head is the one
    # above, model state)
    from prefill_only_shared_gb300.workloads import make_options
    owl = make_options(seed=0, hidden=sh.hidden, vocab=sh.vocab, with_W=False)
    o_h = owl.h_rows.to(dev)
    o_off = torch.from_numpy(owl.opt_off).to(dev)
    o_tok = torch.from_numpy(owl.tokens).to(dev)
    o_q = torch.from_numpy(owl.q_off).to(dev)
    o_prior = torch.from_numpy(owl.prior).to(dev)
    for _ in range(args.warmup):
        clf.options(o_h, W, o_off, o_tok, o_q, o_prior, stream)
    torch.cuda.synchronize()
    oev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    for i in range(args.steps):
        oev[i][0].record(stream)
        clf.options(o_h, W, o_off, o_tok, o_q, o_prior, stream)
        oev[i][1].record(stream)
    torch.cuda.synchronize()
    sp.sp_check_device_error()
    opt_ms = job_time(statistics.mean(e[0].elapsed_time(e[1]) for e in oev), ws, dev)
    opt_bytes = sh.vocab * sh.hidden * 2 + owl.n_rows * sh.hidden * 2 + owl.n_rows * 8
    opt_launches = clf.last_option_launches

    # ---- continuous batching across requests ----------------------------------
    # (a stream of independent yes/no-shaped requests, each with its own
    # 2000-token prefix and 5 x 48 branches, queued before the timed region;
    # batches of up to 16384 node tokens against one request per batch, the
    # same stream and LM head)
    from prefill_only_shared_gb300.pipeline import ContinuousBatcher
    from prefill_only_shared_gb300.workloads import make_request_stream
    n_stream = 32
    stream_reqs = make_request_stream(n_stream, seed=1, shape=sh)
    staged = [(r.tok_offsets, r.tokens, r.q.to(dev), r.k.to(dev), r.v.to(dev), r.h.to(dev),
               r.label_off, r.label_ids) for r in stream_reqs]
    rows_total = sum(int(r.q.shape[0]) for r in stream_reqs)
    br_total = sum(len(r.tok_offsets) - 1 for r in stream_reqs)
    lab_total = sum(int(r.label_off[-1]) for r in stream_reqs)
    cb_ms, cb_batches = {}, {}
    for mode, (budget, cap) in (("one_request_per_batch", (1, 1)), ("batched", (16384, 64))):
        cb = ContinuousBatcher(clf, W, budget, cap, capacity_rows=rows_total,
                               capacity_branches=br_total, capacity_labels=lab_total,
                               schedule=args.schedule)
        times = []
        for rep in range(args.warmup + 3):
            cb.reset()
            for x in staged:
                cb.submit(*x, stream=stream)
            torch.cuda.synchronize()
            c0 = torch.cuda.Event(enable_timing=True)
            c1 = torch.cuda.Event(enable_timing=True)
            c0.record(stream)
            n_b = cb.run(stream)
            c1.record(stream)
            torch.cuda.synchronize()
            if rep >= args.warmup:
                times.append(c0.elapsed_time(c1))
        sp.sp_check_device_error()
        cb_ms[mode] = job_time(statistics.mean(times), ws, dev)
        cb_batches[mode] = n_b
        del cb
    del staged
    stream_branch_tokens = n_stream * 5 * 48

    # ---- end-to-end through the public call, host buffers --------------------
    pin = lambda x: x.pin_memory()
    hq, hk, hv, hh = pin(wl.q), pin(wl.k), pin(wl.v), pin(wl.h)
    hoff = pin(torch.from_numpy(wl.label_off))
    hids = pin(torch.from_numpy(wl.label_ids))
    out_probs = torch.empty(n_labels, dtype=torch.float32).pin_memory()
    out_am = torch.empty(N, dtype=torch.int32).pin_memory()
    h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv, hh, hoff, hids))
    h2d += wl.tokens.nbytes + wl.tok_offsets.nbytes + wl.req_of_branch.nbytes  # read by the planner
    d2h = out_probs.numel() * 4 + out_am.numel() * 4

    def e2e_step():
        # inputs copied in from pinned host memory every step (on a side stream,
        # overlapping the previous step's kernels), results copied out
        clf.run_from_host(wl.req_of_branch, wl.tok_offsets, wl.tokens, hq, hk, hv, hh, W, hoff,
                          hids, out_probs, out_am, stream, args.schedule)

    e2e_ms = float("nan")
    if args.e2e_steps > 0:
        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        if ws > 1:
            torch.distributed.barrier()
        e0.record(stream)
        clf.copy_stream.wait_event(e0)  # the timed steps' copies start after e0
        for _ in range(args.e2e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = e0.elapsed_time(e1) / args.e2e_steps
    e2e_ms = job_time(e2e_ms, ws, dev)
    sp.sp_check_device_error()

    ms = total_ms / args.steps
    value = job_value(branch_tokens, ws, ms)
    peaks, peak_kind = load_peaks()
    lm_avg = statistics.mean(lm_ms)
    attn_avg = statistics.mean(attn_ms)
    lm_bytes = sh.vocab * sh.hidden * 2 + N * sh.hidden * 2 + n_labels * 8 + N * 4
    lm_flops = 2.0 * N * sh.hidden * sh.vocab
    # the readout's bound: HBM (streaming W) unless its products take longer
    # at the tensor peak than W takes at the copy bandwidth (large N)
    lm_tensor = lm_flops / (peaks["bf16_tflops_sustained"] * 1e12) > lm_bytes / (peaks["hbm_gbs"] * 1e9)
    if lm_tensor:
        achieved = lm_flops / (lm_avg / 1e3) / 1e12
        lm_peak, lm_unit, lm_peak_key = peaks["bf16_tflops_sustained"], "TFLOP/s", "bf16_tflops_sustained"
    else:
        achieved = lm_bytes / (lm_avg / 1e3) / 1e9
        lm_peak, lm_unit, lm_peak_key = peaks["hbm_gbs"], "GB/s", "hbm_gbs"
    attn_flops = f_prefix + f_branch
    attn_peak_key = "bf16_tflops_sustained" if "bf16_tflops_sustained" in peaks else "bf16_tflops"
    attn_achieved = attn_flops / (attn_avg / 1e3) / 1e12
    readout_roofline = {
        "kernel": "lmhead_kernel (the whole sp_label_logprobs call: barrier-counter memset + one cooperative launch)",
        "bound": "tensor" if lm_tensor else "hbm",
        "achieved": round(achieved, 1),
        "peak": lm_peak,
        "unit": lm_unit,
        "frac": round(achieved / lm_peak, 4),
        "traffic": kernel_traffic("lmhead.cu", args.config),
        "peak_source": f"{peak_kind} {lm_peak_key}",
        "algorithmic_bytes_per_launch": lm_bytes,
        "algorithmic_flops_per_launch": lm_flops,
    }
    attention_roofline = {
        "kernel": f"attn_tc_kernel (the whole attention of a step: {attn_launches} "
                  f"launch(es) of the {args.schedule} schedule)",
        "bound": "tensor",
        "achieved": round(attn_achieved, 2),
        "peak": peaks[attn_peak_key],
        "unit": "TFLOP/s",
        "frac": round(attn_achieved / peaks[attn_peak_key], 4),
        "traffic": kernel_traffic("attn.cu", args.config),
        "peak_source": f"{peak_kind} {attn_peak_key}",
        "algorithmic_flops_per_launch": attn_flops,
        "note": "the attention calls of a step incl. KV append and merges",
    }
    # the headline roofline is the dominant kernel's: the phase with the
    # larger share of the step
    dominant = "attention" if attn_avg >= lm_avg else "readout"
    result = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "branch tokens/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": DATA,
        "config": workload_config(args.config, sh, N, stats["logical_tokens"],
                                  stats["computed_tokens"], stats["n_rounds"], branch_tokens, ws,
                                  args.schedule),
        "other_schedules": {o: {"ms_per_step": round(t, 5),
                                "value": round(job_value(branch_tokens, ws, t), 1)}
                            for o, t in others.items()},
        "prefix_cache": {
            "workload": "the same request again with its shared segments kept in the prefix "
                        "cache (hot request): only each branch's own suffix is computed",
            "ms_per_step": round(warm_ms, 5),
            "value": round(job_value(branch_tokens, ws, warm_ms), 1),
            "unit": "branch tokens/s",
            "attention_ms": round(warm_attn, 5),
            "computed_tokens": int(warm_stats["computed_tokens"]),
            "cache_hit_tokens": int(warm_stats["cache_hit_tokens"]),
            "gpu_launches_per_step": int(warm_launches),
        },
        "options": {
            "workload": f"{owl.n_questions} questions of 2..8 options of 1..4 tokens "
                        f"({owl.n_opts} options, {owl.n_rows} option tokens), each token read out "
                        f"at the position before it, calibrated by a per-option prior; "
                        f"H {sh.hidden}, V {sh.vocab}",
            "ms_per_call": round(opt_ms, 5),
            "decisions_per_s": round(owl.n_questions * ws / (opt_ms / 1e3), 1),
            "roofline": {"bound": "hbm",
                         "achieved": round(opt_bytes / (opt_ms / 1e3) / 1e9, 1),
                         "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(opt_bytes / (opt_ms / 1e3) / 1e9 / peaks["hbm_gbs"], 4),
                         "algorithmic_bytes_per_call": opt_bytes,
                         "note": "sp_label_logprobs over the option-token rows plus "
                                 "sp_option_softmax, timed together"},
            "gpu_launches_per_call": int(opt_launches),
        },
        "continuous_batching": {
            "workload": f"{n_stream} independent yes/no-shaped requests (own 2000-token prefix, "
                        f"5 x 48 branches, 2 labels each), queued; batches of up to 16384 node "
                        f"tokens against one request per batch",
            "batched": {"batches": cb_batches["batched"],
                        "ms": round(cb_ms["batched"], 4),
                        "requests_per_s": round(n_stream * ws / (cb_ms["batched"] / 1e3), 1),
                        "decisions_per_s": round(br_total * ws / (cb_ms["batched"] / 1e3), 1),
                        "branch_tokens_per_s": round(stream_branch_tokens * ws /
                                                     (cb_ms["batched"] / 1e3), 1)},
            "one_request_per_batch": {
                "batches": cb_batches["one_request_per_batch"],
                "ms": round(cb_ms["one_request_per_batch"], 4),
                "requests_per_s": round(n_stream * ws / (cb_ms["one_request_per_batch"] / 1e3), 1),
                "decisions_per_s": round(br_total * ws / (cb_ms["one_request_per_batch"] / 1e3), 1)},
            "speedup": round(cb_ms["one_request_per_batch"] / cb_ms["batched"], 3),
        },
        "decisions_per_s": round(N * ws / (ms / 1e3), 1),
        "logical_tokens_per_s": round(stats["logical_tokens"] * ws / (ms / 1e3), 1),
        # the same counts over the phases that compute them: branch tokens
        # and logical tokens over the attention time, decisions over the
        # readout and softmax time (the step-based figures above include
        # every phase)
        "per_phase": {
            "branch_tokens_per_s_attention": round(branch_tokens * ws / (attn_avg / 1e3), 1),
            "logical_tokens_per_s_attention": round(stats["logical_tokens"] * ws / (attn_avg / 1e3), 1),
            "decisions_per_s_readout": round(N * ws / ((lm_avg + statistics.mean(sm_ms)) / 1e3), 1),
        },
        "phase_ms": {"attention": round(attn_avg, 5), "label_logprobs": round(lm_avg, 5),
                     "label_softmax": round(statistics.mean(sm_ms), 5),
                     "plan_and_launch_overhead": round(ms - attn_avg - lm_avg - statistics.mean(sm_ms), 5)},
        "roofline": dict(attention_roofline if dominant == "attention" else readout_roofline),
        "attention_roofline": attention_roofline,
        "readout_roofline": readout_roofline,
        "e2e": {"value": round(branch_tokens * ws / (e2e_ms / 1e3), 1), "unit": "branch tokens/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "ms_per_step": round(e2e_ms, 5)},
        "gpu_launches": int(launches_per_step * args.steps),
        "clocks": clocks,
    }
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(wl, args.config)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return result if rank == 0 else None


def run_phase(args, wl, clf, dev):
    """One phase of the step alone, for kernel profiles on a small device
    footprint: "attention" holds q / k / v and the pool; "readout" holds h, W
    and the labels (the readout and the label softmax).  Returns a timing line
    (CUDA events around each call, after the warm-up calls)."""
    import torch
    from prefill_only_shared_gb300 import sp
    stream = torch.cuda.current_stream(dev)
    sh = wl.shape
    N = wl.n_branches
    if args.only == "attention":
        q, k, v = wl.q.to(dev), wl.k.to(dev), wl.v.to(dev)
        plan = clf.plan(wl.req_of_branch, wl.tok_offsets, wl.tokens)
        call = lambda: clf.attention(plan, q, k, v, stream, args.schedule)
        f_prefix, f_branch = attention_flops(plan.segments(), wl)
        work = {"flops_per_call": f_prefix + f_branch}
    else:
        h, W = wl.h.to(dev), wl.W.to(dev)
        off = torch.from_numpy(wl.label_off).to(dev)
        ids = torch.from_numpy(wl.label_ids).to(dev)
        n_labels = int(wl.label_ids.shape[0])

        def call():
            lp, _ = clf.logprobs(h, W, off, ids, n_labels, stream)
            clf.softmax(lp, off, stream)
        work = {"flops_per_call": 2.0 * N * sh.hidden * sh.vocab,
                "bytes_per_call": sh.vocab * sh.hidden * 2 + N * sh.hidden * 2 + n_labels * 8 + N * 4}
    for _ in range(max(args.warmup, 1)):
        call()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    time.sleep(0.3)
    sampler.mark()
    for e0, e1 in evs:
        e0.record(stream)
        call()
        e1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    sp.sp_check_device_error()
    ms = statistics.median(e0.elapsed_time(e1) for e0, e1 in evs)
    return {"phase": args.only, "config": args.config, "schedule": args.schedule,
            "calls": args.steps, "ms_per_call_median": round(ms, 5), **work, "clocks": clocks}


# --------------------------------------------------------------------------
def oracle_sample(wl, plan, branches):
    """The oracle on a bounded sample: for each branch given, its own suffix
    rows (the branch tokens the metric counts) by unshared attention over its
    whole sequence, then its full-vocabulary readout and label softmax.
    Returns the branch tokens computed."""
    import numpy as np
    from oracle import attention as OA
    from oracle import label_softmax as OL
    from oracle import readout as OR
    toks = 0
    for b in branches:
        leaf = plan.segments[plan.paths[b][-1]]
        rows = list(range(leaf.node_start, leaf.node_start + leaf.length))
        OA.sampled_attention(plan, wl.q, wl.k, wl.v, rows)
        lp, _ = OR.label_logprobs(wl.h, wl.W, wl.label_off, wl.label_ids, branches=[b])
        OL.label_softmax(lp, np.array([0, len(lp)]))
        toks += leaf.length
    return toks


def cpu_baseline(wl, config, min_seconds=10.0, max_seconds=30.0):
    """The oracle timed on the host cores: branches in order (wrapping around)
    until about min_seconds of work (at most max_seconds)."""
    import torch
    from oracle import staging as OS
    torch.set_num_threads(os.cpu_count() or 1)
    plan = OS.build_plan(wl.req_of_branch, wl.tok_offsets, wl.tokens)
    t = time.perf_counter()
    toks = nb = 0
    while True:
        toks += oracle_sample(wl, plan, [nb % wl.n_branches])
        nb += 1
        dt = time.perf_counter() - t
        if dt >= min_seconds or dt + dt / nb > max_seconds:
            break
    return {"value": round(toks / dt, 3), "unit": "branch tokens/s", "cores": os.cpu_count(),
            "kind": "oracle",
            "sample": f"{config}: {nb} branch readouts ({toks} branch tokens), each branch's "
                      f"suffix rows by unshared float64 attention over its whole sequence, "
                      f"full-vocabulary readout and softmax; {dt:.1f} s"}


DATA = "synthetic (seeded, the configuration's shapes; random-init LM head)"
L2_MB = 129  # GB300 L2


def workload_config(name, sh, n_branches, logical, computed, n_rounds, branch_tokens, ws,
                    schedule):
    """The `config` object of both arms' lines."""
    w_mb = sh.vocab * sh.hidden * 2 / 1e6
    return {
        "workload": f"{name}: Hq {sh.n_q_heads}/Hkv {sh.n_kv_heads}/d {sh.head_dim}, "
                    f"{n_branches} branches, {logical} logical tokens, {computed} computed, "
                    f"H {sh.hidden}, V {sh.vocab}",
        "branches": n_branches,
        "branch_tokens_per_step": branch_tokens,
        "logical_tokens_per_step": logical,
        "rounds": n_rounds,
        "l2": (f"inputs larger than L2 (the {w_mb:.0f} MB LM head is streamed every step)"
               if w_mb > L2_MB else
               f"inputs smaller than L2 ({w_mb:.0f} MB LM head), not flushed: cache-warm figures"),
        "parallelism": f"replicas x{ws} (independent workloads per GPU)",
        "attention_schedule": schedule,
    }


def run_reference(args, ws, rank):
    if rank != 0:
        return None
    from prefill_only_shared_gb300.workloads import make_workload
    import torch
    torch.set_num_threads(os.cpu_count() or 1)
    from oracle import staging as OS
    wl = make_workload(args.config, seed=0)
    plan = OS.build_plan(wl.req_of_branch, wl.tok_offsets, wl.tokens)
    ps = OS.plan_stats(plan)
    branch_tokens = (sum(sg.length for sg in plan.segments if not sg.shared)
                     + sum(1 for x in plan.recompute if x))
    for i in range(args.warmup):
        oracle_sample(wl, plan, [i % wl.n_branches])
    t = time.perf_counter()
    toks = 0
    for i in range(args.steps):  # one branch per step, in order
        toks += oracle_sample(wl, plan, [i % wl.n_branches])
    dt = time.perf_counter() - t
    value = toks / dt
    return {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 3), "unit": "branch tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": DATA,
        "config": workload_config(args.config, wl.shape, wl.n_branches, ps["logical_tokens"],
                                  ps["computed_tokens"], ps["n_rounds"], branch_tokens, ws,
                                  args.schedule),
        "cpu_baseline": {"value": round(value, 3), "unit": "branch tokens/s",
                         "cores": os.cpu_count(), "kind": "oracle",
                         "sample": f"{args.config}: 1 branch per step, its suffix rows by "
                                   "unshared float64 attention over its whole sequence, "
                                   "full-vocabulary readout and softmax"},
        "e2e": {"value": round(value, 3), "unit": "branch tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    ws, rank, local = dist_env()
    if args.impl == "reference":
        res = run_reference(args, ws, rank)
    else:
        res = run_libsp(args, ws, rank, local)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()

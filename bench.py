"""Benchmark of one constrained decode step: fill_bitmask -> mask_and_sample -> accept.

Workload (default ``booking_128k``): booking-decision JSON schema automaton,
V = 128256 synthetic tokens, B = 256 rows, bf16 logits N(0, 2) with +4 on 5% of
tokens, temperature 0.7, top-p 0.9.  Rows start in the start state; rows that
finish or reach 2048 tokens are reset by accept.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--prefix P] [--impl ours|reference]

Prints one JSON line.  ``value`` is constrained tokens/s with the step's inputs
already resident in HBM, over a steady-state window: the timed steps come after
an untimed prefix of P steps (default 300) and are named in ``config.window``;
the first steps after the warm-up are timed apart (``fresh_start``).  R
pre-generated logit buffers whose total exceeds 4x the L2 size are used in
rotation, so every step reads its logits from HBM.  Beside the headline:
``workloads`` (the four other synthetic workloads, each with its roofline
fraction; mixed_eval_152k also as a decode loop through the host forced-token
driver), ``bench_gap`` (the step against the same sampling with an all-ones
mask), ``mask_cache_without_prefill`` (misses per step and step times on a
context without prefill), the pushdown rows and speculative verification.
``e2e`` repeats the measurement through cg_step_host: every step's logits are
copied from page-locked host memory (the copy of one step overlapping the
previous step's kernel) and its sampled tokens copied back to host memory.
``--impl reference`` times the CPU oracle (the plain restatement the kernels
are checked against) on a bounded sample of the same workload, on every host
core; ``cpu_baseline`` gives that sample on one thread and on every core.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "constrained tokens/s and µs/step (mask+apply+sample) at V=128256, B=256"
SAMPLE_SOURCES = ["grammar_constrained_decoding_gb300/csrc/kernel_sample.cu",
                  "grammar_constrained_decoding_gb300/csrc/bf16_ops.cuh",
                  "grammar_constrained_decoding_gb300/csrc/device.cuh",
                  "grammar_constrained_decoding_gb300/csrc/row_ops.cuh"]


def _kernel_hash() -> str:
    """Hash of the sampling kernel's code (comments and blank lines removed, so
    that a comment edit keeps a recorded DRAM-traffic figure valid)."""
    import re
    h = hashlib.sha256()
    for p in SAMPLE_SOURCES:
        src = open(os.path.join(ROOT, p), encoding="utf-8").read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        h.update("\n".join(ln.rstrip() for ln in src.splitlines() if ln.strip()).encode())
    return h.hexdigest()[:16]


def _peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


def _traffic_record():
    """DRAM bytes per launch of the sampling kernel from a committed ncu summary,
    valid only while the kernel sources are unchanged."""
    p = os.path.join(ROOT, "profiles", "sample_kernel_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    if d.get("kernel_sha") != _kernel_hash():
        return None
    return d


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms."""
    QUERY = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.samples = []
        self._stop = threading.Event()
        self._proc = None
        try:
            self._proc = subprocess.Popen(["nvidia-smi", f"--id={index}", f"--query-gpu={self.QUERY}",
                                           "--format=csv,noheader,nounits", "-lms", "200"],
                                          stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()

    def _read(self):
        for line in self._proc.stdout:
            self.samples.append((time.time(), [v.strip() for v in line.split(",")]))

    def stop(self):
        if self._proc:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self._proc.kill()

    def summary(self, t0: float, t1: float) -> dict:
        # a sample's line arrives up to one period after it was taken
        inside = [s for t, s in self.samples if t0 <= t <= t1 + 0.2]
        if not inside and self.samples:
            # timed region shorter than the sampling period: nearest samples
            inside = [min(self.samples, key=lambda ts: abs(ts[0] - (t0 + t1) / 2))[1]]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        sm = sorted(float(s[1]) for s in inside if s[1].replace(".", "").isdigit())
        mx = [float(s[2]) for s in inside if s[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in inside for i in range(4) if len(s) > 5 + i and s[5 + i] == "Active"})
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside)}


def _parse_cpulist(txt: str) -> set:
    cpus = set()
    for part in txt.strip().split(","):
        if "-" in part:
            a, b = part.split("-")
            cpus.update(range(int(a), int(b) + 1))
        elif part:
            cpus.add(int(part))
    return cpus


def _numa_bind(index: int) -> dict:
    """Binds this process to the CPUs of the GPU's NUMA node when the system
    reports one, so that the page-locked buffers allocated next are local to
    the GPU's host link, and says what it found."""
    info = {"gpu_numa_node": None, "bound_cpus": None}
    try:
        bus = subprocess.run(["nvidia-smi", f"--id={index}", "--query-gpu=pci.bus_id", "--format=csv,noheader"],
                             capture_output=True, text=True, timeout=30).stdout.strip()
        dom, rest = bus.split(":", 1)
        node = int(open(f"/sys/bus/pci/devices/{(dom[-4:] + ':' + rest).lower()}/numa_node").read())
        info["gpu_numa_node"] = node
        if node >= 0:
            cpus = _parse_cpulist(open(f"/sys/devices/system/node/node{node}/cpulist").read())
            if cpus:
                os.sched_setaffinity(0, cpus)
                info["bound_cpus"] = f"{min(cpus)}-{max(cpus)} ({len(cpus)} cpus)"
    except Exception as e:  # no nvidia-smi, no sysfs entry: report and go on unbound
        info["error"] = f"{type(e).__name__}: {e}"[:160]
    try:
        info["nodes_with_cpus"] = sorted(int(d[4:]) for d in os.listdir("/sys/devices/system/node")
                                         if d.startswith("node") and d[4:].isdigit()
                                         and open(f"/sys/devices/system/node/{d}/cpulist").read().strip())
    except OSError:
        pass
    return info


def _dist():
    from grammar_constrained_decoding_gb300.replicas import rank_info
    return rank_info()


def run_ours(args) -> dict | None:
    import numpy as np
    import torch

    import grammar_constrained_decoding_gb300 as cg
    from workloads import CONFIGS, GRAMMARS, make_vocab
    from workloads.logits import make_logits_device

    from grammar_constrained_decoding_gb300 import replicas
    world, rank, local = _dist()
    torch.cuda.set_device(local)
    pg = replicas.init("nccl", torch.device("cuda", local))  # replicas: rows shard, nothing is exchanged
    cfg = CONFIGS[args.config]
    B, V = cfg.B, cfg.V
    W = (V + 31) // 32
    spec = GRAMMARS[cfg.grammars[0]]
    b = spec.bounds
    grammars = [cg.Grammar.compile(GRAMMARS[n].source, GRAMMARS[n].kind,
                                   cg.Bounds(b.ws_max, b.max_len_default, b.depth_max, b.max_items_default,
                                             b.max_tokens)) for n in cfg.grammars]
    toks = make_vocab(cfg.vocab_kind, V, cfg.vocab_seed)
    stream = torch.cuda.Stream()      # graphs are captured on a side stream
    torch.cuda.set_stream(stream)
    vocab = cg.Vocab(toks)
    ctx = cg.Ctx(grammars, vocab, stream)
    ctx.prefill()   # every mask class computed once, outside the timed steps
    dtype = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    esz = 2 if cfg.dtype == "bf16" else 4
    l2 = torch.cuda.get_device_properties(local).L2_cache_size
    step_bytes = B * V * esz
    R = max(2, -(-4 * l2 // step_bytes))
    gen = torch.Generator(device="cuda")
    gen.manual_seed(replicas.replica_seed(cfg.logit_seed, rank))
    bufs = [make_logits_device(B, V, 0, cfg.sigma, cfg.boost, cfg.boost_frac, cfg.dtype, "cuda", gen)
            for _ in range(R)]
    gid = None
    if len(cfg.grammars) > 1:
        gid = torch.as_tensor((np.arange(B) % len(cfg.grammars)).astype(np.int16)).cuda().view(torch.uint16)
    states = torch.zeros(B, dtype=torch.int32, device="cuda").view(torch.uint32)
    counts = torch.zeros(B, dtype=torch.int32, device="cuda").view(torch.uint32)
    bm = torch.empty((B, W), dtype=torch.int32, device="cuda")
    tok = torch.empty(B, dtype=torch.int32, device="cuda")
    flags = torch.empty(B, dtype=torch.uint8, device="cuda")
    seed = cfg.sample_seed

    def step(i, logits):
        # one call: mask fill, masked sampling and accept (one kernel on this workload)
        ctx.step(states, logits, cfg.temp, cfg.top_p, seed, i, tok, states, flags, gid=gid, counts=counts,
                 max_tokens=b.max_tokens)

    def three_calls(i, logits):
        ctx.fill_bitmask(states, bm, gid=gid)
        ctx.mask_and_sample(logits, bm, cfg.temp, cfg.top_p, seed, i, tok)
        ctx.accept(states, tok.view(torch.uint32), states, flags, gid=gid, counts=counts,
                   max_tokens=b.max_tokens)

    # warm-up (fills the mask cache, sizes the sampling scratch)
    for i in range(args.warmup):
        step(i, bufs[i % R])
    torch.cuda.synchronize()
    if ctx.status() != 0:
        raise RuntimeError("device status after warm-up")
    applied = args.warmup   # steps applied to the rows' states so far

    # fresh-start figure: the next F steps of trajectories that began in the
    # start state, where most rows sit in cheap JSON-structure states
    F = 20
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for i in range(applied, applied + F):
        step(i, bufs[i % R])
    f1.record(stream)
    torch.cuda.synchronize()
    fresh_us = f0.elapsed_time(f1) / F * 1e3
    fresh_window = f"steps {applied}..{applied + F - 1}"
    applied += F
    # steady state: an untimed prefix before the timed window, so that the
    # window sees the workload's own mix of row states (rows restart in the
    # start state when they finish or reach the token cap)
    for i in range(applied, applied + args.prefix):
        step(i, bufs[i % R])
    applied += args.prefix
    torch.cuda.synchronize()
    if ctx.status() != 0:
        raise RuntimeError("device status after the prefix")

    # The timed steps run as CUDA graphs of G steps each (launch-bound host
    # code out of the way); each step of a graph keeps its own step index and
    # logits buffer.  A second set of graphs runs the same steps as the three
    # separate calls (fill_bitmask, mask_and_sample, accept) for comparison.
    G = min(args.steps, 250)
    plan = [G] * (args.steps // G) + ([args.steps % G] if args.steps % G else [])

    def capture(first, n, fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
            for i in range(first, first + n):
                fn(i, bufs[i % R])
        return g

    for i in range(applied, applied + args.warmup):   # the three-call path's buffers and scratch, before capture
        three_calls(i, bufs[i % R])
    applied += args.warmup

    graphs, first = [], applied
    for n in plan:
        graphs.append(capture(first, n, step))
        first += n
    sample_graphs, first = [], applied
    for n in plan:
        sample_graphs.append(capture(first, n, three_calls))
        first += n
    # one untimed replay of the step graphs (first replays upload the graphs)
    for g in graphs:
        g.replay()
    torch.cuda.synchronize()
    if ctx.status() != 0:
        raise RuntimeError("device status after graph warm-up")
    applied += args.steps
    window = (f"steps {applied}..{applied + args.steps - 1} of every row's trajectory from the start state "
              f"(untimed before them: {args.warmup} warm-up, {F} fresh-start, {args.prefix} prefix, "
              f"{args.warmup} three-call warm-up steps and one replay of the step graphs); rows restart in the "
              f"start state when they finish or reach {b.max_tokens} tokens")

    sampler = ClockSampler(local) if rank == 0 else None
    time.sleep(0.25)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    start.record(stream)
    for g in graphs:
        g.replay()
    end.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    if pg:
        pg.barrier()
    ms = start.elapsed_time(end)
    status = ctx.status()
    if status != 0:
        raise RuntimeError(f"device status {status} in the timed region")
    # the same steps as three separate calls
    for g in sample_graphs:
        g.replay()
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    s0.record(stream)
    for g in sample_graphs:
        g.replay()
    s1.record(stream)
    torch.cuda.synchronize()
    three_ms = s0.elapsed_time(s1) / args.steps
    if ctx.status() != 0:
        raise RuntimeError("device status after the three-call steps")
    ms = replicas.max_over_ranks(ms, pg, "cuda")
    time.sleep(0.3)
    clocks = sampler.summary(t0, t1) if sampler else None
    if sampler:
        sampler.stop()
    del graphs, sample_graphs

    if args.step_only:   # a profiling run: the timed steps only
        if rank != 0:
            return None
        per_step = ms / args.steps
        return {"metric": METRIC, "value": round(replicas.job_throughput(B * args.steps, world, ms), 1),
                "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(per_step, 5), "us_per_step": round(per_step * 1e3, 3),
                "higher_is_better": True, "dtype": cfg.dtype, "config": {"workload": cfg.name, "window": window},
                "note": "--step-only: the timed cg_step graphs and the three-call graphs; no other leg ran"}

    # speculative verification (cg_accept_many): drafts of K = 8 tokens taken
    # from the workload's own next 8 steps, verified from the states before them
    K = 8
    s_before = states.clone()
    c_before = counts.clone()
    draft = torch.empty((B, K), dtype=torch.int32, device="cuda")
    for j in range(K):
        step(2 * 10**6 + j, bufs[j % R])
        draft[:, j] = tok
    states.copy_(s_before)
    counts.copy_(c_before)
    dlen = torch.full((B,), K, dtype=torch.int32, device="cuda").view(torch.uint32)
    am_s = torch.empty(B, dtype=torch.int32, device="cuda").view(torch.uint32)
    am_n = torch.empty(B, dtype=torch.int32, device="cuda").view(torch.uint32)
    am_f = torch.empty(B, dtype=torch.uint8, device="cuda")
    am_path = torch.empty((B, K + 1), dtype=torch.int32, device="cuda").view(torch.uint32)
    draft_u = draft.view(torch.uint32)

    def verify():
        ctx.accept_many(states, draft_u, dlen, am_s, am_n, am_f, gid=gid, path=am_path)

    for _ in range(3):
        verify()
    torch.cuda.synchronize()
    n_am = 500
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    for _ in range(n_am):
        verify()
    a1.record(stream)
    torch.cuda.synchronize()
    am_us = a0.elapsed_time(a1) / n_am * 1e3
    am_accepted = float(am_n.view(torch.int32).float().mean().item())
    if ctx.status() != 0:
        raise RuntimeError("device status after accept_many")

    # pushdown rows (cg_pda_*): the recursive JSON grammar with a stack of 32
    # frames on the same vocabulary, rows and logits, as the three calls
    # fill (pushdown) -> mask_and_sample -> accept (pushdown), in graphs
    pda_out = _bench_pushdown(args, cg, ctx, vocab, stream, bufs, R, B, V, W, cfg, seed)
    gap = _bench_gap(ctx, stream, bufs, R, B, V, W, cfg, seed, G, ms / args.steps * 1e3)
    cache = _bench_cache(cg, grammars, vocab, stream, bufs, R, B, cfg, seed, b, fresh_us)

    # host evaluators of the forced-token path, per call through the C ABI
    # (Python's call overhead included) on the pages' examples
    host_eval = {}
    for label, fn, span in (("arith 17 * 23 + 91", lambda x: cg.eval_arith(x, "calc_tag"), b"17 * 23 + 91"),
                            ('strop count("strawberry", "r")', cg.eval_strop, b'count("strawberry", "r")')):
        fn(span)
        t_h = time.perf_counter()
        for _ in range(20000):
            fn(span)
        host_eval[label] = round((time.perf_counter() - t_h) / 20000 * 1e6, 3)

    # end to end through cg_step_host: each step's logits copied from
    # page-locked host memory (overlapping the previous step's kernel) and its
    # ids copied back to host memory
    e2e_steps = min(args.steps, args.e2e_steps)
    nh = 2
    cpus0 = os.sched_getaffinity(0)
    numa = _numa_bind(local)   # page-locked buffers on the GPU's NUMA node, when it has one
    host_bufs = [bufs[i].cpu().pin_memory() for i in range(nh)]
    tok_host = torch.empty(B, dtype=torch.int32, pin_memory=True)
    ctx.step_host(states, host_bufs[0], cfg.temp, cfg.top_p, seed, 10**6, tok_host, states, flags, gid=gid,
                  counts=counts, max_tokens=b.max_tokens)   # sizes the context's logit buffers
    ctx.step_host(states, host_bufs[1], cfg.temp, cfg.top_p, seed, 10**6 + 1, tok_host, states, flags, gid=gid,
                  counts=counts, max_tokens=b.max_tokens)
    ctx.sync()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(e2e_steps):
        ctx.step_host(states, host_bufs[i % nh], cfg.temp, cfg.top_p, seed, 10**6 + 2 + i, tok_host, states,
                      flags, gid=gid, counts=counts, max_tokens=b.max_tokens)
    e1.record(stream)
    ctx.sync()
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    os.sched_setaffinity(0, cpus0)
    workloads = None if args.no_workloads else _bench_workloads(cg, local, _peaks(), args.quick)

    if rank != 0:
        return None
    per_step = ms / args.steps
    k2_avg_ms = per_step   # one kernel per step: the fused step kernel
    alg_bytes = B * (V * esz + W * 4)
    peaks = _peaks()
    achieved = alg_bytes / (k2_avg_ms * 1e-3) / 1e9
    traffic = _traffic_record()
    units = B * args.steps * world   # every rank decodes its own B rows
    info = ctx.info()
    out = {
        "metric": METRIC,
        "value": round(replicas.job_throughput(B * args.steps, world, ms), 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(per_step, 5),
        "us_per_step": round(per_step * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": cfg.dtype,
        "data": "synthetic (seeded vocabulary, logits and grammar; no model)",
        "config": {"workload": f"{cfg.name}: booking-decision JSON schema automaton "
                               f"({grammars[0].info()['n_states']} states), V={V}, B={B}, {cfg.dtype} logits "
                               f"N(0,{cfg.sigma}) +{cfg.boost} on {cfg.boost_frac:.0%}, T={cfg.temp}, "
                               f"top_p={cfg.top_p}",
                   "B": B, "V": V, "l2_policy": f"{R} rotated logit buffers, {R * step_bytes / 2**20:.0f} MiB "
                                                 f">= 4x L2 ({l2 / 2**20:.0f} MiB): every step reads HBM",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "mask_classes": info["n_classes"], "window": window},
        "gpu_launches": args.steps,
        "kernel_us": {"step (cg_step, one fused kernel)": round(per_step * 1e3, 3),
                      "step as three calls (fill_bitmask, mask_and_sample, accept)": round(three_ms * 1e3, 3),
                      "accept_many (B rows, drafts of 8 tokens from the next 8 steps)": round(am_us, 3)},
        "accept_many_mean_accepted": round(am_accepted, 3),
        "fresh_start": {"us_per_step": round(fresh_us, 3), "window": fresh_window,
                        "tokens_per_s": round(B / (fresh_us * 1e-6), 1)},
        "bench_gap": gap,
        "mask_cache_without_prefill": cache,
        "workloads": workloads,
        "pushdown": pda_out,
        "host_eval_us_per_call": host_eval,
        "roofline": {"kernel": "stream_topp_kernel<1> (cg_step)", "bound": "hbm",
                     "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4),
                     "peak_source": f"{peaks['source']} (copy bandwidth)",
                     "algorithmic_bytes_per_launch": alg_bytes,
                     "traffic": traffic["dram_bytes_per_launch"] if traffic else None},
        "e2e": {"value": round(B / (e2e_ms * 1e-3), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": step_bytes, "d2h_bytes_per_step": B * 4, "steps": e2e_steps,
                "h2d_gbs": round(step_bytes / (e2e_ms * 1e-3) / 1e9, 1), "numa": numa},
        "clocks": clocks,
    }
    return out


FORMATS = {"calc_tag": 0, "json_answer": 1, "strop_tag": 2}   # CG_RESULT_* of include/cg.h


def _alg_bytes(B: int, V: int, esz: int) -> int:
    """Algorithmic bytes of one step: every row's logits read once and its
    bitmask words once (the per-unit figure 2V + 4W for bf16)."""
    return B * (V * esz + ((V + 31) // 32) * 4)


def _graph_us(stream, fn, first: int, n: int, reps: int = 1) -> float:
    """Device time per step of n steps fn(i) captured in one CUDA graph (one
    untimed replay first; the steps keep their own indices)."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
        for i in range(first, first + n):
            fn(i)
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    del g
    return e0.elapsed_time(e1) / (n * reps) * 1e3


def _bench_gap(ctx, stream, bufs, R, B, V, W, cfg, seed, n, step_us) -> dict:
    """Enforcement overhead (usetacet.com/docs/grammar, "What it is worth": the
    same calls with the automaton on and off): the constrained step against
    the same sampling with the automaton off (an all-ones mask, no bitmask
    fill, no accept)."""
    import torch
    ones = torch.full((B, W), -1, dtype=torch.int32, device="cuda")
    if V % 32:
        ones[:, W - 1] = (1 << (V % 32)) - 1
    tok = torch.empty(B, dtype=torch.int32, device="cuda")

    def f(i):
        ctx.mask_and_sample(bufs[i % R], ones, cfg.temp, cfg.top_p, seed, i, tok)

    for i in range(3):
        f(i)
    un_us = _graph_us(stream, f, 3, n)
    return {"unconstrained_us_per_step": round(un_us, 3), "constrained_us_per_step": round(step_us, 3),
            "overhead": round(step_us / un_us - 1.0, 4),
            "unconstrained": "cg_mask_and_sample with an all-ones bitmask (no fill, no accept)",
            "constrained": "cg_step (mask fill, masked sampling and accept), steady-state window"}


def _bench_cache(cg, grammars, vocab, stream, bufs, R, B, cfg, seed, b, fresh_us, n=40) -> dict:
    """The fused step on a context without prefill: every class mask is
    computed by the first row that misses it (labs.miniml.ai "Evaluator aware
    decoding", "Where XGrammar-2 could take this", on the token mask cache)."""
    import torch
    ctx = cg.Ctx(grammars, vocab, stream)
    n_cls = ctx.info()["n_classes"]
    states = torch.zeros(B, dtype=torch.int32, device="cuda").view(torch.uint32)
    counts = torch.zeros(B, dtype=torch.int32, device="cuda").view(torch.uint32)
    tok = torch.empty(B, dtype=torch.int32, device="cuda")
    flags = torch.empty(B, dtype=torch.uint8, device="cuda")
    us, misses, ready = [], [], ctx.cache_stats()["ready"]
    for i in range(n):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        ctx.step(states, bufs[i % R], cfg.temp, cfg.top_p, seed, i, tok, states, flags, counts=counts,
                 max_tokens=b.max_tokens)
        e1.record(stream)
        r = ctx.cache_stats()["ready"]   # synchronises the stream
        us.append(e0.elapsed_time(e1) * 1e3)
        misses.append(r - ready)
        ready = r
    if ctx.status() != 0:
        raise RuntimeError("device status in the cache leg")
    return {"n_classes": n_cls, "steps": n, "lookups_per_step": B,
            "misses_per_step_first10": misses[:10], "misses_total": sum(misses), "classes_ready_after": ready,
            "us_step0": round(us[0], 2), "us_per_step_1_9": round(sum(us[1:10]) / 9, 2),
            "us_per_step_10_39": round(sum(us[10:40]) / 30, 2),
            "with_prefill_us_per_step_fresh_start": round(fresh_us, 2),
            "note": "steps from the start state on a fresh context (no cg_ctx_prefill), one CUDA-event pair "
                    "per step; a miss is a class mask computed during that step"}


def _mixed_loop(cg, ctx, vocab, stream, bufs, R, B, cfg, gid_np, gid, specs, max_tokens, prefix, n) -> dict:
    """mixed_eval_152k as a decode loop with the host forced-token driver
    (labs.miniml.ai "Evaluator aware decoding", "The core idea"): every step
    the tokens and flags come back to the host, the driver evaluates the rows
    that closed a span and the next step's forced tokens go back to the device
    (the host round trip the pages' "Why isn't this in production APIs yet?"
    names)."""
    import numpy as np
    import torch
    rules = [(s.span_open, s.span_close, FORMATS[s.result_format]) if s.result_format else (b"", b"", -1)
             for s in specs]
    drv = cg.Driver(vocab, B, gid_np, rules)
    states = torch.zeros(B, dtype=torch.int32, device="cuda").view(torch.uint32)
    counts = torch.zeros(B, dtype=torch.int32, device="cuda").view(torch.uint32)
    tok = torch.empty(B, dtype=torch.int32, device="cuda")
    flags = torch.empty(B, dtype=torch.uint8, device="cuda")
    forced_d = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    tok_h = torch.empty(B, dtype=torch.int32, pin_memory=True)
    flags_h = torch.empty(B, dtype=torch.uint8, pin_memory=True)
    fnext_h = torch.full((B,), -1, dtype=torch.int32, pin_memory=True)
    forced_used = np.full(B, -1, np.int32)
    forced_next = np.full(B, -1, np.int32)
    dev_us, host_us, wall_us, forced_rows, evals = [], [], [], [], []
    for i in range(prefix + n):
        forced_used[:] = forced_next
        t0 = time.perf_counter()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        ctx.step(states, bufs[i % R], cfg.temp, cfg.top_p, cfg.sample_seed, i, tok, states, flags, gid=gid,
                 forced=forced_d, counts=counts, max_tokens=max_tokens)
        e1.record(stream)
        tok_h.copy_(tok, non_blocking=True)
        flags_h.copy_(flags, non_blocking=True)
        stream.synchronize()
        t1 = time.perf_counter()
        ne = drv.update(tok_h.numpy().view(np.uint32), flags_h.numpy(), forced_used, forced_next)
        fnext_h.numpy()[:] = forced_next
        forced_d.copy_(fnext_h, non_blocking=True)
        t2 = time.perf_counter()
        if i >= prefix:
            dev_us.append(e0.elapsed_time(e1) * 1e3)
            host_us.append((t2 - t1) * 1e6)
            wall_us.append((t2 - t0) * 1e6)
            forced_rows.append(int((forced_used >= 0).sum()))
            evals.append(ne)
    torch.cuda.synchronize()
    if ctx.status() != 0:
        raise RuntimeError("device status in the mixed decode loop")
    m = lambda v: round(sum(v) / len(v), 3)
    return {"steps": n, "after_prefix": prefix, "wall_us_per_step": m(wall_us), "device_step_us": m(dev_us),
            "host_us_per_step (driver update + forced-token upload)": m(host_us),
            "forced_rows_per_step": m(forced_rows), "injected_tokens_per_step": m(forced_rows),
            "evaluations_per_step": m(evals), "tokens_per_s_wall": round(B / (m(wall_us) * 1e-6), 1),
            "readback_bytes_per_step": B * 5, "upload_bytes_per_step": B * 4}


def _bench_workloads(cg, local, peaks, quick: bool) -> dict:
    """Per-workload steady-state step time, throughput and HBM roofline
    fraction of the four workloads beside the headline one."""
    import numpy as np
    import torch
    from workloads import CONFIGS, GRAMMARS, make_vocab
    from workloads.logits import make_logits_device
    l2 = torch.cuda.get_device_properties(local).L2_cache_size
    out = {}
    for name in ("tiny", "booking_32k", "reasoning_152k", "mixed_eval_152k"):
        cfg = CONFIGS[name]
        B, V = cfg.B, cfg.V
        esz = 2 if cfg.dtype == "bf16" else 4
        specs = [GRAMMARS[n] for n in cfg.grammars]
        grammars = [cg.Grammar.compile(s.source, s.kind, cg.Bounds(s.bounds.ws_max, s.bounds.max_len_default,
                                                                    s.bounds.depth_max, s.bounds.max_items_default,
                                                                    s.bounds.max_tokens)) for s in specs]
        vocab = cg.Vocab(make_vocab(cfg.vocab_kind, V, cfg.vocab_seed))
        stream = torch.cuda.current_stream()
        ctx = cg.Ctx(grammars, vocab, stream)
        ctx.prefill()
        R = max(2, -(-4 * l2 // (B * V * esz)))
        gen = torch.Generator(device="cuda")
        gen.manual_seed(cfg.logit_seed)
        bufs = [make_logits_device(B, V, 0, cfg.sigma, cfg.boost, cfg.boost_frac, cfg.dtype, "cuda", gen)
                for _ in range(R)]
        gid_np = (np.arange(B) % len(specs)).astype(np.uint16)
        gid = torch.as_tensor(gid_np.astype(np.int16)).cuda().view(torch.uint16) if len(specs) > 1 else None
        if cfg.random_start:
            live = grammars[0].live_states()
            st = live[np.random.default_rng([cfg.logit_seed, 0x5747]).integers(0, len(live), B)].astype(np.uint32)
        else:
            st = np.zeros(B, np.uint32)
        states = torch.from_numpy(st.view(np.int32)).cuda().view(torch.uint32)
        counts = torch.zeros(B, dtype=torch.int32, device="cuda").view(torch.uint32)
        tok = torch.empty(B, dtype=torch.int32, device="cuda")
        flags = torch.empty(B, dtype=torch.uint8, device="cuda")
        mt = specs[0].bounds.max_tokens

        def step(i):
            ctx.step(states, bufs[i % R], cfg.temp, cfg.top_p, cfg.sample_seed, i, tok, states, flags, gid=gid,
                     counts=counts, max_tokens=mt)

        prefix = 20 if quick else (50 if B * V > 10**8 else 100)
        n = 20 if quick else 100
        loop = None
        if any(s.result_format for s in specs):
            # evaluator grammars need the host driver's forced tokens every
            # step: the step is timed inside that decode loop (CUDA events
            # around each cg_step)
            loop = _mixed_loop(cg, ctx, vocab, stream, bufs, R, B, cfg, gid_np, gid, specs, mt, prefix, n)
            us = loop["device_step_us"]
            window = f"steps {prefix}..{prefix + n - 1} of the decode loop (CUDA events around each cg_step)"
        else:
            for i in range(prefix):
                step(i)
            torch.cuda.synchronize()
            us = _graph_us(stream, step, prefix, n)
            window = (f"steps {prefix + n}..{prefix + 2 * n - 1} (after a {prefix}-step prefix and one untimed "
                      f"graph replay)")
        if ctx.status() != 0:
            raise RuntimeError(f"device status in workload {name}")
        ab = _alg_bytes(B, V, esz)
        ach = ab / (us * 1e-6) / 1e9
        if cfg.dtype != "bf16":
            path = "three calls (fill_bitmask, per-row f32 sampler, accept)"
        elif cfg.temp > 0 and cfg.top_p < 1:
            path = "stream_topp_kernel<1> (cg_step, per-row fused top-p)"
        else:
            path = "seg_kernel (cg_step, segmented fused " + ("greedy" if cfg.temp == 0 else "Gumbel-max") + ")"
        res = {"B": B, "V": V, "dtype": cfg.dtype, "temp": cfg.temp, "top_p": cfg.top_p, "path": path,
               "us_per_step": round(us, 3), "tokens_per_s": round(B / (us * 1e-6), 1), "window": window,
               "roofline": {"bound": "hbm", "algorithmic_bytes_per_step": ab, "achieved": round(ach, 1),
                            "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(ach / peaks["hbm_gbs"], 4)}}
        if loop:
            res["decode_loop_with_host_driver"] = loop
        out[name] = res
        del ctx, bufs
        torch.cuda.empty_cache()
    return out



def _bench_pushdown(args, cg, ctx, vocab, stream, bufs, R, B, V, W, cfg, seed) -> dict:
    """The pushdown path on json_nested (stack bound 32): per-step time of
    the three calls, and each kernel launched alone back to back."""
    import torch
    from workloads import PDA_GRAMMARS

    source, depth = PDA_GRAMMARS["json_nested"]
    pg = cg.PdaGrammar(source, depth)
    pda = cg.Pda(ctx, vocab, pg)
    cfg_rows = torch.zeros((B, depth + 2), dtype=torch.int32, device="cuda").view(torch.uint32)
    counts = torch.zeros(B, dtype=torch.int32, device="cuda").view(torch.uint32)
    bm = torch.empty((B, W), dtype=torch.int32, device="cuda")
    tok = torch.empty(B, dtype=torch.int32, device="cuda")
    tok_u = tok.view(torch.uint32)
    flags = torch.empty(B, dtype=torch.uint8, device="cuda")

    def pstep3(i, logits):
        # the three calls
        pda.fill_bitmask(cfg_rows, bm)
        ctx.mask_and_sample(logits, bm, cfg.temp, cfg.top_p, seed, i, tok)
        pda.accept(cfg_rows, tok_u, flags, counts=counts, max_tokens=2048)

    def pstep2(i, logits):
        # two launches: sampling, then accept of this step with the next step's fill
        ctx.mask_and_sample(logits, bm, cfg.temp, cfg.top_p, seed, i, tok)
        pda.accept_fill(cfg_rows, tok_u, flags, bm, counts=counts, max_tokens=2048)

    def pstep(i, logits):
        # one call, one fused kernel per row: mask, sample, accept
        pda.step(cfg_rows, logits, cfg.temp, cfg.top_p, seed, i, tok_u, flags, counts=counts, max_tokens=2048)

    base = 3 * 10**6
    for i in range(max(args.warmup, 3)):      # every path once before capture (scratch sizing)
        pstep3(base + i, bufs[i % R])
    pda.fill_bitmask(cfg_rows, bm)            # the two-launch form samples from the mask accept_fill wrote
    pstep2(base + 50, bufs[0])
    pstep(base + 51, bufs[1])
    n = min(args.steps, 250)
    g3 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g3, stream=stream, capture_error_mode="thread_local"):
        for i in range(n):
            pstep3(base + 100 + i, bufs[i % R])
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g2, stream=stream, capture_error_mode="thread_local"):
        for i in range(n):
            pstep2(base + 100 + n + i, bufs[i % R])
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
        for i in range(n):
            pstep(base + 100 + 2 * n + i, bufs[i % R])
    g3.replay()   # uploads, and rows move past the first steps
    pda.fill_bitmask(cfg_rows, bm)
    g2.replay()
    g.replay()
    torch.cuda.synchronize()
    if ctx.status() != 0:
        raise RuntimeError("device status after the pushdown warm-up")

    def timed(fn, reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps * 1e3

    step3_us = timed(g3.replay, 1) / n
    pda.fill_bitmask(cfg_rows, bm)
    step2_us = timed(g2.replay, 1) / n
    step_us = timed(g.replay, 1) / n
    levels = cfg_rows.view(torch.int32)[:, 1].float()
    mean_level, max_level = float(levels.mean().item()), int(levels.max().item())
    fill_us = timed(lambda: pda.fill_bitmask(cfg_rows, bm), 200)
    sample_us = timed(lambda: ctx.mask_and_sample(bufs[0], bm, cfg.temp, cfg.top_p, seed, 7, tok), 200)
    # accept alone: the rows are put back before every call (a copy of the
    # configurations and counts), and the copies alone are timed apart
    snap, csnap = cfg_rows.clone(), counts.clone()

    def restore():
        cfg_rows.copy_(snap)
        counts.copy_(csnap)

    def restore_accept():
        restore()
        pda.accept(cfg_rows, tok_u, flags, counts=counts, max_tokens=2048)

    def restore_accept_fill():
        restore()
        pda.accept_fill(cfg_rows, tok_u, flags, bm, counts=counts, max_tokens=2048)

    t_restore = timed(restore, 200)
    accept_us = timed(restore_accept, 200) - t_restore
    accept_fill_us = timed(restore_accept_fill, 200) - t_restore
    # speculative verification (cg_pda_accept_many): drafts of K = 8 tokens from
    # the rows' own next 8 fused steps, verified from the configurations before
    # them (restored before every call)
    K = 8
    draft = torch.empty((B, K), dtype=torch.int32, device="cuda")
    restore()
    for j in range(K):
        pstep(base + 10**5 + j, bufs[j % R])
        draft[:, j] = tok
    dlen = torch.full((B,), K, dtype=torch.int32, device="cuda").view(torch.uint32)
    am_n = torch.empty(B, dtype=torch.int32, device="cuda").view(torch.uint32)
    am_f = torch.empty(B, dtype=torch.uint8, device="cuda")
    draft_u = draft.view(torch.uint32)

    def restore_verify():
        restore()
        pda.accept_many(cfg_rows, draft_u, dlen, am_n, am_f, counts=counts, max_tokens=2048)

    am_us = timed(restore_verify, 200) - t_restore
    am_accepted = float(am_n.view(torch.int32).float().mean().item())
    if ctx.status() != 0:
        raise RuntimeError("device status after the pushdown steps")
    info, ginfo = pda.info(), pg.info()
    peaks = _peaks()
    fill_bytes = B * 8 * W   # the cached mask read and the bitmask written, per row
    achieved = fill_bytes / (fill_us * 1e-6) / 1e9
    step_bytes = B * (V * (2 if cfg.dtype == "bf16" else 4) + W * 4)   # logits and masks read, as cg_step
    step_achieved = step_bytes / (step_us * 1e-6) / 1e9
    return {
        "workload": f"json_nested: recursive JSON grammar, stack bound {depth} frames, V={V}, B={B}, "
                    f"{cfg.dtype} logits as the main workload, T={cfg.temp}, top_p={cfg.top_p}",
        "automaton": {"states": ginfo["n_states"], "rules": ginfo["n_rules"], "columns": ginfo["n_cols"],
                      "cached_masks": info["n_masks"], "keys": info["n_keys"],
                      "cache_bytes": info["cache_bytes"], "per_row_tokens": info["n_candidates"]},
        "step_us": round(step_us, 3),
        "step": "cg_pda_step: mask, sample and accept in one fused kernel per row",
        "tokens_per_s": round(B / (step_us * 1e-6), 1),
        "sample_then_accept_fill_step_us": round(step2_us, 3),
        "three_call_step_us": round(step3_us, 3),
        "steps": n,
        "fill_us_alone": round(fill_us, 3),
        "sample_us_alone": round(sample_us, 3),
        "accept_us_alone": round(accept_us, 3),
        "accept_fill_us_alone": round(accept_fill_us, 3),
        "accept_many_us (drafts of 8 tokens from the next 8 steps)": round(am_us, 3),
        "accept_many_mean_accepted": round(am_accepted, 3),
        "stack_level_after": {"mean": round(mean_level, 2), "max": max_level},
        "step_roofline": {"kernel": "stream_topp_kernel<2> (cg_pda_step)", "bound": "hbm",
                          "achieved": round(step_achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                          "frac": round(step_achieved / peaks["hbm_gbs"], 4), "algorithmic_bytes_per_launch": step_bytes},
        "fill_roofline": {"kernel": "pda_fill_kernel", "bound": "hbm", "achieved": round(achieved, 1),
                          "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                          "algorithmic_bytes_per_launch": fill_bytes},
    }


class OracleBench:
    """The oracle stepping rows of the workload, each on its own trajectory from
    the start state (the logits of a row-step are generated outside the timing)."""

    def __init__(self, cfg_name: str, row_ids):
        from oracle.dfa import compile_grammar
        from oracle.driver import OracleRun, Row
        from workloads import CONFIGS, GRAMMARS, make_vocab
        self.cfg = CONFIGS[cfg_name]
        specs = [GRAMMARS[n] for n in self.cfg.grammars]
        dfas = [compile_grammar(s.kind, s.source, s.bounds) for s in specs]
        toks = make_vocab(self.cfg.vocab_kind, self.cfg.V, self.cfg.vocab_seed)
        self.run = OracleRun(dfas, specs, toks, specs[0].bounds.max_tokens)
        self.rows = [Row(b, b % len(specs)) for b in row_ids]
        self.step_of = [0] * len(self.rows)
        self.spent = 0.0
        self.done = 0

    def row_step(self, i: int) -> None:
        import numpy as np
        from workloads import make_logits
        cfg = self.cfg
        r = self.rows[i]
        x, _ = make_logits(cfg.V, [r.b], self.step_of[i], cfg.logit_seed, cfg.sigma, cfg.boost, cfg.boost_frac,
                           cfg.dtype)
        t = time.perf_counter()
        self.run.step_row(r, x[0].astype(np.float64), cfg.temp, cfg.top_p, cfg.sample_seed, self.step_of[i])
        self.spent += time.perf_counter() - t
        self.step_of[i] += 1
        self.done += 1


ORACLE_ROWS = 4   # rows a worker steps round robin


def _oracle_worker(job):
    """One worker of the CPU sample: rows [first, first + ORACLE_ROWS) of the
    batch, stepped round robin for budget_s seconds of oracle work (or exactly
    n_steps row-steps), after `warm` untimed row-steps."""
    cfg_name, first, budget_s, n_steps, warm = job
    ob = OracleBench(cfg_name, range(first, first + ORACLE_ROWS))
    for k in range(warm):
        ob.row_step(k % ORACLE_ROWS)
    ob.spent, ob.done = 0.0, 0
    t0 = time.perf_counter()
    k = warm
    while (ob.spent < budget_s) if n_steps is None else (ob.done < n_steps):
        ob.row_step(k % ORACLE_ROWS)
        k += 1
    return ob.done, ob.spent, time.perf_counter() - t0


def _oracle_pool(cfg_name: str, workers: int, budget_s, n_steps, warm):
    """The CPU sample on `workers` processes (spawned: no fork after CUDA), each
    on its own rows; returns [(row-steps, oracle seconds, wall seconds)]."""
    import multiprocessing as mp
    jobs = [(cfg_name, ORACLE_ROWS * w, budget_s, n_steps, warm) for w in range(workers)]
    if workers == 1:
        return [_oracle_worker(jobs[0])]
    with mp.get_context("spawn").Pool(workers) as pool:
        return pool.map(_oracle_worker, jobs)


def cpu_baseline(cfg_name: str, budget_s: float = 10.0) -> dict:
    """The oracle as it stands on the host cores: one thread, and one process
    per core the process may use (os.sched_getaffinity), each on 4 rows of its
    own from the start state."""
    cores = len(os.sched_getaffinity(0))
    one = _oracle_pool(cfg_name, 1, budget_s, None, 1)[0]
    allc = _oracle_pool(cfg_name, cores, budget_s, None, 1)
    v1 = one[0] / one[1]
    va = sum(d / w for d, _, w in allc)
    return {"value": round(va, 2), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "nproc": os.cpu_count(),
            "sample": f"{cfg_name}: {cores} processes x {ORACLE_ROWS} rows from the start state, round robin, "
                      f"{budget_s:.0f} s of oracle work each ({sum(d for d, _, _ in allc)} row-steps), float64 "
                      f"numpy; logit generation excluded",
            "single_thread": {"value": round(v1, 2), "cores": 1,
                              "sample": f"{one[0]} row-steps of rows 0..{ORACLE_ROWS - 1}, {one[1]:.1f} s"}}


def run_reference(args) -> dict | None:
    world, rank, _ = _dist()
    if rank != 0:
        return None
    from workloads import CONFIGS
    cfg = CONFIGS[args.config]
    cores = len(os.sched_getaffinity(0))
    # one step = one row-step on each of `cores` processes (the cpu_baseline sample)
    res = _oracle_pool(args.config, cores, None, args.steps, args.warmup)
    done = sum(d for d, _, _ in res)
    wall = max(w for _, _, w in res)
    value = round(done / wall, 2)
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(wall / max(1, args.steps) * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded vocabulary, logits and grammar; no model)",
            "config": {"workload": f"{cfg.name}: V={cfg.V}, B={cfg.B}; each step is a bounded sample: one row-step "
                                   f"on each of {cores} processes ({ORACLE_ROWS} rows each, round robin)",
                       "B": cfg.B, "V": cfg.V},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"{done} row-steps on {cores} processes, {wall:.1f} s wall"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="booking_128k")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--prefix", type=int, default=300, help="untimed steps before the timed window")
    ap.add_argument("--no-workloads", action="store_true", help="skip the other four workloads")
    ap.add_argument("--quick", action="store_true", help="short legs (smoke runs)")
    ap.add_argument("--step-only", action="store_true", help="profiling runs: the timed steps, no other leg")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        out = run_reference(args)
    else:
        out = run_ours(args)
        if out is not None and not args.step_only:
            out["cpu_baseline"] = None if args.no_cpu_baseline else cpu_baseline(args.config)
    if out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()

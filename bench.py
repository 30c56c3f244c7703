#!/usr/bin/env python3
"""Benchmark of one MLA decode step (absorb -> RoPE -> latent decode ->
split-KV combine -> up-projection) on B300.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--impl ours|reference] [--quick] [--rope plain|yarn]

Prints ONE JSON line (rank 0).  By default all five workloads are measured in
one process; the headline (``value``, ``roofline``, ``e2e``, ``append``,
``cpu_baseline``) is the largest single-GPU one, 64 sequences of U[1, 32768]
tokens, and ``per_workload`` holds every workload's step and decode times and
roofline fractions.  ``value`` is device time per step (us, lower is better)
with all inputs resident in HBM and L2 flushed between steps; ``e2e`` is the
same step through the C ABI from pinned host memory (one copy of the packed
query inputs in, one copy of the output back) per step.  ``--workload`` limits
the run to one workload.  ``--impl reference`` times the fp64 CPU oracle on a
bounded sample of the headline workload instead.  Under torchrun every rank
runs an independent replica (no collective on the data path).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import tempfile
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from mla_latent_kv_68_b300.inputs import WORKLOADS, bf16_bits, workload_inputs  # noqa: E402

METRIC = "MLA decode µs/step, cache GB/s and TFLOP/s as fraction of B300 roofline"
# The headline is the largest workload that fits one GPU: 64 sequences of
# U[1, 32768] cached tokens (about 1.2 GB of latent cache).
HEADLINE = "varlen_b64_s1_h128_l1to32768"
NOMINAL_HBM_GBS = 8000.0        # the part's nominal HBM3e bandwidth, reported beside the measured peak
NOMINAL_BF16_TFLOPS = 2250.0    # nominal dense bf16
CACHE_BYTES_PER_TOKEN = (512 + 64) * 2
FLOPS_PER_VISIBLE_TOKEN_PER_HEAD = 2 * 576 + 2 * 512
L2_FLUSH_BYTES = 256 << 20


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 6400.0, 1800.0, 1400.0, "fallback"


def _decode_traffic(name):
    """DRAM bytes per decode launch of workload `name` from the committed ncu
    summary, if the decode kernel's sources are the ones that were profiled
    (else None)."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in ("decode.cuh", "sm100.cuh", "splitkv.cuh"):
        with open(os.path.join(ROOT, "mla_latent_kv_68_b300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    key = h.hexdigest()[:16]
    try:
        with open(os.path.join(ROOT, "profiles", f"decode_kernel_{name}.md")) as f:
            m = re.search(r"traffic-key: ([0-9a-f]+) bytes: (\d+)", f.read())
    except OSError:
        return None
    return int(m.group(2)) if m and m.group(1) == key else None


def _work(x):
    """Algorithmic bytes and flops of the decode kernel and of the whole step."""
    B, S, H = x["B"], x["S"], x["H"]
    L = x["seqlens"].to(torch.int64)
    cache = int(L.sum()) * CACHE_BYTES_PER_TOKEN
    vis = int(sum(int(l) - S + s + 1 for l in L.tolist() for s in range(S)))
    rows = B * S * H
    dec_bytes = cache + rows * 576 * 2 + rows * 512 * 2          # cache + q_cat in + o_lat out
    dec_flops = vis * H * FLOPS_PER_VISIBLE_TOKEN_PER_HEAD
    w_bytes = 2 * H * 128 * 512 * 2
    step_bytes = dec_bytes + w_bytes + rows * (128 + 64 + 128) * 2
    step_flops = dec_flops + 2 * (2 * rows * 128 * 512)
    return dict(dec_bytes=dec_bytes, dec_flops=dec_flops, step_bytes=step_bytes,
                step_flops=step_flops, cache_bytes=cache)


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during timing."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        # raw samples; the summary goes into the JSON line
        log_dir = os.environ.get("MLA_BENCH_LOG_DIR", os.path.join(tempfile.gettempdir(), "mla_bench"))
        self.path = os.path.join(log_dir, f"clocks_rank{index}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def _oracle_sample(x, seconds: float, seed: int = 0, rope: str = "plain"):
    """Time the oracle on a bounded random sample of output rows; return the
    extrapolated whole-step time in us, the thread count and the sample text."""
    import oracle
    kw = {}
    if rope == "yarn":
        kw = dict(rope_theta=oracle.yarn_theta(64), softmax_scale=oracle.yarn_softmax_scale(40.0))
    threads = oracle.num_threads()
    b = {k: bf16_bits(x[k]) for k in ("q_nope", "q_rope", "c_kv", "k_r", "W_UK", "W_UV")}
    total = x["B"] * x["S"] * x["H"]
    rng = np.random.default_rng(seed)
    L = x["seqlens"].numpy().astype(np.int64)
    per_row_tokens = np.repeat(L, x["S"] * x["H"]).astype(np.float64)
    # probe one batch of `threads` rows, then size the sample to about `seconds`
    n = min(total, threads)
    rows = rng.choice(total, n, replace=False)
    t0 = time.perf_counter()
    oracle.decode(b["q_nope"], b["q_rope"], b["c_kv"], b["k_r"], b["W_UK"], b["W_UV"],
                  x["seqlens"].numpy(), rows=rows, **kw)
    dt = time.perf_counter() - t0
    if dt < seconds and n < total:
        n2 = int(min(total, max(n, n * seconds / max(dt, 1e-3))))
        rows = rng.choice(total, n2, replace=False)
        t0 = time.perf_counter()
        oracle.decode(b["q_nope"], b["q_rope"], b["c_kv"], b["k_r"], b["W_UK"], b["W_UV"],
                      x["seqlens"].numpy(), rows=rows, **kw)
        dt = time.perf_counter() - t0
        n = n2
    # extrapolate by visible tokens (the oracle's cost is linear in them)
    frac = per_row_tokens[rows].sum() / per_row_tokens.sum()
    us = dt / frac * 1e6
    return us, threads, (f"{n} of {total} output rows (random, seeded), {dt:.1f} s wall; "
                         f"scaled by visible-token share {frac:.4f}")


def run_reference(args, rank, world):
    if rank != 0:
        return
    name = args.workload or HEADLINE
    x = workload_inputs(name)
    per_step = []
    for i in range(args.warmup + args.steps):
        us, threads, sample = _oracle_sample(x, seconds=args.ref_seconds, seed=i, rope=args.rope)
        if i >= args.warmup:
            per_step.append(us)
    v = statistics.mean(per_step)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(v, 3), "unit": "us/step",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(v / 1000, 3), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": _config(args, name, x),
        "cpu_baseline": {"value": round(v, 3), "unit": "us/step", "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(v, 3), "unit": "us/step", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _config(args, name, x):
    w = WORKLOADS[name]
    return {"workload": name, "B": w.B, "S": w.S, "H": w.H,
            "L": w.L if w.L is not None else f"U[{w.L_range[0]},{w.L_range[1]}]",
            "sum_L": int(x["seqlens"].sum()), "d_c": 512, "d_rope": 64,
            "l2": "flushed between timed steps (256 MiB write, then 256 MiB read)",
            "parallelism": f"replicas x{args.gpus}" if args.gpus > 1 else "single GPU",
            "rope": ("yarn (s=40, alpha=1, beta=32, original 4096; score scale 0.1 ln s + 1)"
                     if getattr(args, "rope", "plain") == "yarn" else "plain (base 10000)")}


APPEND_D = 7168  # hidden size of the appended tokens (the pages leave d unstated)


def _time_append(args, x, d, dev, stream, flush_l2, theta, mb):
    """The cache-append step (next to the decode step, not part of its time):
    the step's B*S new tokens, c = W^DKV h and k^R = RoPE(W^KR h) written at
    their positions, recorded in a graph and replayed after an L2 flush."""
    B, S = x["B"], x["S"]
    g = torch.Generator().manual_seed(68100)
    h = torch.randn(B, S, APPEND_D, generator=g).to(torch.bfloat16).to(dev)
    wd = (torch.randn(512, APPEND_D, generator=g) / APPEND_D ** 0.5).to(torch.bfloat16).to(dev)
    wr = (torch.randn(64, APPEND_D, generator=g) / APPEND_D ** 0.5).to(torch.bfloat16).to(dev)
    ws = mb.cache_append_workspace(B, S, APPEND_D, device=dev)
    call = (h, wd, wr, d["seqlens"], d["c_kv"], d["k_r"], ws)
    for _ in range(max(3, args.warmup)):
        mb.cache_append(*call, theta=theta)
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr):
        mb.cache_append(*call, theta=theta)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    torch.cuda.synchronize(dev)
    for e in ev:
        flush_l2()
        e[0].record(stream)
        gr.replay()
        e[1].record(stream)
    torch.cuda.synchronize(dev)
    if mb.read_status(ws) != mb.MLA_OK:
        raise RuntimeError("device status not clean after the cache-append steps")
    us = statistics.mean(e[0].elapsed_time(e[1]) for e in ev) * 1000
    nbytes = (512 + 64) * APPEND_D * 2 + B * S * APPEND_D * 2 + B * S * (512 + 64) * 2
    return {"workload": f"B={B} S={S} new tokens, d={APPEND_D}", "us": round(us, 3), "bytes": nbytes,
            "launches": 1, "form": "one cooperative launch (GEMM, grid barrier, finalize)"}


class Packed:
    """One pinned host buffer and one device buffer holding a step's inputs
    (q_nope, q_rope, seqlens) back to back, 256-byte aligned, so that the
    end-to-end step moves its inputs with a single host-to-device copy.  The
    device views are the tensors the step (and its graphs) read."""

    def __init__(self, x, dev):
        parts = [("q_nope", x["q_nope"]), ("q_rope", x["q_rope"]), ("seqlens", x["seqlens"])]
        offs, off = [], 0
        for _, t in parts:
            offs.append(off)
            off = (off + t.numel() * t.element_size() + 255) // 256 * 256
        self.nbytes = off
        self.host = torch.empty(off, dtype=torch.uint8).pin_memory()
        self.dev = torch.empty(off, dtype=torch.uint8, device=dev)
        self.views = {}
        for (name, t), o in zip(parts, offs):
            n = t.numel() * t.element_size()
            self.host[o:o + n].view(t.dtype).view(t.shape).copy_(t)
            self.views[name] = self.dev[o:o + n].view(t.dtype).view(t.shape)
        self.dev.copy_(self.host)


def _roofline(wk, dec_us, hbm, tf_burst):
    """Roofline of the decode kernel: the slower of its algorithmic bytes at
    measured HBM bandwidth and its flops at the measured bf16 burst peak."""
    t_hbm = wk["dec_bytes"] / (hbm * 1e3)          # us
    t_tc = wk["dec_flops"] / (tf_burst * 1e6)      # us
    bound = "hbm" if t_hbm >= t_tc else "tensor"
    return bound, max(t_hbm, t_tc)


def measure_workload(name, args, world, dev, stream, flush_l2, mb, headline=False):
    """Time one workload's step (and its three phases) as K graph replays after
    an L2 flush each; for the headline also the end-to-end step, the cache
    append and the CPU oracle."""
    x = workload_inputs(name)
    theta = mb.yarn_frequencies() if args.rope == "yarn" else None
    scale = mb.yarn_softmax_scale() if args.rope == "yarn" else mb.SOFTMAX_SCALE
    pk = Packed(x, dev)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v)
         for k, v in x.items() if k not in ("q_nope", "q_rope", "seqlens")}
    d.update(pk.views)
    mb.rope_cache(d["k_r"], d["seqlens"], theta=theta)  # cache fill: keys rotated once (untimed)
    step = mb.DecodeStep(x["B"], x["S"], x["H"], device=dev, rope_theta=theta, softmax_scale=scale)
    args_step = (d["q_nope"], d["q_rope"], d["c_kv"], d["k_r"], d["seqlens"], d["W_UK"], d["W_UV"])
    for _ in range(args.warmup):
        step(*args_step)
    if mb.read_status(step.workspace) != mb.MLA_OK:
        raise RuntimeError(f"{name}: device status not clean after warm-up")
    # CUDA graphs of the library calls: the whole step, and its three phases
    g_all = step.capture(step, *args_step)
    g_q = step.capture(step.queries, d["q_nope"], d["q_rope"], d["seqlens"], d["W_UK"])
    g_a = step.capture(step.attend, d["c_kv"], d["k_r"], d["seqlens"])
    g_p = step.capture(step.project, d["W_UV"])
    for _ in range(args.warmup):
        g_all.replay()

    def timed(body, n_events):
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(n_events)]
              for _ in range(args.steps)]
        _barrier(world)
        torch.cuda.synchronize(dev)
        for i in range(args.steps):
            flush_l2()             # L2 flush between steps; the host runs ahead meanwhile
            body(ev[i])
        torch.cuda.synchronize(dev)
        _barrier(world)
        return ev

    def mean_us(ev, a, b):
        return _max_over_ranks(statistics.mean(e[a].elapsed_time(e[b]) for e in ev) * 1000, world)

    ev_all = timed(lambda e: (e[0].record(stream), g_all.replay(), e[1].record(stream)), 2)
    ev_ph = timed(lambda e: (e[0].record(stream), g_q.replay(), e[1].record(stream),
                             g_a.replay(), e[2].record(stream), g_p.replay(),
                             e[3].record(stream)), 4)
    if mb.read_status(step.workspace) != mb.MLA_OK:
        raise RuntimeError(f"{name}: device status not clean after the timed steps")
    r = {"x": x, "step_us": mean_us(ev_all, 0, 1), "q_us": mean_us(ev_ph, 0, 1),
         "dec_us": mean_us(ev_ph, 1, 2), "p_us": mean_us(ev_ph, 2, 3)}
    if headline:
        # end to end through the public API from pinned host memory: one copy
        # of the packed inputs in, the step's graph, one copy of the output back
        hout = torch.empty(step.out.shape, dtype=torch.bfloat16).pin_memory()

        def e2e_body(e, replay=True):
            e[0].record(stream)
            pk.dev.copy_(pk.host, non_blocking=True)
            if replay:
                g_all.replay()
            else:
                step(*args_step)
            hout.copy_(step.out, non_blocking=True)
            e[1].record(stream)

        r["e2e_us"] = mean_us(timed(e2e_body, 2), 0, 1)
        r["eager_us"] = mean_us(timed(lambda e: e2e_body(e, replay=False), 2), 0, 1)
        r["h2d"], r["d2h"] = pk.nbytes, hout.numel() * 2
        r["append"] = _time_append(args, x, d, dev, stream, flush_l2, theta, mb)
        r["oproj"] = _time_output_project(args, x, dev, stream, flush_l2, mb)
        r["prefill"] = _time_prefill(args, dev, stream, flush_l2, mb)
    del g_all, g_q, g_a, g_p, step, d, pk
    torch.cuda.empty_cache()
    return r


def _time_output_project(args, x, dev, stream, flush_l2, mb):
    """The layer's output projection after the step (not part of its time):
    u = W^O [o_1; ...; o_H] for the step's B*S tokens, W^O [7168, H*128]
    bf16, recorded in a graph and replayed after an L2 flush."""
    B, S, H = x["B"], x["S"], x["H"]
    BS, K = B * S, H * 128
    g = torch.Generator().manual_seed(68200)
    xo = torch.randn(BS, K, generator=g).to(torch.bfloat16).to(dev)
    W = (torch.randn(APPEND_D, K, generator=g) / K ** 0.5).to(torch.bfloat16).to(dev)
    u = torch.empty(BS, APPEND_D, dtype=torch.bfloat16, device=dev)
    ws = mb.output_project_workspace(BS, K, APPEND_D, device=dev)
    for _ in range(max(3, args.warmup)):
        mb.output_project(xo, W, u, ws)
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr):
        mb.output_project(xo, W, u, ws)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    torch.cuda.synchronize(dev)
    for e in ev:
        flush_l2()
        e[0].record(stream)
        gr.replay()
        e[1].record(stream)
    torch.cuda.synchronize(dev)
    if mb.read_status() != mb.MLA_OK:
        raise RuntimeError("device status not clean after the output projection")
    us = statistics.mean(e[0].elapsed_time(e[1]) for e in ev) * 1000
    nbytes = APPEND_D * K * 2 + BS * K * 2 + BS * APPEND_D * 2
    del W, xo, u, ws
    torch.cuda.empty_cache()
    return {"workload": f"{BS} tokens, W^O [{APPEND_D}, {K}]", "us": round(us, 3), "bytes": nbytes,
            "launches": 2}


PREFILL = dict(name="prefill_b4_s4096_h128", B=4, S=4096, H=128)


def _time_prefill(args, dev, stream, flush_l2, mb, batch=None):
    """Prefill of whole prompts (not part of the decode step): B prompts of S
    tokens, every position querying the cache up to itself.  Times the three
    phases (RoPE of the queries, expansion of keys and values per head, causal
    attention) in one graph, and the attention alone in another, each after an
    L2 flush.  Algorithmic flops: 2 x 2 x (B S) x (H 128) x 512 for the
    expansion and 2 x (192 + 128) x H per visible (query, key) pair."""
    from mla_latent_kv_68_b300.inputs import make_inputs
    B, S, H = batch or PREFILL["B"], PREFILL["S"], PREFILL["H"]
    x = make_inputs(B, S, H, [S] * B, seed=68005)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    mb.rope_cache(d["k_r"], d["seqlens"])
    step = mb.PrefillStep(B, S, H, S, device=dev)
    run = lambda: step(d["q_nope"], d["q_rope"], d["c_kv"], d["k_r"], d["seqlens"], d["W_UK"], d["W_UV"])
    attn = lambda: mb.prefill_attention(d["q_nope"], step.q_rot, step.k_c, d["k_r"], step.v_c, d["seqlens"],
                                        step.out)
    for _ in range(max(3, args.warmup)):
        run()
    graphs = []
    for fn in (run, attn):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            fn()
        graphs.append(gr)
    times = []
    for gr in graphs:
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(min(args.steps, 10))]
        torch.cuda.synchronize(dev)
        for e in ev:
            flush_l2()
            e[0].record(stream)
            gr.replay()
            e[1].record(stream)
        torch.cuda.synchronize(dev)
        times.append(statistics.mean(e[0].elapsed_time(e[1]) for e in ev) * 1000)
    if mb.read_status() != mb.MLA_OK:
        raise RuntimeError("device status not clean after the prefill")
    pairs = B * H * S * (S + 1) // 2
    f_attn = pairs * 2 * (192 + 128)
    f_exp = 2 * 2 * B * S * H * 128 * 512
    _, tf_burst, _, _ = _peaks()
    del graphs, step, d, x
    torch.cuda.empty_cache()
    total_us, attn_us = times
    name = PREFILL["name"] if B == PREFILL["B"] else f"prefill_b{B}_s{S}_h{H}"
    return {"workload": f"{name}: {B} prompts of {S} tokens, {H} heads, causal",
            "us": round(total_us, 3), "attention_us": round(attn_us, 3),
            "flops": f_attn + f_exp, "attention_flops": f_attn,
            "tflops": round((f_attn + f_exp) / (total_us * 1e-6) / 1e12, 1),
            "attention_tflops": round(f_attn / (attn_us * 1e-6) / 1e12, 1),
            "frac": round((f_attn + f_exp) / (total_us * 1e-6) / 1e12 / tf_burst, 4),
            "attention_frac": round(f_attn / (attn_us * 1e-6) / 1e12 / tf_burst, 4),
            "peak_tflops": tf_burst, "launches": 3}


def run_ours(args, rank, world, local_rank):
    from mla_latent_kv_68_b300 import binding as mb

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    mb.lib()
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_read = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_sink = torch.empty(1, dtype=torch.float32, device=dev)

    def flush_l2():
        """Write a buffer twice the size of L2, then read another one, so that
        no line of the inputs stays cached and no dirty line of the flush is
        left to be written back inside the timed step."""
        flush.zero_()
        torch.sum(flush_read.view(1, -1), dim=1, out=flush_sink)

    names = [args.workload] if args.workload else [HEADLINE] + [n for n in WORKLOADS if n != HEADLINE]
    head = names[0]
    res = {}
    with ClockSampler(local_rank) as clocks:
        for n in names:
            res[n] = measure_workload(n, args, world, dev, stream, flush_l2, mb, headline=(n == head))
    if rank != 0:
        return
    hbm, tf_burst, tf_sust, src = _peaks()
    per = {}
    for n in names:
        r = res[n]
        wk = _work(r["x"])
        bound, t_roof = _roofline(wk, r["dec_us"], hbm, tf_burst)
        t_step_roof = max(wk["step_bytes"] / (hbm * 1e3), wk["step_flops"] / (tf_burst * 1e6))
        per[n] = {"step_us": round(r["step_us"], 3), "queries_us": round(r["q_us"], 3),
                  "decode_us": round(r["dec_us"], 3), "combine_project_us": round(r["p_us"], 3),
                  "decode_bound": bound, "decode_roofline_us": round(t_roof, 3),
                  "decode_frac": round(t_roof / r["dec_us"], 4),
                  "decode_hbm_gbs": round(wk["dec_bytes"] / (r["dec_us"] * 1e-6) / 1e9, 1),
                  "decode_tflops": round(wk["dec_flops"] / (r["dec_us"] * 1e-6) / 1e12, 1),
                  "step_roofline_us": round(t_step_roof, 3),
                  "step_frac": round(t_step_roof / r["step_us"], 4)}
    r = res[head]
    wk = _work(r["x"])
    bound, t_roof = _roofline(wk, r["dec_us"], hbm, tf_burst)
    if bound == "hbm":
        achieved = wk["dec_bytes"] / (r["dec_us"] * 1e-6) / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(achieved / hbm, 4),
                "frac_vs_nominal": round(achieved / NOMINAL_HBM_GBS, 4), "nominal_peak": NOMINAL_HBM_GBS}
    else:
        achieved = wk["dec_flops"] / (r["dec_us"] * 1e-6) / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": tf_burst, "unit": "TFLOP/s",
                "frac": round(achieved / tf_burst, 4),
                "frac_vs_nominal": round(achieved / NOMINAL_BF16_TFLOPS, 4),
                "nominal_peak": NOMINAL_BF16_TFLOPS}
    roof.update({"kernel": "mla_decode (the decode kernel, which plans its own split)",
                 "traffic": _decode_traffic(head), "peak_source": src,
                 "algorithmic_bytes": wk["dec_bytes"], "algorithmic_flops": wk["dec_flops"],
                 "launch_us": round(r["dec_us"], 3)})
    app = r["append"]
    line = {
        "metric": METRIC, "value": round(r["step_us"], 3), "unit": "us/step", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(r["step_us"] / 1000, 5),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; random-init weights of the pages' MLA dimensions)",
        "config": _config(args, head, r["x"]),
        "roofline": roof,
        "kernels": {"queries_us": round(r["q_us"], 3), "decode_us": round(r["dec_us"], 3),
                    "combine_project_us": round(r["p_us"], 3), "step_us": round(r["step_us"], 3),
                    "step_roofline_us": per[head]["step_roofline_us"],
                    "algorithmic_decode_bytes": wk["dec_bytes"],
                    "algorithmic_decode_flops": wk["dec_flops"]},
        "per_workload": per,
        "e2e": {"value": round(r["e2e_us"], 3), "unit": "us/step", "h2d_bytes_per_step": r["h2d"],
                "d2h_bytes_per_step": r["d2h"],
                "path": "pinned host -> one H2D copy of the packed inputs -> step graph -> one D2H copy",
                "eager_calls_value": round(r["eager_us"], 3)},
        "append": {**app, "achieved_gbs": round(app["bytes"] / (app["us"] * 1e-6) / 1e9, 1),
                   "frac": round(app["bytes"] / (app["us"] * 1e-6) / 1e9 / hbm, 4)},
        "output_projection": {**r["oproj"],
                              "achieved_gbs": round(r["oproj"]["bytes"] / (r["oproj"]["us"] * 1e-6) / 1e9, 1),
                              "frac": round(r["oproj"]["bytes"] / (r["oproj"]["us"] * 1e-6) / 1e9 / hbm, 4)},
        "prefill": r["prefill"],
        "gpu_launches": mb.DecodeStep.LAUNCHES_PER_STEP * args.steps,
        "clocks": clocks.summary(),
    }
    if not args.quick and world == 1:
        us, threads, sample = _oracle_sample(r["x"], seconds=args.ref_seconds, rope=args.rope)
        line["cpu_baseline"] = {"value": round(us, 1), "unit": "us/step", "cores": threads,
                                "kind": "oracle", "sample": sample, "workload": head}
    print(json.dumps(line), flush=True)


def _barrier(world):
    if world > 1:
        torch.distributed.barrier()


def _max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    t = torch.tensor([v], dtype=torch.float64,
                     device="cuda" if torch.distributed.get_backend() == "nccl" else "cpu")
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=None, choices=list(WORKLOADS),
                    help="measure only this workload (default: all five, headline first)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--quick", action="store_true", help="skip the CPU-baseline timing")
    ap.add_argument("--ref-seconds", type=float, default=12.0)
    ap.add_argument("--rope", default="plain", choices=["plain", "yarn"],
                    help="RoPE frequencies of the step (yarn: the long-context setting)")
    ap.add_argument("--prefill-only", action="store_true",
                    help="measure only the prefill (its JSON object), for profiling")
    ap.add_argument("--prefill-batch", type=int, default=PREFILL["B"],
                    help="prompts of the prefill workload (4096 tokens each)")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be >= 3")
    if args.prefill_only:
        from mla_latent_kv_68_b300 import binding as mb
        dev = torch.device("cuda", 0)
        mb.lib()
        flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        print(json.dumps(_time_prefill(args, dev, torch.cuda.current_stream(dev), flush.zero_, mb,
                                       batch=args.prefill_batch)), flush=True)
        return 0

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        if args.impl == "reference" and rank != 0:
            return 0
        if args.impl == "ours":
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if backend == "nccl":
                torch.cuda.set_device(local_rank)
            torch.distributed.init_process_group(backend)
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local_rank)
    if world > 1 and args.impl == "ours":
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())

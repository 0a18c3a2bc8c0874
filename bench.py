#!/usr/bin/env python
"""Decode-attention throughput of the FADE tiered KV cache on one GB300 per rank.

Workload (default): the Llama-3-8B-shaped aggressive-mode sweep — 32 layers, batch 64,
32 query / 8 KV heads, head_dim 128, 32768-token context per row, n_sink 4, recent window 64,
middle tier INT4 K / INT2 V (group 32, fp16 scales), position eviction to int4_budget 4096.
Synthetic seeded data (no weights, no dataset).

A timed step is one pass of the whole hot path over all layers: RoPE of the step's q and k,
demote + quantise-pack, evict + re-RoPE, append, split-KV decode attention + combine (and
H2O/EMA accumulation for the policies that use it). ``value`` = batch x steps x ranks /
(max over ranks of the device time of the timed steps). The compressed cache (8 GB) is far
larger than L2, so no L2 flush is needed between steps.

Besides the contract keys, the line carries: ``roofline_by_call`` (attention and eviction,
and score accumulation under H2O / EMA, each against its bound, with the recorded DRAM
traffic of the current sources), ``attention_only`` (decode-attention tokens/s),
``per_step_ms`` (median and p90 of separately timed steps), ``per_call_overlapped_ms``, and
``cpu_baseline``. Options: ``--workload`` (1, 2, 3, 4, 5, 5b), ``--v-codec pq`` (product-
quantised middle V), ``--shared-rows`` (batch-shared tier decisions), ``--no-graph``,
``--no-pipeline``, ``--side-streams``.

--impl reference runs the oracle (plain numpy CPU restatement of the method) on the same
workload: one single-threaded process per host core, each stepping one full-size (layer,
row, KV head) unit, the unit time scaled to a whole step by the number of units.
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

METRIC = "decode-attn tokens/s (batch×steps) and achieved HBM GB/s vs GB300 peak"
PQ_CALIB_ROWS, PQ_ITERS = 4096, 8   # --v-codec pq: calibration rows and k-means rounds
_T0 = time.perf_counter()


def progress(msg):
    """Stage marks on stderr (stdout carries only the JSON line)."""
    print(f"[bench +{time.perf_counter() - _T0:7.1f}s] {msg}", file=sys.stderr, flush=True)


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="4")
    p.add_argument("--layers", type=int, default=None,
                   help="override the layer count (profiling captures only; the headline "
                        "line always runs every layer of the workload)")
    p.add_argument("--batch", type=int, default=None,
                   help="override the batch (profiling captures of a reduced case only)")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-graph", action="store_true", help="launch every kernel (no CUDA graph)")
    p.add_argument("--side-streams", type=int, default=0,
                   help="streams that take the layers' maintenance in turn (pipelined schedule); "
                        "0 = one when a layer's middle tier fills the GPU (at least 2^20 "
                        "token-heads), else two")
    p.add_argument("--shared-rows", action="store_true",
                   help="the rows share their tier decisions (row-summed scores; rows of equal "
                        "length)")
    p.add_argument("--v-codec", default="int", choices=["int", "pq"],
                   help="middle-tier V: INT codes with scales, or product-quantised (a codebook "
                        "trained on the GPU from synthetic calibration rows before timing)")
    p.add_argument("--k-bits", type=int, default=None, choices=[2, 4],
                   help="middle-tier K code width instead of the workload's (a custom variant "
                        "of the workload, named with a _k<bits> suffix; no CPU baseline)")
    p.add_argument("--no-pipeline", action="store_true",
                   help="in the graph, run each layer's maintenance before its attention instead "
                        "of overlapping it with the following layers")
    p.add_argument("--no-cpu-baseline", action="store_true")
    return p.parse_args()


def workload(key):
    from synth import get_workload

    return get_workload(int(key) if key.isdigit() else key)


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples (every 200 ms) while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
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
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- bytes
def mid_token_bytes(cfg):
    """Bytes of one middle token: packed K with its scales, and V as INT codes with scales or
    as d/4 PQ code bytes (the per-layer codebook comes from L2, not counted per token)."""
    d = cfg.head_dim
    if cfg.v_codec == "pq":
        return d * cfg.middle_k_bits // 8 + 2 * (d // 32) + d // 4
    return d * (cfg.middle_k_bits + cfg.middle_v_bits) // 8 + 2 * 2 * (d // 32)


def attention_bytes(cfg, layer):
    """Algorithmic bytes of one fade_decode_attention call: every held token once (middle at
    its packed size with scales, FP16 tiers at 4d) plus q read and out written."""
    d = cfg.head_dim
    mid_tok = mid_token_bytes(cfg)
    units_fp16 = int((layer.h_n_sink + layer.h_n_recent).sum()) * cfg.num_kv_heads
    units_mid = int(layer.h_n_mid.sum()) * cfg.num_kv_heads
    return units_mid * mid_tok + units_fp16 * 4 * d + 2 * cfg.batch * cfg.num_q_heads * d * 2


def accumulate_bytes(cfg, layer):
    """Algorithmic bytes of one fade_h2o_accumulate call: each held token's G logits read and
    its score read and written, plus the (M, L) of every query head."""
    held = int((layer.h_n_sink + layer.h_n_mid + layer.h_n_recent).sum()) * cfg.num_kv_heads
    G = cfg.num_q_heads // cfg.num_kv_heads
    return held * (4 * G + 8) + cfg.batch * cfg.num_q_heads * 8


def evict_bytes(cfg, layer, n_ev=1):
    """Algorithmic bytes of one steady-state fade_evict_rerope call: the middle tier (codes,
    scales, scores) read once and its survivors written once to the other buffer, plus the
    recent keys read and rewritten in place."""
    d = cfg.head_dim
    mid_tok = mid_token_bytes(cfg) + 4
    H = cfg.num_kv_heads
    n_mid_after = int(layer.h_n_mid.sum())
    read = (n_mid_after + n_ev * cfg.batch) * mid_tok * H
    write = n_mid_after * mid_tok * H
    rec = int(layer.h_n_recent.sum()) * H * d * 2 * 2
    return read + write + rec


# DRAM bytes per launch from an ncu capture (profiles/dram_traffic.json), keyed by the SHA-256
# of the kernel sources they were taken on: a figure whose sources changed is reported as null.
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.json")
CSRC = os.path.join(ROOT, "tiered_mixed_precision_gb300", "csrc")
TRAFFIC_SOURCES = {
    "attention": ["attention_mma.cuh", "attention_mma.cu", "attention_mma_k2.cu", "attention.cu",
                  "fade_internal.cuh"],
    "evict_rerope": ["cache.cu", "fade_internal.cuh"],
}


def sources_sha256(call):
    import hashlib

    h = hashlib.sha256()
    for f in TRAFFIC_SOURCES[call]:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def measured_traffic(call, workload_name):
    try:
        rec = json.load(open(TRAFFIC_FILE))[call]
    except (OSError, ValueError, KeyError):
        return None
    if rec.get("workload") != workload_name or rec.get("sources_sha256") != sources_sha256(call):
        return None
    return rec.get("dram_bytes_per_launch")


# fp32 operations the method performs per re-positioned key (head_dim d): dequantise d codes
# (one multiply each), un-RoPE and re-RoPE (d/2 pairs x 2 rotations x 4 multiplies + 2 adds),
# the fp16 cast (d), the group absmax (d comparisons), the requantising division and rounding
# (2 d). Recent-ring keys are fp16 (no dequantisation or requantisation): rotations and cast.
def evict_alu_ops(cfg, layer):
    d = cfg.head_dim
    mid_key = d + 2 * (d // 2) * 6 + d + d + 2 * d
    rec_key = 2 * (d // 2) * 6 + d
    H = cfg.num_kv_heads
    n_mid = int(layer.h_n_mid.sum()) * H
    n_rec = int(layer.h_n_recent.sum()) * H
    return n_mid * mid_key + n_rec * rec_key


def alu_peak_derived(dev, peaks):
    """The same rate from unit counts and clocks: SMs x 128 fp32 lanes x the maximum SM
    clock (T operations/s), reported beside the measured one."""
    import torch

    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    mhz = (peaks or {}).get("sm_max_mhz", 2070.0)
    return sms * 128 * mhz * 1e6 / 1e12


def alu_peak_tops(dev):
    """The device's rate of separately rounded fp32 operations, measured: a library kernel
    runs independent chains of packed fp32 multiplies (the form the re-positioning arithmetic
    uses) on registers, 8 CTAs of 256 threads per SM; best of 5 timed launches (CUDA events,
    after 2 warm-up launches). Returns (T operations/s, description)."""
    import torch

    from tiered_mixed_precision_gb300 import fade as F

    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    sink = torch.zeros(256, dtype=torch.float32, device=dev)
    blocks, iters = 8 * sms, 4096
    for _ in range(2):
        F.fade_measure_fp32_rate(blocks, iters, sink)
    best = None
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        ops = F.fade_measure_fp32_rate(blocks, iters, sink)
        e1.record()
        e1.synchronize()
        r = ops / (e0.elapsed_time(e1) / 1e3) / 1e12
        best = r if best is None else max(best, r)
    return best, (f"measured: packed fp32 multiply chains (mul.rn.f32x2), {blocks} CTAs x 256 "
                  f"threads, best of 5 CUDA-event timings")


def load_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        return None


# ----------------------------------------------------------------------------- CPU oracle
_CPU_SNIPPET = r"""
import json, sys, time
sys.path.insert(0, {root!r})
import numpy as np
from oracle.cache import Params, UnitCache
from oracle.rope import RopeTable
from synth import draw_vectors, get_workload
wl = get_workload({key!r})
P = int({P})
u = UnitCache(Params.from_workload(wl), RopeTable.from_workload(wl, P + 4096))
k = draw_vectors(wl, "k", (P, wl.head_dim), "cpu_sample", {worker})
v = draw_vectors(wl, "v", (P, wl.head_dim), "cpu_sample", {worker})
u.prefill(k, v, mass=np.ones(P) if wl.policy == "h2o" else None)
steps, warm, budget_s = {steps}, {warmup}, {budget_s}
G = wl.group
times = []
i = 0
t_start = time.perf_counter()
while True:
    q = draw_vectors(wl, "q", (G, wl.head_dim), "cpu_step", {worker}, i)
    kk = draw_vectors(wl, "k", (wl.head_dim,), "cpu_step", {worker}, i)
    vv = draw_vectors(wl, "v", (wl.head_dim,), "cpu_step", {worker}, i)
    t0 = time.perf_counter()
    u.step(q, kk, vv)
    dt = time.perf_counter() - t0
    if i >= warm:
        times.append(dt)
    i += 1
    if len(times) >= steps or (time.perf_counter() - t_start > budget_s and len(times) >= 1):
        break
print(json.dumps({{"unit_step_s": float(np.mean(times)), "n": len(times)}}))
"""


def run_oracle_sample(key, steps, warmup, budget_s=25.0, workers=None):
    """The oracle's decode step on the host cores: one single-threaded process per core, each
    stepping its own full-size (layer, row, KV head) unit (units are independent), all at
    once; the mean per-unit step time under that load, times the units of a whole step and
    divided by the processes, gives the whole-step time."""
    wl = workload(key)
    P = wl.ragged[1] if wl.ragged else wl.prompt_len
    if workers is None:
        workers = max(1, int(os.environ.get("FADE_CPU_WORKERS", os.cpu_count() or 1)))
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    procs = []
    for w in range(workers):
        code = _CPU_SNIPPET.format(root=ROOT, key=key if not key.isdigit() else int(key), P=P,
                                   steps=steps, warmup=warmup, budget_s=budget_s, worker=w)
        procs.append(subprocess.Popen([sys.executable, "-c", code], stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True, env=env))
    res = []
    for pr in procs:
        out, err = pr.communicate(timeout=900)
        if pr.returncode != 0:
            raise RuntimeError("oracle sample failed: " + err[-2000:])
        res.append(json.loads(out.strip().splitlines()[-1]))
    unit_step_s = float(np.mean([r["unit_step_s"] for r in res]))
    n = min(r["n"] for r in res)
    units = wl.layers * wl.batch * wl.num_kv_heads
    step_s = unit_step_s * units / workers
    return {
        "value": wl.batch / step_s, "unit": "tokens/s", "cores": workers, "kind": "oracle",
        "sample": (f"{n} decode steps of one full-size (layer, row, KV head) unit (prompt {P}) "
                   f"in each of {workers} single-threaded processes running at once (one per "
                   f"host core); mean unit-step time x {units} units / {workers} = one whole "
                   f"step"),
        "ms_per_step": step_s * 1e3,
    }


# ----------------------------------------------------------------------------- GPU arm
def run_ours(args, rank, world):
    import torch

    from tiered_mixed_precision_gb300 import Config, build
    from tiered_mixed_precision_gb300.model import FadeCache
    from synth import draw_prompt, draw_vectors, ragged_context_lengths
    from synth.draws import pq_calibration, pq_init_indices

    build.build()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    wl = workload(args.workload)
    if world > 1:
        wl = wl.scaled(seed=wl.seed + 1000 * rank)   # weak scaling: each rank its own batch
    if args.layers:
        wl = wl.scaled(layers=args.layers)
    if args.batch:
        wl = wl.scaled(batch=args.batch)
    if args.k_bits:
        wl = wl.scaled(middle_k_bits=args.k_bits, name=f"{wl.name}_k{args.k_bits}")
    lens = ragged_context_lengths(wl)
    maxP = int(lens.max())
    K, W = args.steps, args.warmup
    # timed, per-step spread, e2e, a possible eager timing pass, probe and warm-up
    nsteps = 4 * K + W + 8
    if wl.policy != "none" and wl.int4_budget >= 0:
        cfg = Config.from_workload(wl)
    else:  # without eviction the middle tier grows by one token per step
        cfg = Config.from_workload(
            wl, mid_capacity=max(1, maxP + nsteps - wl.n_sink - wl.recent_window))
    if args.shared_rows:
        import dataclasses

        cfg = dataclasses.replace(cfg, shared_rows=True)
    if args.v_codec == "pq":
        import dataclasses

        cfg = dataclasses.replace(cfg, v_codec="pq")
    max_pos = maxP + nsteps + 16
    fc = FadeCache(cfg, wl.layers, maxP, max_pos, dev)
    progress(f"cache allocated: {wl.name}, {wl.layers} layers")
    if args.v_codec == "pq":   # one codebook, trained on the GPU, shared by every layer
        calib = pq_calibration(wl, PQ_CALIB_ROWS, backend="torch", device=dev)
        fc.train_pq_codebook(calib, pq_init_indices(PQ_CALIB_ROWS, wl.seed), PQ_ITERS)
        del calib
        progress("PQ codebook trained")
    h2o = wl.policy == "h2o" and wl.int4_budget >= 0
    for layer in range(wl.layers):
        # H2O: the prefill attention mass is computed on the GPU from the prompt's queries
        pr = draw_prompt(wl, layer, maxP, with_q=h2o, backend="torch", device=dev)
        fc.prefill(layer, pr["k"], pr["v"], lens, None, q_raw=pr.get("q"))
        del pr
    torch.cuda.synchronize()
    torch.cuda.empty_cache()   # drop the prompt draws: only the cache stays resident
    progress("prefill done")
    L, B, Hq, Hkv, d = wl.layers, wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.head_dim
    q_all = draw_vectors(wl, "q", (K + W, L, B, Hq, d), "bench", backend="torch", device=dev)
    k_all = draw_vectors(wl, "k", (K + W, L, B, Hkv, d), "bench", backend="torch", device=dev)
    v_all = draw_vectors(wl, "v", (K + W, L, B, Hkv, d), "bench", backend="torch", device=dev)
    out = torch.empty((L, B, Hq, d), dtype=torch.float16, device=dev)

    def step(s):
        fc.step_all(q_all[s], k_all[s], v_all[s], out)

    for s in range(W):
        step(s)
    torch.cuda.synchronize()
    progress(f"{W} warm-up steps done")

    # Steady state (a step leaves every tier count unchanged): the whole step is captured
    # once as a CUDA graph (without timing nodes: per-call times come from separately
    # captured graphs after the timed region) and replayed on fixed input buffers (each
    # step's inputs are copied in first, inside the timed region).
    before = fc.mirror()
    step(W - 1 if W > 0 else 0)
    steady = all((x == y).all() for a, b in zip(before, fc.mirror()) for x, y in zip(a, b))
    graph = None
    qb, kb, vb = q_all[0].clone(), k_all[0].clone(), v_all[0].clone()
    fc.timers = None
    fc.launches = 0
    pipelined = steady and not args.no_graph and not args.no_pipeline
    n_side = args.side_streams
    if n_side <= 0:  # concurrent compactions of large layers compete; short ones fill gaps
        n_side = 1 if B * Hkv * max(wl.int4_budget, 0) >= (1 << 20) else 2
    side = [torch.cuda.Stream() for _ in range(n_side)] if pipelined else None
    # a cache that grows every step (no eviction): a captured step replayed with the positions
    # copied in and the host mirror advanced, captured again whenever the tensor-core
    # attention kernel's schedule changes (a row's middle tier reaching a new tile); those
    # captures inside the timed region are timed with it
    growing = not steady and not args.no_graph and fc.growing_graph_ok()
    if growing:
        fc.timers = None   # per-call events come from eager steps after the timed region
        fc.launches = 0
        qb.copy_(q_all[W - 1 if W > 0 else 0])
        kb.copy_(k_all[W - 1 if W > 0 else 0])
        vb.copy_(v_all[W - 1 if W > 0 else 0])
        fc.growing_step(qb, kb, vb, out)
        launches_per_step = fc.launches
        graph = fc  # not None: the replays go through fc.growing_step
        torch.cuda.synchronize()
        progress("growing-cache graph captured and replayed once")
    captures_before = fc.growing_captures
    if steady and not args.no_graph:
        if pipelined:
            # prologue: the coming step's maintenance of every layer; from here on each step
            # issues a layer's maintenance for the next step right after that layer's attention
            fc.maintain_all()
            torch.cuda.synchronize()
            fc.launches = 0
        graph = fc.capture_step(qb, kb, vb, out, side)
        launches_per_step = fc.launches
        graph.replay()
        torch.cuda.synchronize()
        progress("graph captured and replayed once")
    barrier(world)
    clocks = ClockSampler(dev.index)
    clocks.start()
    if graph is None:
        fc.timers = None  # no per-call events inside the timed region (they cost host time)
        fc.launches = 0
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for s in range(W, W + K):
        if graph is not None:
            qb.copy_(q_all[s], non_blocking=True)
            kb.copy_(k_all[s], non_blocking=True)
            vb.copy_(v_all[s], non_blocking=True)
            if growing:
                fc.growing_step(qb, kb, vb, out)
            else:
                graph.replay()
        else:
            step(s)
    e1.record()
    torch.cuda.synchronize()
    timed_captures = fc.growing_captures - captures_before
    clk = clocks.stop()
    progress(f"{K} timed steps done")
    launches = launches_per_step * K if graph is not None else fc.launches
    # spread of the step time: K more steps, each between its own events (outside the
    # timed region, in the same launch mode)
    fc.timers, saved_timers = None, fc.timers
    spread = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(K)]
    for i, (sa, sb) in enumerate(spread):
        s = W + i
        sa.record()
        if graph is not None:
            qb.copy_(q_all[s], non_blocking=True)
            kb.copy_(k_all[s], non_blocking=True)
            vb.copy_(v_all[s], non_blocking=True)
            if growing:
                fc.growing_step(qb, kb, vb, out)
            else:
                graph.replay()
        else:
            step(s)
        sb.record()
    torch.cuda.synchronize()
    fc.timers = saved_timers
    per_step = sorted(sa.elapsed_time(sb) for sa, sb in spread)
    per_step_ms = {"median": float(np.median(per_step)),
                   "p90": float(np.percentile(per_step, 90)), "n": K,
                   "note": "per-step events after the timed region"}
    ms = e0.elapsed_time(e1)
    ms_max = max_over_ranks(ms, world)
    # per-call durations: from graphs of the same step captured with timing events as nodes,
    # replayed after the timed region (or from eager steps)
    timing_note = "events of an instrumented replay after the timed region"
    per_call_overlapped = None
    ms_iso = None
    try:
        if graph is None or growing:  # per-call events come from extra eager steps below
            raise RuntimeError("eager launches" if graph is None else "growing-cache graph")
        fc.timers = {}
        inst = fc.capture_step(qb, kb, vb, out, side)   # same schedule, with timing nodes
        inst.replay()
        torch.cuda.synchronize()
        per_call = {name: [a.elapsed_time(b) for a, b in pairs]
                    for name, pairs in fc.timers.items()}
        del inst
        if pipelined:
            # Overlapped calls share the GPU, so their events do not give a kernel's own
            # duration: replay the same step order with the maintenance inline (no overlap)
            # and take the per-call durations and the roofline from that replay.
            per_call_overlapped = {n: float(np.mean(v)) for n, v in per_call.items()}
            fc.timers = {}
            iso = fc.capture_step(qb, kb, vb, out, None, pipelined=True)
            iso.replay()
            torch.cuda.synchronize()
            g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            g0.record()
            iso.replay()
            g1.record()
            torch.cuda.synchronize()
            ms_iso = g0.elapsed_time(g1)
            per_call = {name: [a.elapsed_time(b) for a, b in pairs]
                        for name, pairs in fc.timers.items()}
            timing_note = ("events of a replay after the timed region with each layer's "
                           f"maintenance inline (not overlapped; {ms_iso:.3f} ms per step)")
            del iso
    except Exception as exc:  # eager run, or timing nodes unavailable: time eager steps instead
        timing_note = ("events of eager steps after the timed region" if graph is None else
                       f"eager steps after the timed region ({type(exc).__name__})")
        progress(f"per-call timing from eager steps ({exc})")
        fc.timers = {}
        for s in range(W, W + K):
            if pipelined:
                fc.step_all_pipelined(q_all[s], k_all[s], v_all[s], out, None)
            else:
                step(s)
        torch.cuda.synchronize()
        per_call = {name: [a.elapsed_time(b) for a, b in pairs]
                    for name, pairs in fc.timers.items()}
    fc.timers = None
    # time shares are taken against the step that produced the per-call events
    step_ms_for_share = ms_iso if ms_iso is not None else ms / K

    # roofline of the attention call and of the eviction call
    peaks = load_peaks()
    peak = peaks["hbm_gbs"] if peaks else 6800.0
    peak_src = "measured" if peaks else "fallback"
    lay0 = fc.layers[0]
    traffic_key = wl.name if args.v_codec == "int" else wl.name + "+pq"
    rl = {}
    attn_b = attention_bytes(cfg, lay0)
    if "attention" in per_call:
        t = float(np.mean(per_call["attention"])) / 1e3
        rl["attention"] = {"bound": "hbm", "achieved": attn_b / t / 1e9, "peak": peak,
                           "unit": "GB/s", "frac": attn_b / t / 1e9 / peak,
                           "traffic": measured_traffic("attention", traffic_key),
                           "bytes_per_launch": attn_b, "ms_per_launch": t * 1e3,
                           "peak_source": peak_src,
                           "time_share": float(np.mean(per_call["attention"])) * L / step_ms_for_share}
    if "attention" in rl and fc.needs_logits:   # H2O / EMA: the call also writes its logits
        held = int((lay0.h_n_sink + lay0.h_n_mid + lay0.h_n_recent).sum()) * Hkv
        rl["attention"]["logits_written_bytes"] = held * 4 * (Hq // Hkv)
    if "accumulate" in per_call:   # H2O / EMA: the score update reads the step's logits
        ab = accumulate_bytes(cfg, lay0)
        t = float(np.mean(per_call["accumulate"])) / 1e3
        rl["accumulate"] = {"bound": "hbm", "achieved": ab / t / 1e9, "peak": peak,
                            "unit": "GB/s", "frac": ab / t / 1e9 / peak, "traffic": None,
                            "bytes_per_launch": ab, "ms_per_launch": t * 1e3,
                            "peak_source": peak_src,
                            "time_share": float(np.mean(per_call["accumulate"])) * L /
                            step_ms_for_share}
    if "evict" in per_call:
        eb = evict_bytes(cfg, lay0)
        t = float(np.mean(per_call["evict"])) / 1e3
        hbm = {"bound": "hbm", "achieved": eb / t / 1e9, "peak": peak,
               "unit": "GB/s", "frac": eb / t / 1e9 / peak,
               "traffic": measured_traffic("evict_rerope", traffic_key),
               "bytes_per_launch": eb, "ms_per_launch": t * 1e3,
               "peak_source": peak_src,
               "time_share": float(np.mean(per_call["evict"])) * L / step_ms_for_share}
        if wl.policy == "position":
            # every survivor (middle and recent) is re-positioned: the method's fp32 arithmetic
            # per key against the FP32 lanes of the device at the maximum SM clock
            ops = evict_alu_ops(cfg, lay0)
            apeak, apeak_src = alu_peak_tops(dev)
            rl["evict_rerope"] = {"bound": "alu", "achieved": ops / t / 1e12, "peak": apeak,
                                  "unit": "TOP/s", "frac": ops / t / 1e12 / apeak,
                                  "traffic": hbm["traffic"], "ops_per_launch": ops,
                                  "ms_per_launch": t * 1e3, "peak_source": apeak_src,
                                  "derived_peak": alu_peak_derived(dev, peaks),
                                  "time_share": hbm["time_share"], "hbm_view": hbm}
        else:
            rl["evict_rerope"] = hbm
    dominant = max(rl, key=lambda n: rl[n]["time_share"]) if rl else None

    # end to end: inputs copied from pinned host memory and outputs read back every step
    e2e = None
    if not args.no_e2e:
        qh = q_all[W:].cpu().pin_memory()
        kh = k_all[W:].cpu().pin_memory()
        vh = v_all[W:].cpu().pin_memory()
        oh = torch.empty((K, L, B, Hq, d), dtype=torch.float16).pin_memory()
        qd, kd, vd = torch.empty_like(q_all[0]), torch.empty_like(k_all[0]), torch.empty_like(v_all[0])
        torch.cuda.synchronize()
        barrier(world)
        pipelined_host = graph is not None and not growing
        if pipelined_host:           # the two graphs of the host-fed pipeline, captured untimed
            fc.timers = None         # (without timing nodes)
            fc.prepare_host_pipeline(side)
            torch.cuda.synchronize()
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record()
        if pipelined_host:           # copies of step s+1 in and step s-1 out overlap step s
            fc.run_from_host(qh, kh, vh, oh, side)
        for s in range(0 if pipelined_host else K):
            if graph is not None:    # the graph reads its fixed input buffers
                qb.copy_(qh[s], non_blocking=True)
                kb.copy_(kh[s], non_blocking=True)
                vb.copy_(vh[s], non_blocking=True)
                if growing:
                    fc.growing_step(qb, kb, vb, out)
                else:
                    graph.replay()
            else:
                qd.copy_(qh[s], non_blocking=True)
                kd.copy_(kh[s], non_blocking=True)
                vd.copy_(vh[s], non_blocking=True)
                fc.step_all(qd, kd, vd, out)
            oh[s].copy_(out, non_blocking=True)
        f1.record()
        torch.cuda.synchronize()
        ems = max_over_ranks(f0.elapsed_time(f1), world)
        e2e = {"value": B * K * world / (ems / 1e3), "unit": "tokens/s",
               "h2d_bytes_per_step": int(qd.nbytes + kd.nbytes + vd.nbytes),
               "d2h_bytes_per_step": int(out.nbytes), "ms_per_step": ems / K}
        progress("end-to-end steps done")

    value = B * K * world / (ms_max / 1e3)
    res = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": ms_max / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": wl.name, "layers": L, "batch": B, "num_q_heads": Hq,
                   "num_kv_heads": Hkv, "head_dim": d, "context": maxP, "n_sink": wl.n_sink,
                   "recent_window": wl.recent_window, "int4_budget": wl.int4_budget,
                   "policy": wl.policy, "k_bits": wl.middle_k_bits, "v_bits": wl.middle_v_bits,
                   "shared_rows": bool(args.shared_rows), "v_codec": args.v_codec,
                   "storage": (f"fp16 sinks/recent, packed INT{wl.middle_k_bits} K / "
                               f"INT{wl.middle_v_bits} V middle"
                               if args.v_codec == "int" else
                               f"fp16 sinks/recent, packed INT{wl.middle_k_bits} K / PQ V middle "
                               f"(256 centroids per 4-channel sub-space, codebook trained on "
                               f"{PQ_CALIB_ROWS} synthetic rows, {PQ_ITERS} rounds)"),
                   "l2": "no flush: the compressed cache read per step is far larger than L2",
                   "parallelism": f"replicas x{world} (rows independent, no collective)",
                   "launch": (f"cuda graph per step (growing cache: positions copied in, host "
                              f"mirror advanced per replay; {timed_captures} re-captures in the "
                              f"timed region)" if growing else
                              "cuda graph per step" if graph is not None else "eager launches") +
                             (f"; each layer's maintenance overlaps the next layers "
                              f"({len(side)} side streams taken in turn)" if pipelined else ""),
                   "per_call_timing": timing_note},
        "per_step_ms": per_step_ms,
        "roofline": dict(rl[dominant], kernel=dominant) if dominant else None,
        "roofline_by_call": rl,
        # decode-attention calls alone: B tokens per step over L attention launches
        "attention_only": {
            "value": B * world / (float(np.mean(per_call.get("attention", [np.nan]))) * L / 1e3),
            "unit": "tokens/s", "gbs": rl.get("attention", {}).get("achieved")},
        # mean per-call event durations while maintenance overlaps attention (ms)
        "per_call_overlapped_ms": per_call_overlapped,
        "e2e": e2e, "gpu_launches": launches, "clocks": clk,
    }
    return res


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x, world):
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    if args.impl == "reference":
        if rank == 0:
            ref = run_oracle_sample(args.workload, args.steps, args.warmup)
            wl = workload(args.workload)
            line = {"impl": "reference", "metric": METRIC, "value": ref["value"],
                    "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
                    "warmup": args.warmup, "ms_per_step": ref["ms_per_step"],
                    "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                    "dtype": "f64", "data": "synthetic",
                    "config": {"workload": wl.name},
                    "cpu_baseline": {k: ref[k] for k in ("value", "unit", "cores", "kind", "sample")},
                    "e2e": {"value": ref["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                            "d2h_bytes_per_step": 0}}
            print(json.dumps(line), flush=True)
        return
    res = run_ours(args, rank, world)
    progress("GPU arm done")
    if rank == 0:
        if not args.no_cpu_baseline and not args.k_bits:
            cb = run_oracle_sample(args.workload, steps=3, warmup=1, budget_s=20.0)
            progress("oracle sample done")
            res["cpu_baseline"] = {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample")}
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()

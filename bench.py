#!/usr/bin/env python3
"""Benchmark: INT8 paged decode attention, effective KV GB/s (and the rest of the path).

Workload (N = 1): single-sequence decode with 24 query / 4 KV heads, head_dim
256, block size 16, histories 8192, 16384 and 32768 (K with 4 outlier channels
per KV head x20, V N(0,1), seeded), i.e. the long-history decode configuration.
One step = one new token through the 16 full-attention layers of the pages'
model: for every (layer, history) one i8kv_int8_decode_step call quantizes the
new token's K/V into that layer's paged INT8 cache (the producer's rule, bit for
bit), quantizes its query and attends over the whole history, then its merge
kernel runs.  Each layer owns its cache, so a step streams 16 x 56K tokens x
2080 B = 1.9 GB and L2 (129 MB) holds none of it between steps.  All K timed
steps run as one CUDA graph with timing events around it.  The dominant
kernel's own average duration comes from a second graph of the same K x 48
calls back to back.  The producer + plain decode pair (two calls) is timed per
history among the secondary results.

  value     = KV bytes read by the decode launches / timed wall time (GB/s)
  roofline  = same bytes / the decode-step calls' own time (second graph), against the
              measured HBM copy bandwidth (MEASURED_PEAKS.json)
  e2e       = the same step through the C ABI with pinned host buffers: the new
              tokens' q/k/v copied host->device and every output copied back,
              inside the timed graph
  secondary = per-history decode times, BF16-KV comparison decode, prefix chunk
              TOPS, producer throughput (measured after the main timed region)

--impl reference times the CPU oracle instead (bounded samples of the same
decode), on the host cores, and prints the same JSON line with "impl".
Multi-GPU (torchrun): every rank runs the same per-GPU workload (weak scaling,
no collective on the data path); rank 0 prints the max-over-ranks time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "INT8 paged decode attn effective KV GB/s (% HBM peak); prefix-chunk INT8 TOPS"
HISTORIES = (8192, 16384, 32768)
LAYERS = 16          # full-attention layers of the pages' model
FALLBACK_HBM_GBS = 6800.0


# ----------------------------------------------------------------------------- helpers
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", 0.0)), "measured"
    return FALLBACK_HBM_GBS, 1900.0, "fallback"


def kernel_hash(*rel):
    """Hash of the kernel sources' code: comments and whitespace are dropped, so
    a comment edit does not void a recorded ncu figure."""
    h = hashlib.sha256()
    for r in rel:
        with open(os.path.join(ROOT, r), encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(kind: str, src_hash: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source (same hash); else None."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 3 and parts[0] == kind and parts[1] == src_hash:
                return float(parts[2])
    return None


class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled every 100 ms while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.samples = []
        self.proc = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        if gpu_id:
            cmd += ["-i", gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        rows = [s for (t, s) in self.samples if t0 <= t <= t1]
        window = "timed"
        if not rows:
            rows = [s for (_, s) in self.samples]
            window = "whole run (timed region shorter than one sample)"
        mhz, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            f = [x.strip() for x in r.split(",")]
            if len(f) < 8:
                continue
            try:
                mhz.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(mhz), "window": window}


def max_over_ranks(torch, dist, ms: float, device) -> float:
    """The slowest rank's time: the whole job ends when it does."""
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(world: int, steps: int, bytes_per_step: int, ms: float) -> float:
    """Replicas (weak scaling): every rank streams bytes_per_step per step."""
    return world * steps * bytes_per_step / (ms / 1e3) / 1e9


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), for the CPU baseline."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "hardware", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ----------------------------------------------------------------------------- reference (oracle) arm
def headline_config(world: int, layers: int) -> dict:
    """The headline workload's `config` object, shared by both arms."""
    return {"workload": f"decode_outlier: single-sequence decode, 24 q / 4 kv heads, head_dim 256, "
                        f"block 16, histories {list(HISTORIES)}, x{layers} layers per step",
            "global_batch": world, "seq_len": list(HISTORIES), "parallelism": f"replicas x{world}",
            "l2": "inputs larger than L2 (each layer has its own cache; 1.9 GB per step)"}


def oracle_decode_sample(L: int = HISTORIES[0]):
    """The oracle's inputs for one (layer, history L) decode of the workload."""
    from oracle import oracle as orc
    w = wl.decode_outlier(L)
    k, v = w.kv(0)
    cache = orc.kv_quant_write(k, v, w.slots(0), w.num_blocks, w.block_size)
    q = w.q()
    q_i8 = np.empty(q.shape, np.int8)
    q_s = np.empty(q.shape[:2], np.float32)
    for h in range(q.shape[1]):
        q_i8[0, h], q_s[0, h] = orc.quantize_vector(q[0, h])
    return w, cache, q_i8, q_s


def time_oracle(budget_s: float, nthreads: int):
    """Oracle decode of the 8192-token history (all 24 heads), repeated for about budget_s."""
    from oracle import oracle as orc
    w, cache, q_i8, q_s = oracle_decode_sample()
    reps, t_total = 0, 0.0
    while t_total < budget_s or reps == 0:
        t0 = time.perf_counter()
        orc.decode_attn(q_i8, q_s, cache, w.block_tables, w.seq_lens, w.block_size, nthreads=nthreads)
        t_total += time.perf_counter() - t0
        reps += 1
    gbs = reps * w.kv_bytes_int8() / t_total / 1e9
    return gbs, reps, t_total


def time_oracle_prefix(budget_s: float, nthreads: int):
    """Oracle prefix chunk (16384 history + 2048 chunk, 24 q / 4 KV heads, head_dim
    256) on a bounded sample of chunk rows (all 24 heads each, evenly spaced
    over the chunk), repeated for about budget_s; returns INT8 TOPS over the
    sampled rows' causal pairs (4 D ops each), the rows and the time."""
    from oracle import oracle as orc
    w = wl.prefix_chunk()
    k, v = w.kv()
    cache = orc.kv_quant_write(k, v, w.slots(), w.num_blocks, w.block_size)
    q = w.q()
    n_rows = max(1, min(w.chunk, 2 * nthreads))
    rows = np.linspace(0, w.chunk - 1, n_rows).astype(np.int32)
    q_i8 = np.empty(q.shape, np.int8)
    q_s = np.empty(q.shape[:2], np.float32)
    for j in rows:
        for h in range(w.Hq):
            q_i8[j, h], q_s[j, h] = orc.quantize_vector(q[j, h])
    ops = sum(w.Hq * (w.history + int(j) + 1) * 4 * w.D for j in rows)
    reps, t_total = 0, 0.0
    while t_total < budget_s or reps == 0:
        t0 = time.perf_counter()
        orc.prefix_attn(q_i8, q_s, cache, w.block_table, w.history, w.block_size, rows=rows, nthreads=nthreads)
        t_total += time.perf_counter() - t0
        reps += 1
    return reps * ops / t_total / 1e12, len(rows), reps, t_total


def cpu_baseline(seconds: float):
    """The oracle on this host: the decode sample on all cores and on one thread,
    and a prefix-chunk sample on all cores."""
    cores = cpu_cores()
    gbs, reps, el = time_oracle(seconds, cores)
    gbs1, reps1, el1 = time_oracle(seconds, 1)
    tops, nrows, preps, pel = time_oracle_prefix(seconds, cores)
    return {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle", "cpu_model": cpu_model(),
            "sample": f"{reps} oracle decodes of the 8192-token history (24 heads) in {el:.1f} s on {cores} threads",
            "single_thread": {"value": gbs1, "unit": "GB/s", "cores": 1,
                              "sample": f"{reps1} oracle decodes of the same history in {el1:.1f} s on 1 thread"},
            "prefix": {"value": tops, "unit": "INT8 TOPS", "cores": cores,
                       "sample": f"{preps} x {nrows} chunk rows (24 heads each) of the 16384 + 2048 chunk in "
                                 f"{pel:.1f} s on {cores} threads"}}


def run_reference(args):
    from oracle import oracle as orc
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    orc.build()
    cores = cpu_cores()
    # A step is a bounded sample of the headline step: one layer at each of the
    # three histories (the headline step runs every layer), over the first
    # kv_heads KV heads and their query heads.
    samples = [oracle_decode_sample(L) for L in HISTORIES]
    # one probe pass over all 24 heads fixes how many query heads a step samples,
    # so that the whole run (warm-up + steps) stays within about two minutes
    t0 = time.perf_counter()
    for w, cache, q_i8, q_s in samples:
        orc.decode_attn(q_i8, q_s, cache, w.block_tables, w.seq_lens, w.block_size, nthreads=cores)
    t_full = time.perf_counter() - t0
    per_step_budget = 120.0 / max(1, args.steps + args.warmup)
    heads = int(max(1, min(24, 24 * per_step_budget / max(t_full, 1e-6))))
    kv_heads = (heads + 5) // 6
    subs = []
    for w, cache, q_i8, q_s in samples:
        sub = cache if kv_heads == 4 else _sub_cache(cache, kv_heads)
        subs.append((w, sub, np.ascontiguousarray(q_i8[:, : 6 * kv_heads]),
                     np.ascontiguousarray(q_s[:, : 6 * kv_heads])))

    def step():
        for w, sub, qs, qss in subs:
            orc.decode_attn(qs, qss, sub, w.block_tables, w.seq_lens, w.block_size, nthreads=cores)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    bytes_step = sum(HISTORIES) * kv_heads * (2 * 256 + 8)
    value = args.steps * bytes_step / el / 1e9
    sample = (f"oracle decode of one layer at each history {list(HISTORIES)}, {kv_heads * 6} query heads over "
              f"{kv_heads} KV head(s) per step, {cores} threads")
    line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "impl": "reference",
            "config": headline_config(args.gpus, args.layers),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample,
                             "cpu_model": cpu_model()},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def _sub_cache(cache, kv_heads):
    """The oracle cache restricted to the first kv_heads KV heads (contiguous copies)."""
    return dict(k_cache=np.ascontiguousarray(cache["k_cache"][:, :kv_heads]),
                v_cache=np.ascontiguousarray(cache["v_cache"][:, :kv_heads]),
                k_scale=np.ascontiguousarray(cache["k_scale"][:, :, :kv_heads]),
                v_scale=np.ascontiguousarray(cache["v_scale"][:, :, :kv_heads]))


# ----------------------------------------------------------------------------- our arm
class DecodeLayer:
    """One layer's INT8 cache at one history, plus the new token's buffers."""

    def __init__(self, i8, torch, base, w: wl.DecodeWorkload, k_new, v_new, q_new):
        self.w = w
        self.cache = {n: t.clone() for n, t in base.items()}
        dev = "cuda"
        self.k = k_new
        self.v = v_new
        self.q = q_new
        L = int(w.seq_lens[0])
        self.slot = torch.tensor(w.slots(0, L - 1, L), dtype=torch.int32, device=dev)
        self.q_i8 = torch.empty((1, w.Hq, w.D), dtype=torch.int8, device=dev)
        self.q_scale = torch.empty((1, w.Hq), dtype=torch.float32, device=dev)
        self.out = torch.empty((1, w.Hq, w.D), dtype=torch.float32, device=dev)
        self.bt = torch.from_numpy(w.block_tables).cuda()
        self.sl = torch.from_numpy(w.seq_lens).cuda()

    def step(self, i8, ws):
        """Producer + attention for the new token in one call (the timed path)."""
        c = self.cache
        i8.int8_decode_step(self.out, self.q, self.k.view(1, *self.k.shape[1:]), self.v.view(1, *self.v.shape[1:]),
                            c["k_cache"], c["v_cache"], c["k_scale"], c["v_scale"], self.bt, self.sl, ws)

    def produce(self, i8):
        i8.kv_quant_write(self.k, self.v, self.slot, **self.cache, q=self.q, q_i8=self.q_i8, q_scale=self.q_scale)

    def decode(self, i8, ws):
        c = self.cache
        i8.int8_paged_decode_attn(self.out, self.q_i8, self.q_scale, c["k_cache"], c["v_cache"], c["k_scale"],
                                  c["v_scale"], self.bt, self.sl, ws)


def to_dev(torch, a):
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run_ours(args):
    import torch
    import torch.distributed as dist

    from int8_kv_cache_token_gb300 import build as ibuild
    ibuild.build()
    import int8_kv_cache_token_gb300 as i8

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")
    hbm_peak, tensor_peak, peak_kind = measured_peaks()
    stream = torch.cuda.current_stream()

    # ---- inputs: one seeded history per length, cloned into every layer ----
    layers = []
    for L in HISTORIES:
        w = wl.decode_outlier(L)
        k, v = w.kv(0)
        base = i8.alloc_int8_cache(w.num_blocks, w.Hkv, w.D)
        i8.kv_quant_write(to_dev(torch, k), to_dev(torch, v), to_dev(torch, w.slots(0)), **base)
        k_new, v_new = to_dev(torch, k[L - 1:L]), to_dev(torch, v[L - 1:L])
        q_new = to_dev(torch, w.q())
        for _ in range(args.layers):
            layers.append(DecodeLayer(i8, torch, base, w, k_new, v_new, q_new))
        del base
    torch.cuda.synchronize()
    ws = {L: i8.decode_workspace(1, 24, 4, 256, wl.decode_outlier(L).block_tables.shape[1]) for L in HISTORIES}
    bytes_per_step = sum(ly.w.kv_bytes_int8() for ly in layers)
    launches_per_step = 2 * len(layers)  # decode step (producer work + attention), merge

    def step():
        for ly in layers:
            ly.step(i8, ws[int(ly.w.seq_lens[0])])

    for _ in range(max(args.warmup, 1)):
        step()
    torch.cuda.synchronize()
    assert i8.device_error() == 0, "kernel error during warm-up"

    # ---- capture the K timed steps as one CUDA graph ----
    g = capture_graph(torch, lambda: [step() for _ in range(args.steps)])
    g.replay()  # one untimed replay of the captured graph (warm)
    torch.cuda.synchronize()

    gpu_id = None
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(local).uuid)
    except Exception:
        pass
    sampler = ClockSampler(gpu_id) if rank == 0 else None
    time.sleep(0.25 if sampler else 0)
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.time()
    t_start.record()
    g.replay()
    t_end.record()
    torch.cuda.synchronize()
    wall1 = time.time()
    if world > 1:
        dist.barrier()
    if sampler:
        sampler.stop()
    ms = t_start.elapsed_time(t_end)
    if world > 1:
        ms = max_over_ranks(torch, dist, ms, "cuda")
    err = i8.device_error()
    assert err == 0, f"kernel error {err} in the timed region"
    value = whole_job_gbs(world, args.steps, bytes_per_step, ms)

    # ---- the dominant kernel alone: the same K x 48 decode-step calls back to back ----
    # (one graph, events around it; a call is the decode-step attention kernel plus
    # its merge kernel).  Then per history, the 16 layers x K calls of that length,
    # for the step and for the plain decode (the producer run separately).
    dec_ms = time_graph(torch, lambda: [ly.step(i8, ws[int(ly.w.seq_lens[0])]) for ly in layers], args.steps)
    n_dec = len(layers)
    achieved = bytes_per_step / (dec_ms / 1e3) / 1e9
    avg_launch_us = dec_ms / n_dec * 1e3
    by_len, step_by_len = {}, {}
    for L in HISTORIES:
        sub = [ly for ly in layers if int(ly.w.seq_lens[0]) == L]
        ms_l = time_graph(torch, lambda: [ly.decode(i8, ws[L]) for ly in sub], args.steps)
        by_len[L] = ms_l / len(sub)
        ms_s = time_graph(torch, lambda: [ly.step(i8, ws[L]) for ly in sub], args.steps)
        step_by_len[L] = ms_s / len(sub)
    src = kernel_hash("int8_kv_cache_token_gb300/csrc/decode.cu", "int8_kv_cache_token_gb300/csrc/common.cuh")
    traffic = recorded_traffic("int8_decode_step", src)
    roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                "frac": (achieved / hbm_peak) if achieved else None, "traffic": traffic,
                "kernel": "decode_kernel<256, INT8, STEP> + decode_merge_kernel",
                "peak_kind": f"of {peak_kind} (HBM copy bandwidth)",
                "avg_launch_us": avg_launch_us,
                "algorithmic_bytes_per_launch": bytes_per_step / len(layers),
                "method": "K x 48 decode-step calls (attention + merge kernel) replayed back to back in one CUDA "
                          "graph, CUDA events around the graph"}

    # ---- e2e: the same steps through the C ABI with pinned host buffers ----
    e2e = run_e2e(args, torch, i8, layers, ws, bytes_per_step, world)

    secondary = {}
    if rank == 0:
        secondary["decode_by_history"] = {
            str(L): {"us": v * 1e3, "gb_s": wl.decode_outlier(L).kv_bytes_int8() / (v / 1e3) / 1e9,
                     "frac_hbm": wl.decode_outlier(L).kv_bytes_int8() / (v / 1e3) / 1e9 / hbm_peak}
            for L, v in by_len.items()}
        secondary["decode_step_by_history"] = {
            str(L): {"us": v * 1e3} for L, v in step_by_len.items()}
        if not args.quick:
            secondary.update(run_secondary(torch, i8, hbm_peak, tensor_peak, peak_kind))
            try:
                secondary["decode_other_workloads"] = run_batch_decodes(torch, i8, hbm_peak)
            except Exception as e:  # pragma: no cover - report, do not hide
                secondary["decode_other_workloads"] = {"error": str(e)[:200]}
            try:
                secondary["decode_u8_probs_by_history"] = run_u8p_comparison(torch, i8, hbm_peak)
            except Exception as e:  # pragma: no cover - report, do not hide
                secondary["decode_u8_probs_by_history"] = {"error": str(e)[:200]}
            try:
                secondary["prefix_int8_vs_bf16_kv_by_history"] = run_prefix_by_history(torch, i8, tensor_peak,
                                                                                        peak_kind)
            except Exception as e:  # pragma: no cover - report, do not hide
                secondary["prefix_int8_vs_bf16_kv_by_history"] = {"error": str(e)[:200]}
            try:
                secondary["bf16_kv_decode_by_history"] = run_bf16_comparison(
                    torch, i8, hbm_peak, {L: v * 1e3 for L, v in by_len.items()})
            except Exception as e:  # pragma: no cover - report, do not hide
                secondary["bf16_kv_decode_by_history"] = {"error": str(e)[:200]}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline(args.cpu_seconds)

    if rank == 0:
        clocks = sampler.summary(wall0, wall1) if sampler else None
        line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "s8/s32 (fp32 softmax)", "data": "synthetic (seeded)",
                "config": headline_config(world, args.layers),
                "gpu_launches": args.steps * launches_per_step,
                "e2e": e2e, "roofline": roofline, "cpu_baseline": cpu, "clocks": clocks,
                "secondary": secondary}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_e2e(args, torch, i8, layers, ws, bytes_per_step, world):
    """Per step: one H2D copy of every layer's new q/k/v (packed in one pinned host
    buffer), the 48 decode-step calls on views of the device copy, one D2H copy of
    every output; captured with the steps in one graph."""
    k_n, v_n, q_n = layers[0].k.numel(), layers[0].v.numel(), layers[0].q.numel()
    per = k_n + v_n + q_n
    n = len(layers)
    host_in = torch.empty(n * per, dtype=torch.bfloat16).pin_memory()
    for i, ly in enumerate(layers):
        host_in[i * per:i * per + k_n].copy_(ly.k.reshape(-1).cpu())
        host_in[i * per + k_n:i * per + k_n + v_n].copy_(ly.v.reshape(-1).cpu())
        host_in[i * per + k_n + v_n:(i + 1) * per].copy_(ly.q.reshape(-1).cpu())
    dev_in = torch.empty(n * per, dtype=torch.bfloat16, device="cuda")
    dev_out = torch.empty((n,) + tuple(layers[0].out.shape[1:]), dtype=torch.float32, device="cuda")
    host_out = torch.empty(dev_out.shape, dtype=torch.float32).pin_memory()
    views = []
    for i, ly in enumerate(layers):
        base = i * per
        views.append((dev_in[base:base + k_n].view(1, *ly.k.shape[1:]),
                      dev_in[base + k_n:base + k_n + v_n].view(1, *ly.v.shape[1:]),
                      dev_in[base + k_n + v_n:base + per].view(ly.q.shape), dev_out[i:i + 1]))
    h2d = host_in.numel() * host_in.element_size()
    d2h = host_out.numel() * host_out.element_size()
    stream = torch.cuda.current_stream()
    g = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        with torch.cuda.graph(g, stream=cap):
            for _ in range(args.steps):
                dev_in.copy_(host_in, non_blocking=True)
                for ly, (kv, vv, qv, ov) in zip(layers, views):
                    c = ly.cache
                    i8.int8_decode_step(ov, qv, kv, vv, c["k_cache"], c["v_cache"], c["k_scale"], c["v_scale"], ly.bt,
                                        ly.sl, ws[int(ly.w.seq_lens[0])])
                host_out.copy_(dev_out, non_blocking=True)
    stream.wait_stream(cap)
    g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    a.record()
    g.replay()
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b)
    if world > 1:
        ms = max_over_ranks(torch, dist, ms, "cuda")
    return {"value": whole_job_gbs(world, args.steps, bytes_per_step, ms), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms / args.steps}


def capture_graph(torch, fn):
    """fn() captured once into a CUDA graph (on a side stream, as torch requires)."""
    stream = torch.cuda.current_stream()
    g = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        with torch.cuda.graph(g, stream=cap):
            fn()
    stream.wait_stream(cap)
    return g


def time_graph(torch, fn, reps: int):
    """Average ms of fn() captured reps times in one graph."""
    stream = torch.cuda.current_stream()
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        with torch.cuda.graph(g, stream=cap):
            for _ in range(reps):
                fn()
    stream.wait_stream(cap)
    g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    g.replay()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


def time_rotating(torch, calls, reps: int):
    """Average ms per call of `calls` (a list of closures over distinct caches whose
    total size exceeds L2), replayed round-robin `reps` times in one graph."""
    return time_graph(torch, lambda: [c() for c in calls], reps) / len(calls)


def run_bf16_comparison(torch, i8, hbm_peak, int8_us: dict):
    """BF16-KV decode over the same histories (the pages' BF16 control): µs, GB/s
    at 4096 B per cached token, and the INT8 speedup over it."""
    res = {}
    for L in HISTORIES:
        w = wl.decode_outlier(L)
        k, v = w.kv(0)
        base = i8.alloc_bf16_cache(w.num_blocks, w.Hkv, w.D)
        i8.bf16_kv_write(to_dev(torch, k), to_dev(torch, v), to_dev(torch, w.slots(0)), **base)
        copies = max(2, int(np.ceil(400e6 / w.kv_bytes_bf16())))
        caches = [{n: t.clone() for n, t in base.items()} for _ in range(copies)]
        del base
        q = to_dev(torch, w.q())
        out = torch.empty((1, w.Hq, w.D), dtype=torch.float32, device="cuda")
        ws = i8.decode_workspace(1, w.Hq, w.Hkv, w.D, w.block_tables.shape[1])
        bt, sl = to_dev(torch, w.block_tables), to_dev(torch, w.seq_lens)
        calls = [(lambda c=c: i8.bf16_paged_decode_attn(out, q, c["k_cache"], c["v_cache"], bt, sl, ws)) for c in caches]
        ms = time_rotating(torch, calls, 20)
        gbs = w.kv_bytes_bf16() / (ms / 1e3) / 1e9
        res[str(L)] = {"us": ms * 1e3, "gb_s": gbs, "frac_hbm": gbs / hbm_peak,
                       "int8_speedup": (ms * 1e3) / int8_us[L] if L in int8_us else None}
        del caches
        torch.cuda.empty_cache()
    return res


def run_u8p_comparison(torch, i8, hbm_peak):
    """Decode with UINT8 probability codes against the signed codes, each timed
    the same way (rotating cache copies past L2, one graph): µs and the ratio."""
    res = {}
    for L in HISTORIES:
        w = wl.decode_outlier(L)
        k, v = w.kv(0)
        base = i8.alloc_int8_cache(w.num_blocks, w.Hkv, w.D)
        i8.kv_quant_write(to_dev(torch, k), to_dev(torch, v), to_dev(torch, w.slots(0)), **base)
        copies = max(2, int(np.ceil(400e6 / w.kv_bytes_int8())))
        caches = [{n: t.clone() for n, t in base.items()} for _ in range(copies)]
        del base
        q_i8 = torch.empty((1, w.Hq, w.D), dtype=torch.int8, device="cuda")
        q_s = torch.empty((1, w.Hq), dtype=torch.float32, device="cuda")
        dummy = torch.zeros((1, w.Hkv, w.D), dtype=torch.bfloat16, device="cuda")
        i8.kv_quant_write(dummy, dummy, torch.full((1,), -1, dtype=torch.int32, device="cuda"), **caches[0],
                          q=to_dev(torch, w.q()), q_i8=q_i8, q_scale=q_s)
        out = torch.empty((1, w.Hq, w.D), dtype=torch.float32, device="cuda")
        ws = i8.decode_workspace(1, w.Hq, w.Hkv, w.D, w.block_tables.shape[1])
        bt, sl = to_dev(torch, w.block_tables), to_dev(torch, w.seq_lens)
        r = {}
        for name, u8 in (("s8_codes", False), ("u8_codes", True)):
            calls = [(lambda c=c, u8=u8: i8.int8_paged_decode_attn(out, q_i8, q_s, c["k_cache"], c["v_cache"],
                                                                   c["k_scale"], c["v_scale"], bt, sl, ws,
                                                                   u8_probs=u8)) for c in caches]
            r[name + "_us"] = time_rotating(torch, calls, 20) * 1e3
        r["u8_over_s8_time"] = r["u8_codes_us"] / r["s8_codes_us"]
        res[str(L)] = r
        del caches
        torch.cuda.empty_cache()
    return res


def run_batch_decodes(torch, i8, hbm_peak):
    """The other decode workloads, timed only (their parity is in the tests): a
    single sequence at 4096 tokens (24 q / 4 KV heads, head_dim 256), 64 sequences
    with lengths uniform in [1024, 32768] (same heads) and batch 16 at 32768 with
    32 q / 8 KV heads, head_dim 128.  Shapes, lengths and paging come from
    workloads.py; the K/V values are drawn on the device (torch generator, seed 0)
    and written through the producer, the query quantized by its query path.
    Each cache exceeds L2 except the 4096-token one's, which rotates copies."""
    res = {}
    gen = torch.Generator(device="cuda")
    gen.manual_seed(0)
    for name, w in (("decode_single_4096", wl.decode_4k()), ("decode_batch64_mixed_lengths", wl.decode_batch()),
                    ("decode_gqa128_batch16_32768", wl.producer_gqa_decode())):
        try:
            cache = i8.alloc_int8_cache(w.num_blocks, w.Hkv, w.D)
            for b in range(w.B):
                L = int(w.seq_lens[b])
                k = torch.randn((L, w.Hkv, w.D), generator=gen, device="cuda").to(torch.bfloat16)
                v = torch.randn((L, w.Hkv, w.D), generator=gen, device="cuda").to(torch.bfloat16)
                i8.kv_quant_write(k, v, to_dev(torch, w.slots(b)), **cache)
                del k, v
            q = torch.randn((w.B, w.Hq, w.D), generator=gen, device="cuda").to(torch.bfloat16)
            q_i8 = torch.empty((w.B, w.Hq, w.D), dtype=torch.int8, device="cuda")
            q_s = torch.empty((w.B, w.Hq), dtype=torch.float32, device="cuda")
            dummy = torch.zeros((w.B, w.Hkv, w.D), dtype=torch.bfloat16, device="cuda")
            i8.kv_quant_write(dummy, dummy, torch.full((w.B,), -1, dtype=torch.int32, device="cuda"), **cache, q=q,
                              q_i8=q_i8, q_scale=q_s)
            out = torch.empty((w.B, w.Hq, w.D), dtype=torch.float32, device="cuda")
            ws = i8.decode_workspace(w.B, w.Hq, w.Hkv, w.D, w.block_tables.shape[1])
            bt, sl = to_dev(torch, w.block_tables), to_dev(torch, w.seq_lens)
            nbytes = w.kv_bytes_int8()
            copies = max(1, int(np.ceil(400e6 / nbytes)))
            caches = [cache] + [{n: t.clone() for n, t in cache.items()} for _ in range(copies - 1)]
            calls = [(lambda c=c: i8.int8_paged_decode_attn(out, q_i8, q_s, c["k_cache"], c["v_cache"], c["k_scale"],
                                                            c["v_scale"], bt, sl, ws)) for c in caches]
            ms = time_rotating(torch, calls, 10 if nbytes > 1e9 else 20)
            torch.cuda.synchronize()
            assert i8.device_error() == 0
            gbs = nbytes / (ms / 1e3) / 1e9
            res[name] = {"us": ms * 1e3, "kv_bytes": nbytes, "gb_s": gbs, "frac_hbm": gbs / hbm_peak,
                         "batch": w.B, "heads": f"{w.Hq}/{w.Hkv}/{w.D}"}
            del caches, cache
            torch.cuda.empty_cache()
        except Exception as e:  # pragma: no cover - report, do not hide
            res[name] = {"error": str(e)[:200]}
    return res


def hbm_roofline(moved: int, ms: float, peak: float, kind: str, kernel: str) -> dict:
    gbs = moved / (ms / 1e3) / 1e9
    return {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
            "peak_kind": f"of {kind} (HBM copy bandwidth)", "kernel": kernel, "algorithmic_bytes_per_launch": moved}


def run_secondary(torch, i8, hbm_peak, tensor_peak=0.0, peak_kind="measured"):
    """Other rows of the path, each timed on its own (after the main region)."""
    res = {}
    # producer: 8192 new tokens, 8 KV heads, head_dim 128, 32 query heads
    try:
        p = wl.producer_tokens()
        cache = i8.alloc_int8_cache(p["num_blocks"], p["Hkv"], p["D"])
        k, v, q, s = (to_dev(torch, p[n]) for n in ("k", "v", "q", "slots"))
        q_i8 = torch.empty(q.shape, dtype=torch.int8, device="cuda")
        q_s = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
        ms = time_graph(torch, lambda: i8.kv_quant_write(k, v, s, **cache, q=q, q_i8=q_i8, q_scale=q_s), 20)
        T, Hkv, Hq, D = 8192, p["Hkv"], p["Hq"], p["D"]
        moved = T * (2 * Hkv * D * 2 + 2 * Hkv * D + 2 * Hkv * 4) + T * Hq * (2 * D + D + 4)
        res["producer_8192x8x128"] = {"us": ms * 1e3, "gb_s": moved / (ms / 1e3) / 1e9,
                                      "frac_hbm": moved / (ms / 1e3) / 1e9 / hbm_peak,
                                      "roofline": hbm_roofline(moved, ms, hbm_peak, peak_kind,
                                                               "kv_quant_write_kernel<128, plain>")}
    except Exception as e:  # pragma: no cover - report, do not hide
        res["producer_8192x8x128"] = {"error": str(e)[:200]}
    # fused producer: the same tokens at positions 0..8191 with Q/K RMSNorm and
    # full-width RoPE (table rows read once per token, 512 B each)
    try:
        p = wl.producer_rope_tokens()
        cache = i8.alloc_int8_cache(p["num_blocks"], p["Hkv"], p["D"])
        k, v, q, s, pos, cs, qw, kw = (to_dev(torch, p[n]) for n in ("k", "v", "q", "slots", "positions", "cos_sin",
                                                                  "q_norm_weight", "k_norm_weight"))
        q_i8 = torch.empty(q.shape, dtype=torch.int8, device="cuda")
        q_s = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
        ms = time_graph(torch, lambda: i8.kv_rope_quant_write(k, v, s, **cache, positions=pos, cos_sin=cs,
                                                              rotary_dim=p["rotary_dim"], q=q, q_i8=q_i8, q_scale=q_s,
                                                              q_norm_weight=qw, k_norm_weight=kw), 20)
        T, Hkv, Hq, D, rd = 8192, p["Hkv"], p["Hq"], p["D"], p["rotary_dim"]
        moved = (T * (2 * Hkv * D * 2 + 2 * Hkv * D + 2 * Hkv * 4) + T * Hq * (2 * D + D + 4) + T * (rd * 4 + 4))
        res["producer_rope_norm_8192x8x128"] = {"us": ms * 1e3, "gb_s": moved / (ms / 1e3) / 1e9,
                                                "frac_hbm": moved / (ms / 1e3) / 1e9 / hbm_peak,
                                                "roofline": hbm_roofline(moved, ms, hbm_peak, peak_kind,
                                                                         "kv_quant_write_kernel<128, fused>")}
    except Exception as e:  # pragma: no cover
        res["producer_rope_norm_8192x8x128"] = {"error": str(e)[:200]}
    # prefix chunk: 2048 queries after 16384 cached tokens, 24 q / 4 kv heads, head_dim 256.
    # Three copies of the whole call's state (cache, operand-tile workspace,
    # query, output: about 150 MB each, 3x L2) rotate inside one graph, so no
    # call finds its tiles in L2; the unit timed is the whole call (tiles,
    # attention, merge of the split last wave).
    try:
        w = wl.prefix_chunk()
        k, v = w.kv()
        base = i8.alloc_int8_cache(w.num_blocks, w.Hkv, w.D)
        i8.kv_quant_write(to_dev(torch, k), to_dev(torch, v), to_dev(torch, w.slots()), **base)
        qd = to_dev(torch, w.q())
        dummy = torch.zeros((w.chunk, w.Hkv, w.D), dtype=torch.bfloat16, device="cuda")
        none = torch.full((w.chunk,), -1, dtype=torch.int32, device="cuda")
        bt = to_dev(torch, w.block_table)
        sets = []
        for _ in range(3):
            cache = {n: t.clone() for n, t in base.items()}
            q_i8 = torch.empty(qd.shape, dtype=torch.int8, device="cuda")
            q_s = torch.empty(qd.shape[:2], dtype=torch.float32, device="cuda")
            i8.kv_quant_write(dummy, dummy, none, **cache, q=qd, q_i8=q_i8, q_scale=q_s)
            out = torch.empty((w.chunk, w.Hq, w.D), dtype=torch.float32, device="cuda")
            sets.append((cache, q_i8, q_s, out, i8.prefix_workspace(w.history, w.chunk, w.Hkv, w.D)))
        del base
        calls = [(lambda c=c, qi=qi, qs=qs, o=o, ws=ws: i8.int8_prefix_attn(
            o, qi, qs, c["k_cache"], c["v_cache"], c["k_scale"], c["v_scale"], bt, w.history, workspace=ws))
            for (c, qi, qs, o, ws) in sets]
        ms = time_rotating(torch, calls, 4)
        torch.cuda.synchronize()
        assert i8.device_error() == 0
        tops = w.int8_ops() / (ms / 1e3) / 1e12
        res["prefix_16384+2048"] = {
            "ms": ms, "int8_tops": tops, "pairs": w.pairs(), "ops": w.int8_ops(),
            "roofline": {"bound": "tensor", "achieved": tops, "peak": tensor_peak, "unit": "TFLOP/s",
                         "frac": tops / tensor_peak if tensor_peak else None,
                         "peak_kind": f"of {peak_kind} dense bf16 (burst): the INT8 codes run exactly on the "
                                      "tcgen05 f16 path, which has the bf16 rate",
                         "kernel": "prefix_tiles_kernel + prefix_attn_kernel<256, INT8> + prefix_merge_kernel",
                         "algorithmic_ops_per_launch": w.int8_ops(),
                         "traffic": recorded_traffic("int8_prefix", kernel_hash(
                             "int8_kv_cache_token_gb300/csrc/prefix.cu", "int8_kv_cache_token_gb300/csrc/common.cuh")),
                         "method": "3 rotating copies of cache + workspace + query + output (3x L2), 12 calls in "
                                   "one CUDA graph, CUDA events around it"}}
        del sets, calls
        torch.cuda.empty_cache()
    except Exception as e:  # pragma: no cover
        res["prefix_16384+2048"] = {"error": str(e)[:200]}
    # first prefill chunk, 0 + 4096 tokens, 24 / 4 heads, head_dim 256: the routed
    # entry on the high-precision path (producer + bf16 attention) and forced onto
    # INT8 (producer with the query + INT8 attention), as the pages compare them
    try:
        w = wl.PrefixWorkload("first_chunk", 24, 4, 256, 0, 4096, seed=5)
        k, v = w.kv()
        kd, vd, qd, sd = to_dev(torch, k), to_dev(torch, v), to_dev(torch, w.q()), to_dev(torch, w.slots())
        cache = i8.alloc_int8_cache(w.num_blocks, w.Hkv, w.D)
        out = torch.empty((w.chunk, w.Hq, w.D), dtype=torch.float32, device="cuda")
        q_i8 = torch.empty((w.chunk, w.Hq, w.D), dtype=torch.int8, device="cuda")
        q_s = torch.empty((w.chunk, w.Hq), dtype=torch.float32, device="cuda")
        bt = to_dev(torch, w.block_table)
        pws = i8.prefix_workspace(0, w.chunk, w.Hkv, w.D)
        flops = w.int8_ops()
        first = {}
        for name, thr in (("bf16", 4096), ("int8", 0)):
            ms = time_graph(torch, lambda thr=thr: i8.prefill_chunk(out, qd, kd, vd, sd, cache["k_cache"],
                                                                    cache["v_cache"], cache["k_scale"],
                                                                    cache["v_scale"], bt, 0, int8_min_history=thr,
                                                                    q_i8=q_i8, q_scale=q_s, workspace=pws), 5)
            first[name] = {"ms": ms, "tflops": flops / (ms / 1e3) / 1e12}
        first["bf16_over_int8_time"] = first["bf16"]["ms"] / first["int8"]["ms"]
        res["prefill_first_chunk_0+4096"] = first
    except Exception as e:  # pragma: no cover
        res["prefill_first_chunk_0+4096"] = {"error": str(e)[:200]}
    return res


PREFIX_HISTORIES = ((4096, 4096), (8192, 4096), (12288, 2242), (16384, 2048))


def run_prefix_by_history(torch, i8, tensor_peak, peak_kind):
    """The prefix chunk on the INT8 path and on the BF16-KV comparison path (every
    key from a bf16 paged cache), at the pages' history/chunk pairs and the
    16384 + 2048 chunk, 24 q / 4 KV heads, head_dim 256.  Each call is timed
    whole (operand tiles + attention + merge of a split last wave), two copies of
    its state rotating inside one graph."""
    res = {}
    for H, C in PREFIX_HISTORIES:
        w = wl.PrefixWorkload(f"prefix_{H}+{C}", 24, 4, 256, H, C, seed=0)
        k, v = w.kv()
        kd, vd, sd, qd = to_dev(torch, k), to_dev(torch, v), to_dev(torch, w.slots()), to_dev(torch, w.q())
        bt = to_dev(torch, w.block_table)
        dummy = torch.zeros((C, w.Hkv, w.D), dtype=torch.bfloat16, device="cuda")
        none = torch.full((C,), -1, dtype=torch.int32, device="cuda")
        int8_calls, bf16_calls = [], []
        for _ in range(2):
            c8 = i8.alloc_int8_cache(w.num_blocks, w.Hkv, w.D)
            i8.kv_quant_write(kd, vd, sd, **c8)
            q_i8 = torch.empty(qd.shape, dtype=torch.int8, device="cuda")
            q_s = torch.empty(qd.shape[:2], dtype=torch.float32, device="cuda")
            i8.kv_quant_write(dummy, dummy, none, **c8, q=qd, q_i8=q_i8, q_scale=q_s)
            cb = i8.alloc_bf16_cache(w.num_blocks, w.Hkv, w.D)
            i8.bf16_kv_write(kd, vd, sd, **cb)
            out = torch.empty((C, w.Hq, w.D), dtype=torch.float32, device="cuda")
            ws = i8.prefix_workspace(H, C, w.Hkv, w.D)
            int8_calls.append(lambda c=c8, qi=q_i8, qs=q_s, o=out, ws=ws: i8.int8_prefix_attn(
                o, qi, qs, c["k_cache"], c["v_cache"], c["k_scale"], c["v_scale"], bt, H, workspace=ws))
            bf16_calls.append(lambda c=cb, o=out, ws=ws: i8.bf16_kv_prefix_attn(
                o, qd, c["k_cache"], c["v_cache"], bt, H, workspace=ws))
        ms8 = time_rotating(torch, int8_calls, 3)
        msb = time_rotating(torch, bf16_calls, 3)
        torch.cuda.synchronize()
        assert i8.device_error() == 0
        ops = w.int8_ops()
        res[f"{H}+{C}"] = {"int8_ms": ms8, "int8_tops": ops / (ms8 / 1e3) / 1e12,
                           "int8_frac": ops / (ms8 / 1e3) / 1e12 / tensor_peak if tensor_peak else None,
                           "bf16_kv_ms": msb, "bf16_kv_tflops": ops / (msb / 1e3) / 1e12,
                           "int8_speedup": msb / ms8, "peak_kind": f"of {peak_kind} dense bf16 (burst)"}
        del int8_calls, bf16_calls
        torch.cuda.empty_cache()
    return res


def run_profile(args):
    """Decode launches only, for profilers: `--layers` copies of each history (each
    its own cache; the set exceeds L2), launched eagerly in the order 8192, 16384,
    32768, 8192, ...: `--warmup` then `--steps` launches."""
    import torch

    from int8_kv_cache_token_gb300 import build as ibuild
    ibuild.build()
    import int8_kv_cache_token_gb300 as i8
    rounds = []
    ws = {}
    for L in HISTORIES:
        w = wl.decode_outlier(L)
        k, v = w.kv(0)
        base = i8.alloc_int8_cache(w.num_blocks, w.Hkv, w.D)
        i8.kv_quant_write(to_dev(torch, k), to_dev(torch, v), to_dev(torch, w.slots(0)), **base)
        k_new, v_new, q_new = to_dev(torch, k[L - 1:L]), to_dev(torch, v[L - 1:L]), to_dev(torch, w.q())
        rounds.append([DecodeLayer(i8, torch, base, w, k_new, v_new, q_new) for _ in range(args.layers)])
        ws[L] = i8.decode_workspace(1, 24, 4, 256, w.block_tables.shape[1])
        del base
    for grp in rounds:
        for ly in grp:
            ly.produce(i8)
    torch.cuda.synchronize()
    order = [rounds[j % len(HISTORIES)][(j // len(HISTORIES)) % args.layers]
             for j in range(args.warmup + args.steps)]
    for ly in order:
        if args.profile_step:
            ly.step(i8, ws[int(ly.w.seq_lens[0])])
        else:
            ly.decode(i8, ws[int(ly.w.seq_lens[0])])
    torch.cuda.synchronize()
    assert i8.device_error() == 0
    print(json.dumps({"profile": "int8_decode_step" if args.profile_step else "int8_decode",
                      "histories": list(HISTORIES), "launches": len(order),
                      "bytes_per_launch": {str(L): wl.decode_outlier(L).kv_bytes_int8() for L in HISTORIES}}))
    return 0


def run_profile_prefix(args):
    """Prefix-chunk launches only, for profilers: the 16384 + 2048 chunk (24 q / 4 KV
    heads, head_dim 256), `--warmup` then `--steps` launches."""
    import torch

    from int8_kv_cache_token_gb300 import build as ibuild
    ibuild.build()
    import int8_kv_cache_token_gb300 as i8
    w = wl.prefix_chunk()
    k, v = w.kv()
    cache = i8.alloc_int8_cache(w.num_blocks, w.Hkv, w.D)
    i8.kv_quant_write(to_dev(torch, k), to_dev(torch, v), to_dev(torch, w.slots()), **cache)
    qd = to_dev(torch, w.q())
    q_i8 = torch.empty(qd.shape, dtype=torch.int8, device="cuda")
    q_s = torch.empty(qd.shape[:2], dtype=torch.float32, device="cuda")
    dummy = torch.zeros((w.chunk, w.Hkv, w.D), dtype=torch.bfloat16, device="cuda")
    none = torch.full((w.chunk,), -1, dtype=torch.int32, device="cuda")
    i8.kv_quant_write(dummy, dummy, none, **cache, q=qd, q_i8=q_i8, q_scale=q_s)
    out = torch.empty((w.chunk, w.Hq, w.D), dtype=torch.float32, device="cuda")
    bt = to_dev(torch, w.block_table)
    pws = i8.prefix_workspace(w.history, w.chunk, w.Hkv, w.D)
    torch.cuda.synchronize()
    for _ in range(args.warmup + args.steps):
        i8.int8_prefix_attn(out, q_i8, q_s, cache["k_cache"], cache["v_cache"], cache["k_scale"], cache["v_scale"],
                            bt, w.history, workspace=pws)
    torch.cuda.synchronize()
    assert i8.device_error() == 0
    print(json.dumps({"profile": "int8_prefix", "history": w.history, "chunk": w.chunk,
                      "launches": args.warmup + args.steps, "int8_ops_per_launch": w.int8_ops()}))
    return 0


def run_profile_gqa128(args):
    """Decode launches at head_dim 128 for profilers: batch 4 at 32768 with 32 q /
    8 KV heads (the batch-16 decode's shape at a quarter of its batch, 277 MB of
    cache, above L2); device-drawn seeded values; `--warmup` then `--steps` launches."""
    import torch

    from int8_kv_cache_token_gb300 import build as ibuild
    ibuild.build()
    import int8_kv_cache_token_gb300 as i8
    w = wl.producer_gqa_decode(B=4)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(0)
    cache = i8.alloc_int8_cache(w.num_blocks, w.Hkv, w.D)
    for b in range(w.B):
        L = int(w.seq_lens[b])
        k = torch.randn((L, w.Hkv, w.D), generator=gen, device="cuda").to(torch.bfloat16)
        v = torch.randn((L, w.Hkv, w.D), generator=gen, device="cuda").to(torch.bfloat16)
        i8.kv_quant_write(k, v, to_dev(torch, w.slots(b)), **cache)
    q = torch.randn((w.B, w.Hq, w.D), generator=gen, device="cuda").to(torch.bfloat16)
    q_i8 = torch.empty((w.B, w.Hq, w.D), dtype=torch.int8, device="cuda")
    q_s = torch.empty((w.B, w.Hq), dtype=torch.float32, device="cuda")
    dummy = torch.zeros((w.B, w.Hkv, w.D), dtype=torch.bfloat16, device="cuda")
    i8.kv_quant_write(dummy, dummy, torch.full((w.B,), -1, dtype=torch.int32, device="cuda"), **cache, q=q,
                      q_i8=q_i8, q_scale=q_s)
    out = torch.empty((w.B, w.Hq, w.D), dtype=torch.float32, device="cuda")
    ws = i8.decode_workspace(w.B, w.Hq, w.Hkv, w.D, w.block_tables.shape[1])
    bt, sl = to_dev(torch, w.block_tables), to_dev(torch, w.seq_lens)
    torch.cuda.synchronize()
    for _ in range(args.warmup + args.steps):
        i8.int8_paged_decode_attn(out, q_i8, q_s, cache["k_cache"], cache["v_cache"], cache["k_scale"],
                                  cache["v_scale"], bt, sl, ws)
    torch.cuda.synchronize()
    assert i8.device_error() == 0
    print(json.dumps({"profile": "int8_decode_gqa128", "batch": w.B, "kv_bytes": w.kv_bytes_int8(),
                      "launches": args.warmup + args.steps}))
    return 0


def run_profile_first_chunk(args):
    """High-precision first-chunk launches only, for profilers: 0 + 4096 tokens (24 q /
    4 KV heads, head_dim 256), `--warmup` then `--steps` calls (tiles + attention)."""
    import torch

    from int8_kv_cache_token_gb300 import build as ibuild
    ibuild.build()
    import int8_kv_cache_token_gb300 as i8
    w = wl.PrefixWorkload("first_chunk", 24, 4, 256, 0, 4096, seed=5)
    k, v = w.kv()
    kd, vd, qd = to_dev(torch, k), to_dev(torch, v), to_dev(torch, w.q())
    out = torch.empty((w.chunk, w.Hq, w.D), dtype=torch.float32, device="cuda")
    pws = i8.prefix_workspace(0, w.chunk, w.Hkv, w.D)
    torch.cuda.synchronize()
    for _ in range(args.warmup + args.steps):
        i8.bf16_prefix_attn(out, qd, kd, vd, workspace=pws)
    torch.cuda.synchronize()
    assert i8.device_error() == 0
    print(json.dumps({"profile": "bf16_first_chunk", "chunk": w.chunk, "launches": args.warmup + args.steps,
                      "flops_per_launch": w.int8_ops()}))
    return 0


def run_profile_producer(args):
    """Producer launches only, for profilers: 8192 tokens, 32 q / 8 KV heads, head_dim
    128; each round launches the plain producer, then the fused one (Q/K RMSNorm and
    full-width RoPE); `--warmup` then `--steps` rounds."""
    import torch

    from int8_kv_cache_token_gb300 import build as ibuild
    ibuild.build()
    import int8_kv_cache_token_gb300 as i8
    p = wl.producer_rope_tokens()
    cache = i8.alloc_int8_cache(p["num_blocks"], p["Hkv"], p["D"])
    k, v, q, s, pos, cs, qw, kw = (to_dev(torch, p[n]) for n in ("k", "v", "q", "slots", "positions", "cos_sin",
                                                              "q_norm_weight", "k_norm_weight"))
    q_i8 = torch.empty(q.shape, dtype=torch.int8, device="cuda")
    q_s = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    for _ in range(args.warmup + args.steps):
        i8.kv_quant_write(k, v, s, **cache, q=q, q_i8=q_i8, q_scale=q_s)
        i8.kv_rope_quant_write(k, v, s, **cache, positions=pos, cos_sin=cs, rotary_dim=p["rotary_dim"], q=q,
                               q_i8=q_i8, q_scale=q_s, q_norm_weight=qw, k_norm_weight=kw)
    torch.cuda.synchronize()
    assert i8.device_error() == 0
    print(json.dumps({"profile": "producer", "tokens": 8192, "rounds": args.warmup + args.steps}))
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--layers", type=int, default=LAYERS)
    ap.add_argument("--quick", action="store_true", help="skip the secondary measurements")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--cpu-seconds", type=float, default=8.0,
                    help="seconds of each of the three CPU oracle samples")
    ap.add_argument("--profile", action="store_true",
                    help="decode launches only (the three histories round-robin, --layers caches each) for ncu")
    ap.add_argument("--profile-step", action="store_true",
                    help="with --profile: the one-launch decode step instead of the plain decode")
    ap.add_argument("--profile-prefix", action="store_true",
                    help="prefix-chunk launches only (16384 + 2048 chunk) for ncu")
    ap.add_argument("--profile-gqa128", action="store_true",
                    help="decode launches at head_dim 128 (batch 4 x 32768, 32/8 heads) for ncu")
    ap.add_argument("--profile-first-chunk", action="store_true",
                    help="high-precision first-chunk launches only (0 + 4096) for ncu")
    ap.add_argument("--profile-producer", action="store_true",
                    help="plain and fused producer launches only (8192 tokens) for ncu")
    args = ap.parse_args()
    if args.profile_first_chunk:
        return run_profile_first_chunk(args)
    if args.profile_gqa128:
        return run_profile_gqa128(args)
    if args.profile_producer:
        return run_profile_producer(args)
    if args.profile:
        return run_profile(args)
    if args.profile_prefix:
        return run_profile_prefix(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())

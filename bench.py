#!/usr/bin/env python3
"""Throughput of the Code Predictor frame loop on GB300.

One step = one qp_predict_frames call: the whole 15-step loop for a batch of
B frames whose inputs are already resident in HBM.  Prints ONE JSON line
(rank 0).  ``--impl reference`` times the CPU oracle instead, on the same
workload and metric.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config C] [--impl ours|reference]

Configs (B frames): 1 = B1 greedy, 2 = B32 greedy (default), 3 = B128 greedy,
4 = B256 top-k 50 sampling, 5 = B1024 greedy with Q8_0 weights.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import glob
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "code-predictor frames/s (15 steps each) at batch B on 1 GB300; µs/step at B=1"
L2_FLUSH_BYTES = 512 << 20
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=2)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-sweep", action="store_true", help="skip the per-configuration summary")
    ap.add_argument("--step-calls", action="store_true",
                    help="time only the state-slot step calls and print their rows (a profiling entry)")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


# ---------------------------------------------------------------------------
# algorithmic work of one call: weight bytes of the whole loop plus frame I/O,
# and the FLOPs of every position's GEMMs, heads and attention
# ---------------------------------------------------------------------------

def work_of(g, B: int, gemm_format: str, sampling: bool):
    """(bytes, flops) one call must move / compute at minimum."""
    d, qw, kvw, F, V, th = g.hidden, g.n_q_heads * g.head_dim, g.n_kv_heads * g.head_dim, g.ffn, g.vocab, g.talker_hidden
    layer_params = (qw + 2 * kvw) * d + d * qw + 2 * F * d + d * F
    head_params = V * d
    proj_params = d * th
    wb = 2.0 if gemm_format == "bf16" else 34.0 / 32.0
    weight_bytes = wb * (g.n_steps * (g.layers * layer_params + head_params) + proj_params)
    io = B * (th * 4 + 4 + g.n_steps * 4          # H, q0, codes
              + th * 2 + (g.n_steps - 1) * d * 2)  # E0 row and the code-embedding rows gathered
    if sampling:
        io += B * g.n_steps * V * 4
    positions = g.n_steps + 1
    flops = B * (2 * positions * g.layers * layer_params + 2 * g.n_steps * head_params + 2 * 2 * proj_params)
    for p in range(positions):   # attention: q.k and p.v over p+1 keys, every q head
        flops += B * g.layers * g.n_q_heads * (p + 1) * g.head_dim * 4
    return weight_bytes + io, float(flops)


def _strip_comments(text: str) -> str:
    """C/C++ source without its comments (string and character literals are
    kept as they are, so a '//' inside a literal is not taken for one)."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
            out.append(" ")
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return "".join(out)


def source_hash():
    """Hash of what the kernels are built from: the CUDA sources and headers
    with comments and blank space removed (so a recorded traffic figure stays
    valid across comment-only edits) and the compiler's command-line flags."""
    from codebook_rvq_code_gb300 import build as qb
    h = hashlib.sha256()
    for f in sorted(glob.glob(os.path.join(ROOT, "codebook_rvq_code_gb300", "csrc", "*"))
                    + glob.glob(os.path.join(ROOT, "include", "*.h"))):
        h.update(" ".join(_strip_comments(open(f, encoding="utf-8").read()).split()).encode())
    h.update(" ".join(f.replace(ROOT, "<repo>") for f in qb.ARCH + qb.NVCC_FLAGS).encode())   # not where the repo sits
    return h.hexdigest()[:16]


def recorded_traffic(config_name: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current sources."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    e = d.get(config_name)
    if not e or e.get("source_hash") != source_hash():
        return None
    return e.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline and the reference arm)
# ---------------------------------------------------------------------------

def oracle_threads():
    """Threads the oracle's matrix products run on (numpy's BLAS pool)."""
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n and n[0]:
            return int(n[0])
    except Exception:
        pass
    return os.cpu_count() or 1


def cpu_model() -> str:
    """The host CPU's model name, as the kernel reports it."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def host_cpu():
    return {"cpu_model": cpu_model(), "host_cores": os.cpu_count() or 1}


_SINGLE_THREAD = """
import json, sys, time
sys.path.insert(0, {root!r})
import bench, synthetic as S
g = S.Geometry()
w = S.make_workload({cfg}, g)
rate, done, el = bench.time_oracle(g, S.workload_weights(w, g), w, {frames}, {budget})
print(json.dumps([rate, done, el]))
"""


def oracle_rate(g, raw, w, frames: int, budget_s: float, cfg=None, single_thread=False):
    """frames/s of the oracle over the first `frames` frames of the workload
    (one batch per pass, passes until about budget_s).  single_thread: in a
    fresh process whose BLAS pool is held to one thread by the environment
    (the pool size is fixed when numpy loads).  Returns (rate, frames done,
    seconds, threads used)."""
    if not single_thread:
        rate, done, el = time_oracle(g, raw, w, frames, budget_s)
        return rate, done, el, oracle_threads()
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               BLIS_NUM_THREADS="1", VECLIB_MAXIMUM_THREADS="1")
    code = _SINGLE_THREAD.format(root=ROOT, cfg=cfg, frames=frames, budget=budget_s)
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
    rate, done, el = json.loads(r.stdout.strip().splitlines()[-1])
    return rate, done, el, 1


def time_oracle(g, raw, w, frames: int, budget_s: float):
    """Run the oracle on the first `frames` frames of the workload until
    about budget_s seconds have passed; frames/s."""
    import oracle as O
    P = O.Predictor.from_raw(g, raw)
    H, q0 = w.H[:frames], w.q0[:frames]
    gum = None if w.gumbel is None else w.gumbel[:frames]
    done, t0 = 0, time.perf_counter()
    while True:
        O.predict_frames(P, H, q0, w.temperature, w.top_k, gum)
        done += frames
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return done / el, done, el


def config_of(g, w, world: int):
    """The workload's config, the same on both arms."""
    return {"workload": w.name, "B": w.B, "steps_per_frame": g.n_steps, "engine": engine_of(w.B, w.gemm_format, w.temperature > 0),
            "l2": f"flushed between timed iterations ({L2_FLUSH_BYTES >> 20} MB write)",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def reference_arm(args, g, raw, w):
    import oracle as O
    P = O.Predictor.from_raw(g, raw)
    frames = min(w.B, 8)
    H, q0 = w.H[:frames], w.q0[:frames]
    gum = None if w.gumbel is None else w.gumbel[:frames]
    for _ in range(args.warmup):
        O.predict_frames(P, H, q0, w.temperature, w.top_k, gum)
    times = []
    for _ in range(args.steps):
        t = time.perf_counter()
        O.predict_frames(P, H, q0, w.temperature, w.top_k, gum)
        times.append(time.perf_counter() - t)
    sec = sum(times)
    fps = frames * args.steps / sec
    cores = oracle_threads()
    sample = (f"first {frames} of the {w.B} frames of {w.name}, full 15-step loop, per step; "
              f"{cores} BLAS threads on {cpu_model()} ({os.cpu_count()} host cores)")
    return {
        "impl": "reference", "metric": METRIC, "value": fps, "unit": "frames/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sec / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": config_of(g, w, args.gpus),
        "cpu_baseline": {"value": fps, "unit": "frames/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": fps, "unit": "frames/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def roofline_of(g, B, gemm_format, sampling, ms_per_call, hbm, tf):
    nbytes, flops = work_of(g, B, gemm_format, sampling)
    sec = ms_per_call / 1e3
    if nbytes / (hbm * 1e9) >= flops / (tf * 1e12):
        ach, peak, unit, bound = nbytes / sec / 1e9, hbm, "GB/s", "hbm"
    else:
        ach, peak, unit, bound = flops / sec / 1e12, tf, "TFLOP/s", "tensor"
    return {"bound": bound, "achieved": ach, "peak": peak, "unit": unit, "frac": ach / peak}


def whole_job(local_ms: float, frames_per_step: int, steps: int, world: int, device=None):
    """The job's time and throughput over all ranks: each rank timed its own
    `steps` calls of `frames_per_step` frames (weak scaling, no collective on
    the data path); the job took as long as the slowest rank, and processed
    every rank's frames.  With world > 1 the max is taken with one all_reduce
    on `device` (the rank's GPU under NCCL, the CPU under gloo)."""
    total_ms = float(local_ms)
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([total_ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
    return total_ms, world * frames_per_step * steps / (total_ms / 1e3)


def engine_of(B: int, gemm_format: str, sampled: bool = False) -> str:
    """The schedule QP_ENGINE_AUTO picks (include/qp_debug.h) at the 1.7B
    geometry (either table width): the cluster engine for greedy calls of at
    most 32 frames (either weight format), else the small-batch engine for
    calls of at most 40 frames, else the tile engine."""
    if not sampled and B <= 32:
        return "cluster"
    return "small" if B <= 40 else "tile"


def median_call_ms(fn, steps, flush, stream):
    """Median CUDA-event time in ms of `steps` calls of fn, each after an L2
    flush (the rows beside the headline: the median keeps one disturbed call,
    another process's work or a clock dip, out of the figure)."""
    import statistics
    import torch
    ts = []
    for i in range(steps):
        flush.fill_(float(i))
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    return statistics.median(ts)


def sweep(g, dev, stream, steps, hbm, tf):
    """Every batch configuration once more: ms per call, frames/s, us/step
    and roofline fraction (each call a full 15-step loop, L2 flushed)."""
    import torch
    import synthetic as S
    import codebook_rvq_code_gb300 as qpk
    out = {}
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    raw_cache = {}
    for cfg in (1, 2, 3, 4, 5):
        w = S.make_workload(cfg, g)
        if w.gemm_format not in raw_cache:
            raw_cache[w.gemm_format] = S.workload_weights(w, g)
        cp = qpk.CodePredictor(g, max_batch=w.B)
        cp.load_raw_weights(raw_cache[w.gemm_format], device=dev)
        H = torch.from_numpy(w.H).to(dev)
        q0 = torch.from_numpy(w.q0).to(dev)
        samp = None if w.gumbel is None else (w.temperature, w.top_k, torch.from_numpy(w.gumbel).to(dev))
        codes = torch.empty((w.B, g.n_steps), dtype=torch.int32, device=dev)
        for _ in range(3):
            cp.predict(H, q0, out_codes=codes, sampling=samp, stream=stream)
        torch.cuda.synchronize()
        ms = median_call_ms(lambda: cp.predict(H, q0, out_codes=codes, sampling=samp, stream=stream), steps, flush,
                            stream)
        st = cp.device_status()
        cp.close()
        roof = roofline_of(g, w.B, w.gemm_format, samp is not None, ms, hbm, tf)
        out[w.name] = {"B": w.B, "engine": engine_of(w.B, w.gemm_format, w.temperature > 0), "ms_per_call": ms,
                       "frames_per_s": w.B / (ms / 1e3),
                       "us_per_step": 1e3 * ms / g.n_steps, "roofline_bound": roof["bound"],
                       "roofline_frac": roof["frac"], "device_status": st}
    return out


def cpu_sweep(g, per_config):
    """The oracle beside each configuration's GPU row: frames/s on a bounded
    sample of that configuration (its first frames, at most 32 per pass, on
    the BLAS pool's threads), and for configuration 1 also single-threaded
    at B = 1, with the µs per step that gives."""
    import synthetic as S
    raw_cache = {}
    for cfg in (1, 2, 3, 4, 5):
        w = S.make_workload(cfg, g)
        row = per_config.get(w.name)
        if row is None:
            continue
        if w.gemm_format not in raw_cache:
            raw_cache[w.gemm_format] = S.workload_weights(w, g)
        raw = raw_cache[w.gemm_format]
        frames = min(w.B, 32)
        fps, done, el, used = oracle_rate(g, raw, w, frames, 4.0)
        cb = {"value": fps, "unit": "frames/s", "cores": used, "kind": "oracle",
              "sample": f"{done} frames ({frames} per pass) of {w.name} in {el:.1f} s"}
        if cfg == 1:
            fps1, done1, el1, used1 = oracle_rate(g, raw, w, 1, 4.0, cfg=1, single_thread=True)
            cb["single_thread_B1"] = {"value": fps1, "unit": "frames/s", "cores": used1,
                                      "us_per_step": 1e6 / fps1 / g.n_steps,
                                      "sample": f"{done1} frames (1 per pass) in {el1:.1f} s"}
        row["cpu_baseline"] = dict(cb, **host_cpu())
        row["gpu_over_cpu"] = row["frames_per_s"] / fps


def deterministic_rows(g, dev, stream, steps, per_config):
    """What the deterministic mode (include/qp.h, qp_set_deterministic)
    costs: configurations 1, 2 and 4 timed again with it on, beside their
    ordinary rows."""
    import torch
    import synthetic as S
    import codebook_rvq_code_gb300 as qpk
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    raw = None
    out = {}
    for cfg in (1, 2, 4):
        w = S.make_workload(cfg, g)
        raw = raw or S.workload_weights(w, g)
        cp = qpk.CodePredictor(g, max_batch=w.B)
        cp.load_raw_weights(raw, device=dev)
        cp.set_deterministic(True)
        H = torch.from_numpy(w.H).to(dev)
        q0 = torch.from_numpy(w.q0).to(dev)
        samp = None if w.gumbel is None else (w.temperature, w.top_k, torch.from_numpy(w.gumbel).to(dev))
        codes = torch.empty((w.B, g.n_steps), dtype=torch.int32, device=dev)
        for _ in range(3):
            cp.predict(H, q0, out_codes=codes, sampling=samp, stream=stream)
        torch.cuda.synchronize()
        ms = median_call_ms(lambda: cp.predict(H, q0, out_codes=codes, sampling=samp, stream=stream), steps, flush,
                            stream)
        base = per_config.get(w.name, {}).get("ms_per_call")
        out[f"deterministic_{w.name}"] = {"ms_per_call": ms, "us_per_step": 1e3 * ms / g.n_steps,
                                          "frames_per_s": w.B / (ms / 1e3), "ordinary_ms_per_call": base,
                                          "cost": (ms / base - 1.0) if base else None,
                                          "device_status": cp.device_status()}
        cp.close()
    return out


def work_exporter(g, B: int):
    """(bytes, flops) of one call in the exporter's model layout: Talker-wide
    code tables projected at every step, Q8_0 projection and layer matrices
    (34 B per 32 weights), f16 heads and tables."""
    d, qw, kvw, F, V, th = g.hidden, g.n_q_heads * g.head_dim, g.n_kv_heads * g.head_dim, g.ffn, g.vocab, g.talker_hidden
    layer_params = (qw + 2 * kvw) * d + d * qw + 2 * F * d + d * F
    head_params, proj_params = V * d, d * th
    weight_bytes = 34.0 / 32.0 * g.n_steps * (g.layers * layer_params + proj_params) + 2.0 * g.n_steps * head_params
    io = B * (th * 4 + 4 + g.n_steps * 4 + th * 2 + (g.n_steps - 1) * g.code_embed_dim * 2)
    positions = g.n_steps + 1
    flops = B * (2 * positions * g.layers * layer_params + 2 * g.n_steps * head_params + 2 * positions * proj_params)
    for p_ in range(positions):
        flops += B * g.layers * g.n_q_heads * (p_ + 1) * g.head_dim * 4
    return weight_bytes + io, float(flops)


def exporter_rows(dev, stream, steps, hbm, tc):
    """The exporter's model layout (2048-wide code tables through small_to_mtp,
    Q8_0 matrices, f16 heads and tables), random weights, greedy, at one frame
    (the cluster engine, which streams each Q8_0 matrix as its f16 hi and lo
    images: 4 B per weight against the blocks' 1.0625) and at 256 frames (the
    tile engine, which streams the blocks and dequantises on chip)."""
    import dataclasses
    import torch
    import codebook_rvq_code_gb300 as qpk
    import synthetic as S
    g = dataclasses.replace(S.Geometry(), code_embed_dim=S.Geometry().talker_hidden)
    raw = S.make_weights(g, seed=0, gemm_format="q8_0", head_format="f16", embed_format="f16")
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    out = {}
    for B in (1, 256):
        cp = qpk.CodePredictor(g, max_batch=B)
        cp.load_raw_weights(raw, device=dev)
        H, q0 = S.toy_inputs(g, B, seed=100 + B)
        tH = torch.from_numpy(H).to(dev)
        tq = torch.from_numpy(q0).to(dev)
        codes = torch.empty((B, g.n_steps), dtype=torch.int32, device=dev)
        for _ in range(3):
            cp.predict(tH, tq, out_codes=codes, stream=stream)
        torch.cuda.synchronize()
        ms = median_call_ms(lambda: cp.predict(tH, tq, out_codes=codes, stream=stream), steps, flush, stream)
        nbytes, flops = work_exporter(g, B)
        t_hbm, t_tc = nbytes / (hbm * 1e9), flops / (tc * 1e12)
        bound = "hbm" if t_hbm >= t_tc else "tensor"
        out[f"exporter_layout_B{B}"] = {
            "workload": f"{B} frames, 1.7B geometry, 2048-wide code tables projected each step, "
                        "Q8_0 matrices, f16 heads and tables, greedy",
            "ms_per_call": ms, "us_per_step": 1e3 * ms / g.n_steps, "frames_per_s": B / (ms / 1e3),
            "engine": engine_of(B, "q8_0"),
            "device_status": cp.device_status(),
            "roofline": {"bound": bound, "frac": (t_hbm if bound == "hbm" else t_tc) / (ms / 1e3),
                         "algorithmic_bytes": nbytes, "algorithmic_flops": flops}}
        cp.close()
    return out


def work_step_call(g, B: int, n_groups: int, ctx: float):
    """Algorithmic bytes of one state-slot step call: one step's layer
    weights, one head per distinct step among the rows, each row's KV reads
    (ctx positions on average) and appended position, input code, output
    code and logits."""
    d, qw, kvw, F, V = g.hidden, g.n_q_heads * g.head_dim, g.n_kv_heads * g.head_dim, g.ffn, g.vocab
    layer_bytes = 2 * ((qw + 2 * kvw) * d + d * qw + 2 * F * d + d * F)
    kv = B * g.layers * (ctx + 1) * 2 * kvw * 2
    io = B * (4 + 4 + V * 4 + d * 2)
    return g.layers * layer_bytes + n_groups * V * d * 2 + kv + io


def sched_rows(dev, stream, steps, hbm):
    """State-slot step calls (include/qp_sched.h): B rows at mixed steps
    2..15 (one head per distinct step), each call one step of each row; the
    begin call of B new frames beside it.  L2 flushed between calls."""
    import numpy as np
    import torch
    import codebook_rvq_code_gb300 as qpk
    import synthetic as S
    g = S.Geometry()
    raw = S.make_weights(g, seed=0)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    cp = qpk.CodePredictor(g, max_batch=64)
    cp.load_raw_weights(raw, device=dev)
    out = {}

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        return median_call_ms(fn, steps, flush, stream)

    for B in (1, 32, 64):
        H, q0 = S.toy_inputs(g, B, seed=700 + B)
        tH, tq = torch.from_numpy(H).to(dev), torch.from_numpy(q0).to(dev)
        slots = list(range(B))
        q1 = torch.empty(B, dtype=torch.int32, device=dev)
        ms_begin = timed(lambda: cp.begin_frames(slots, tH, tq, out_q1=q1, stream=stream))
        st = [8] if B == 1 else [2 + b % (g.n_steps - 1) for b in range(B)]
        codes = torch.empty(B, dtype=torch.int32, device=dev)
        ms_step = timed(lambda: cp.step_frames(slots, st, q1, out_codes=codes, stream=stream))
        n_groups = len(set(st))
        ctx = float(np.mean(st))
        nbytes = work_step_call(g, B, n_groups, ctx)
        out[f"step_call_B{B}"] = {
            "workload": f"{B} rows at steps {sorted(set(st))} ({n_groups} step groups), 1.7B geometry, bf16, greedy",
            "ms_per_call": ms_step, "rows_per_s": B / (ms_step / 1e3), "begin_ms_per_call": ms_begin,
            "device_status": cp.device_status(),
            "roofline": {"bound": "hbm", "frac": nbytes / (hbm * 1e9) / (ms_step / 1e3), "algorithmic_bytes": nbytes,
                         "traffic": recorded_traffic(f"step_call_B{B}")}}
    cp.close()
    return out


def rvq_rows(dev, stream, steps, hbm):
    """The RVQ codebook kernels (include/qp_rvq.h) on a codec-sized workload:
    16 EMA codebooks of 2048 x 512 and 16384 frames' codes.  The codec's
    codebook width is not on the pages; 512 is this measurement's choice.
    Roofline: HBM, with the unique bytes each call must move (the decode
    gathers 16 rows per frame, but from a 64 MB table that stays in L2)."""
    import numpy as np
    import torch
    import codebook_rvq_code_gb300 as qpk
    Q, K, D, N = 16, 2048, 512, 16384
    rng = np.random.default_rng(5)
    usage = torch.from_numpy(rng.uniform(0.0, 50.0, size=(Q, K)).astype(np.float32)).to(dev)
    es = torch.from_numpy(rng.standard_normal((Q, K, D)).astype(np.float32)).to(dev) * usage[:, :, None]
    codes = torch.from_numpy(rng.integers(0, K, size=(N, Q), dtype=np.int32)).to(dev)
    cbs = torch.empty_like(es)
    out = torch.empty((N, D), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        return median_call_ms(fn, steps, flush, stream)

    # frame-feedback embeddings (qp_code_embeddings) of configuration 5's batch:
    # 1024 frames x 15 codes, bf16 rows in, f32 rows out
    import synthetic as S
    g = S.Geometry()
    Bf = 1024
    cp = qpk.CodePredictor(g, max_batch=1)
    cp.load_raw_weights(S.make_weights(g, seed=0), device=dev)
    fcodes = torch.from_numpy(rng.integers(0, g.vocab, size=(Bf, g.n_steps), dtype=np.int32)).to(dev)
    fout = torch.empty((Bf, g.n_steps, g.hidden), dtype=torch.float32, device=dev)
    ms_f = timed(lambda: cp.code_embeddings(fcodes, out=fout, stream=stream))
    fst = cp.device_status()
    cp.close()
    fb = Bf * g.n_steps * (g.hidden * 2 + g.hidden * 4 + 4)
    ms_n = timed(lambda: qpk.rvq_normalize(es, usage, out=cbs, stream=stream))
    ms_d = timed(lambda: qpk.rvq_decode(cbs, codes, out=out, stream=stream))
    nb = 2 * Q * K * D * 4 + Q * K * 4
    db = Q * K * D * 4 + N * Q * 4 + N * D * 4
    return {
        "code_embeddings": {"workload": f"{Bf} frames x {g.n_steps} codes, {g.hidden}-wide bf16 tables -> f32",
                            "ms": ms_f, "frames_per_s": Bf / (ms_f / 1e3), "device_status": fst,
                            "roofline": {"bound": "hbm", "achieved": fb / (ms_f / 1e3) / 1e9, "peak": hbm,
                                         "unit": "GB/s", "frac": fb / (ms_f / 1e3) / 1e9 / hbm, "bytes": fb}},
        "rvq_normalize": {"workload": f"{Q} EMA codebooks x {K} x {D} f32", "ms": ms_n,
                          "roofline": {"bound": "hbm", "achieved": nb / (ms_n / 1e3) / 1e9, "peak": hbm,
                                       "unit": "GB/s", "frac": nb / (ms_n / 1e3) / 1e9 / hbm, "bytes": nb}},
        "rvq_decode": {"workload": f"{N} frames x {Q} codes into {K} x {D} f32 codebooks", "ms": ms_d,
                       "frames_per_s": N / (ms_d / 1e3),
                       "gathered_GB_per_s": N * Q * D * 4 / (ms_d / 1e3) / 1e9,
                       "roofline": {"bound": "hbm", "achieved": db / (ms_d / 1e3) / 1e9, "peak": hbm,
                                    "unit": "GB/s", "frac": db / (ms_d / 1e3) / 1e9 / hbm, "bytes": db}},
    }


# ---------------------------------------------------------------------------

def main():
    args = parse()
    import numpy as np
    import synthetic as S

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    g = S.Geometry()
    w = S.make_workload(args.config, g)

    if args.impl == "reference":
        if rank != 0:
            return
        raw = S.workload_weights(w, g)
        print(json.dumps(reference_arm(args, g, raw, w)), flush=True)
        return

    import torch
    import torch.distributed as dist
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if args.step_calls:
        from codebook_rvq_code_gb300 import build as qb
        qb.build()
        rows = sched_rows(dev, torch.cuda.current_stream(dev), max(1, args.steps), peaks()[0])
        if rank == 0:
            print(json.dumps({"step_calls": rows}), flush=True)
        return

    from codebook_rvq_code_gb300 import build as qb
    qb.build()
    import codebook_rvq_code_gb300 as qpk

    raw = S.workload_weights(w, g)
    cp = qpk.CodePredictor(g, max_batch=w.B)
    cp.load_raw_weights(raw, device=dev)
    B = w.B
    H = torch.from_numpy(w.H).to(dev)
    q0 = torch.from_numpy(w.q0).to(dev)
    codes = torch.empty((B, g.n_steps), dtype=torch.int32, device=dev)
    samp = None
    if w.gumbel is not None:
        samp = (w.temperature, w.top_k, torch.from_numpy(w.gumbel).to(dev))
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def call():
        cp.predict(H, q0, out_codes=codes, sampling=samp, stream=stream)

    for _ in range(max(3, args.warmup)):
        call()
    torch.cuda.synchronize()
    if cp.device_status() != 0:
        raise RuntimeError("device status set during warm-up")
    if world > 1:
        dist.barrier()

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(local_rank) as clk:
        torch.cuda.synchronize()
        for i in range(args.steps):
            flush.fill_(float(i))          # evict the previous call's lines from L2
            starts[i].record(stream)
            call()
            ends[i].record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms, value = whole_job(sum(step_ms), B, args.steps, world, dev if world > 1 else None)
    ms_per_step = total_ms / args.steps
    launches = cp.launches_per_call(B, samp is not None) * args.steps

    # end to end through the host-buffer entry point: pinned H/q0 in, codes out
    e2e = None
    if not args.no_e2e:
        Hh = torch.from_numpy(w.H).pin_memory()
        qh = torch.from_numpy(w.q0).pin_memory()
        ch = torch.empty((B, g.n_steps), dtype=torch.int32).pin_memory()
        for _ in range(2):
            cp.predict_host(Hh, qh, ch, sampling=samp, stream=stream)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            cp.predict_host(Hh, qh, ch, sampling=samp, stream=stream)
        el = time.perf_counter() - t0
        e2e = {"value": world * B * args.steps / el, "unit": "frames/s",
               "h2d_bytes_per_step": int(Hh.numel() * 4 + qh.numel() * 4),
               "d2h_bytes_per_step": int(ch.numel() * 4)}

    if rank != 0:
        cp.close()
        if world > 1:
            dist.destroy_process_group()
        return

    # One call is one kernel launch of at most a few ms, timed on its own:
    # the burst tensor-core peak is its ceiling (the sustained one is for
    # kernels timed inside a seconds-long loop).
    hbm, tf_burst, tf_sust, peak_src = peaks()
    nbytes, flops = work_of(g, B, w.gemm_format, samp is not None)
    sec = ms_per_step / 1e3
    t_hbm, t_tc = nbytes / (hbm * 1e9), flops / (tf_burst * 1e12)
    if t_hbm >= t_tc:
        roof = {"bound": "hbm", "achieved": nbytes / sec / 1e9, "peak": hbm, "unit": "GB/s"}
    else:
        roof = {"bound": "tensor", "achieved": flops / sec / 1e12, "peak": tf_burst, "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["peak_source"] = f"{peak_src} (MEASURED_PEAKS.json)" if peak_src == "measured" else "fallback"
    roof["algorithmic_bytes_per_launch"] = nbytes
    roof["algorithmic_flops_per_launch"] = flops
    roof["traffic"] = recorded_traffic(w.name)

    line = {
        "metric": METRIC, "value": value, "unit": "frames/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16",
        "arithmetic": ("tensor-core operands f16 (bf16 weights converted exactly; Q8_0 weights as an exact f16 "
                       "pair hi + lo), f32 accumulation; norms, softmax and decisions f32"),
        "weights": w.gemm_format,
        "data": "synthetic",
        "config": config_of(g, w, world),
        "us_per_step": 1e3 * ms_per_step / g.n_steps,
        "roofline": roof,
        "gpu_launches": launches,
        "clocks": clk.summary(),
    }
    if e2e:
        line["e2e"] = e2e
    if not args.no_sweep and world == 1:
        line["per_config"] = sweep(g, dev, stream, max(5, min(args.steps, 20)), hbm, tf_burst)
        b1 = [v for v in line["per_config"].values() if v["B"] == 1]
        if b1:
            line["us_per_step_at_B1"] = b1[0]["us_per_step"]
        line["next_rows"] = rvq_rows(dev, stream, max(5, min(args.steps, 20)), hbm)
        line["next_rows"].update(exporter_rows(dev, stream, max(5, min(args.steps, 20)), hbm, tf_burst))
        line["next_rows"].update(sched_rows(dev, stream, max(5, min(args.steps, 20)), hbm))
        line["next_rows"].update(deterministic_rows(g, dev, stream, max(5, min(args.steps, 20)), line["per_config"]))
    if not args.no_cpu_baseline:
        frames = min(B, 32)
        fps, done, el, used = oracle_rate(g, raw, w, frames, 10.0)
        line["cpu_baseline"] = dict({"value": fps, "unit": "frames/s", "cores": used, "kind": "oracle",
                                     "sample": f"{done} frames ({frames} per pass) of {w.name} in {el:.1f} s"},
                                    **host_cpu())
        if not args.no_sweep and world == 1:
            cpu_sweep(g, line["per_config"])
    cp.close()
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

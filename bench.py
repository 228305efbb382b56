#!/usr/bin/env python3
"""Benchmark of one CfC K-loop training step (forward + BPTT + dW/db/du/dh0) on GB300.

A step is one pass of the whole hot path over one batch: cfc_forward (persistent cluster
recurrence), then cfc_backward (reverse-time recurrence, the weight-gradient contraction,
the reduce_axis0 bias sum, du), captured once into a CUDA graph and replayed.  The workload is
the pages' shape (B=32 sequences, K=64 steps, C=128 hidden channels, n_x=48 inputs; page
"K-loop Parallelization -- Block-per-Batch Kernel Refactor", section "Problem") with seeded
synthetic inputs.  Printed: one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload I] [--impl ours|reference]

--impl reference times the fp64 CPU oracle (a plain, deliberately slow program) on a bounded
sample of the same workload on the host cores.  Under torchrun each rank runs its own replica
(weak scaling, no data-path collective) and rank 0 prints the max-over-ranks time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "CfC fwd+BPTT seq·steps/s at B=32,K=64,C=128; % of HBM & tensor-pipe roofline"
UNIT = "seq·steps/s"
L2_FLUSH_BYTES = 256 << 20  # > 129 MB L2


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", type=int, default=1)
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's B (a smaller case of it, e.g. for profiling)")
    ap.add_argument("--seq", type=int, default=None, help="override the workload's K")
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="CPU work budget of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-largest", action="store_true",
                    help="skip the record of the largest (2048 x 128 x 256) workload")
    ap.add_argument("--dw-modes", default="0,1,2",
                    help="tensor-core weight-gradient modes timed on the largest workload")
    ap.add_argument("--profile", action="store_true",
                    help="only run --steps eager training steps of the workload (for ncu "
                         "captures: the step's kernels and nothing else), print nothing")
    ap.add_argument("--dw-mode", type=int, default=0, help="weight-gradient mode (--profile)")
    return ap.parse_args()


def workload(args):
    """The selected workload, with B / K overridden when asked (renamed after its sizes)."""
    import dataclasses

    from recurrent_cfc_cell_gb300 import inputs

    w = inputs.CONFIGS[args.workload]
    if args.batch is None and args.seq is None:
        return w
    B = args.batch if args.batch is not None else w.B
    K = args.seq if args.seq is not None else w.K
    name = f"{w.name.split('_')[0]}_B{B}_K{K}_nx{w.n_x}_C{w.C}"
    return dataclasses.replace(w, name=name, B=B, K=K)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            d = json.load(fh)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "sm_max_mhz": d.get("sm_max_mhz", 2070.0), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "sm_max_mhz": 2070.0, "source": "fallback"}


# ---------------------------------------------------------------- algorithmic work per unit
def fwd_fused(w) -> bool:
    """cfc_forward forms the input projection inside the tensor-core recurrence (B >= 384 at
    C = 256, B >= 768 at C = 128, n_x <= 64): one launch, no X in memory."""
    return w.C in (128, 256) and w.B >= (384 if w.C == 256 else 768) and w.n_x <= 64


def work_per_unit(w):
    """FLOPs and HBM bytes per (batch row, step) of each stage (fp32 = 4 bytes)."""
    C, n_x, n_in = w.C, w.n_x, w.n_in
    return {
        # input projection W_u u + b for all steps: reads u, writes the 4C values X in place
        "proj": {"flop": 8 * C * n_x, "bytes": 4 * (n_x + 4 * C)},
        # forward recurrence: W_h h_{t-1} (4C x C); reads X and ts, writes h_t and the cache
        "fwd_rec": {"flop": 8 * C * C, "bytes": 4 * (4 * C + 1 + 4 * C)},
        # the whole forward as cfc_forward runs it: projection and recurrence; where the
        # tensor-core recurrence forms the projection itself X never goes through memory
        # (reads u and ts, writes h_t and the cache), otherwise both stages' bytes
        "fwd": {"flop": 8 * C * n_x + 8 * C * C,
                "bytes": (4 * (n_x + 1 + 4 * C) if fwd_fused(w)
                          else 4 * (n_x + 4 * C) + 4 * (4 * C + 1 + 4 * C))},
        # BPTT recurrence: W_h^T d_pre (4C x C); reads dH, cache, ts; writes d_pre
        "bwd_rec": {"flop": 8 * C * C, "bytes": 4 * (C + 3 * C + 1 + 4 * C)},
        # dW contraction (4C x n_in per row) + du (4C x n_x) + db; reads d_pre, u, h
        "grad": {"flop": 8 * C * n_in + 8 * C * n_x + 4 * C,
                 "bytes": 4 * (4 * C + n_x + C) + 4 * 4 * C + 4 * n_x},
    }


def source_digest(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def workload_tag(w) -> str:
    """Short workload name used in the profile summaries' file names (e.g. pages_B32_K64)."""
    return "_".join(w.name.split("_")[:3])


def profiled_traffic(kernel: str, sources: list[str], workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it matches the current source."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(path):
        return None
    fields = {}
    with open(path) as fh:
        for line in fh:
            if ":" in line and line.startswith("- "):
                k, v = line[2:].split(":", 1)
                v = v.strip()
                m = re.match(r"`([^`]*)`", v)  # a backticked value may carry a note after it
                fields[k.strip()] = m.group(1) if m else v.split()[0] if v else v
    if fields.get("source_sha256_16") != source_digest(sources):
        return None
    try:
        return float(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------- clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.remove(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- reference arm (oracle)
def run_reference(args, rank, world):
    if rank != 0:
        return 0
    import oracle
    from recurrent_cfc_cell_gb300 import inputs

    w = workload(args)
    inp = inputs.make_inputs(w)
    # calibrate one single-row oracle step, then size each step's sample so the whole run
    # stays near a minute of CPU work
    one = {k: (v[:, :1] if k in ("u", "ts", "dH") else v[:1] if k == "h0" else v)
           for k, v in inp.items()}
    t0 = time.perf_counter()
    oracle.step(one)
    t_row = max(time.perf_counter() - t0, 1e-4)
    budget = 60.0 / max(1, args.steps + args.warmup)
    rows = max(1, min(w.B, int(budget / t_row)))
    sample = {k: (v[:, :rows] if k in ("u", "ts", "dH") else v[:rows] if k == "h0" else v)
              for k, v in inp.items()}
    for _ in range(args.warmup):
        oracle.step(sample)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.step(sample)
    dt = time.perf_counter() - t0
    units = rows * w.K * args.steps
    value = units / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": dict(w.describe()),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{rows} of {w.B} batch rows x K={w.K} per step, fp64 C, "
                                   "single thread"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def _oracle_shard(w, r0: int, r1: int, seconds: float):
    """Run the oracle on batch rows r0..r1 of the workload for `seconds`; (units, seconds)."""
    import oracle
    from recurrent_cfc_cell_gb300 import inputs

    inp = inputs.make_inputs(w)
    sub = {k: (v[:, r0:r1] if k in ("u", "ts", "dH") else v[r0:r1] if k == "h0" else v)
           for k, v in inp.items()}
    n = 0
    t0 = time.perf_counter()
    while True:
        oracle.step(sub)
        n += 1
        dt = time.perf_counter() - t0
        if dt >= seconds:
            return n * (r1 - r0) * w.K, dt


def cpu_baseline(w, seconds: float) -> dict:
    """The oracle on the host cores: single-threaded on the whole workload, and on all cores
    with the batch rows (independent sequences) split over spawned processes; the all-core
    figure is the reported one."""
    import concurrent.futures
    import multiprocessing

    # The single-thread leg on at most 128 rows: one oracle step of the whole largest workload
    # (2048 rows x 128 steps) would take minutes; rows are independent, so the rate per row-step
    # is the same.
    units1, dt1 = _oracle_shard(w, 0, min(w.B, 128), seconds)
    single = units1 / dt1
    cores = min(os.cpu_count() or 1, w.B)
    bounds = [(w.B * i // cores, w.B * (i + 1) // cores) for i in range(cores)]
    ctx = multiprocessing.get_context("spawn")
    with concurrent.futures.ProcessPoolExecutor(max_workers=cores, mp_context=ctx) as ex:
        res = list(ex.map(_oracle_shard, [w] * cores, [b[0] for b in bounds],
                          [b[1] for b in bounds], [seconds] * cores))
    total = sum(u for u, _ in res) / max(dt for _, dt in res)
    return {"value": total, "unit": UNIT, "cores": cores, "kind": "oracle",
            "single_thread_value": single,
            "sample": f"the workload (B={w.B}, K={w.K}) split by batch rows over {cores} "
                      f"processes, each running fp64 C oracle steps on its rows for "
                      f"{seconds:.0f} s; single thread on {min(w.B, 128)} rows: "
                      f"{single:.0f} {UNIT}"}


# ---------------------------------------------------------------- parity (oracle leg)
def _bf16_bits_to_f32(a):
    import numpy as np

    return (np.asarray(a).astype(np.uint16).astype(np.uint32) << 16).view(np.float32)


def decode_dpre(raw, C: int, dw_mode: int):
    """The workspace head after cfc_backward -> fp32-valued d_pre [K, B, 4, C] (the layout the
    public header documents for each mode)."""
    import numpy as np

    raw = np.asarray(raw)
    if dw_mode in (2, 3):
        return raw
    K, B = raw.shape[:2]
    d = _bf16_bits_to_f32(raw[:, :, 0, : 4 * C]).astype(np.float64)
    if dw_mode == 0:
        d = d + _bf16_bits_to_f32(raw[:, :, 1, : 4 * C])
    return d.reshape(K, B, 4, C)


def oracle_parity(inp: dict, gpu: dict, rows=None) -> dict:
    """Part of the CPU-baseline leg: one more run of the oracle (on all rows, or on the listed
    rows when the workload is too large for a bounded sample), compared with the GPU's outputs
    of the timed step: max|x - y| / max|y| per tensor (dW and db only on all rows)."""
    import numpy as np

    import oracle

    if rows is not None:
        rows = np.asarray(rows)
        inp = {k: (np.ascontiguousarray(v[:, rows]) if k in ("u", "ts", "dH")
                   else np.ascontiguousarray(v[rows]) if k == "h0" else v)
               for k, v in inp.items()}
        gpu = {k: (v[:, rows] if k in ("H", "cache", "d_pre", "du") else v[rows] if k == "dh0"
                   else None) for k, v in gpu.items()}
    ref = oracle.step(inp)
    ref["cache"] = np.stack([ref["ff1"], ref["ff2"], ref["gate"]], axis=2)
    out = {}
    for k in ("H", "cache", "d_pre", "du", "dh0", "dW", "db"):
        if gpu.get(k) is None or k not in ref:
            continue
        out[k] = oracle.rel_err(gpu[k], ref[k])
    return {"max_rel_err": out, "rows": "all" if rows is None else [int(r) for r in rows],
            "metric": "max|x-y| / max|y| per tensor against the fp64 oracle"}


# ---------------------------------------------------------------- measured peaks
def measure_peaks(torch, _lib, dev) -> dict:
    """fp32 FMA rate and L2 read bandwidth from the library's probes, dense tf32 from a cuBLAS
    matmul (torch, TF32 allowed), the SM count; best of several CUDA-event-timed runs."""
    props = torch.cuda.get_device_properties(dev)
    sms = props.multi_processor_count
    stream = torch.cuda.current_stream()

    def best(fn, reps=5):
        ts = []
        for k in range(reps + 2):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            work = fn()
            b.record(stream)
            torch.cuda.synchronize()
            if k >= 2:
                ts.append((a.elapsed_time(b), work))
        return min(ts)

    out = torch.empty(sms * 8 * 256, dtype=torch.float32, device=dev)
    ms, flop = best(lambda: _lib.probe_fma(out, sms * 8, 20000))
    fma = flop / (ms * 1e-3) / 1e12
    buf = torch.ones(8 << 20, dtype=torch.float32, device=dev)  # 32 MB, inside the 129 MB L2
    ms, nbytes = best(lambda: _lib.probe_l2_read(buf, 40, out, sms * 8))
    l2 = nbytes / (ms * 1e-3) / 1e9
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = True
    try:
        a = torch.randn(8192, 8192, device=dev)
        b = torch.randn(8192, 8192, device=dev)
        ms, fl = best(lambda: (torch.matmul(a, b), 2.0 * 8192 ** 3)[1])
        tf32 = fl / (ms * 1e-3) / 1e12
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev
    del a, b, buf, out
    return {"sms": sms, "fp32_fma_tflops": fma, "l2_read_gbs": l2, "tf32_tflops": tf32,
            "how": "fp32: cfc_probe_fma (8 packed-FMA chains per thread, 8 CTAs of 256 per SM); "
                   "L2: cfc_probe_l2_read over a 32 MB buffer, 40 passes; tf32: torch.matmul "
                   "8192^3 with TF32 allowed (cuBLAS); best of 5, CUDA events"}


# ---------------------------------------------------------------- stage timing
def stage_times(torch, _lib, st, flush, stream, n: int) -> dict:
    """Device time of each stage of one step, CUDA events between the stage calls, L2 flushed
    before each group: the whole forward (cfc_forward, as the step runs it), then its two stage
    entry points (the projection, the forward recurrence), the BPTT recurrence (into an
    fp32 d_pre at the workspace head, the same kernels as in the step), the standalone gradient
    stage (cfc_weight_grad from that fp32 d_pre), and the whole cfc_backward.  "grad" is the
    gradient chain as cfc_backward runs it (BPTT writing the contraction's operand rows
    directly): cfc_backward minus the BPTT stage."""
    i = st.inputs
    n_bptt = _lib.bptt_workspace_bytes(st.B, st.K, st.C, st.n_x)
    bptt_ws = torch.empty(n_bptt, dtype=torch.uint8, device=st.device) if n_bptt else None
    d32 = st.d_pre_fp32_view
    stages = [
        ("fwd", lambda: st.forward()),
        ("proj", lambda: _lib.cfc_input_projection(i["u"], i["W"], i["b"], st.H, st.cache)),
        ("fwd_rec", lambda: _lib.cfc_forward_recurrence(i["h0"], i["W"], i["ts"], st.H,
                                                       st.cache, ws=st.fws)),
        ("bwd_rec", lambda: _lib.cfc_backward_recurrence_ws(i["dH"], i["W"], i["ts"], st.cache,
                                                           d32, st.dh0, bptt_ws)),
        ("grad_standalone", lambda: _lib.cfc_weight_grad(d32, i["u"], i["h0"], i["W"], st.H,
                                                         st.dW, st.db, st.du, st.ws,
                                                         dw_mode=st.dw_mode)),
        ("bwd", lambda: st.backward()),
    ]
    marks = [[torch.cuda.Event(enable_timing=True) for _ in range(len(stages) + 1)]
             for _ in range(n)]
    for ev in marks:
        flush.zero_()
        ev[0].record(stream)
        for j, (_, fn) in enumerate(stages):
            fn()
            ev[j + 1].record(stream)
    torch.cuda.synchronize()
    out = {name: sum(ev[j].elapsed_time(ev[j + 1]) for ev in marks) / n
           for j, (name, _) in enumerate(stages)}
    out["grad"] = max(out["bwd"] - out["bwd_rec"], 1e-6)
    return out


def kernel_table(w, stage_ms: dict, pk: dict, mp: dict | None) -> dict:
    wpu = work_per_unit(w)
    fp32_peak = mp["fp32_fma_tflops"] if mp else None
    tab = {}
    for name in ("fwd", "proj", "fwd_rec", "bwd_rec", "grad"):
        t = stage_ms[name]
        flop = wpu[name]["flop"] * w.units
        byt = wpu[name]["bytes"] * w.units
        e = {"ms": t, "tflops": flop / (t * 1e-3) / 1e12, "gbs": byt / (t * 1e-3) / 1e9}
        e["hbm_frac"] = e["gbs"] / pk["hbm_gbs"]
        e["bf16_frac"] = e["tflops"] / pk["bf16_tflops"]
        if fp32_peak:
            e["fp32_frac"] = e["tflops"] / fp32_peak
        tab[name] = e
    return tab


def timed_replays(torch, st, flush, stream, steps: int) -> float:
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for k in range(steps):
        flush.zero_()
        starts[k].record(stream)
        st.replay()
        ends[k].record(stream)
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in zip(starts, ends)) / steps


class _Bf16StateStep:
    """The bf16-state training step (cfc_forward_bf16 + cfc_backward_bf16) in one CUDA graph."""

    def __init__(self, torch, _lib, w, d, dev):
        B, K, C, n_x = w.B, w.K, w.C, w.n_x
        self.H = torch.empty((K, B, C), dtype=torch.bfloat16, device=dev)
        self.cache = torch.empty((K, B, 3, C), dtype=torch.bfloat16, device=dev)
        self.fws = torch.empty(_lib.forward_bf16_workspace_bytes(B, K, C, n_x),
                               dtype=torch.uint8, device=dev)
        self.ws = torch.empty(_lib.workspace_bytes(B, K, C, n_x, _lib.CFC_DW_BF16),
                              dtype=torch.uint8, device=dev)
        f32 = dict(dtype=torch.float32, device=dev)
        self.out = {"dW": torch.empty((4, C, n_x + C), **f32), "db": torch.empty((4, C), **f32),
                    "du": torch.empty((K, B, n_x), **f32), "dh0": torch.empty((B, C), **f32)}
        self.d, self._lib, self.torch = d, _lib, torch
        self.run()  # eager first: sets the kernels' attributes before capture
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self.run()
        torch.cuda.current_stream().wait_stream(s)
        with torch.cuda.graph(self.graph):
            self.run()

    def run(self):
        d, o, L = self.d, self.out, self._lib
        L.cfc_forward_bf16(d["u"], d["h0"], d["W"], d["b"], d["ts"], self.H, self.cache, self.fws)
        L.cfc_backward_bf16(d["dH"], d["u"], d["h0"], d["W"], d["ts"], self.H, self.cache,
                            o["dW"], o["db"], o["du"], o["dh0"], self.ws)

    def replay(self):
        self.graph.replay()


def bf16_state_record(torch, _lib, w, d, dev, flush, stream, steps: int) -> dict:
    """Step time of the bf16-state variant on workload `w` (graph replays, L2 flushed), and the
    bytes of the activations kept from forward to backward (H and the cache) in each dtype."""
    sb = _Bf16StateStep(torch, _lib, w, d, dev)
    for _ in range(3):
        flush.zero_()
        sb.replay()
    torch.cuda.synchronize()
    ms = timed_replays(torch, sb, flush, stream, steps)
    status = _lib.device_status()
    act = w.units * 4 * w.C
    return {"ms_per_step": ms, "value": w.units / (ms * 1e-3), "unit": UNIT, "steps": steps,
            "activation_bytes_bf16": 2 * act, "activation_bytes_fp32": 4 * act,
            "device_status": status}


class _DecayStep:
    """One training step of the pages' tau-decay cell (cfc_decay_forward + cfc_decay_backward)."""

    def __init__(self, torch, _lib, w, d, dev):
        B, K, C, n_x = w.B, w.K, w.C, w.n_x
        f32 = dict(dtype=torch.float32, device=dev)
        self.H = torch.empty((K, B, C), **f32)
        self.E = torch.empty((K, B, C), **f32)
        self.out = {"dW": torch.empty((C, n_x + C), **f32), "db": torch.empty((C,), **f32),
                    "dtau": torch.empty((C,), **f32), "dx": torch.empty((K, B, n_x), **f32),
                    "dh0": torch.empty((B, C), **f32)}
        self.ws = torch.empty(_lib.decay_workspace_bytes(B, K, C, n_x), dtype=torch.uint8,
                              device=dev)
        self.d, self._lib, self.graph = d, _lib, None

    def forward(self):
        d = self.d
        self._lib.cfc_decay_forward(d["x"], d["h0"], d["W"], d["b"], d["tau"], d["ts"], self.H,
                                    self.E)

    def backward(self):
        d, o = self.d, self.out
        self._lib.cfc_decay_backward(d["dH"], d["x"], d["h0"], d["W"], d["tau"], d["ts"], self.H,
                                     self.E, o["dW"], o["db"], o["dtau"], o["dx"], o["dh0"],
                                     self.ws)

    def run(self):
        self.forward()
        self.backward()

    def capture(self, torch):
        self.run()
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self.run()
        torch.cuda.current_stream().wait_stream(s)
        with torch.cuda.graph(self.graph):
            self.run()

    def replay(self):
        self.graph.replay()


def _timed(torch, fn, flush, stream, n: int) -> float:
    """Mean ms of fn() over n calls, each after an L2 flush, CUDA events on `stream`."""
    tot = 0.0
    for _ in range(n):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        torch.cuda.synchronize()
        tot += a.elapsed_time(b)
    return tot / n


def decay_record(torch, _lib, inputs, dev, flush, stream, mp, steps: int,
                 with_parity: bool) -> list:
    """The pages' tau-decay cell on its pages-shaped and larger-batch workloads: step time
    (graph replays, L2 flushed), the two stages, the recurrences against the measured FP32 FMA
    rate, and the oracle comparison of every output on the pages-shaped workload."""
    recs = []
    for w in inputs.DECAY_CONFIGS[1:]:
        inp = inputs.make_decay_inputs(w)
        d = {k: torch.from_numpy(v).to(dev).contiguous() for k, v in inp.items()}
        st = _DecayStep(torch, _lib, w, d, dev)
        st.capture(torch)
        for _ in range(3):
            flush.zero_()
            st.replay()
        torch.cuda.synchronize()
        ms = timed_replays(torch, st, flush, stream, steps)
        fwd_ms = _timed(torch, st.forward, flush, stream, 20)
        bwd_ms = _timed(torch, st.backward, flush, stream, 20)
        # Per (b, t) unit: the recurrent mat-vec (2 C^2 flop) in each direction, the projection
        # (2 C n_x), and the weight and input gradients (2 C (n_in + 1) + 2 C n_x).
        C, n_x = w.C, w.n_x
        rec_flop = 2.0 * C * C * w.units
        peak = mp["fp32_fma_tflops"] if mp else None
        fwd_tf = rec_flop / (fwd_ms * 1e-3) / 1e12
        bwd_tf = rec_flop / (bwd_ms * 1e-3) / 1e12
        rec = {"workload": w.name, "config": w.describe(), "ms_per_step": ms,
               "value": w.units / (ms * 1e-3), "unit": UNIT, "steps": steps,
               "stages_ms": {"forward": fwd_ms, "backward": bwd_ms},
               "recurrence_tflops": {"forward": fwd_tf, "backward": bwd_tf},
               "fp32_fma_frac": ({"forward": fwd_tf / peak, "backward": bwd_tf / peak}
                                 if peak else None),
               "flop_per_unit": {"recurrences": 4.0 * C * C, "projection": 2.0 * C * n_x,
                                 "gradients": 2.0 * C * (n_x + C + 1) + 2.0 * C * n_x},
               "device_status": _lib.device_status()}
        if with_parity and w.units <= 4096:
            import oracle
            import oracle.decay

            ref = oracle.decay.step(inp)
            got = {"H": st.H.cpu().numpy(), "E": st.E.cpu().numpy()}
            got.update({k: v.cpu().numpy() for k, v in st.out.items()})
            rec["parity"] = {"max_rel_err": {k: oracle.rel_err(got[k], ref[k]) for k in got},
                             "metric": "max|x-y| / max|y| per tensor against the fp64 oracle"}
        recs.append(rec)
        del st
        torch.cuda.empty_cache()
    return recs


def outputs_np(st) -> dict:
    out = {k: v.cpu().numpy() for k, v in st.outputs().items()}
    out["d_pre"] = decode_dpre(out["d_pre"], st.C, st.dw_mode)
    return out


def largest_record(torch, _lib, inputs, KLoopStep, to_device, dev, flush, stream, pk, mp,
                   modes, local: int, with_parity: bool) -> dict:
    """The largest workload (B=2048, K=128, n_x=64, C=256), measured in this run: step time
    (graph replays, L2 flushed), stage times, each stage's fractions, clocks, and the weight-
    gradient stage in each tensor-core mode with its tensor-pipe fraction."""
    w = inputs.CONFIGS[4]
    inp = inputs.make_inputs(w)
    dinp = to_device(inp, dev)
    st = KLoopStep(w.B, w.K, w.C, w.n_x, device=dev).bind(**dinp)
    st.capture()
    for _ in range(3):
        flush.zero_()
        st.replay()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    ms = timed_replays(torch, st, flush, stream, 10)
    clock_info = clocks.stop()
    parity = None
    if with_parity:
        gpu = outputs_np(st)
        parity = oracle_parity(inp, gpu, rows=[0, 777, 1500, w.B - 1])
        del gpu
    stg = stage_times(torch, _lib, st, flush, stream, 5)
    kern = kernel_table(w, stg, pk, mp)
    # The contraction stage per mode: flops of dW (with db) and du, against the peak of the
    # operand type; accurate mode issues three products per algorithmic one.
    wpu = work_per_unit(w)
    flop = wpu["grad"]["flop"] * w.units
    contraction = {}
    names = {0: "accurate", 1: "bf16", 2: "tf32"}
    del st
    torch.cuda.empty_cache()
    bf16 = bf16_state_record(torch, _lib, w, dinp, dev, flush, stream, 10)
    torch.cuda.empty_cache()
    for m in modes:
        sm = KLoopStep(w.B, w.K, w.C, w.n_x, dw_mode=m, device=dev).bind(**dinp)
        sm.forward()
        t = stage_times(torch, _lib, sm, flush, stream, 5)
        peak = mp["tf32_tflops"] if (m == 2 and mp) else pk["bf16_tflops"]
        ach = flop / (t["grad"] * 1e-3) / 1e12
        issued = 3 if m == 0 else 1
        contraction[names[m]] = {
            "grad_ms": t["grad"], "grad_standalone_ms": t["grad_standalone"],
            "achieved_tflops": ach, "peak_tflops": peak, "frac": ach / peak,
            "issued_frac": issued * ach / peak,
            "peak_note": ("measured tf32 (cuBLAS)" if m == 2 else "measured dense bf16 burst")}
        del sm
        torch.cuda.empty_cache()
    return {"workload": w.name, "ms_per_step": ms, "value": w.units / (ms * 1e-3), "unit": UNIT,
            "steps": 10, "warmup": 3, "stages": stg, "kernels": kern,
            "contraction": contraction, "clocks": clock_info, "parity_sampled": parity,
            "bf16_state": bf16}


# ---------------------------------------------------------------- our arm
def main():
    args = parse_args()
    rank, world, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, rank, world)

    import torch
    import torch.distributed as dist

    from recurrent_cfc_cell_gb300 import _lib, build, inputs
    from recurrent_cfc_cell_gb300.step import KLoopStep, to_device

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    if rank == 0:
        build.build()
    if world > 1:
        dist.barrier()
    _lib.load()

    w = workload(args)
    inp = inputs.make_inputs(w)
    dinp = to_device(inp, dev)
    if args.profile:
        st = KLoopStep(w.B, w.K, w.C, w.n_x, dw_mode=args.dw_mode, device=dev).bind(**dinp)
        for _ in range(args.steps):
            st.run()
        torch.cuda.synchronize()
        return 0 if _lib.device_status() == 0 else 1
    st = KLoopStep(w.B, w.K, w.C, w.n_x, device=dev).bind(**dinp)
    st.capture()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        st.replay()
    torch.cuda.synchronize()

    # ---- timed region: K graph replays, L2 flushed between them (flush outside the events)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    for k in range(args.steps):
        flush.zero_()
        starts[k].record(stream)
        st.replay()
        ends[k].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clock_info = clocks.stop()
    ms = sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / args.steps
    if world > 1:
        t = torch.tensor([ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    units_per_step = w.units * world
    value = units_per_step / (ms * 1e-3)
    launches_per_step = _lib.step_launches(w.B, w.K, w.C, w.n_x)

    pk = peaks()
    mp = measure_peaks(torch, _lib, dev)
    stage_ms = stage_times(torch, _lib, st, flush, stream, min(args.steps, 200))
    kernels = kernel_table(w, stage_ms, pk, mp)
    n_bptt_ws = _lib.bptt_workspace_bytes(w.B, w.K, w.C, w.n_x)
    # The dominant kernel: the larger of the two recurrences (each stage is one launch).
    # (Where the forward forms the projection itself, its stage is the whole cfc_forward.)
    fwd_key = "fwd" if fwd_fused(w) else "fwd_rec"
    dominant = max((fwd_key, "bwd_rec"), key=lambda k: stage_ms[k])
    # Which kernel that stage ran: the tensor-core recurrences serve batches of at least 384
    # (forward) or 129 (BPTT) rows at C = 256, 768 or 513 at C = 128; the CUDA-core ones
    # the rest.
    tc_fwd = w.C in (128, 256) and w.B >= (384 if w.C == 256 else 768)
    tc = tc_fwd if dominant == fwd_key else n_bptt_ws > 0
    kname = {("fwd_rec", False): "cfc_fwd_kernel", ("bwd_rec", False): "cfc_bwd_kernel",
             ("fwd_rec", True): "cfc_fwd_tc_kernel", ("fwd", True): "cfc_fwd_tc_kernel",
             ("bwd_rec", True): "cfc_bwd_l2x_kernel"}[(dominant, tc)]
    ksrc = ["recurrent_cfc_cell_gb300/csrc/" + kname[: -len("_kernel")] + ".cu",
            "recurrent_cfc_cell_gb300/csrc/cfc_ptx.cuh",
            "recurrent_cfc_cell_gb300/csrc/cfc_kernels.h"]
    achieved = kernels[dominant]["tflops"]
    if tc:
        # Algorithmic fp32-equivalent flops against the dense bf16 tensor peak; each product
        # is issued as 3 MMAs (hi*hi, hi*lo, lo*hi of the fp16 terms) in both recurrences.
        n_mma = 3
        roofline = {"bound": "tensor", "achieved": achieved, "peak": pk["bf16_tflops"],
                    "unit": "TFLOP/s", "frac": achieved / pk["bf16_tflops"],
                    "traffic": profiled_traffic(kname, ksrc, workload_tag(w)),
                    "kernel": kname,
                    "peak_note": f"dense bf16 burst, {pk['source']}; {n_mma} MMAs per product, "
                                 f"issued frac {n_mma * achieved / pk['bf16_tflops']:.3f}",
                    "hbm_frac": kernels[dominant]["gbs"] / pk["hbm_gbs"]}
    else:
        peak = mp["fp32_fma_tflops"]
        roofline = {"bound": "alu", "achieved": achieved, "peak": peak,
                    "unit": "TFLOP/s", "frac": achieved / peak,
                    "traffic": profiled_traffic(kname, ksrc, workload_tag(w)),
                    "kernel": kname,
                    "peak_note": "fp32 FMA rate measured in this run by cfc_probe_fma",
                    "hbm_frac": kernels[dominant]["gbs"] / pk["hbm_gbs"]}

    # ---- end to end through the public API with host buffers: every step copies its inputs
    # in from pinned host memory and its gradients out to pinned host memory (one packed copy
    # each way by the library's copy kernel, captured with the step's kernels in one graph).
    ste = KLoopStep(w.B, w.K, w.C, w.n_x, device=dev).stage_host()
    for k, v in inp.items():
        ste.host_in[k].copy_(torch.from_numpy(v))
    h2d, d2h = ste.io_bytes()
    n_e2e = min(args.steps, 200)
    ste.capture(with_host_io=True)
    for _ in range(3):
        ste.replay()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n_e2e)]
    for a, b in ev:
        flush.zero_()
        a.record(stream)
        ste.replay()
        b.record(stream)
    torch.cuda.synchronize()
    e2e_ms = sum(a.elapsed_time(b) for a, b in ev) / n_e2e
    if world > 1:
        t = torch.tensor([e2e_ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_ms = float(t.item())
    e2e = {"value": units_per_step / (e2e_ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms}
    status = _lib.device_status()
    gpu_out = outputs_np(st) if rank == 0 else None
    del ste
    bf16 = bf16_state_record(torch, _lib, w, dinp, dev, flush, stream, min(args.steps, 200))
    status = status or bf16["device_status"]
    decay = decay_record(torch, _lib, inputs, dev, flush, stream, mp, min(args.steps, 200),
                         rank == 0 and not args.no_cpu_baseline)
    status = status or max(r["device_status"] for r in decay)
    largest = None
    if not args.no_largest and w.name != inputs.CONFIGS[4].name:
        modes = [int(m) for m in args.dw_modes.split(",") if m.strip()]
        largest = largest_record(torch, _lib, inputs, KLoopStep, to_device, dev, flush, stream,
                                 pk, mp, modes, local, rank == 0 and world == 1)
        status = status or _lib.device_status()

    if rank == 0:
        cpu = None
        parity = None
        if not args.no_cpu_baseline and world == 1:
            cpu = cpu_baseline(w, args.cpu_seconds)
            # the oracle once more on the whole workload when that is a bounded sample
            parity = oracle_parity(inp, gpu_out) if w.units <= 65536 else oracle_parity(
                inp, gpu_out, rows=[0, w.B // 2, w.B - 1])
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": dict(w.describe(), parallelism=f"replicas{world}",
                           l2="flushed between timed steps (256 MB write)",
                           graph="one CUDA graph per step", dw_mode="accurate"),
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps, "clocks": clock_info,
            "kernels": kernels, "stages_ms": stage_ms, "parity": parity,
            "measured_peaks": mp, "largest_config": largest, "bf16_state": bf16,
            "decay_cell": decay,
            "device_status": status, "peaks_source": pk["source"],
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())

#!/usr/bin/env python
"""Benchmark of the cartridge-attention hot path on GB300.

One step = one pass over every step of the path on synthetic data:
  a1  cartridge write: f32 leaf rows -> bf16 shadow        (cart_attn_fwd given
      the f32 leaves: its prep launch writes the shadow into the workspace)
  a2-a4  training forward (RoPE at p+i, end-aligned mask)  (cart_attn_fwd)
  a5-a8  training backward into the cartridge rows          (cart_attn_bwd, reading
      the forward's workspace)
         [N > 1: all-reduce(SUM) of the cartridge gradients]
  a9  one decode step of 64 conversations behind a shared cartridge
                                                            (cart_attn_decode)
Workloads: self-study training B=4, Hq=32, Hkv=8, d=128, p=2048 (row 0
frozen), n=1024, bf16 Q/K/V with f32 cartridge leaves; serving decode B=64,
p=4096 shared, private lengths ~U{0..1024}.  `--workload longctx` swaps the
training part for B=1, Hq=64, p=8192, n=4096.

`value` is the training fwd+bwd throughput in algorithmic TFLOP/s (4*d FLOPs
per visible (query, key) pair forward, 2.5x that backward), summed over
ranks; the decode throughput (algorithmic HBM GB/s, the shared cartridge
counted once) is reported under "decode".  L2 is flushed between timed steps,
outside the timed events: a 256 MiB write, then a 256 MiB read of another
buffer, so that no dirty line of the flush is written back inside a timed
kernel (decode.dirty_l2 reports the decode after the write alone).

`--impl reference` times the fp64 CPU oracle on the host cores instead, on a
bounded sample of the same workload.
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
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "cartridge-attn fwd+bwd TFLOP/s and decode HBM GB/s (% of GB300 roofline)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", choices=("selfstudy", "longctx"), default="selfstudy")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--workload-steps", type=int, default=10,
                    help="timed steps of the other training workloads (long-context fwd+bwd, "
                         "equivalence-gate fwd; 0: skip)")
    ap.add_argument("--record-traffic", metavar="CSV",
                    help="write profiles/dram_traffic.json from an ncu CSV of DRAM bytes and exit")
    ap.add_argument("--traffic-steps", type=int, default=1,
                    help="whole bench steps the --record-traffic capture covers")
    ap.add_argument("--traffic-command", default="", help="the command that made the capture")
    ap.add_argument("--ext-steps", type=int, default=20,
                    help="timed steps of the packed-training and span-decode lines (0: skip)")
    ap.add_argument("--profile-only", action="store_true",
                    help="run --steps untimed steps of the headline step (training step + "
                         "decode step) after --warmup ones and exit: the command ncu captures")
    return ap.parse_args()


# ------------------------------------------------------------------ peaks ----
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return {k: float(pk[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_src_sha(name: str) -> str:
    csrc = os.path.join(ROOT, "trained_kv_prefix_gb300", "csrc")
    files = {"bwd_dkdv": ["bwd.cu"], "bwd_dq": ["bwd.cu"], "fwd": ["fwd.cu"],
             "decode": ["decode.cu", "fwd.cu"]}
    f = files.get(name)
    if f is None:
        return ""
    h = hashlib.sha256()
    for part in f + ["ptx.cuh", "internal.cuh"]:
        with open(os.path.join(csrc, part), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:12]


TRAFFIC_JSON = os.path.join(ROOT, "profiles", "dram_traffic.json")
def ncu_key(name: str):
    """The bench's kernel key of an ncu kernel name (demangled); the decode
    step's kernels (the cartridge pass is fwd_kernel in decode mode, template
    mode 2) all count under "decode"."""
    m = re.search(r"(\w+_kernel)<([^>]*)>", name)
    if not m:
        return None
    base, targs = m.group(1), [t.strip() for t in m.group(2).split(",")]
    if base == "fwd_kernel":
        return "decode" if len(targs) > 1 and targs[1] == "2" else "fwd"
    return {"dkdv_kernel": "bwd_dkdv", "dq_kernel": "bwd_dq",
            "decode_private_kernel": "decode", "decode_merge_kernel": "decode"}.get(base)


def ncu_traffic(kernel: str, workload: str):
    """Per-launch DRAM bytes of `kernel` on `workload`, from the data file that
    `--record-traffic` writes from an ncu capture, when it was taken on the
    current source of that kernel (else None)."""
    try:
        with open(TRAFFIC_JSON) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    ent = rec.get("kernels", {}).get(f"{kernel}@{workload}")
    if not ent or ent.get("src_sha") != kernel_src_sha(kernel):
        return None
    return int(ent["bytes"])


def record_traffic(csv_path: str, steps: int, workloads: dict, command: str):
    """Parse an ncu --csv capture of dram__bytes_read.sum and
    dram__bytes_write.sum covering `steps` whole bench steps and write the
    per-step DRAM bytes of each bench kernel (summed over its launches in a
    step) into profiles/dram_traffic.json, with the hash of the sources they
    were taken on.  `workloads` maps a kernel key to its workload name."""
    import csv
    with open(csv_path, newline="") as f:
        rows = [r for r in csv.reader(f) if r]
    hdr = next(i for i, r in enumerate(rows) if "Kernel Name" in r and "Metric Name" in r)
    cols = rows[hdr]
    ki, mi, vi = cols.index("Kernel Name"), cols.index("Metric Name"), cols.index("Metric Value")
    ui = cols.index("Metric Unit") if "Metric Unit" in cols else None
    scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "KB": 1024, "MB": 1 << 20,
             "GB": 1 << 30}
    tot = {}
    for r in rows[hdr + 1:]:
        if len(r) <= max(ki, mi, vi) or not r[mi].startswith("dram__bytes_"):
            continue
        key = ncu_key(r[ki])
        if key is None:
            continue
        unit = r[ui] if ui is not None else "byte"
        tot[key] = tot.get(key, 0.0) + float(r[vi].replace(",", "")) * scale.get(unit, 1)
    try:
        with open(TRAFFIC_JSON) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        rec = {}
    rec["what"] = ("DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of each bench "
                   "kernel per step (the decode entry sums the kernels of one decode step), "
                   "from one ncu capture; bench.py uses an entry while src_sha matches")
    kern = rec.setdefault("kernels", {})
    for key, b in tot.items():
        kern[f"{key}@{workloads.get(key, '')}"] = {
            "bytes": int(round(b / max(1, steps))), "src_sha": kernel_src_sha(key),
            "command": command}
    with open(TRAFFIC_JSON, "w") as f:
        json.dump(rec, f, indent=1, sort_keys=True)
        f.write("\n")
    return rec


# ----------------------------------------------------------------- clocks ----
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.25)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                self.out = ""
        return False

    def summary(self):
        rows = []
        for line in (self.out or "").splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append(dict(sm=float(parts[0]), smax=float(parts[1]), power=float(parts[2]),
                                 hw=parts[4], hwt=parts[5], swt=parts[6], swp=parts[7]))
            except ValueError:
                continue
        if not rows:
            return None
        load = [r for r in rows if r["power"] > 200.0] or rows
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in load),
                "sm_max_mhz": max(r["smax"] for r in rows), "samples": len(rows),
                "samples_under_load": len(load), "reasons": sorted(reasons)}


# --------------------------------------------------------------- L2 flush ----
class L2Flush:
    """Between timed steps no input may sit in L2 (129 MB on GB300).  Calling
    the object writes a 256 MiB buffer (the flush) and then reads a second
    256 MiB buffer, so that L2 holds clean lines of that buffer: the dirty
    lines the write leaves behind are written back here, outside the timed
    region, instead of inside the next timed kernel (where they would cost
    HBM write bandwidth that belongs to the flush, not to the kernel).
    `dirty()` is the write alone, for comparison."""

    def __init__(self, dev):
        import torch
        self.buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        self.clean_buf = torch.ones(32 << 20, dtype=torch.int64, device=dev)

    def __call__(self):
        self.buf.zero_()
        self.sink = self.clean_buf.sum()

    def dirty(self):
        self.buf.zero_()


# ------------------------------------------------------------- accounting ----
def decode_bytes(s, lens) -> int:
    """Algorithmic HBM bytes of one decode step: the shared cartridge once,
    each conversation's private rows 0..L_b (K and V), q / k_new / v_new / o,
    and the appended row."""
    import numpy as np
    row = s.Hkv * s.d * 2
    L = np.asarray(lens, dtype=np.int64)
    cart = 2 * s.p * row
    priv = 2 * int((L + 1).sum()) * row
    io = s.B * (2 * s.Hq * s.d * 2 + 2 * s.Hkv * s.d * 2) + 2 * s.B * row + s.B * 4
    return cart + priv + io


def kernel_work(name, ts, ds, lens):
    """(amount, unit) of algorithmic work one launch of `name` performs."""
    pairs = ts.B * ts.Hq * ts.pairs_per_head()
    if name == "fwd":
        return 4.0 * ts.d * pairs, "flop"
    if name == "bwd_dkdv":   # S^T, dP^T, dV, dK: 4 of the 5 algorithmic GEMMs
        return 8.0 * ts.d * pairs, "flop"
    if name == "bwd_dq":     # dQ (the S and dP it recomputes are not counted)
        return 2.0 * ts.d * pairs, "flop"
    if name == "decode":     # the whole step: its kernels overlap by design
        return float(decode_bytes(ds, lens)), "byte"
    return None, None


# ------------------------------------------------------------- reference ----
def oracle_sample_flops(ts, heads, rows):
    pairs = 0
    for i in range(rows[0], rows[1]):
        pairs += ts.p + i + 1
    pairs *= ts.B * heads
    return 4.0 * ts.d * pairs * 3.5   # fwd + bwd (2.5x)


def run_oracle_sample(ts, inp64, kv_heads, rows):
    import oracle
    G = ts.Hq // ts.Hkv
    oracle.fwd(inp64["q"], inp64["k"], inp64["v"], inp64["kc"], inp64["vc"], theta=ts.theta,
               heads=(kv_heads[0] * G, kv_heads[1] * G), rows=rows)
    oracle.bwd(inp64["q"], inp64["k"], inp64["v"], inp64["kc"], inp64["vc"], inp64["do"],
               theta=ts.theta, kv_heads=kv_heads, rows=rows)


def cpu_baseline(ts, target_s=15.0):
    """The oracle as it stands, timed on this host's cores on a bounded sample
    (query rows at the end of the sequence, half of the kv groups, every
    sequence), sized for roughly `target_s` seconds."""
    import oracle
    from trained_kv_prefix_gb300 import synth
    inp = synth.train_inputs(ts)
    a = {k: synth.f64(v) for k, v in inp.items()}
    kvh = (0, max(1, ts.Hkv // 2))
    heads = (kvh[1] - kvh[0]) * (ts.Hq // ts.Hkv)
    probe = (ts.n - 16, ts.n)
    t0 = time.perf_counter()
    run_oracle_sample(ts, a, kvh, probe)
    dt = time.perf_counter() - t0
    per_row = max(dt / 16, 1e-6)
    nrows = int(max(16, min(ts.n, target_s / per_row)))
    rows = (ts.n - nrows, ts.n)
    t0 = time.perf_counter()
    run_oracle_sample(ts, a, kvh, rows)
    dt = time.perf_counter() - t0
    flops = oracle_sample_flops(ts, heads, rows)
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle", "seconds": round(dt, 2),
            "sample": (f"{ts.name} fwd+bwd, fp64 oracle, all {ts.B} sequences, kv groups "
                       f"{kvh[0]}..{kvh[1] - 1} ({heads} query heads), query rows "
                       f"{rows[0]}..{rows[1] - 1} of {ts.n}; algorithmic FLOPs of the sample")}


def reference_arm(args, ts):
    import oracle
    from trained_kv_prefix_gb300 import dist as cdist, synth
    rank, world, _ = cdist.env_rank_world()
    if rank != 0:
        return
    oracle.build()
    inp = synth.train_inputs(ts)
    a = {k: synth.f64(v) for k, v in inp.items()}
    kvh = (0, max(1, ts.Hkv // 2))
    heads = (kvh[1] - kvh[0]) * (ts.Hq // ts.Hkv)
    # size one step so that warmup + steps stay within ~150 s of CPU time
    t0 = time.perf_counter()
    run_oracle_sample(ts, a, kvh, (ts.n - 8, ts.n))
    per_row = max((time.perf_counter() - t0) / 8, 1e-6)
    budget = 150.0 / max(1, args.steps + args.warmup)
    nrows = int(max(1, min(ts.n, budget / per_row)))
    rows = (ts.n - nrows, ts.n)
    for _ in range(args.warmup):
        run_oracle_sample(ts, a, kvh, rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run_oracle_sample(ts, a, kvh, rows)
    dt = time.perf_counter() - t0
    flops = oracle_sample_flops(ts, heads, rows) * args.steps
    value = flops / dt / 1e12
    sample = (f"{ts.name} fwd+bwd, fp64 oracle, all {ts.B} sequences, {heads} query heads, "
              f"query rows {rows[0]}..{rows[1] - 1} per step")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_name(ts), "sample": sample},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def measure_extensions(args, ts, ds, dev, rank, peaks, flush):
    """The packed-segment training step and the span-verify decode step,
    each timed alone (CUDA events on the launch stream, L2 flushed outside
    the events between steps).  Packed: ts's heads and cartridge, 8
    segments of U{1..n} tokens (the longest n); work = 3.5 x 4d x Hq x the
    visible pairs of every segment.  Span: the serving decode workload with
    4 new tokens per conversation; bytes = the shared cartridge once + every
    conversation's private rows 0..L+3 (K and V) + q/k/v/o of the span."""
    import numpy as np
    import torch
    from trained_kv_prefix_gb300 import cartattn, synth

    stream = torch.cuda.current_stream(dev)

    def timed(fn, steps):
        for _ in range(3):
            flush()
            fn()
        torch.cuda.synchronize(dev)
        tot = 0.0
        for _ in range(steps):
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            e1.synchronize()
            tot += e0.elapsed_time(e1)
        return tot / steps  # ms

    out = {}
    segs = 8
    lens = synth.packed_lengths(ts.n, segs, seed=ts.seed + 1000 * rank)
    pin = synth.packed_inputs(ts, lens, seed=ts.seed + 1000 * rank)
    g = {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in pin.items()}
    kcb = g["kc"].to(torch.bfloat16)
    vcb = g["vc"].to(torch.bfloat16)
    n = g["max_seqlen"]
    o, lse = cartattn.cart_attn_fwd_packed(g["q"], g["k"], g["v"], kcb, vcb, g["cu"], n,
                                           frozen_prefix=ts.frozen_prefix, theta=ts.theta)

    def packed_step():
        cartattn.cart_attn_fwd_packed(g["q"], g["k"], g["v"], kcb, vcb, g["cu"], n,
                                      frozen_prefix=ts.frozen_prefix, theta=ts.theta, o=o, lse=lse)
        cartattn.cart_attn_bwd_packed(g["q"], g["k"], g["v"], kcb, vcb, o, lse, g["do"], g["cu"], n,
                                      frozen_prefix=ts.frozen_prefix, theta=ts.theta)

    L = lens.astype(np.float64)
    flops = 3.5 * 4.0 * ts.d * ts.Hq * float((L * ts.p + L * (L + 1) / 2).sum())
    ms = timed(packed_step, args.ext_steps)
    tf = flops / (ms * 1e-3) / 1e12
    out["packed_train"] = {
        "metric": "packed-segment fwd+bwd TFLOP/s", "value": tf, "unit": "TFLOP/s",
        "frac": tf / peaks["bf16_tflops"], "ms_per_step": ms,
        "config": {"segments": segs, "tokens": int(L.sum()), "max_seqlen": n,
                   "lengths": [int(x) for x in lens], "Hq": ts.Hq, "Hkv": ts.Hkv, "d": ts.d,
                   "cartridge_rows": ts.p}}
    span = 4
    din = {k: v.to(dev) for k, v in synth.decode_span_inputs(ds, span, seed=ds.seed + 1000 * rank).items()}
    ws = torch.empty(cartattn.decode_span_workspace_size(ds.B, span, ds.Hq, ds.Hkv, ds.d, ds.p,
                                                         ds.cache_rows), dtype=torch.uint8,
                     device=dev)
    od = torch.empty_like(din["q"])

    def span_step():
        cartattn.cart_attn_decode_span(din["q"], din["k_new"], din["v_new"], din["kc"], din["vc"],
                                       din["k_cache"], din["v_cache"], din["lens"], theta=ds.theta,
                                       o=od, workspace=ws)

    ms = timed(span_step, args.ext_steps)
    Ls = din["lens"].cpu().numpy().astype(np.int64)
    row = ds.Hkv * ds.d * 2
    byts = 2 * ds.p * row + int((Ls + span).sum()) * 2 * row + ds.B * span * (
        2 * ds.Hq * ds.d * 2 + 2 * row + 2 * row)
    out["span_decode"] = {
        "metric": "span-verify decode HBM GB/s", "value": byts / (ms * 1e-3) / 1e9, "unit": "GB/s",
        "frac": byts / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], "ms_per_step": ms,
        "tokens_per_s": ds.B * span / (ms * 1e-3),
        "config": {"conversations": ds.B, "span": span, "cartridge_rows": ds.p,
                   "bytes_per_step": byts}}
    assert cartattn.device_status() == 0
    return out


def measure_train_workload(ts, dev, rank, peaks, flush, steps, bwd=True):
    """One more training workload timed alone: `steps` passes of the
    cartridge write + forward (+ backward), CUDA events on the launch stream
    around each pass, L2 flushed outside the events.  Work = 4d FLOPs per
    visible (query, key) pair forward and 2.5x that backward.  Per-kernel
    figures come from the library's launch trace over as many passes again
    (its events, between launches, cost time and end the kernels'
    programmatic chaining, so the timed passes run without it)."""
    import torch
    from trained_kv_prefix_gb300 import cartattn, synth

    stream = torch.cuda.current_stream(dev)
    tin = {k: v.to(dev) for k, v in synth.train_inputs(ts, seed=ts.seed + 1000 * rank).items()}
    o = torch.empty_like(tin["q"])
    lse = torch.empty((ts.B, ts.Hq, ts.n), dtype=torch.float32, device=dev)
    g = cartattn.geom(ts.B, ts.n, ts.Hq, ts.Hkv, ts.d, ts.p, ts.frozen_prefix, None, ts.theta)
    # f32 cartridge leaves: the forward's prep launch writes their bf16 shadow
    ws_f = torch.empty(cartattn.fwd_workspace_size(g, 0, cartattn.CART_F32), dtype=torch.uint8,
                       device=dev)
    grads = None
    if bwd:
        grads = dict(dq=torch.empty_like(tin["q"]), dk=torch.empty_like(tin["k"]),
                     dv=torch.empty_like(tin["v"]),
                     dkc=torch.empty((ts.p, ts.Hkv, ts.d), dtype=torch.float32, device=dev),
                     dvc=torch.empty((ts.p, ts.Hkv, ts.d), dtype=torch.float32, device=dev))
        ws_b = torch.empty(cartattn.bwd_reuse_workspace_size(g, 0, cartattn.CART_F32),
                           dtype=torch.uint8, device=dev)

    def step():
        cartattn.cart_attn_fwd(tin["q"], tin["k"], tin["v"], tin["kc"], tin["vc"],
                               frozen_prefix=ts.frozen_prefix, theta=ts.theta, o=o, lse=lse,
                               workspace=ws_f)
        if bwd:
            cartattn.cart_attn_bwd(tin["q"], tin["k"], tin["v"], tin["kc"], tin["vc"], o, lse,
                                   tin["do"],
                                   frozen_prefix=ts.frozen_prefix, theta=ts.theta,
                                   workspace=ws_b, fwd_workspace=ws_f, **grads)

    for _ in range(3):
        flush()
        step()
    torch.cuda.synchronize(dev)
    tot = 0.0
    for _ in range(steps):
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step()
        e1.record(stream)
        e1.synchronize()
        tot += e0.elapsed_time(e1)
    cartattn.trace_read(True)  # drop older records
    cartattn.trace_enable(True)
    for _ in range(steps):
        flush()
        step()
    torch.cuda.synchronize(dev)
    cartattn.trace_enable(False)
    trace = cartattn.trace_read(True)
    assert cartattn.device_status() == 0
    ms = tot / steps
    flops = ts.fwd_flops() + (ts.bwd_flops() if bwd else 0.0)
    tf = flops / (ms * 1e-3) / 1e12
    per = {}
    for name, t in trace:
        e = per.setdefault(name, [0, 0.0])
        e[0] += 1
        e[1] += t
    kernels = {}
    for name, (cnt, t) in per.items():
        ent = {"launches": cnt, "avg_us": round(t / cnt * 1e3, 2)}
        amt, unit = kernel_work(name, ts, None, None)
        if amt is not None and unit == "flop":
            ach = amt / (t / cnt * 1e-3) / 1e12
            ent.update(achieved=ach, unit="TFLOP/s", frac=ach / peaks["bf16_tflops"])
        kernels[name] = ent
    return {"metric": ("fwd+bwd" if bwd else "fwd") + " TFLOP/s", "value": tf, "unit": "TFLOP/s",
            "frac": tf / peaks["bf16_tflops"], "ms_per_step": ms, "steps": steps,
            "flops_per_step": flops,
            "config": {"workload": workload_name(ts, decode=False), "B": ts.B, "n": ts.n,
                       "Hq": ts.Hq, "Hkv": ts.Hkv, "d": ts.d, "cartridge_rows": ts.p,
                       "pairs_per_head": ts.pairs_per_head()},
            "kernels": kernels}


def workload_name(ts, decode=True):
    name = (f"{ts.name}-train B={ts.B} Hq={ts.Hq} Hkv={ts.Hkv} d={ts.d} p={ts.p} "
            f"(row 0 frozen) n={ts.n} bf16/f32-leaves")
    return name + (" + serving-decode B=64 Hq=32 Hkv=8 d=128 p=4096 L~U{0..1024}" if decode else "")


# ------------------------------------------------------------------ ours ----
def main():
    args = parse_args()
    from trained_kv_prefix_gb300 import synth
    if args.record_traffic:
        ts = synth.SELFSTUDY if args.workload == "selfstudy" else synth.LONGCTX
        wl = {"fwd": ts.name, "bwd_dkdv": ts.name, "bwd_dq": ts.name, "decode": synth.DECODE.name}
        rec = record_traffic(args.record_traffic, args.traffic_steps, wl, args.traffic_command)
        print(json.dumps(rec, indent=1))
        return
    ts = synth.SELFSTUDY if args.workload == "selfstudy" else synth.LONGCTX
    if args.impl == "reference":
        reference_arm(args, ts)
        return

    import numpy as np
    import torch
    from trained_kv_prefix_gb300 import build as cbuild
    from trained_kv_prefix_gb300 import cartattn
    from trained_kv_prefix_gb300 import dist as cdist

    rank, world, local = cdist.env_rank_world()
    has_pg = cdist.init_from_env("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        cbuild.build()
    cdist.barrier(dev)
    cartattn.lib()
    peaks, peaks_src = load_peaks()
    ds = synth.DECODE

    # ---- inputs (per-rank seeds: every rank trains on its own sequences)
    tin = {k: v.to(dev) for k, v in synth.train_inputs(ts, seed=ts.seed + 1000 * rank).items()}
    din = {k: v.to(dev) for k, v in synth.decode_inputs(ds, seed=ds.seed + 1000 * rank).items()}
    lens = din["lens"].cpu().numpy()
    o = torch.empty_like(tin["q"])
    lse = torch.empty((ts.B, ts.Hq, ts.n), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(tin["q"]), torch.empty_like(tin["k"]), torch.empty_like(tin["v"])
    dkc = torch.empty((ts.p, ts.Hkv, ts.d), dtype=torch.float32, device=dev)
    dvc = torch.empty_like(dkc)
    od = torch.empty_like(din["q"])
    g = cartattn.geom(ts.B, ts.n, ts.Hq, ts.Hkv, ts.d, ts.p, ts.frozen_prefix, None, ts.theta)
    # f32 cartridge leaves: the forward's prep launch writes their bf16 shadow
    # into ws_f, where the backward reads it
    ws_f = torch.empty(cartattn.fwd_workspace_size(g, 0, cartattn.CART_F32), dtype=torch.uint8,
                       device=dev)
    ws_b = torch.empty(cartattn.bwd_reuse_workspace_size(g, 0, cartattn.CART_F32),
                       dtype=torch.uint8, device=dev)
    ws_d = torch.empty(cartattn.decode_workspace_size(ds.B, ds.Hq, ds.Hkv, ds.d, ds.p,
                                                      ds.cache_rows), dtype=torch.uint8, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)

    def train_part():
        cartattn.cart_attn_fwd(tin["q"], tin["k"], tin["v"], tin["kc"], tin["vc"],
                               frozen_prefix=ts.frozen_prefix, theta=ts.theta, o=o, lse=lse,
                               workspace=ws_f)
        cartattn.cart_attn_bwd(tin["q"], tin["k"], tin["v"], tin["kc"], tin["vc"], o, lse, tin["do"],
                               frozen_prefix=ts.frozen_prefix, theta=ts.theta, dq=dq, dk=dk, dv=dv,
                               dkc=dkc, dvc=dvc, workspace=ws_b, fwd_workspace=ws_f)
        cdist.allreduce_cartridge_grads(dkc, dvc)

    def decode_part():
        cartattn.cart_attn_decode(din["q"], din["k_new"], din["v_new"], din["kc"], din["vc"],
                                  din["k_cache"], din["v_cache"], din["lens"], theta=ds.theta,
                                  o=od, workspace=ws_d)

    if args.profile_only:
        # exactly warmup + steps headline steps of the library's kernels
        for _ in range(args.warmup + args.steps):
            flush()
            train_part()
            decode_part()
        torch.cuda.synchronize(dev)
        assert cartattn.device_status() == 0
        if rank == 0:
            print(json.dumps({"profile_only": True, "steps": args.steps, "warmup": args.warmup}))
        return

    for _ in range(max(args.warmup, 3)):
        flush()
        train_part()
        decode_part()
    torch.cuda.synchronize(dev)
    assert cartattn.device_status() == 0

    # ---- timed region
    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    cdist.barrier(dev)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        wall0 = time.perf_counter()
        for i in range(K):
            flush()
            evs[i][0].record(stream)
            train_part()
            evs[i][1].record(stream)
            decode_part()
            evs[i][2].record(stream)
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - wall0
    cdist.barrier(dev)
    torch.cuda.synchronize(dev)
    status = cartattn.device_status()
    train_ms = sum(e[0].elapsed_time(e[1]) for e in evs)
    dec_ms = sum(e[1].elapsed_time(e[2]) for e in evs)
    # the per-kernel figures: the same K steps again under the library's
    # launch trace (events on the launch streams around each launch; they
    # cost time between launches and end the programmatic chaining of the
    # training kernels, so the timed steps above run without them)
    cartattn.trace_read(True)
    cartattn.trace_enable(True)
    for i in range(K):
        flush()
        train_part()
        decode_part()
    torch.cuda.synchronize(dev)
    cartattn.trace_enable(False)
    status |= cartattn.device_status()
    trace = cartattn.trace_read(True)
    # one trace record per launch, except the decode step: its three kernels
    # (cartridge pass, private pass, merge) are chained and traced as one
    n_launch = sum(3 if name == "decode" else 1 for name, _ in trace)
    train_ms, dec_ms = cdist.max_over_ranks([train_ms, dec_ms], dev)

    flops_step = ts.fwd_flops() + ts.bwd_flops()
    value = world * flops_step * K / (train_ms * 1e-3) / 1e12
    dbytes = decode_bytes(ds, lens)
    dec_gbs = world * dbytes * K / (dec_ms * 1e-3) / 1e9

    # the decode step after a write-only flush (its dirty lines are written
    # back while the decode reads), for comparison with the headline
    dirty_ms = 0.0
    for _ in range(K):
        flush.dirty()
        d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        d0.record(stream)
        decode_part()
        d1.record(stream)
        d1.synchronize()
        dirty_ms += d0.elapsed_time(d1)
    dirty_ms = cdist.max_over_ranks([dirty_ms], dev)[0]
    dec_dirty = {"value": world * dbytes * K / (dirty_ms * 1e-3) / 1e9, "unit": "GB/s",
                 "ms_per_step": dirty_ms / K,
                 "l2": "256 MiB write between steps, no clean read after it"}

    # ---- per-kernel device times from the trace (events on the launch stream)
    per = {}
    for name, ms in trace:
        t = per.setdefault(name, [0, 0.0])
        t[0] += 1
        t[1] += ms
    total_ms = sum(v[1] for v in per.values()) or 1.0
    kernels = []
    for name, (cnt, ms) in sorted(per.items(), key=lambda kv: -kv[1][1]):
        amt, unit = kernel_work(name, ts, ds, lens)
        ent = {"name": name, "launches": cnt, "total_ms": round(ms, 4),
               "share": round(ms / total_ms, 4), "avg_us": round(ms / cnt * 1e3, 2)}
        if amt is not None:
            avg_s = ms / cnt * 1e-3
            if unit == "flop":
                ent.update(achieved=amt / avg_s / 1e12, unit="TFLOP/s",
                           frac=amt / avg_s / 1e12 / peaks["bf16_tflops"])
            else:
                ent.update(achieved=amt / avg_s / 1e9, unit="GB/s",
                           frac=amt / avg_s / 1e9 / peaks["hbm_gbs"])
        kernels.append(ent)

    def roofline_for(name):
        ent = next((k for k in kernels if k["name"] == name), None)
        if ent is None or "achieved" not in ent:
            return None
        tensor = ent["unit"] == "TFLOP/s"
        amt, _ = kernel_work(name, ts, ds, lens)
        rf = {"kernel": name, "bound": "tensor" if tensor else "hbm",
              "achieved": ent["achieved"],
              "peak": peaks["bf16_tflops"] if tensor else peaks["hbm_gbs"],
              "unit": ent["unit"], "frac": ent["frac"],
              "traffic": ncu_traffic(name, ts.name if tensor else ds.name),
              "work_per_launch": amt, "work_unit": "FLOP" if tensor else "byte",
              "peak_source": f"{peaks_src} (MEASURED_PEAKS.json bf16 burst)" if tensor
              else f"{peaks_src} (MEASURED_PEAKS.json hbm_gbs)"}
        if tensor:
            rf["frac_of_sustained"] = ent["achieved"] / peaks["bf16_tflops_sustained"]
        return rf

    # bwd_dq runs on the library's side stream next to bwd_dkdv: its event
    # span includes the time it waits for SMs that bwd_dkdv holds, so it is
    # not a candidate for the dominant kernel (its serialized duration is in
    # the ncu launch list under profiles/).
    train_kernels = [k for k in kernels if k["name"] in ("fwd", "bwd_dkdv")]
    dominant = train_kernels[0]["name"] if train_kernels else kernels[0]["name"]
    dec_dom = "decode" if any(k["name"] == "decode" for k in kernels) else None

    # ---- end to end through the public API with host buffers
    e2e = None
    dec_e2e = None
    if args.e2e_steps > 0:
        host = {k: v.cpu().pin_memory() for k, v in synth.train_inputs(
            ts, seed=ts.seed + 1000 * rank).items()}
        outs_h = {"dq": torch.empty_like(dq, device="cpu").pin_memory(),
                  "dk": torch.empty_like(dk, device="cpu").pin_memory(),
                  "dv": torch.empty_like(dv, device="cpu").pin_memory(),
                  "dkc": torch.empty_like(dkc, device="cpu").pin_memory(),
                  "dvc": torch.empty_like(dvc, device="cpu").pin_memory()}
        h2d = sum(v.numel() * v.element_size() for v in host.values())
        d2h = sum(v.numel() * v.element_size() for v in outs_h.values())
        # A pipelined trainer: inputs and gradients are double-buffered on the
        # device; step i's host-to-device copy runs on a copy stream while
        # step i-1's kernels run, and step i's gradients go back to the host
        # on another stream while step i+1's kernels run.  Events keep each
        # buffer's reuse in order.  Every step still copies all its inputs in
        # and all its gradients out inside the timed region.
        dev_in = [{k: torch.empty_like(v, device=dev) for k, v in host.items()} for _ in range(2)]
        dev_out = [{k: torch.empty_like(t) for k, t in (("dq", dq), ("dk", dk), ("dv", dv),
                                                          ("dkc", dkc), ("dvc", dvc))}
                   for _ in range(2)]
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev = {n: [torch.cuda.Event() for _ in range(2)]
              for n in ("in_ready", "in_free", "out_ready", "out_free")}

        def e2e_step(i):
            b = i % 2
            x, y = dev_in[b], dev_out[b]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev["in_free"][b])  # step i-2's kernels are done with x
                for k2, v in host.items():
                    x[k2].copy_(v, non_blocking=True)
                ev["in_ready"][b].record(s_in)
            stream.wait_event(ev["in_ready"][b])
            if i >= 2:
                stream.wait_event(ev["out_free"][b])  # step i-2's gradients have left y
            cartattn.cart_attn_fwd(x["q"], x["k"], x["v"], x["kc"], x["vc"],
                                   frozen_prefix=ts.frozen_prefix, theta=ts.theta,
                                   o=o, lse=lse, workspace=ws_f)
            cartattn.cart_attn_bwd(x["q"], x["k"], x["v"], x["kc"], x["vc"], o, lse, x["do"],
                                   frozen_prefix=ts.frozen_prefix, theta=ts.theta,
                                   dq=y["dq"], dk=y["dk"], dv=y["dv"], dkc=y["dkc"],
                                   dvc=y["dvc"], workspace=ws_b, fwd_workspace=ws_f)
            cdist.allreduce_cartridge_grads(y["dkc"], y["dvc"])
            ev["in_free"][b].record(stream)
            ev["out_ready"][b].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev["out_ready"][b])
                for k2, t in y.items():
                    outs_h[k2].copy_(t, non_blocking=True)
                ev["out_free"][b].record(s_out)

        for i in range(2):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        cdist.barrier(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s_in)
        for i in range(args.e2e_steps):
            e2e_step(i)
        e1.record(s_out)
        torch.cuda.synchronize(dev)
        e_ms = cdist.max_over_ranks([e0.elapsed_time(e1)], dev)[0]
        e2e = {"value": world * flops_step * args.e2e_steps / (e_ms * 1e-3) / 1e12,
               "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e_ms / args.e2e_steps,
               "pipelined": "inputs and gradients double-buffered: step i's host-to-device "
                            "copy overlaps step i-1's kernels, its device-to-host copy step "
                            "i+1's; events from the first input copy to the last gradient copy"}
        # decode end to end: the new token's q/k/v and lengths in, o out
        dhost = {k: din[k].cpu().pin_memory() for k in ("q", "k_new", "v_new", "lens")}
        od_h = torch.empty_like(od, device="cpu").pin_memory()

        def dec_e2e_step():
            for k2, v in dhost.items():
                din[k2].copy_(v, non_blocking=True)
            decode_part()
            od_h.copy_(od, non_blocking=True)

        dec_e2e_step()
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(args.e2e_steps):
            flush()
            dec_e2e_step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        dflush = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        dflush[0].record(stream)
        for _ in range(args.e2e_steps):
            flush()
        dflush[1].record(stream)
        torch.cuda.synchronize(dev)
        d_ms = max(e0.elapsed_time(e1) - dflush[0].elapsed_time(dflush[1]), 1e-6)
        d_ms = cdist.max_over_ranks([d_ms], dev)[0]
        dec_e2e = {"value": world * dbytes * args.e2e_steps / (d_ms * 1e-3) / 1e9, "unit": "GB/s",
                   "h2d_bytes_per_step": sum(v.numel() * v.element_size() for v in dhost.values()),
                   "d2h_bytes_per_step": od_h.numel() * od_h.element_size()}

    ext = measure_extensions(args, ts, ds, dev, rank, peaks, flush) if args.ext_steps > 0 else None
    more = None
    if args.workload_steps > 0:
        other = synth.LONGCTX if ts is synth.SELFSTUDY else synth.SELFSTUDY
        more = {f"{other.name}_train": measure_train_workload(other, dev, rank, peaks, flush,
                                                              args.workload_steps),
                "equiv_fwd": measure_train_workload(synth.EQUIV, dev, rank, peaks, flush,
                                                    max(args.workload_steps, 20), bwd=False)}
        more["equiv_fwd"]["config"]["values"] = (
            "random inputs of the equivalence gate's shapes (the forward's work does not "
            "depend on the values)")

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(ts)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": (train_ms + dec_ms) / K,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": workload_name(ts), "global_batch": ts.B * world,
                       "seq_len": ts.n, "cartridge_rows": ts.p,
                       "decode_conversations": ds.B * world, "parallelism": f"dp{world}",
                       "l2": ("flushed between timed steps, outside the events: a 256 MiB "
                              "write, then a 256 MiB read of a second buffer (the write's "
                              "dirty lines go back to HBM before the timed kernels); "
                              "decode.dirty_l2 times the decode after the write alone"),
                       "train_ms_per_step": train_ms / K, "decode_ms_per_step": dec_ms / K,
                       "wall_s": round(wall, 3)},
            "roofline": roofline_for(dominant),
            "decode": {"metric": "decode HBM GB/s (shared cartridge counted once)",
                       "value": dec_gbs, "unit": "GB/s", "bytes_per_step": dbytes,
                       "frac": dec_gbs / world / peaks["hbm_gbs"],
                       "roofline": roofline_for(dec_dom) if dec_dom else None, "e2e": dec_e2e,
                       "dirty_l2": dec_dirty},
            "extensions": ext,
            "workloads": more,
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": n_launch,
            "clocks": clk.summary(), "kernels": kernels, "device_status": status,
        }
        print(json.dumps(line), flush=True)
    if has_pg:
        import torch.distributed as tdist
        tdist.destroy_process_group()


if __name__ == "__main__":
    main()

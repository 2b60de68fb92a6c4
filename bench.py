#!/usr/bin/env python
"""Causal prefill attention throughput on GB300.

One step = one causal forward pass (all of: K/V streaming, S = QK^T, online
softmax, P V, epilogue) over the synthetic workload, inputs resident in HBM.
The metric is causal TFLOP/s, counting 2*B*H*(S^2/2)*(d_qk+d_v) FLOPs, and
its fraction of the GB300 dense tensor peak of the input type.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun each rank runs the same workload on its own GPU (independent
problems, no collective on the data path: weak scaling); rank 0 prints one
JSON line.  ``--impl reference`` times the float64 CPU oracle on a bounded
sample of the same workload instead.
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
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads  # noqa: E402

METRIC = "causal fwd TFLOP/s and % of GB300 dense BF16/FP8 tensor peak, 1 GPU"
DEFAULT_WORKLOAD = "bf16_gqa_b1_h32kv8_s16384_d128"
ALSO_WORKLOADS = ["fp8_gqa_b1_h32kv8_s16384_d128"]
L2_FLUSH_BYTES = 512 << 20
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
KERNEL_SOURCES = ["causal_flashattention_prefill_gb300/csrc/fwd_sm103.cu",
                  "causal_flashattention_prefill_gb300/csrc/zyfa_ptx.cuh"]


def _code_only(text: str) -> str:
    """Source text without comments and with whitespace collapsed, so that
    the hash changes with the code, not with its comments."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def tensor_peak(dtype: str, peaks: dict) -> float:
    """Dense peak in TFLOP/s for the input type: BF16 measured burst; FP8 =
    BF16 x 2 (the nominal dense ratio, 4.5 / 2.25 PFLOP/s)."""
    bf16 = float(peaks["bf16_tflops"])
    return bf16 if dtype == "bf16" else 2.0 * bf16


def load_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        t = json.load(f)
    e = t.get(workload)
    if not e or e.get("kernel_hash") != kernel_hash():
        return None
    return float(e["bytes_per_launch"])


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clock and throttle samples taken during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"zyfa_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return None
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append(dict(sm=float(parts[1]), max=float(parts[2]),
                                     power=float(parts[3]), hw=parts[5], hwt=parts[6],
                                     swt=parts[7], pcap=parts[8]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return None
        loaded = [r for r in rows if r["power"] > 300.0]
        note = None
        if not loaded:
            note = ("no nvidia-smi sample fell under load (the timed region is shorter "
                    "than the 100 ms sampling interval); figures are of all samples")
            loaded = rows
        reasons = set()
        for r in loaded:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        out = {"sm_mhz": statistics.median(r["sm"] for r in loaded),
               "sm_max_mhz": max(r["max"] for r in rows),
               "power_w_max": max(r["power"] for r in rows),
               "samples": len(rows), "samples_under_load": 0 if note else len(loaded),
               "reasons": sorted(reasons), "source": "nvidia-smi -lms 100"}
        if note:
            out["note"] = note
        return out


class NvmlClockSampler:
    """SM clock, power and clock-event reasons read through NVML (ctypes on the
    driver's libnvidia-ml) every ~2 ms on a background thread, from just
    before to just after the timed region, so that a region of a few tens of
    milliseconds still holds samples taken while the kernels run."""

    # nvmlClocksEventReasons bits (nvml.h)
    REASONS = ((0x4, "sw_power_cap"), (0x8, "hw_slowdown"), (0x20, "sw_thermal_slowdown"),
               (0x40, "hw_thermal_slowdown"), (0x80, "hw_power_brake_slowdown"))

    def __init__(self, device):
        import ctypes
        self.c = ctypes
        self.ok = False
        self.samples = []
        self.stop = False
        try:
            import torch
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            p = torch.cuda.get_device_properties(device)
            bus = f"{p.pci_domain_id:08x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0".encode()
            self.h = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByPciBusId_v2(bus, ctypes.byref(self.h)) != 0:
                return
            self.reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx)) != 0:   # NVML_CLOCK_SM
                return
            self.max_mhz = mx.value
            self.nv = nv
            self.ok = True
        except (OSError, AttributeError, RuntimeError):
            self.ok = False

    def _read(self):
        c = self.c
        mhz, pw, rs = c.c_uint(), c.c_uint(), c.c_ulonglong()
        self.nv.nvmlDeviceGetClockInfo(self.h, 1, c.byref(mhz))
        self.nv.nvmlDeviceGetPowerUsage(self.h, c.byref(pw))
        self.reasons_fn(self.h, c.byref(rs))
        return time.perf_counter(), mhz.value, pw.value / 1000.0, rs.value

    def _loop(self):
        while not self.stop:
            self.samples.append(self._read())
            time.sleep(0.002)

    def __enter__(self):
        import threading
        if self.ok:
            self.samples.append(self._read())
            self.th = threading.Thread(target=self._loop, daemon=True)
            self.th.start()
        return self

    def __exit__(self, *exc):
        if self.ok:
            self.stop = True
            self.th.join(timeout=2)

    def summary(self):
        if not self.ok or not self.samples:
            return None
        reasons = set()
        for _, _, _, r in self.samples:
            for bit, name in self.REASONS:
                if r & bit:
                    reasons.add(name)
        sm = [m for _, m, _, _ in self.samples]
        return {"sm_mhz": statistics.median(sm), "sm_mhz_min": min(sm), "sm_max_mhz": self.max_mhz,
                "power_w_max": max(p for _, _, p, _ in self.samples),
                "samples": len(self.samples), "samples_under_load": len(self.samples),
                "reasons": sorted(reasons),
                "source": "NVML every ~2 ms during the timed region (power is NVML's "
                          "running average)"}


# -------------------------------------------------------------- GPU timing

def time_kernel(w, steps, warmup, device):
    """Per-launch device time (CUDA events on the launching stream) with the
    L2 flushed between launches; returns (ms list, result tensors)."""
    import torch
    import causal_flashattention_prefill_gb300 as zf

    t = workloads.make_inputs(w)
    q, k, v = (t[n].to(device) for n in ("q", "k", "v"))
    ds = [None] * 3
    if w.dtype == "fp8":
        ds = [torch.tensor([t[n + "_descale"]], dtype=torch.float32, device=device)
              for n in ("q", "k", "v")]
    out_shape = (w.B, w.S, w.H, w.d_v) if w.layout == "bshd" else (w.B, w.H, w.S, w.d_v)
    out = torch.empty(out_shape, dtype=torch.bfloat16, device=device)
    lse = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device=device)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)

    def launch():
        zf.attention(q, k, v, out=out, lse=lse, q_descale=ds[0], k_descale=ds[1],
                     v_descale=ds[2], layout=w.layout, return_lse=True,
                     stream=stream.cuda_stream)

    for _ in range(warmup):
        flush.zero_()
        launch()
    torch.cuda.synchronize(device)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    return t, (q, k, v, ds, out, lse), launch, flush, starts, ends


def run_timed(launch, flush, starts, ends, device):
    import torch
    torch.cuda.synchronize(device)
    t0 = time.perf_counter()
    for s, e in zip(starts, ends):
        flush.zero_()
        s.record()
        launch()
        e.record()
    torch.cuda.synchronize(device)
    wall = time.perf_counter() - t0
    return [s.elapsed_time(e) for s, e in zip(starts, ends)], wall


def time_rotate_quantize(w, steps, warmup, device, peaks, peak_src):
    """The FP8 input step with rotation (rotate + quantise q of the workload
    through zyfa_fp8_quantize_rotated), timed like the attention kernel.  HBM
    bound: the algorithmic bytes are one read of x and one write of the codes
    (3 bytes per BF16 element); the kernel reads x twice (max pass, then
    quantise pass)."""
    import torch
    import causal_flashattention_prefill_gb300 as zf

    t = workloads.make_inputs(w)
    x = t["q"].to(device)                         # BF16 (B, S, H, d)
    d = x.shape[-1]
    rows = x.numel() // d
    signs = zf.hadamard_signs(d, seed=0, device=device)
    x8 = torch.empty(x.shape, dtype=torch.uint8, device=device)
    ds = torch.empty(1, dtype=torch.float32, device=device)
    ws = torch.empty(zf.zyfa_fp8_quantize_workspace_bytes(), dtype=torch.uint8, device=device)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device).cuda_stream

    def launch():
        st = zf.zyfa_fp8_quantize_rotated(x.data_ptr(), rows, d, zf.ZYFA_BF16, signs.data_ptr(),
                                          x8.data_ptr(), ds.data_ptr(), ws.data_ptr(), stream)
        if st != zf.ZYFA_OK:
            raise zf.ZyfaError(st)

    for _ in range(warmup):
        flush.zero_()
        launch()
    torch.cuda.synchronize(device)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ms, _ = run_timed(launch, flush, starts, ends, device)
    mean_ms = statistics.mean(ms)
    algo_bytes = 3.0 * x.numel()
    gbs = algo_bytes / (mean_ms * 1e-3) / 1e9
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    return {"workload": f"fp8_quantize_rotated on q of {w.name} (d={d}, BF16 in)",
            "value": gbs, "unit": "GB/s", "ms_per_launch": mean_ms, "gpu_launches": 2 * steps,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                         "frac": gbs / hbm, "traffic": None,
                         "algorithmic_bytes_per_launch": algo_bytes,
                         "peak_source": f"{peak_src} copy bandwidth"}}


def sampled_parity(w, t, out, lse, n_rows=64):
    """Checks a few rows of the timed launch against the oracle before timing."""
    import oracle
    rows = np.unique(np.concatenate([np.arange(4), np.array([w.S // 2, w.S - 1]),
                                     np.random.default_rng(5).integers(0, w.S, n_rows)]))
    heads = [0, w.H - 1]
    q, k, v = (workloads.codes(t[n]) for n in ("q", "k", "v"))
    worst = 0.0
    worst_lse = 0.0
    group = w.H // w.Hkv
    for h in heads:
        hk = h // group
        sl_q = (slice(None), slice(None), [h]) if w.layout == "bshd" else (slice(None), [h])
        sl_k = (slice(None), slice(None), [hk]) if w.layout == "bshd" else (slice(None), [hk])
        O, L = oracle.attention_rows_f64(q[sl_q], k[sl_k], v[sl_k], rows, dtype=w.dtype,
                                         layout=w.layout, q_descale=t["q_descale"],
                                         k_descale=t["k_descale"], v_descale=t["v_descale"])
        o = out.float().cpu().numpy()
        og = o[:, rows, h] if w.layout == "bshd" else o[:, h, rows]
        worst = max(worst, float(np.abs(og - O[:, 0]).max()))
        worst_lse = max(worst_lse, float(np.abs(lse[:, h, rows].cpu().numpy() - L[:, 0]).max()))
    tol = (1e-2, 1e-3) if w.dtype == "bf16" else (4e-2, 5e-3)
    return {"rows": int(len(rows)), "heads": heads, "max_abs_dO": worst,
            "max_abs_dLSE": worst_lse, "ok": bool(worst <= tol[0] and worst_lse <= tol[1])}


def e2e_measure(w, t, steps, device):
    """Same metric through the public API with host buffers: every step copies
    q, k, v (and descales) from pinned host memory, runs the pass, and reads
    O and LSE back to pinned host memory; all of it inside the timed region.

    Steps are pipelined the way a serving loop overlaps requests: two sets of
    device buffers, the uploads on one stream, the attention calls on a
    second and the downloads on a third, ordered by events (step i+1 uploads
    while step i computes and step i-1 downloads).  `serial_value` is the
    same measurement one step at a time on one stream."""
    import torch
    import causal_flashattention_prefill_gb300 as zf

    hq, hk, hv = (t[n].pin_memory() for n in ("q", "k", "v"))
    fp8 = w.dtype == "fp8"
    hds = [torch.tensor([t[n + "_descale"]], dtype=torch.float32).pin_memory()
           for n in ("q", "k", "v")] if fp8 else [None] * 3
    out_shape = (w.B, w.S, w.H, w.d_v) if w.layout == "bshd" else (w.B, w.H, w.S, w.d_v)

    def buffers():
        d = {n: torch.empty_like(x, device=device) for n, x in (("q", hq), ("k", hk), ("v", hv))}
        d["ds"] = [torch.empty(1, dtype=torch.float32, device=device) for _ in range(3)] \
            if fp8 else [None] * 3
        d["out"] = torch.empty(out_shape, dtype=torch.bfloat16, device=device)
        d["lse"] = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device=device)
        d["hout"] = torch.empty(out_shape, dtype=torch.bfloat16).pin_memory()
        d["hlse"] = torch.empty((w.B, w.H, w.S), dtype=torch.float32).pin_memory()
        return d

    sets = [buffers(), buffers()]
    s_in, s_comp, s_out = (torch.cuda.Stream(device) for _ in range(3))
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "comp", "out")}

    def upload(d):
        for n, h in (("q", hq), ("k", hk), ("v", hv)):
            d[n].copy_(h, non_blocking=True)
        if fp8:
            for dd, h in zip(d["ds"], hds):
                dd.copy_(h, non_blocking=True)

    def compute(d):
        zf.attention(d["q"], d["k"], d["v"], out=d["out"], lse=d["lse"], q_descale=d["ds"][0],
                     k_descale=d["ds"][1], v_descale=d["ds"][2], layout=w.layout,
                     return_lse=True)

    def download(d):
        d["hout"].copy_(d["out"], non_blocking=True)
        d["hlse"].copy_(d["lse"], non_blocking=True)

    def pipelined_step(i):
        b = i & 1
        d = sets[b]
        with torch.cuda.stream(s_in):
            s_in.wait_event(ev["comp"][b])    # step i-2 has read these inputs
            upload(d)
            ev["in"][b].record(s_in)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(ev["in"][b])
            s_comp.wait_event(ev["out"][b])   # step i-2's results are read back
            compute(d)
            ev["comp"][b].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev["comp"][b])
            download(d)
            ev["out"][b].record(s_out)

    def serial_step(_):
        d = sets[0]
        upload(d)
        compute(d)
        download(d)

    def timed(fn, n):
        for i in range(2):
            fn(i)
        torch.cuda.synchronize(device)
        t0 = time.perf_counter()
        for i in range(n):
            fn(i)
        torch.cuda.synchronize(device)
        return (time.perf_counter() - t0) / n

    dt = timed(pipelined_step, steps)
    dt_serial = timed(serial_step, max(3, steps // 2))
    h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv))
    h2d += 12 if fp8 else 0
    d2h = sets[0]["hout"].numel() * 2 + sets[0]["hlse"].numel() * 4
    return {"value": w.flops / dt / 1e12, "unit": "TFLOP/s", "ms_per_step": dt * 1e3,
            "steps": steps, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "pipelined": "two buffer sets; uploads, attention calls and downloads on three "
                         "streams; every step's copies inside the timed region",
            "serial_value": w.flops / dt_serial / 1e12, "serial_ms_per_step": dt_serial * 1e3}


# ------------------------------------------------------------ CPU oracle

def oracle_sample(w, budget_s: float = 15.0, t=None):
    """Times the float64 oracle on a bounded sample of the workload: 256-row
    blocks of query rows taken from the end of the sequence backwards (the
    longest causal rows first), each over every (batch, head) slice in turn,
    until about ``budget_s`` seconds of CPU work have been spent."""
    import oracle
    if t is None:
        t = workloads.make_inputs(w)
    q, k, v = (workloads.codes(t[n]) for n in ("q", "k", "v"))
    group = w.H // w.Hkv
    R = min(w.S, 256)
    n_blocks = (w.S + R - 1) // R
    elapsed = 0.0
    flops = 0.0
    slices = 0
    blocks_used = 0
    for blk in range(n_blocks):
        hi = w.S - blk * R
        rows = np.arange(max(0, hi - R), hi)
        block_flops = float(sum(2.0 * (i + 1) * (w.d_qk + w.d_v) for i in rows))
        blocks_used = blk + 1
        for bh in range(w.B * w.H):
            if elapsed >= budget_s:
                break
            b, h = divmod(bh, w.H)
            hk = h // group
            if w.layout == "bshd":
                qs, ks, vs = q[b:b + 1, :, h:h + 1], k[b:b + 1, :, hk:hk + 1], v[b:b + 1, :, hk:hk + 1]
            else:
                qs, ks, vs = q[b:b + 1, h:h + 1], k[b:b + 1, hk:hk + 1], v[b:b + 1, hk:hk + 1]
            t0 = time.perf_counter()
            oracle.attention_rows_f64(qs, ks, vs, rows, dtype=w.dtype, layout=w.layout,
                                      q_descale=t["q_descale"], k_descale=t["k_descale"],
                                      v_descale=t["v_descale"])
            elapsed += time.perf_counter() - t0
            flops += block_flops
            slices += 1
        if elapsed >= budget_s:
            break
    cores = len(os.sched_getaffinity(0))
    return {"value": flops / elapsed / 1e12, "unit": "TFLOP/s", "cores": cores,
            "kind": "oracle", "seconds": elapsed,
            "sample": f"{slices} (batch, head, {R}-row block) slices from the last {blocks_used} "
                      f"query blocks of {w.name} (numpy float64, materialised masked scores, "
                      f"{cores} host threads available to BLAS)"}


# ------------------------------------------------------------------ main

def job_mean_ms(local_mean_ms: float, world: int, device) -> float:
    """Mean step time of the whole job: the slowest rank's (max over ranks,
    on whatever process group is initialised; the identity on one rank)."""
    if world <= 1:
        return local_mean_ms
    import torch
    import torch.distributed as dist
    tt = torch.tensor([local_mean_ms], dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def job_tflops(flops_per_rank: float, mean_ms: float, world: int) -> float:
    """Whole-job TFLOP/s: each of the `world` ranks ran its own problem of
    `flops_per_rank` within `mean_ms` (weak scaling, no data-path exchange)."""
    return world * flops_per_rank / (mean_ms * 1e-3) / 1e12


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def sweep_todo(path: str, names, khash: str) -> list:
    """Workloads of `names` (in order) that `path` holds no result line for
    with kernel source hash `khash`; lines that do not parse are ignored."""
    done = set()
    if os.path.exists(path):
        with open(path) as f:
            for raw in f:
                try:
                    d = json.loads(raw)
                except ValueError:
                    continue
                if d.get("kernel_hash") == khash and "workload" in d.get("config", {}):
                    done.add(d["config"]["workload"])
    return [n for n in names if n not in done]


def run_sweep(path: str, names, steps: int, warmup: int) -> int:
    """Times each workload in its own process (kernel only, no extra legs)
    and appends its JSON line to `path`, skipping workloads already recorded
    for the current kernel source, so an interrupted sweep resumes where it
    stopped.  Returns the number of workloads that failed."""
    failed = 0
    for name in sweep_todo(path, names, kernel_hash()):
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--workload", name,
                            "--steps", str(steps), "--warmup", str(warmup), "--no-extras"],
                           capture_output=True, text=True)
        lines = [x for x in r.stdout.splitlines() if x.startswith("{")]
        if r.returncode != 0 or not lines:
            failed += 1
            print(json.dumps({"workload": name, "failed": r.returncode,
                              "tail": r.stderr[-400:]}), flush=True)
            continue
        with open(path, "a") as f:
            f.write(lines[-1] + "\n")
        print(lines[-1], flush=True)
    return failed


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the e2e, FP8 and CPU-baseline legs")
    ap.add_argument("--sweep", metavar="FILE",
                    help="time every workload (or --workloads) into FILE, one JSON line each, "
                         "resuming after those already recorded for this kernel source")
    ap.add_argument("--workloads", help="comma-separated workload names for --sweep")
    args = ap.parse_args()
    if args.sweep:
        names = args.workloads.split(",") if args.workloads else sorted(workloads.WORKLOADS)
        for n in names:
            if n not in workloads.WORKLOADS:
                raise SystemExit(f"unknown workload {n}")
        raise SystemExit(1 if run_sweep(args.sweep, names, args.steps, max(3, args.warmup)) else 0)
    warmup = max(3, args.warmup)
    world, rank, local = dist_setup()
    w = workloads.WORKLOADS[args.workload]

    if args.impl == "reference":
        if rank != 0:
            return
        per_step = []
        t = workloads.make_inputs(w)
        # each step is one bounded sample, sized so the whole run stays within
        # a few minutes
        budget = max(0.05, min(20.0, 150.0 / (args.steps + warmup)))
        for _ in range(warmup):
            oracle_sample(w, budget_s=budget, t=t)
        for _ in range(args.steps):
            per_step.append(oracle_sample(w, budget_s=budget, t=t))
        value = statistics.mean(s["value"] for s in per_step)
        cpu = dict(per_step[0])
        cpu["value"] = value
        line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": warmup,
                "ms_per_step": 1e3 * statistics.mean(s["seconds"] for s in per_step),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f64", "data": "synthetic",
                "config": {"workload": w.name, "B": w.B, "S": w.S, "H": w.H, "Hkv": w.Hkv,
                           "d_qk": w.d_qk, "d_v": w.d_v, "layout": w.layout,
                           "sample": cpu["sample"]},
                "cpu_baseline": cpu,
                "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    import torch
    import causal_flashattention_prefill_gb300 as zf
    from causal_flashattention_prefill_gb300 import build as zbuild

    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    device = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(device)
    zbuild.build()
    zf.load()

    peaks, peak_src = load_peaks()
    t, bufs, launch, flush, starts, ends = time_kernel(w, args.steps, warmup, device)
    parity = sampled_parity(w, t, bufs[4], bufs[5]) if rank == 0 else None

    if world > 1:
        dist.barrier()
    visible = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")
    gpu_index = int(visible[device.index]) if len(visible) > device.index and \
        visible[device.index].strip().isdigit() else device.index
    clk = NvmlClockSampler(device)
    if not clk.ok:
        clk = ClockSampler(gpu_index)
    with clk:
        ms, wall = run_timed(launch, flush, starts, ends, device)
    if world > 1:
        dist.barrier()
    mean_ms = job_mean_ms(statistics.mean(ms), world, device)
    value = job_tflops(w.flops, mean_ms, world)
    per_gpu = w.flops / (mean_ms * 1e-3) / 1e12
    peak = tensor_peak(w.dtype, peaks)
    traffic = load_traffic(w.name)

    st, status_word = zf.zyfa_device_status()
    extras = {}
    if rank == 0 and not args.no_extras:
        also = []
        for name in ALSO_WORKLOADS:
            w2 = workloads.WORKLOADS[name]
            t2, b2, l2, f2, s2, e2 = time_kernel(w2, max(20, args.steps // 5), warmup, device)
            par2 = sampled_parity(w2, t2, b2[4], b2[5])
            ms2, _ = run_timed(l2, f2, s2, e2, device)
            v2 = w2.flops / (statistics.mean(ms2) * 1e-3) / 1e12
            p2 = tensor_peak(w2.dtype, peaks)
            also.append({"workload": name, "dtype": w2.dtype, "value": v2, "unit": "TFLOP/s",
                         "ms_per_launch": statistics.mean(ms2), "peak": p2,
                         "frac": v2 / p2, "parity": par2})
            del t2, b2
        if w.d_qk in (128, 192):
            also.append(time_rotate_quantize(w, max(20, args.steps // 5), warmup, device, peaks,
                                             peak_src))
        extras["also"] = also
        extras["e2e"] = e2e_measure(w, t, max(20, min(100, args.steps)), device)
        if world == 1:
            extras["cpu_baseline"] = oracle_sample(w, budget_s=15.0, t=t)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": warmup, "ms_per_step": mean_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w.dtype, "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "S": w.S, "H": w.H, "Hkv": w.Hkv,
                       "d_qk": w.d_qk, "d_v": w.d_v, "layout": w.layout,
                       "values": "N(0,1) q, k, v" if w.values == "gaussian" else w.values,
                       "l2": f"flushed between steps ({L2_FLUSH_BYTES >> 20} MiB write, "
                             "outside the timed events)",
                       "pct_of_peak": 100.0 * per_gpu / peak,
                       "timed_wall_s": wall},
            "roofline": {"bound": "tensor", "achieved": per_gpu, "peak": peak,
                         "unit": "TFLOP/s", "frac": per_gpu / peak, "traffic": traffic,
                         "peak_source": f"{peak_src} bf16 burst"
                                        + (" x 2 (nominal FP8/BF16 ratio)" if w.dtype != "bf16"
                                           else "")},
            "gpu_launches": args.steps,
            "parity_sample": parity,
            "device_status_word": status_word,
            "clocks": clk.summary(),
            "kernel_hash": kernel_hash(),
        }
        if "e2e" in extras:
            line["e2e"] = extras["e2e"]
        if "cpu_baseline" in extras:
            line["cpu_baseline"] = extras["cpu_baseline"]
        if "also" in extras:
            line["also"] = extras["also"]
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

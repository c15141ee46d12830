"""Benchmark of the linear-recurrence state update on GB300.

One step = both tier-1 scan forms (FMA and gated) over the large elementwise
workload B=8 T=8192 N=2048 (inputs resident in HBM, 1.6 GB per form, larger
than L2), through the C ABI.  Prints ONE JSON line with the contract keys,
the roofline of the dominant kernel, the CPU-oracle baseline, the
end-to-end figure (pinned host buffers, copies inside the timed region) and,
under "forms", every other workload measured the same way.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun each rank runs the same workload on its own GPU (independent
channels need no collective): "scaling": "weak", value = all ranks' bytes /
the slowest rank's time.
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

import synth  # noqa: E402

SCAN = synth.CONFIGS["scan_large"]
GB = 1e9


def scan_bytes(B, T, N, has_s0=True):
    """Algorithmic bytes of one scan: read a and b|u, write s_t (12 B per
    element) plus s0 in and s_final out (8 B per channel)."""
    return 12 * B * T * N + (8 if has_s0 else 4) * B * N


# Per-workload algorithmic bytes and flops: every input read once and every
# output written once per token and head (q, k, per-key decays, v in; o out;
# per-head scalars 4 bytes; grouped k and q shared by H / G heads), plus the
# final state written (and, for a decode, the initial state read).  Flops per
# state entry and step: diag 5 (k v product, decay FMA, readout FMA), delta 6
# (two dot-product FMAs and the update FMA), RWKV-7 7 (plus the decay).
def matrix_cost(name):
    c = synth.CONFIGS[name]
    B, T, H, dk, dv = c["B"], c["T"], c["H"], c["dk"], c["dv"]
    th = B * T * H
    state = B * H * dk * dv * 4
    if name in ("gla", "gated_memory"):
        per_th, flop_e, s_in = (3 * dk + 2 * dv) * 4, 5, 0
    elif name == "mamba2":
        G = c["G"]
        per_th, flop_e, s_in = (2 * dv + 1) * 4 + 2 * dk * 4 * G / H, 5, 0
    elif name == "deltanet":
        per_th, flop_e, s_in = (2 * dk + 2 * dv + 1) * 4, 6, 0
    elif name == "rwkv7_prefill":
        per_th, flop_e, s_in = (3 * dk + 2 * dv) * 4, 7, 0
    else:  # rwkv7_decode: random initial state read and written
        per_th, flop_e, s_in = (3 * dk + 2 * dv) * 4, 7, state
    nbytes = th * per_th + state + s_in
    flops = th * dk * dv * flop_e
    return th, nbytes, flops


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "sm_max_mhz": 2070.0}, "fallback"


def traffic_record(kernel):
    """dram bytes per launch of `kernel` from the committed ncu summary, if the
    kernel source is unchanged since the capture (else None)."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return None
    for line in open(path):
        if line.startswith("#"):
            continue
        f = dict(kv.split("=", 1) for kv in line.split() if "=" in kv)
        if f.get("kernel") != kernel or "src" not in f:
            continue
        src = os.path.join(ROOT, f["src"])
        if os.path.exists(src) and hashlib.sha256(open(src, "rb").read()).hexdigest()[:16] == f.get("src_sha"):
            return float(f["dram_bytes_per_launch"])
    return None


# ---------------------------------------------------------------- ranks
def max_over_ranks(ms, device="cpu"):
    """Largest per-rank time; the identity without a process group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbps(step_bytes, steps, world, ms_total):
    """Whole-job throughput: every rank moves `step_bytes` per step (weak
    scaling), timed by the slowest rank."""
    return world * steps * step_bytes / (ms_total / 1e3) / GB


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t_on = self.t_off = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "20",
                 "-i", str(self.gpu)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, on):
        if on:
            self.t_on = time.time()
        else:
            self.t_off = time.time()

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(ts=ts, sm=float(parts[1]), max=float(parts[2]),
                                 hw=parts[5].lower() == "active", hwt=parts[6].lower() == "active",
                                 swt=parts[7].lower() == "active", pcap=parts[8].lower() == "active"))
            except ValueError:
                continue
        return clock_summary(rows, self.t_on, self.t_off, "nvidia-smi, 20 ms")


def clock_summary(rows, t_on, t_off, source):
    """Median SM clock, its maximum and the throttle reasons seen, from the
    samples inside the timed region [t_on, t_off] (else those within 0.1 s of
    it, when the region is shorter than the sampling period, else all)."""
    if not rows:
        return None
    inwin = [r for r in rows if t_on and t_off and t_on <= r["ts"] <= t_off]
    near = [r for r in rows if t_on and t_off and t_on - 0.1 <= r["ts"] <= t_off + 0.1]
    use = inwin or near or rows
    reasons = [name for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                                      ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap"))
               if any(r[key] for r in use)]
    return {"sm_mhz": statistics.median(r["sm"] for r in use), "sm_max_mhz": max(r["max"] for r in use),
            "reasons": reasons, "samples": len(use), "in_timed_region": bool(inwin),
            "within_0.1s_of_timed_region": bool(inwin or near),
            "timed_region_ms": round((t_off - t_on) * 1e3, 1) if t_on and t_off else None, "source": source}


class NvmlClockSampler:
    """The same record read in-process through NVML (read-only queries, by
    ctypes) every PERIOD_S, so that samples fall inside a timed region of a
    few milliseconds.  The device is found by the UUID CUDA reports for it."""
    PERIOD_S = 0.002
    # clock-event reason bits of NVML's current-clocks query
    BITS = {"pcap": 0x4, "hw": 0x8, "swt": 0x20, "hwt": 0x40}

    def __init__(self, torch, cuda_index):
        import ctypes
        self.ct = ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        uuid = "GPU-" + str(torch.cuda.get_device_properties(cuda_index).uuid)
        self.h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.h)) != 0:
            raise OSError("no NVML device with the CUDA device's UUID")
        self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
        if self.reasons_fn is None:
            self.reasons_fn = lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self.lib = lib
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx)) != 0:   # 1: the SM clock
            raise OSError("max clock query failed")
        self.max = float(mx.value)
        self.rows = []
        self.t_on = self.t_off = None
        self.stop_flag = False
        self.thread = None

    def _sample(self):
        ct = self.ct
        clk, rs = ct.c_uint(), ct.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.h, 1, ct.byref(clk)) != 0 or \
                self.reasons_fn(self.h, ct.byref(rs)) != 0:
            return
        r = dict(ts=time.time(), sm=float(clk.value), max=self.max)
        r.update({k: bool(rs.value & bit) for k, bit in self.BITS.items()})
        self.rows.append(r)

    def _loop(self):
        while not self.stop_flag:
            self._sample()
            time.sleep(self.PERIOD_S)

    def start(self):
        self.thread = threading.Thread(target=self._loop, daemon=True)
        self.thread.start()

    def mark(self, on):
        if on:
            self.t_on = time.time()
        else:
            self.t_off = time.time()

    def stop(self):
        self.stop_flag = True
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self):
        return clock_summary(self.rows, self.t_on, self.t_off, f"NVML, {self.PERIOD_S * 1e3:g} ms")


def make_clock_sampler(torch, cuda_index, smi_index):
    """The in-process NVML sampler, else the nvidia-smi one."""
    try:
        return NvmlClockSampler(torch, cuda_index)
    except (OSError, AttributeError, TypeError, ValueError):
        return ClockSampler(smi_index)


# ---------------------------------------------------------------- CPU oracle record
# The oracle runs on the machine's host cores in two ways (the pages time their C
# scan single-threaded, one subprocess per cell with the median of repeated
# runs, "SunnyNet 工程化实录" §2.3):
#   * all cores: the workload split into independent units -- (batch row,
#     block of 128 channels) for the scans, (batch, head) for the matrix
#     recurrences, batch blocks for single-step decodes -- on one thread per
#     logical CPU (ctypes releases the GIL inside the oracle);
#   * one thread: the median of repeated runs of one unit.
# The fp64 all-core run also supplies the reference the GPU outputs are
# measured against.
SCAN_BLOCK = 128
PAGES_ERR = {   # the pages' own accuracy figures (max |diff| on O(1) data), for context
    "scan": (7.63e-06, "SunnyNet 工程化实录 §2.3 (C scan against torch)"),
    "deltanet": (4.6e-05, "SunnyNet 工程化实录 §4.2 (DeltaNet against its reference)"),
    "gla": (2.05e-05, "SunnyNet 工程化实录 §4.3 (GLA against its reference)"),
}


def host_cores():
    return os.cpu_count() or 1


def run_pool(tasks, threads):
    """Run zero-argument callables on `threads` threads; results in order and
    wall seconds."""
    import concurrent.futures as cf
    t0 = time.perf_counter()
    if threads <= 1:
        res = [t() for t in tasks]
    else:
        with cf.ThreadPoolExecutor(threads) as ex:
            res = list(ex.map(lambda f: f(), tasks))
    return res, time.perf_counter() - t0


class OracleJob:
    """A workload cut into independent oracle units.  `units` is a list of
    (slices, fn) with fn(prec) running the oracle on that unit; `place`
    copies a unit's fp64 result into the full reference arrays; `nbytes` and
    `tok_heads` are the algorithmic bytes and token-heads of the whole job and
    `unit_share` the fraction one unit holds."""

    def __init__(self, units, outputs, place, nbytes, tok_heads=None, what=""):
        self.units, self.outputs, self.place = units, outputs, place
        self.nbytes, self.tok_heads, self.what = nbytes, tok_heads, what
        self.unit_share = 1.0 / len(units)

    def run_all(self, prec, threads):
        res, secs = run_pool([(lambda f=f: f(prec)) for _, f in self.units], threads)
        return res, secs

    def reference(self, threads):
        """fp64 all-core run: (reference arrays, seconds)."""
        import numpy as np
        res, secs = self.run_all("f64", threads)
        ref = {k: np.empty(shape, np.float64) for k, shape in self.outputs.items()}
        for (sl, _), r in zip(self.units, res):
            self.place(ref, sl, r)
        return ref, secs

    def one_thread(self, prec, reps):
        f = self.units[0][1]
        f(prec)                                  # warm (library loaded, pages touched)
        ts = []
        for _ in range(reps):
            t0 = time.perf_counter()
            f(prec)
            ts.append(time.perf_counter() - t0)
        return statistics.median(ts)

    def rate(self, secs, share=1.0):
        r = {"GBps": round(self.nbytes * share / secs / GB, 4), "s": round(secs, 4)}
        if self.tok_heads is not None:
            r["tok_heads_per_s"] = round(self.tok_heads * share / secs, 1)
        return r


def scan_job(a, rhs, s0, forms=("fma", "gated"), block=SCAN_BLOCK):
    """The elementwise scans cut into (batch row, block of channels) units; a
    unit runs every form in `forms` (rhs maps a form to its b or u array).
    Single steps (T = 1) are cut into blocks of batch rows instead."""
    import numpy as np

    import oracle
    B, T, N = a.shape
    fns = {"fma": oracle.scan_fma, "gated": oracle.scan_gated}
    units = []

    def make(sl, au, ru, su):
        return lambda prec: [fns[f](au, ru[f], su, prec=prec) for f in forms]

    if T == 1:
        step = max(1, B // 64)
        for b0 in range(0, B, step):
            b1 = min(B, b0 + step)
            sl = (b0, b1, 0, N)
            units.append((sl, make(sl, a[b0:b1], {f: rhs[f][b0:b1] for f in forms},
                                   None if s0 is None else s0[b0:b1])))
    else:
        for b in range(B):
            for n0 in range(0, N, block):
                n1 = min(N, n0 + block)
                sl = (b, b + 1, n0, n1)
                au = np.ascontiguousarray(a[b:b + 1, :, n0:n1])
                ru = {f: np.ascontiguousarray(rhs[f][b:b + 1, :, n0:n1]) for f in forms}
                su = None if s0 is None else np.ascontiguousarray(s0[b:b + 1, n0:n1])
                units.append((sl, make(sl, au, ru, su)))

    def place(ref, sl, r):
        b0, b1, n0, n1 = sl
        for f, (so, sf) in zip(forms, r):
            ref[f"s_{f}"][b0:b1, :, n0:n1] = so
            ref[f"s_final_{f}"][b0:b1, n0:n1] = sf

    outputs = {}
    for f in forms:
        outputs[f"s_{f}"] = (B, T, N)
        outputs[f"s_final_{f}"] = (B, N)
    unit_what = "batch-row blocks" if T == 1 else f"(batch row, {block}-channel block) units"
    return OracleJob(units, outputs, place, len(forms) * scan_bytes(B, T, N, s0 is not None),
                     what=f"{unit_what}, forms {'+'.join(forms)}")


def scan_bwd_job(a, s, s0, gs, u=None, block=SCAN_BLOCK):
    """The reverse scan of one form (gated when u is given), cut like the
    forward scans; used for its fp64 reference only."""
    import numpy as np

    import oracle
    B, T, N = a.shape
    kind = "fma" if u is None else "gated"
    units = []
    for b in range(B):
        for n0 in range(0, N, block):
            n1 = min(N, n0 + block)
            cut = lambda x: None if x is None else np.ascontiguousarray(x[b:b + 1, ..., n0:n1])
            args = (cut(a), cut(s), cut(s0), cut(gs), cut(u))
            units.append(((b, n0, n1), lambda prec, q=args: oracle.scan_backward(
                kind, q[0], q[1], q[2], q[3], None, q[4], prec=prec)))

    def place(ref, sl, r):
        b, n0, n1 = sl
        ref["grad_a"][b, :, n0:n1] = r[0][0]
        ref["grad_bu"][b, :, n0:n1] = r[1][0]
        ref["grad_s0"][b, n0:n1] = r[2][0]

    nb = (20 if u is None else 24) * B * T * N + 8 * B * N
    return OracleJob(units, {"grad_a": (B, T, N), "grad_bu": (B, T, N), "grad_s0": (B, N)}, place, nb,
                     what=f"(batch row, {block}-channel block) units")


def matrix_job(kind, x, B, T, H, dk, dv, nbytes, G=None):
    """A matrix recurrence cut into (batch, head) units, or into batch blocks
    of all heads for a single step.  kind: diag | delta | rwkv7; x holds host
    float32 arrays q, k, v, g (decays, beta or w) and optional S0, plus
    decay_kind and scale for diag."""
    import numpy as np

    import oracle
    G = G or H
    S_shape = (B, H, dv, dk) if kind == "rwkv7" else (B, H, dk, dv)
    S0 = x.get("S0")

    def call(q, k, v, g, s0, Hu, Gu, prec):
        if kind == "diag":
            return oracle.recur_diag(q, k, v, g, s0, H=Hu, G=Gu, decay_kind=x["decay_kind"], scale=x["scale"],
                                     prec=prec)
        if kind == "delta":
            return oracle.recur_delta(q, k, v, g, s0, scale=x["scale"], prec=prec)
        return oracle.recur_rwkv7(q, k, v, g, s0, prec=prec)

    units = []
    if T == 1:
        step = max(1, B // 64)
        for b0 in range(0, B, step):
            b1 = min(B, b0 + step)
            args = [x[n][b0:b1] for n in ("q", "k", "v", "g")] + [None if S0 is None else S0[b0:b1]]
            units.append((("b", b0, b1), lambda prec, a=args: call(*a, H, G, prec)))
    else:
        for b in range(B):
            for h in range(H):
                gi = h // (H // G)
                qk = [np.ascontiguousarray(x[n][b:b + 1, :, gi:gi + 1]) for n in ("q", "k")]
                vu = np.ascontiguousarray(x["v"][b:b + 1, :, h:h + 1])
                gu = np.ascontiguousarray(x["g"][b:b + 1, :, h:h + 1])   # per key (B,T,H,dk) or per head (B,T,H)
                su = None if S0 is None else np.ascontiguousarray(S0[b:b + 1, h:h + 1])
                units.append((("bh", b, h), lambda prec, a=(qk[0], qk[1], vu, gu, su): call(*a, 1, 1, prec)))

    def place(ref, sl, r):
        o, S = r
        if sl[0] == "b":
            ref["o"][sl[1]:sl[2]] = o
            ref["S"][sl[1]:sl[2]] = S
        else:
            ref["o"][sl[1]:sl[1] + 1, :, sl[2]:sl[2] + 1] = o
            ref["S"][sl[1]:sl[1] + 1, sl[2]:sl[2] + 1] = S

    what = "batch blocks of all heads" if T == 1 else "(batch, head) units"
    return OracleJob(units, {"o": (B, T, H, dv), "S": S_shape}, place, nbytes, tok_heads=B * T * H, what=what)


def err_pair(y, r):
    """(normwise, elementwise) error of y against the fp64 reference r:
    max|y - r| / max|r|, and max |y - r| / max(|r|, 1e-3 max|r|)."""
    import numpy as np
    y = np.asarray(y, np.float64)
    r = np.asarray(r, np.float64)
    m = float(np.max(np.abs(r))) if r.size else 0.0
    d = np.abs(y - r)
    nw = float(np.max(d)) / max(m, 1e-300)
    ew = float(np.max(d / np.maximum(np.abs(r), 1e-3 * m + 1e-300)))
    return nw, ew


def errors(outs, ref, tol, pages=None):
    """Per-output error figures against the fp64 oracle, with the bound."""
    rec = {"err_normwise": {}, "err_elementwise": {}, "tolerance": tol, "tolerance_on": "err_normwise"}
    for k, y in outs.items():
        nw, ew = err_pair(y, ref[k])
        rec["err_normwise"][k] = float(f"{nw:.3e}")
        rec["err_elementwise"][k] = float(f"{ew:.3e}")
    rec["within_tolerance"] = all(v <= tol for v in rec["err_normwise"].values())
    if pages is not None:
        rec["pages_max_abs_diff"] = {"value": pages[0], "where": pages[1]}
    return rec


def cpu_record(job, reps_1t=3, want_ref=True):
    """The four CPU oracle figures of one workload and (optionally) its fp64
    reference.  Returns (record, reference or None)."""
    cores = host_cores()
    threads = min(len(job.units), cores)
    ref, s64 = job.reference(threads) if want_ref else (None, None)
    if s64 is None:
        _, s64 = job.run_all("f64", threads)
    _, s32 = job.run_all("f32", threads)
    t64 = job.one_thread("f64", reps_1t)
    t32 = job.one_thread("f32", reps_1t)
    hinfo = {"threads": threads, "logical_cpus": cores, "cpu_model": cpu_model()}
    rec = {
        "cpu_fp64_all": dict(job.rate(s64), **hinfo, sample=f"the whole workload, {len(job.units)} {job.what}"),
        "cpu_fp32_all": dict(job.rate(s32), **hinfo, sample=f"the whole workload, {len(job.units)} {job.what}"),
        "cpu_fp64_1t": dict(job.rate(t64, job.unit_share), threads=1, cpu_model=hinfo["cpu_model"],
                            sample=f"one unit ({job.unit_share:.3g} of the workload), median of {reps_1t}"),
        "cpu_fp32_1t": dict(job.rate(t32, job.unit_share), threads=1, cpu_model=hinfo["cpu_model"],
                            sample=f"one unit ({job.unit_share:.3g} of the workload), median of {reps_1t}"),
    }
    return rec, ref


def cpu_model():
    """The host CPU's name from /proc/cpuinfo (model name, or the Arm
    implementer / part codes), else the platform string."""
    import platform
    try:
        info = open("/proc/cpuinfo").read().splitlines()
    except OSError:
        return platform.processor() or platform.machine()
    fields = {}
    for line in info:
        if ":" in line:
            k, v = line.split(":", 1)
            fields.setdefault(k.strip(), v.strip())
    if "model name" in fields:
        return fields["model name"]
    if "CPU part" in fields:
        return f"{platform.machine()} implementer {fields.get('CPU implementer', '?')} part {fields['CPU part']}"
    return platform.processor() or platform.machine()


def run_reference(args):
    """The reference arm: the CPU oracle as it stands, on this arm's workload
    (the full B=8 T=8192 N=2048 scan, both forms, inputs drawn on the CPU),
    fp64, the workload's independent units on every host core."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    x = synth.config_inputs("scan_large")
    a, b, u, s0 = (x[n].numpy() for n in ("a", "b", "u", "s0"))
    B, T, N = a.shape
    job = scan_job(a, {"fma": b, "gated": u}, s0)
    threads = min(len(job.units), host_cores())
    for _ in range(args.warmup):
        job.run_all("f64", threads)
    times = [job.run_all("f64", threads)[1] for _ in range(args.steps)]
    per_step_bytes = 2 * scan_bytes(B, T, N)
    total = sum(times)
    value = args.steps * per_step_bytes / total / GB
    sample = (f"the full workload B=8 T=8192 N=2048 per step, both forms, fp64 oracle, {len(job.units)} "
              f"{job.what} on {threads} threads ({cpu_model()})")
    line = {
        "impl": "reference", "metric": "recurrence_scan_GBps", "value": round(value, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * total / args.steps, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "scan_large B=8 T=8192 N=2048, FMA + gated forms"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU arm
def link_bandwidth(torch, dev, nbytes=1 << 30, reps=4):
    """Pinned host <-> device copy rates of this machine (GB/s): each direction
    alone and both at once on two streams.  They bound the end-to-end step."""
    n = nbytes // 4
    h_in, h_out = torch.empty(n, pin_memory=True), torch.empty(n, pin_memory=True)
    d_in, d_out = torch.empty(n, device=dev), torch.empty(n, device=dev)
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def timed(fn):
        fn()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(reps):
            fn()
        torch.cuda.synchronize()
        return (time.perf_counter() - t0) / reps

    def h2d():
        with torch.cuda.stream(s1):
            d_in.copy_(h_in, non_blocking=True)

    def d2h():
        with torch.cuda.stream(s2):
            h_out.copy_(d_out, non_blocking=True)

    def both():
        h2d()
        d2h()

    gb = nbytes / 1e9
    out = {"h2d_GBps": round(gb / timed(h2d), 1), "d2h_GBps": round(gb / timed(d2h), 1),
           "concurrent_each_GBps": round(gb / timed(both), 1)}
    del h_in, h_out, d_in, d_out
    return out


def time_form(torch, fn, warmup, reps, stream, flush=None):
    """Median ms of `fn` over `reps` launches (CUDA events on `stream`).
    `flush` (a tensor larger than L2) is overwritten on the stream before every
    timed launch, outside the events, for workloads that would fit in L2."""
    for _ in range(warmup):
        fn()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    torch.cuda.synchronize()
    for s, e in ev:
        if flush is not None:
            with torch.cuda.stream(stream):
                flush.fill_(1.0)
        s.record(stream)
        fn()
        e.record(stream)
    torch.cuda.synchronize()
    ts = sorted(s.elapsed_time(e) for s, e in ev)
    return ts[len(ts) // 2]


GRAPH_CALLS = 16   # scan calls captured in one CUDA graph for the small-workload latency


def host(t):
    """A device tensor's values as a host numpy array (None stays None)."""
    return None if t is None else t.detach().cpu().numpy()


def bench_forms(torch, sr, ctx, dev, stream, fp32_peak_tflops, hbm_peak, cpu=True, scan_ref=None,
                warmup=3, reps=20):
    """Every other workload, each on its own inputs, outside the main timed
    region.  With `cpu`, each workload also gets its CPU-oracle figures and
    the error of every GPU output against the fp64 oracle (`scan_ref` is the
    large scan's fp64 reference, computed by the caller).  Returns a dict of
    per-form results."""
    import numpy as np
    out = {}
    s = stream
    flush = torch.empty(64 << 20, device=dev)          # 256 MB, larger than L2
    with torch.cuda.stream(stream):
        # the small scan workload (0.4 MB, fits in L2): per-call latency of both
        # forms, launched directly and replayed from a CUDA graph of GRAPH_CALLS
        # calls; L2 is flushed before every timed call or replay.  The
        # single-step scans (T = 1) are measured the same way.
        c = synth.CONFIGS["scan_small"]
        for label, (Bs, Ts, Ns), maker in (
                ("scan_small", (c["B"], c["T"], c["N"]), lambda: synth.config_inputs("scan_small", device=dev)),
                ("scan_step_B1024", (1024, 1, 2048),
                 lambda: synth.scan_inputs(1024, 1, 2048, large=True, cid=31, device=dev)),
                ("scan_step_B1", (1, 1, 2048), lambda: synth.scan_inputs(1, 1, 2048, large=True, cid=32, device=dev))):
            xs = maker()
            sos = {f: torch.empty((Bs, Ts, Ns), device=dev) for f in ("fma", "gated")}
            sfs = {f: torch.empty((Bs, Ns), device=dev) for f in ("fma", "gated")}
            nb = scan_bytes(Bs, Ts, Ns, xs["s0"] is not None)
            rec = {"workload": f"B={Bs} T={Ts} N={Ns}", "bytes_per_call": nb, "l2": "flushed",
                   "graph_calls": GRAPH_CALLS}
            for form, rhs in (("fma", "b"), ("gated", "u")):
                f = sr.sn_scan_fma if form == "fma" else sr.sn_scan_gated
                call = lambda: f(ctx.handle, Bs, Ts, Ns, xs["a"], xs[rhs], xs["s0"], sfs[form], sos[form], s)
                direct = time_form(torch, call, warmup, reps, s, flush=flush)
                torch.cuda.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=s):
                    for _ in range(GRAPH_CALLS):
                        call()
                replay = time_form(torch, g.replay, warmup, reps, s, flush=flush)
                rec[form] = {"us_per_call": round(direct * 1e3, 2),
                             "us_per_call_graph": round(replay * 1e3 / GRAPH_CALLS, 2),
                             "GBps": round(nb / direct / 1e6, 1),
                             "GBps_graph": round(nb / (replay / GRAPH_CALLS) / 1e6, 1)}
                del g
            if cpu:
                xh = {n: host(xs[n]) for n in ("a", "b", "u", "s0")}
                job = scan_job(xh["a"], {"fma": xh["b"], "gated": xh["u"]}, xh["s0"])
                crec, ref = cpu_record(job, reps_1t=10)
                rec.update(crec)
                rec.update(errors({f"s_{f}": host(sos[f]) for f in ("fma", "gated")} |
                                  {f"s_final_{f}": host(sfs[f]) for f in ("fma", "gated")}, ref, 1e-5,
                                  PAGES_ERR["scan"]))
            out[label] = rec
            del xs, sos, sfs
        # the chunked look-back kernel on the same large scan workload
        x = synth.config_inputs("scan_large", device=dev)
        B, T, N = SCAN["B"], SCAN["T"], SCAN["N"]
        ctx.ensure_workspace(B, T, N)
        so = torch.empty((B, T, N), device=dev)
        sf = torch.empty((B, N), device=dev)
        ctx.set_option(sr.SN_OPT_SCAN_KERNEL, sr.SN_SCAN_KERNEL_LOOKBACK)
        for form, rhs in (("fma", "b"), ("gated", "u")):
            f = sr.sn_scan_fma if form == "fma" else sr.sn_scan_gated
            ms = time_form(torch, lambda: f(ctx.handle, B, T, N, x["a"], x[rhs], x["s0"], sf, so, s), warmup, reps, s)
            nb = scan_bytes(B, T, N)
            r = {"ms": round(ms, 4), "GBps": round(nb / ms / 1e6, 1),
                 "hbm_frac": round(nb / ms / 1e6 / hbm_peak, 3), "bound": "hbm"}
            if scan_ref is not None:
                r.update(errors({"s": host(so), "s_final": host(sf)},
                                {"s": scan_ref[f"s_{form}"], "s_final": scan_ref[f"s_final_{form}"]}, 1e-5))
            out[f"scan_{form}_lookback"] = r
        ctx.set_option(sr.SN_OPT_SCAN_KERNEL, sr.SN_SCAN_KERNEL_AUTO)
        # few channels, long T (B=1 T=262144 N=64, the chunked kernels' regime):
        # the automatic choice (the fused one-launch kernel), reduce-then-scan,
        # the look-back kernel and the sequential kernel
        Bf, Tf, Nf = 1, 262144, 64
        xf = synth.scan_inputs(Bf, Tf, Nf, large=True, cid=6)
        af, bf, s0f = xf["a"].to(dev), xf["b"].to(dev), xf["s0"].to(dev)
        sof = torch.empty_like(af)
        sff = torch.empty_like(s0f)
        ctx.ensure_workspace(Bf, Tf, Nf)
        few = {"workload": f"B={Bf} T={Tf} N={Nf}", "bytes_per_call": scan_bytes(Bf, Tf, Nf)}
        fref = None
        if cpu:
            fjob = scan_job(xf["a"].numpy(), {"fma": xf["b"].numpy()}, xf["s0"].numpy(), forms=("fma",), block=1)
            fref, _ = fjob.reference(min(len(fjob.units), host_cores()))
        for label, kern in (("fused", sr.SN_SCAN_KERNEL_FUSED), ("reduce_scan", sr.SN_SCAN_KERNEL_REDUCE_SCAN),
                            ("lookback", sr.SN_SCAN_KERNEL_LOOKBACK), ("sequential", sr.SN_SCAN_KERNEL_SEQUENTIAL)):
            ctx.set_option(sr.SN_OPT_SCAN_KERNEL, kern)
            ms = time_form(torch, lambda: sr.sn_scan_fma(ctx.handle, Bf, Tf, Nf, af, bf, s0f, sff, sof, s), warmup,
                           reps, s)
            few[label] = {"ms": round(ms, 4), "GBps": round(scan_bytes(Bf, Tf, Nf) / ms / 1e6, 1),
                          "hbm_frac": round(scan_bytes(Bf, Tf, Nf) / ms / 1e6 / hbm_peak, 3)}
            if fref is not None:
                few[label].update(errors({"s": host(sof), "s_final": host(sff)},
                                         {"s": fref["s_fma"], "s_final": fref["s_final_fma"]}, 1e-5))
        ctx.set_option(sr.SN_OPT_SCAN_KERNEL, sr.SN_SCAN_KERNEL_AUTO)
        few["auto_picks"] = "fused"
        out["scan_fma_few_channels"] = few
        # and its reverse scan (read a, s, ds; write da, db): sequential against chunked
        sr.sn_scan_fma(ctx.handle, Bf, Tf, Nf, af, bf, s0f, sff, sof, s)
        gsf = torch.empty_like(af).normal_(generator=torch.Generator(dev).manual_seed(78))
        daf, dbf, d0f = torch.empty_like(af), torch.empty_like(af), torch.empty_like(s0f)
        nbb = 20 * Bf * Tf * Nf + 8 * Bf * Nf
        fewb = {"workload": f"B={Bf} T={Tf} N={Nf}", "bytes_per_call": nbb}
        bref = None
        if cpu:
            bjob = scan_bwd_job(host(af), host(sof), host(s0f), host(gsf), block=1)
            bref, _ = bjob.reference(min(len(bjob.units), host_cores()))
        for label, kern in (("chunked", sr.SN_SCAN_KERNEL_REDUCE_SCAN), ("sequential", sr.SN_SCAN_KERNEL_SEQUENTIAL)):
            ctx.set_option(sr.SN_OPT_SCAN_KERNEL, kern)
            ms = time_form(torch, lambda: sr.sn_scan_fma_backward(ctx.handle, Bf, Tf, Nf, af, s0f, sof, gsf, None,
                                                                   daf, dbf, d0f, s), warmup, reps, s)
            fewb[label] = {"ms": round(ms, 4), "GBps": round(nbb / ms / 1e6, 1),
                           "hbm_frac": round(nbb / ms / 1e6 / hbm_peak, 3)}
            if bref is not None:
                fewb[label].update(errors({"grad_a": host(daf), "grad_b": host(dbf), "grad_s0": host(d0f)},
                                          {"grad_a": bref["grad_a"], "grad_b": bref["grad_bu"],
                                           "grad_s0": bref["grad_s0"]}, 1e-5))
        ctx.set_option(sr.SN_OPT_SCAN_KERNEL, sr.SN_SCAN_KERNEL_AUTO)
        fewb["auto_picks"] = "chunked"
        out["scan_fma_backward_few_channels"] = fewb
        del xf, af, bf, s0f, sof, sff, gsf, daf, dbf, d0f, fref, bref
        # reverse scans (backward pass) on the same workload: read a, s, ds (+u),
        # write da, db|du
        gs_ = torch.empty((B, T, N), device=dev).normal_(generator=torch.Generator(dev).manual_seed(77))
        da = torch.empty((B, T, N), device=dev)
        db = torch.empty((B, T, N), device=dev)
        d0 = torch.empty((B, N), device=dev)
        for form in ("fma", "gated"):
            if form == "fma":
                sr.sn_scan_fma(ctx.handle, B, T, N, x["a"], x["b"], x["s0"], sf, so, s)
                f = lambda: sr.sn_scan_fma_backward(ctx.handle, B, T, N, x["a"], x["s0"], so, gs_, None, da, db, d0, s)
                nb = 20 * B * T * N + 8 * B * N
            else:
                sr.sn_scan_gated(ctx.handle, B, T, N, x["a"], x["u"], x["s0"], sf, so, s)
                f = lambda: sr.sn_scan_gated_backward(ctx.handle, B, T, N, x["a"], x["u"], x["s0"], so, gs_, None, da,
                                                      db, d0, s)
                nb = 24 * B * T * N + 8 * B * N
            ms = time_form(torch, f, warmup, reps, s)
            r = {"ms": round(ms, 4), "GBps": round(nb / ms / 1e6, 1),
                 "hbm_frac": round(nb / ms / 1e6 / hbm_peak, 3), "bound": "hbm"}
            if cpu:
                bjob = scan_bwd_job(host(x["a"]), host(so), host(x["s0"]), host(gs_),
                                    u=host(x["u"]) if form == "gated" else None)
                bref, _ = bjob.reference(min(len(bjob.units), host_cores()))
                r.update(errors({"grad_a": host(da), "grad_bu": host(db), "grad_s0": host(d0)}, bref, 1e-5))
                del bref
            out[f"scan_{form}_backward"] = r
        del x, so, sf, gs_, da, db, d0
        for name in ("gla", "mamba2", "deltanet", "rwkv7_prefill", "rwkv7_decode", "gated_memory"):
            c = synth.CONFIGS[name]
            x = synth.config_inputs(name, device=dev)
            Bc, Tc, H, dk, dv = c["B"], c["T"], c["H"], c["dk"], c["dv"]
            o = torch.empty((Bc, Tc, H, dv), device=dev)
            if name in ("gla", "mamba2", "gated_memory"):
                kind, gname = "diag", "d"
                S = torch.empty((Bc, H, dk, dv), device=dev)
                fn = lambda: sr.sn_recur_diag(ctx.handle, Bc, Tc, H, x["G"], dk, dv, x["decay_kind"], x["scale"],
                                              x["q"], x["k"], x["v"], x["d"], None, S, o, s)
            elif name == "deltanet":
                kind, gname = "delta", "beta"
                S = torch.empty((Bc, H, dk, dv), device=dev)
                fn = lambda: sr.sn_recur_delta(ctx.handle, Bc, Tc, H, dk, dv, x["scale"], x["q"], x["k"], x["v"],
                                               x["beta"], None, S, o, s)
            else:
                kind, gname = "rwkv7", "w"
                S = torch.empty((Bc, H, dv, dk), device=dev)
                fn = lambda: sr.sn_recur_rwkv7(ctx.handle, Bc, Tc, H, dk, dv, x["q"], x["k"], x["v"], x["w"],
                                               x["S0"], S, o, s)
            st = fn()
            if st != sr.SN_OK:
                out[name] = {"error": sr.sn_status_str(st)}
                continue
            ms = time_form(torch, fn, warmup, reps, s)
            th, nb, fl = matrix_cost(name)
            gbps = nb / ms / 1e6
            tflops = fl / ms / 1e9
            r = {"ms": round(ms, 4), "tok_heads_per_s": round(th / ms * 1e3, 1), "GBps": round(gbps, 1),
                 "hbm_frac": round(gbps / hbm_peak, 3), "TFLOPs_fp32": round(tflops, 2),
                 "fp32_frac": round(tflops / fp32_peak_tflops, 3)}
            r["bound"] = "hbm" if name == "rwkv7_decode" else "alu"
            out[name] = r
            torch.cuda.synchronize()
            got = {"o": host(o), "S": host(S)}
            chunked = None
            if name in ("gla", "mamba2", "gated_memory", "deltanet"):
                # the chunked tensor-core form of the same workload (tf32 operands)
                if name == "deltanet":
                    ctx.ensure_workspace_bytes(sr.sn_recur_delta_chunked_workspace_bytes(Bc, Tc, H, dk, dv))
                    fc = lambda: sr.sn_recur_delta_chunked(ctx.handle, Bc, Tc, H, dk, dv, x["scale"], x["q"], x["k"],
                                                           x["v"], x["beta"], None, S, o, s)
                    tflop = delta_tensor_flops(Bc, Tc, H, dk, dv)
                else:
                    ctx.ensure_workspace_bytes(sr.sn_recur_chunked_workspace_bytes(Bc, Tc, H, dk, dv))
                    fc = lambda: sr.sn_recur_diag_chunked(ctx.handle, Bc, Tc, H, x["G"], dk, dv, x["decay_kind"],
                                                          x["scale"], x["q"], x["k"], x["v"], x["d"], None, S, o, s)
                    tflop = chunked_tensor_flops(Bc, Tc, H, dk, dv)
                st = fc()
                if st != sr.SN_OK:
                    out[name + "_chunked_tc"] = {"error": sr.sn_status_str(st)}
                else:
                    ms = time_form(torch, fc, warmup, reps, s)
                    tf = tflop / ms / 1e9
                    out[name + "_chunked_tc"] = {
                        "ms": round(ms, 4), "tok_heads_per_s": round(th / ms * 1e3, 1),
                        "GBps": round(nb / ms / 1e6, 1), "hbm_frac": round(nb / ms / 1e6 / hbm_peak, 3),
                        "TFLOPs_tf32": round(tf, 2), "tf32_frac": round(tf / tf32_peak_tflops(), 4),
                        "speedup_vs_sequence_kernel": round(r["ms"] / ms, 2), "bound": "latency",
                        "tolerance": 2e-3}
                    torch.cuda.synchronize()
                    chunked = {"o": host(o), "S": host(S)}
                assert ctx.last_error() == sr.SN_OK
            if cpu:
                xh = {"q": host(x["q"]), "k": host(x["k"]), "v": host(x["v"]), "g": host(x[gname]),
                      "S0": host(x.get("S0")), "scale": x.get("scale", 1.0), "decay_kind": x.get("decay_kind")}
                job = matrix_job(kind, xh, Bc, Tc, H, dk, dv, nb, G=x.get("G", H))
                crec, ref = cpu_record(job)
                r.update(crec)
                pages = PAGES_ERR.get("gla" if name == "gla" else name)
                r.update(errors(got, ref, 1e-4, pages))
                if chunked is not None:
                    out[name + "_chunked_tc"].update(errors(chunked, ref, 2e-3))
                del ref, xh, job
            del x, o, S, got, chunked
        # single-step decode of the other kinds (column decode kernel), B=1024 T=1,
        # random states: each step reads and writes every state once
        for name, maker, (Bc, H, G, dk, dv) in (
                ("gla_decode", lambda c: synth.gla_inputs(1024, 1, 4, 128, 128, cid=c, device=dev), (1024, 4, 4, 128, 128)),
                ("mamba2_decode", lambda c: synth.mamba2_inputs(1024, 1, 24, 1, 128, 64, cid=c, device=dev),
                 (1024, 24, 1, 128, 64)),
                ("deltanet_decode", lambda c: synth.deltanet_inputs(1024, 1, 8, 128, 128, cid=c, device=dev),
                 (1024, 8, 8, 128, 128))):
            x = maker(97)
            S0 = torch.empty((Bc, H, dk, dv), device=dev).normal_(generator=torch.Generator(dev).manual_seed(98))
            S = S0.clone()
            o = torch.empty((Bc, 1, H, dv), device=dev)
            if name == "deltanet_decode":
                call = lambda Si, So: sr.sn_recur_delta(ctx.handle, Bc, 1, H, dk, dv, x["scale"], x["q"], x["k"],
                                                        x["v"], x["beta"], Si, So, o, s)
                gname, kind = "beta", "delta"
            else:
                call = lambda Si, So: sr.sn_recur_diag(ctx.handle, Bc, 1, H, G, dk, dv, x["decay_kind"], x["scale"],
                                                       x["q"], x["k"], x["v"], x["d"], Si, So, o, s)
                gname, kind = "d", "diag"
            gbytes = x[gname].numel() * 4
            nb = 2 * S.numel() * 4 + (x["q"].numel() + x["k"].numel() + x["v"].numel() + o.numel()) * 4 + gbytes
            ms = time_form(torch, lambda: call(S, S), warmup, reps, s)   # in place: the states (>= 268 MB) exceed L2
            r = {"ms": round(ms, 4), "tok_heads_per_s": round(Bc * H / ms * 1e3, 1),
                 "GBps": round(nb / ms / 1e6, 1), "hbm_frac": round(nb / ms / 1e6 / hbm_peak, 3),
                 "bound": "hbm", "workload": f"B={Bc} T=1 H={H} dk={dk} dv={dv}"}
            assert ctx.last_error() == sr.SN_OK
            if cpu:
                # one step from the stored initial states (out of place) against the oracle
                call(S0, S)
                torch.cuda.synchronize()
                got = {"o": host(o), "S": host(S)}
                xh = {"q": host(x["q"]), "k": host(x["k"]), "v": host(x["v"]), "g": host(x[gname]),
                      "S0": host(S0), "scale": x["scale"], "decay_kind": x.get("decay_kind")}
                job = matrix_job(kind, xh, Bc, 1, H, dk, dv, nb, G=G)
                crec, ref = cpu_record(job)
                r.update(crec)
                r.update(errors(got, ref, 1e-4))
                del ref, xh, job, got
            out[name] = r
            del x, S, S0, o
        # readout epilogues on the GLA and Mamba-2 output shapes (12 B per element);
        # L2 is flushed before each timed launch (the GLA tensors fit in it)
        gen = torch.Generator(dev).manual_seed(91)
        for name, (Bc, Tc, H, dv) in (("gla_readout_norm_gate", (4, 4096, 4, 128)),
                                      ("mamba2_readout_dskip", (4, 4096, 24, 64))):
            o = torch.empty((Bc, Tc, H, dv), device=dev).normal_(generator=gen)
            z = torch.empty((Bc, Tc, H, dv), device=dev).normal_(generator=gen)
            y = torch.empty_like(o)
            if name.endswith("norm_gate"):
                w = torch.ones(dv, device=dev)
                fn = lambda: sr.sn_readout_norm_gate(ctx.handle, Bc, Tc, H, dv, o, z, w, 1e-6, y, s)
            else:
                D = torch.ones(H, device=dev)
                fn = lambda: sr.sn_readout_dskip(ctx.handle, Bc, Tc, H, dv, o, z, D, y, s)
            st = fn()
            if st != sr.SN_OK:
                out[name] = {"error": sr.sn_status_str(st)}
                continue
            ms = time_form(torch, fn, warmup, reps, s, flush=flush)
            nb = 12 * o.numel()
            r = {"ms": round(ms, 4), "GBps": round(nb / ms / 1e6, 1),
                 "hbm_frac": round(nb / ms / 1e6 / hbm_peak, 3), "bound": "hbm", "l2": "flushed"}
            if cpu:
                import oracle
                torch.cuda.synchronize()
                oh, zh = host(o), host(z)
                if name.endswith("norm_gate"):
                    tasks = [lambda b=b: oracle.readout_norm_gate(oh[b:b + 1], zh[b:b + 1], host(w), eps=1e-6)
                             for b in range(Bc)]
                else:
                    tasks = [lambda b=b: oracle.readout_dskip(oh[b:b + 1], zh[b:b + 1], host(D)) for b in range(Bc)]
                parts, _ = run_pool(tasks, min(Bc, host_cores()))
                r.update(errors({"y": host(y)}, {"y": np.concatenate(parts, axis=0)}, 1e-5))
            out[name] = r
            del o, z, y
        del flush
    return out


CHUNK = 128


def chunked_tensor_flops(B, T, H, dk, dv):
    """Tensor-core flops of the chunked form: per chunk of C tokens the
    products Q K^T (C x C x dk), Q S (C x dv x dk), A V (C x dv x C) and
    Khat^T V (dk x dv x C)."""
    nch = B * H * ((T + CHUNK - 1) // CHUNK)
    C = CHUNK
    return nch * 2 * (C * C * dk + C * dv * dk + C * dv * C + dk * dv * C)


def delta_tensor_flops(B, T, H, dk, dv):
    """Tensor-core flops of the chunked delta rule per chunk of C tokens: the
    Gram matrix K K^T three times (hi/lo split), W = T K, U = T V, W S_n,
    K^T Delta, and the output products Q K^T, Q S_n and A Delta."""
    nch = B * H * ((T + CHUNK - 1) // CHUNK)
    C = CHUNK
    prep = 3 * C * C * dk + C * C * dk + C * C * dv
    chain = C * dk * dv + dk * C * dv
    out = C * C * dk + C * dk * dv + C * C * dv
    return nch * 2 * (prep + chain + out)


def tf32_peak_tflops():
    """Dense tf32 peak: the measured bf16 burst peak times the nominal
    tf32 / bf16 ratio (1.1 / 2.25 PFLOP/s)."""
    return load_peaks()[0]["bf16_tflops"] * (1.1 / 2.25)


def run_ours(args):
    import torch

    import scan_runtime_gb300 as sr

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    sr.build()
    torch.cuda.set_device(local)
    dev = torch.device(f"cuda:{local}")
    ctx = sr.Context(local)
    stream = torch.cuda.Stream(dev)
    peaks, peak_src = load_peaks()
    hbm_peak = float(peaks["hbm_gbs"])
    props = torch.cuda.get_device_properties(dev)
    sm_count = props.multi_processor_count
    fp32_peak = sm_count * 128 * 2 * float(peaks.get("sm_max_mhz", 2070.0)) * 1e6 / 1e12   # TFLOP/s

    B, T, N = SCAN["B"], SCAN["T"], SCAN["N"]
    x = synth.config_inputs("scan_large", device=dev)
    so_f = torch.empty((B, T, N), device=dev)
    so_g = torch.empty((B, T, N), device=dev)
    sf_f = torch.empty((B, N), device=dev)
    sf_g = torch.empty((B, N), device=dev)
    h = ctx.handle
    per_form_bytes = scan_bytes(B, T, N)
    step_bytes = 2 * per_form_bytes

    def step(evs=None):
        if evs is not None:
            evs[0].record(stream)
        st1 = sr.sn_scan_fma(h, B, T, N, x["a"], x["b"], x["s0"], sf_f, so_f, stream)
        if evs is not None:
            evs[1].record(stream)
        st2 = sr.sn_scan_gated(h, B, T, N, x["a"], x["u"], x["s0"], sf_g, so_g, stream)
        if evs is not None:
            evs[2].record(stream)
        if st1 != sr.SN_OK or st2 != sr.SN_OK:
            raise RuntimeError(f"scan failed: {st1} {st2}")

    torch.cuda.synchronize()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    clk = make_clock_sampler(torch, torch.cuda.current_device(), local)
    clk.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clk.mark(True)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    clk.mark(False)
    if world > 1:
        torch.distributed.barrier()
    time.sleep(0.1)
    clk.stop()
    ms_total = max_over_ranks(t_start.elapsed_time(t_end), dev)
    launch_ms = [e[0].elapsed_time(e[1]) for e in evs] + [e[1].elapsed_time(e[2]) for e in evs]
    avg_launch_ms = sum(launch_ms) / len(launch_ms)
    value = whole_job_gbps(step_bytes, args.steps, world, ms_total)
    achieved = per_form_bytes / (avg_launch_ms / 1e3) / GB

    # end to end through the C ABI's host-buffer call (sn_scan_host): pinned host inputs
    # in, both forms' s_t and s_final out, every step; wall clock per step
    e2e = None
    if not args.no_e2e:
        hbuf = {n: torch.empty_like(x[n], device="cpu").pin_memory() for n in ("a", "b", "u", "s0")}
        for n in hbuf:
            hbuf[n].copy_(x[n])
        hout = {f: (torch.empty((B, T, N), pin_memory=True), torch.empty((B, N), pin_memory=True))
                for f in ("fma", "gated")}

        def e2e_step():
            ctx.scan_host(hbuf["a"], hbuf["b"], hbuf["u"], hbuf["s0"], out=hout, rows_per_chunk=1)

        n_e2e = max(3, min(args.steps, 20))
        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            e2e_step()
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks((time.perf_counter() - t0) * 1e3 / n_e2e, dev)
        h2d = 3 * B * T * N * 4 + B * N * 4
        d2h = 2 * B * T * N * 4 + 2 * B * N * 4
        link = link_bandwidth(torch, dev)
        # the step cannot beat moving its bytes over the host link, both directions at once
        bound_ms = max(h2d, d2h) / (link["concurrent_each_GBps"] * 1e6)
        e2e = {"value": round(whole_job_gbps(step_bytes, 1, world, e2e_ms), 2), "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 3),
               "api": "sn_scan_host (C ABI, host buffers; 3 pipeline streams, one batch row per chunk)",
               "link": link, "link_bound_ms_per_step": round(bound_ms, 3),
               "link_frac": round(bound_ms / e2e_ms, 3)}
        del hbuf, hout

    # CPU baseline: the oracle on this run's own inputs (the full workload,
    # copied to the host), rank 0 at N=1 only: fp64 and fp32, on every host
    # core and on one thread.  The fp64 run is also the reference the GPU
    # outputs are measured against (here and in the forms).
    cpu = None
    scan_rec = scan_ref = None
    do_cpu = rank == 0 and world == 1 and not args.no_cpu
    if do_cpu:
        xh = {n: x[n].cpu().numpy() for n in ("a", "b", "u", "s0")}
        job = scan_job(xh["a"], {"fma": xh["b"], "gated": xh["u"]}, xh["s0"])
        crec, scan_ref = cpu_record(job, reps_1t=5)
        got = {"s_fma": host(so_f), "s_final_fma": host(sf_f), "s_gated": host(so_g), "s_final_gated": host(sf_g)}
        scan_rec = dict(crec)
        scan_rec.update(errors(got, scan_ref, 1e-5, PAGES_ERR["scan"]))
        a64 = crec["cpu_fp64_all"]
        cpu = {"value": a64["GBps"], "unit": "GB/s", "cores": a64["threads"], "kind": "oracle",
               "sample": f"the full workload B=8 T=8192 N=2048 (this run's inputs), both forms, fp64 oracle, "
                         f"{len(job.units)} {job.what} on {a64['threads']} threads, {a64['s']:.2f} s",
               "detail": {"cpu_model": a64["cpu_model"], "logical_cpus": a64["logical_cpus"],
                          "fp64_all_threads_GBps": a64["GBps"],
                          "fp64_1_thread_GBps": crec["cpu_fp64_1t"]["GBps"],
                          "fp32_all_threads_GBps": crec["cpu_fp32_all"]["GBps"],
                          "fp32_1_thread_GBps": crec["cpu_fp32_1t"]["GBps"],
                          "sample_1_thread": crec["cpu_fp64_1t"]["sample"]}}
        del xh, job, got

    forms = None
    if not args.no_forms:
        forms = bench_forms(torch, sr, ctx, dev, stream, fp32_peak, hbm_peak, cpu=do_cpu, scan_ref=scan_ref)
        if scan_rec is not None:
            forms["scan_large"] = scan_rec
    scan_ref = None

    assert ctx.last_error() == sr.SN_OK
    clocks = clk.summary()
    traffic = traffic_record("scan_seq_tma")
    line = {
        "metric": "recurrence_scan_GBps", "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_total / args.steps, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": "scan_large B=8 T=8192 N=2048, FMA + gated forms (sequential-in-T kernel)",
                   "B": B, "T": T, "N": N, "bytes_per_step": step_bytes,
                   "l2": "inputs (1.07 GB per form) larger than L2; no flush",
                   "parallelism": f"dp{world}" if world > 1 else "single"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(achieved / hbm_peak, 4),
                     "traffic": traffic, "kernel": "scan_seq_tma", "peak_source": f"{peak_src} hbm_gbs"},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
        "forms": forms,
        "fp32_peak_tflops": round(fp32_peak, 1),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    ctx.close()
    if world > 1:
        torch.distributed.destroy_process_group()


# ---------------------------------------------------------------- profiling cases
PROFILE_CASES = {
    # name: (description, workload builder)
    "scan_seq": "sequential scan (FMA), B=8 T=2048 N=2048 (402 MB moved, > L2)",
    "scan_seq_full": "sequential scan (FMA), full workload B=8 T=8192 N=2048 (1.61 GB moved)",
    "scan_lookback": "look-back scan (FMA), B=8 T=2048 N=2048",
    "scan_few_channels": "fused chunked scan (FMA, the automatic choice), few channels B=1 T=262144 N=64",
    "scan_bwd_fma": "reverse scan (FMA form), B=8 T=2048 N=2048 (20 B per element)",
    "scan_bwd_gated": "reverse scan (gated form), B=8 T=2048 N=2048 (24 B per element)",
    "gla": "diag per-key, full GLA workload B=4 T=4096 H=4 dk=dv=128",
    "mamba2": "diag per-head, full Mamba-2 workload B=4 T=4096 H=24 dk=128 dv=64",
    "deltanet": "delta rule, full DeltaNet workload B=4 T=4096 H=8 dk=dv=128",
    "rwkv7_prefill": "RWKV-7 sequence kernel, full prefill workload B=16 T=4096 H=12 64x64",
    "rwkv7_decode": "RWKV-7 decode kernel, full decode workload B=1024 T=1 H=12 64x64",
    "gla_decode": "decode ring kernel, GLA single step B=1024 T=1 H=4 128x128, states in place",
    "deltanet_decode": "decode ring kernel, DeltaNet single step B=1024 T=1 H=8 128x128, states in place",
    "gla_chunked": "chunked tensor-core form, full GLA workload B=4 T=4096 H=4 dk=dv=128",
    "mamba2_chunked": "chunked tensor-core form, full Mamba-2 workload B=4 T=4096 H=24 dk=128 dv=64",
    "deltanet_chunked": "chunked tensor-core delta rule, full DeltaNet workload B=4 T=4096 H=8 dk=dv=128",
    "readout_norm_gate": "GLA readout epilogue RMSNorm(o)*w*silu(g), B=4 T=4096 H=24 dv=128 (fills past L2)",
    "readout_dskip": "Mamba-2 skip connection o + D*x, B=4 T=4096 H=24 dv=64",
}


def run_profile_case(args):
    """Run one kernel `--steps` times after `--warmup` on its profiling case and
    print its median time; used as the command under ncu."""
    import torch

    import scan_runtime_gb300 as sr
    sr.build()
    dev = torch.device("cuda:0")
    ctx = sr.Context(0)
    s = torch.cuda.Stream(dev)
    name = args.profile_case
    h = ctx.handle
    if name == "scan_few_channels":
        B, T, N = 1, 262144, 64
        x = synth.scan_inputs(B, T, N, large=True, cid=6, device=dev)
        so = torch.empty((B, T, N), device=dev)
        sf = torch.empty((B, N), device=dev)
        ctx.ensure_workspace(B, T, N)
        fn = lambda: sr.sn_scan_fma(h, B, T, N, x["a"], x["b"], x["s0"], sf, so, s)
        nbytes = scan_bytes(B, T, N)
    elif name.startswith("scan_bwd"):
        B, T, N = 8, 2048, 2048
        x = synth.scan_inputs(B, T, N, large=True, device=dev)
        so = torch.empty((B, T, N), device=dev)
        sf = torch.empty((B, N), device=dev)
        sr.sn_scan_fma(h, B, T, N, x["a"], x["b"], x["s0"], sf, so, s)
        gs_ = torch.empty((B, T, N), device=dev).normal_(generator=torch.Generator(dev).manual_seed(77))
        da, db = torch.empty((B, T, N), device=dev), torch.empty((B, T, N), device=dev)
        d0 = torch.empty((B, N), device=dev)
        if name.endswith("gated"):
            fn = lambda: sr.sn_scan_gated_backward(h, B, T, N, x["a"], x["u"], x["s0"], so, gs_, None, da, db, d0, s)
            nbytes = 24 * B * T * N + 8 * B * N
        else:
            fn = lambda: sr.sn_scan_fma_backward(h, B, T, N, x["a"], x["s0"], so, gs_, None, da, db, d0, s)
            nbytes = 20 * B * T * N + 8 * B * N
    elif name.startswith("scan"):
        B, T, N = (8, 8192, 2048) if name.endswith("_full") else (8, 2048, 2048)
        x = synth.scan_inputs(B, T, N, large=True, device=dev)
        so = torch.empty((B, T, N), device=dev)
        sf = torch.empty((B, N), device=dev)
        if name == "scan_lookback":
            ctx.set_option(sr.SN_OPT_SCAN_KERNEL, sr.SN_SCAN_KERNEL_LOOKBACK)
            ctx.ensure_workspace(B, T, N)
        else:
            ctx.set_option(sr.SN_OPT_SCAN_KERNEL, sr.SN_SCAN_KERNEL_SEQUENTIAL)
        fn = lambda: sr.sn_scan_fma(h, B, T, N, x["a"], x["b"], x["s0"], sf, so, s)
        nbytes = scan_bytes(B, T, N)
    elif name.startswith("readout_"):
        Bc, Tc, H, dv = (4, 4096, 24, 128) if name.endswith("norm_gate") else (4, 4096, 24, 64)
        gen = torch.Generator(dev).manual_seed(92)
        o = torch.empty((Bc, Tc, H, dv), device=dev).normal_(generator=gen)
        z = torch.empty((Bc, Tc, H, dv), device=dev).normal_(generator=gen)
        y = torch.empty_like(o)
        if name.endswith("norm_gate"):
            w = torch.ones(dv, device=dev)
            fn = lambda: sr.sn_readout_norm_gate(h, Bc, Tc, H, dv, o, z, w, 1e-6, y, s)
        else:
            D = torch.ones(H, device=dev)
            fn = lambda: sr.sn_readout_dskip(h, Bc, Tc, H, dv, o, z, D, y, s)
        nbytes = 12 * o.numel()
    elif name in ("gla_decode", "deltanet_decode"):
        if name == "gla_decode":
            Bc, H, dk, dv = 1024, 4, 128, 128
            x = synth.gla_inputs(Bc, 1, H, dk, dv, cid=97, device=dev)
        else:
            Bc, H, dk, dv = 1024, 8, 128, 128
            x = synth.deltanet_inputs(Bc, 1, H, dk, dv, cid=97, device=dev)
        S = torch.empty((Bc, H, dk, dv), device=dev).normal_(generator=torch.Generator(dev).manual_seed(98))
        o = torch.empty((Bc, 1, H, dv), device=dev)
        if name == "gla_decode":
            fn = lambda: sr.sn_recur_diag(h, Bc, 1, H, H, dk, dv, x["decay_kind"], x["scale"], x["q"], x["k"],
                                          x["v"], x["d"], S, S, o, s)
            gbytes = x["d"].numel() * 4
        else:
            fn = lambda: sr.sn_recur_delta(h, Bc, 1, H, dk, dv, x["scale"], x["q"], x["k"], x["v"], x["beta"],
                                           S, S, o, s)
            gbytes = x["beta"].numel() * 4
        nbytes = 2 * S.numel() * 4 + (x["q"].numel() + x["k"].numel() + x["v"].numel() + o.numel()) * 4 + gbytes
    elif name == "deltanet_chunked":
        c = synth.CONFIGS["deltanet"]
        x = synth.config_inputs("deltanet", device=dev)
        Bc, Tc, H, dk, dv = c["B"], c["T"], c["H"], c["dk"], c["dv"]
        o = torch.empty((Bc, Tc, H, dv), device=dev)
        S = torch.empty((Bc, H, dk, dv), device=dev)
        ctx.ensure_workspace_bytes(sr.sn_recur_delta_chunked_workspace_bytes(Bc, Tc, H, dk, dv))
        fn = lambda: sr.sn_recur_delta_chunked(h, Bc, Tc, H, dk, dv, x["scale"], x["q"], x["k"], x["v"], x["beta"],
                                               None, S, o, s)
        nbytes = matrix_cost("deltanet")[1]
    elif name.endswith("_chunked"):
        base = name[:-len("_chunked")]
        c = synth.CONFIGS[base]
        x = synth.config_inputs(base, device=dev)
        Bc, Tc, H, dk, dv = c["B"], c["T"], c["H"], c["dk"], c["dv"]
        o = torch.empty((Bc, Tc, H, dv), device=dev)
        S = torch.empty((Bc, H, dk, dv), device=dev)
        ctx.ensure_workspace_bytes(sr.sn_recur_chunked_workspace_bytes(Bc, Tc, H, dk, dv))
        fn = lambda: sr.sn_recur_diag_chunked(h, Bc, Tc, H, x["G"], dk, dv, x["decay_kind"], x["scale"], x["q"],
                                              x["k"], x["v"], x["d"], None, S, o, s)
        nbytes = matrix_cost(base)[1]
    else:
        c = synth.CONFIGS[name]
        x = synth.config_inputs(name, device=dev)
        Bc, Tc, H, dk, dv = c["B"], c["T"], c["H"], c["dk"], c["dv"]
        o = torch.empty((Bc, Tc, H, dv), device=dev)
        if name in ("gla", "mamba2"):
            S = torch.empty((Bc, H, dk, dv), device=dev)
            fn = lambda: sr.sn_recur_diag(h, Bc, Tc, H, x["G"], dk, dv, x["decay_kind"], x["scale"], x["q"], x["k"],
                                          x["v"], x["d"], None, S, o, s)
        elif name == "deltanet":
            S = torch.empty((Bc, H, dk, dv), device=dev)
            fn = lambda: sr.sn_recur_delta(h, Bc, Tc, H, dk, dv, x["scale"], x["q"], x["k"], x["v"], x["beta"],
                                           None, S, o, s)
        else:
            S = torch.empty((Bc, H, dv, dk), device=dev)
            fn = lambda: sr.sn_recur_rwkv7(h, Bc, Tc, H, dk, dv, x["q"], x["k"], x["v"], x["w"], x["S0"], S, o, s)
        nbytes = matrix_cost(name)[1]
    torch.cuda.synchronize()
    def call():
        st = fn()
        if st != sr.SN_OK:
            raise RuntimeError(f"{name}: {sr.sn_status_str(st)}")

    ms = time_form(torch, call, args.warmup, args.steps, s)
    assert ctx.last_error() == sr.SN_OK
    print(json.dumps({"profile_case": name, "what": PROFILE_CASES[name], "median_ms": round(ms, 4),
                      "GBps": round(nbytes / ms / 1e6, 1)}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-forms", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--profile-case", choices=sorted(PROFILE_CASES), default=None,
                    help="run only this kernel on its profiling case (for ncu)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.profile_case:
        run_profile_case(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

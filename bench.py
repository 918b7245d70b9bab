"""Benchmark: attention forward useful TFLOP/s on one GB300 (per process), JSON line on rank 0.

Workload (default): causal MHA prefill B=2, H=32, S=4096, d=128, bf16, seeded
synthetic N(0,1) inputs with query heads 16-31 doubled.  Useful FLOPs count 4*d
per allowed (i, j) pair only (masked pairs are not counted).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

A decode workload name (decode_* / cross_*) times one decode step instead: S_q new
query rows per sequence against a key/value cache resident in HBM (same metric,
useful TFLOP/s; its roofline is HBM bandwidth over the algorithmic bytes).

Each timed step is one attn_forward over the whole batch (all heads, all rows);
L2 is flushed before every step (a 256 MiB buffer written, then read back) and
the step is timed with CUDA events on the launching stream.  Under torchrun every rank runs its own
replica of the workload (the forward pass has no exchange step); the reported
value is all ranks' useful FLOPs over the slowest rank's time.
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

import workloads as wl  # noqa: E402

METRIC = "attention fwd useful TFLOP/s and % of GB300 dense BF16 tensor peak"
NOMINAL_BF16_TFLOPS = 2250.0
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_SOURCES = ["transformer_self_attention_gb300/csrc/attn_fwd_tc.cu",
                  "transformer_self_attention_gb300/csrc/sm103_ptx.h",
                  "transformer_self_attention_gb300/csrc/kernels.h"]
DECODE_KERNEL_SOURCES = ["transformer_self_attention_gb300/csrc/attn_decode.cu",
                         "transformer_self_attention_gb300/csrc/sm103_ptx.h",
                         "transformer_self_attention_gb300/csrc/kernels.h"]


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK), "fallback"


def kernel_hash(sources=KERNEL_SOURCES) -> str:
    h = hashlib.sha256()
    for rel in sources:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload_name: str, kernel: str = "attn_fwd_tc", sources=KERNEL_SOURCES):
    """DRAM bytes per launch of the dominant kernel from the committed ncu summary, if current."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload_name}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_hash = re.search(r"kernel_source_hash:\s*([0-9a-f]+)", text)
    m_bytes = re.search(r"dram_bytes_per_full_launch:\s*([0-9.eE+]+)", text)
    if not m_hash or not m_bytes or m_hash.group(1) != kernel_hash(sources):
        return None
    return float(m_bytes.group(1))


# The NVML sampler that ClockSampler runs in a child process (no torch import, so it starts in
# milliseconds).  It reads the SM clock and the clock event reasons (the power draw every 16th
# time, the maximum clock once), sleeping `interval` seconds between readings, stamped with
# CLOCK_MONOTONIC, until its standard input closes.
_NVML_SAMPLER = r"""
import ctypes, sys, time, select
bus, interval = sys.argv[1].encode(), float(sys.argv[2])
nv = ctypes.CDLL("libnvidia-ml.so.1")
assert nv.nvmlInit_v2() == 0
h = ctypes.c_void_p()
assert nv.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(h)) == 0
get_reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or nv.nvmlDeviceGetCurrentClocksThrottleReasons
mhz, mx, mw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))
print("ready", flush=True)
out = []
k = 0
while True:
    t = time.monotonic()
    nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(mhz))       # NVML_CLOCK_SM
    get_reasons(h, ctypes.byref(rs))
    if k % 16 == 0:                                          # the power reading is slower: every 16th
        nv.nvmlDeviceGetPowerUsage(h, ctypes.byref(mw))
    k += 1
    out.append("%.6f %d %d %d %d" % (t, mhz.value, mx.value, mw.value, rs.value))
    if select.select([sys.stdin], [], [], 0)[0] and not sys.stdin.readline():
        break
    time.sleep(interval)
print("\n".join(out), flush=True)
nv.nvmlShutdown()
"""

# NVML clock event reason bits (nvml.h)
_REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown"}


class ClockSampler:
    """SM clock and throttle reasons sampled during the timed region.

    NVML in a child process about every 0.1-0.2 ms (its readings are stamped with the monotonic clock, and
    the summary keeps those between mark_start() and mark_end(), weighting each reading by the
    time until the next); nvidia-smi every 200 ms when NVML cannot be loaded.
    """
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, device=None):
        self.proc, self.kind, self.t0, self.t1 = None, None, None, None
        try:
            import torch
            pr = torch.cuda.get_device_properties(device if device is not None else gpu_index)
            bus = "%08x:%02x:%02x.0" % (pr.pci_domain_id, pr.pci_bus_id, pr.pci_device_id)
            self.proc = subprocess.Popen([sys.executable, "-c", _NVML_SAMPLER, bus, "0.0001"], stdin=subprocess.PIPE,
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            if self.proc.stdout.readline().strip() == "ready":
                self.kind = "nvml"
            else:
                self.proc.kill()
                self.proc = None
        except Exception:
            self.proc = None
        if self.proc is None:
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                     "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
                self.kind = "nvidia-smi"
            except (FileNotFoundError, OSError):
                self.proc = None

    def mark_start(self):
        self.t0 = time.monotonic()

    def mark_end(self):
        self.t1 = time.monotonic()

    def stop(self):
        if self.proc is None:
            return None
        if self.kind == "nvml":
            try:
                out, _ = self.proc.communicate(input="", timeout=10)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                return None
            return self._summary_nvml(out)
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        return self._summary_smi(out)

    def _summary_nvml(self, out):
        rows = []
        for line in out.strip().splitlines():
            parts = line.split()
            if len(parts) == 5:
                rows.append((float(parts[0]), float(parts[1]), float(parts[2]), float(parts[3]), int(parts[4])))
        if not rows:
            return None
        t0 = self.t0 if self.t0 is not None else rows[0][0]
        t1 = self.t1 if self.t1 is not None else rows[-1][0]
        # readings inside the timed region, plus the last one before it (in force at its start)
        inside = [r for r in rows if t0 <= r[0] <= t1]
        before = [r for r in rows if r[0] < t0]
        sel = ([before[-1]] if before else []) + inside
        if not sel:
            return None
        # time-weighted median of the SM clock over [t0, t1]
        spans = []
        for k, r in enumerate(sel):
            a = max(r[0], t0)
            b = sel[k + 1][0] if k + 1 < len(sel) else t1
            spans.append((r[1], max(0.0, b - a)))
        total = sum(w for _, w in spans)
        acc, med = 0.0, spans[0][0]
        for mhz, wgt in sorted(spans):
            acc += wgt
            if acc >= 0.5 * total:
                med = mhz
                break
        reasons = set()
        for r in sel:
            for bit, name in _REASON_BITS.items():
                if r[4] & bit:
                    reasons.add(name)
        return {"sm_mhz": med, "sm_max_mhz": max(r[2] for r in sel), "reasons": sorted(reasons),
                "samples": len(inside), "sampler": "NVML about every 0.1-0.2 ms in a child process",
                "sm_mhz_time_weighted_median": med, "sm_mhz_min": min(r[1] for r in sel),
                "power_w_max": max(r[3] for r in sel) / 1000.0, "timed_region_s": t1 - t0}

    def _summary_smi(self, out):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        loaded = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "sampler": "nvidia-smi every 200 ms"}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


_INPUTS = {}


def _oracle_inputs(w: wl.Workload):
    if w.name not in _INPUTS:
        Qc, Kc, Vc = wl.make_inputs(w)
        _INPUTS[w.name] = (Qc.float().numpy(), Kc.float().numpy(), Vc.float().numpy())
    return _INPUTS[w.name]


def make_bias_matrix(w: wl.Workload):
    """The per-head bias matrix [1, Hq, S, S] of `--bias`: bf16 N(0, 2^2), seeded by the workload."""
    import torch
    g = torch.Generator(device="cpu").manual_seed(w.seed + 2)
    return (torch.randn(1, w.Hq, w.S, w.S, generator=g) * 2).to(torch.bfloat16)


def score_bias_host(args, w: wl.Workload):
    """The score bias of the command line as the oracle takes it: (ALiBi slopes [Hq] or None,
    float32 bias matrix [1, Hq, S, S] or None), the values the GPU arm sets."""
    alibi = wl.alibi_slopes(w.Hq) if getattr(args, "alibi", False) else None
    bias = None
    if getattr(args, "bias", False):
        key = ("bias", w.name)
        if key not in _INPUTS:
            _INPUTS[key] = make_bias_matrix(w).float().numpy()
        bias = _INPUTS[key]
    return alibi, bias


def cpu_baseline(w: wl.Workload, target_s: float = 12.0, frac: float | None = None, sb=(None, None)):
    """The fp64 oracle, as it stands, on a strided sample of the workload's rows (with the
    score bias sb = (slopes, bias matrix) of the timed configuration)."""
    import numpy as np
    n_cores = len(os.sched_getaffinity(0))
    os.environ.setdefault("OMP_NUM_THREADS", str(n_cores))
    import oracle
    oracle.build()
    Qf, Kf, Vf = _oracle_inputs(w)
    pairs = wl.allowed_pairs_per_head(w)

    def run(stride):
        bb, aa, ii = np.meshgrid(np.arange(w.B), np.arange(w.Hq), np.arange(0, w.S, stride), indexing="ij")
        rb, ra, ri = bb.ravel(), aa.ravel(), ii.ravel()
        t0 = time.perf_counter()
        oracle.attention_rows(Kf, Vf, w.Hq, w.scale, w.kind, w.window, list(w.globals_idx), Qf[rb, ra, ri],
                              rb, ra, ri, alibi=sb[0], bias=sb[1])
        dt = time.perf_counter() - t0
        # useful flops of the sampled rows: rows are strided uniformly, so the sample holds 1/stride of the pairs
        rows_frac = len(ri) / (w.B * w.Hq * w.S)
        return dt, 4.0 * w.d * pairs * w.B * w.Hq * rows_frac, len(ri)

    if frac is None:
        dt, fl, _ = run(64)
        rate = fl / max(dt, 1e-6)
        want = min(1.0, rate * target_s / wl.useful_flops(w))
        stride = max(1, int(round(1.0 / max(want, 1e-9))))
    else:
        stride = max(1, int(round(1.0 / frac)))
    dt, fl, n = run(stride)
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": int(os.environ["OMP_NUM_THREADS"]),
            "kind": "oracle", "seconds": round(dt, 3),
            "sample": f"every {stride}th query row of every (batch, head): {n} rows, "
                      f"{fl / 1e9:.1f} useful GFLOP, fp64 C oracle with OpenMP"}


def fwd_config(args, w, world: int = 1) -> dict:
    """The workload description both arms print (identical keys and values for one command line)."""
    return {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "S": w.S, "d": w.d,
            "mask": wl.MASK_NAMES[w.kind], "window": w.window, "n_global": len(w.globals_idx),
            "useful_gflop_per_step": wl.useful_flops(w) / 1e9,
            "l2": L2Flush.NOTE,
            "score_bias": ("alibi, slopes 2^(-8(a+1)/H)" if args.alibi else
                           "matrix [1, Hq, S, S] bf16 N(0, 2^2)" if args.bias else "none"),
            "inputs": "E4M3, per-tensor scales" if args.fp8 else w.dtype,
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def run_reference(args, w):
    world, rank, _ = dist_setup()
    if rank != 0:
        return 0
    n_cores = len(os.sched_getaffinity(0))
    os.environ.setdefault("OMP_NUM_THREADS", str(n_cores))
    # one calibration sample fixes the per-step sample so the whole run takes a few minutes
    sb = score_bias_host(args, w)
    cal = cpu_baseline(w, target_s=max(2.0, 150.0 / max(1, args.steps + args.warmup)), sb=sb)
    frac_stride = int(re.search(r"every (\d+)th", cal["sample"]).group(1))
    times, flops = [], 0.0
    for s in range(args.warmup + args.steps):
        r = cpu_baseline(w, frac=1.0 / frac_stride, sb=sb)
        if s >= args.warmup:
            times.append(r["seconds"])
            flops = r["value"] * r["seconds"] * 1e12
    t = sum(times) / len(times)
    value = flops / t / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": fwd_config(args, w, max(1, args.gpus)),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": int(os.environ["OMP_NUM_THREADS"]),
                             "kind": "oracle", "sample": r["sample"]},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


class L2Flush:
    """Evicts the step's inputs from L2 (129 MB) before a timed step: a 256 MiB buffer is written,
    then read back.  The write alone leaves about L2's worth of dirty lines, and the next kernel
    would pay for writing them back to HBM inside its own time (18 us of a 142 us decode step);
    the read pass has them written back before the timed region and leaves only clean lines of
    the buffer in L2."""

    BYTES = 256 * 1024 * 1024
    NOTE = "flushed before every GPU step (256 MiB written, then read back)"

    def __init__(self, dev):
        import torch
        self.buf = torch.empty(self.BYTES, dtype=torch.uint8, device=dev)
        self.words = self.buf.view(torch.int64)

    def __call__(self):
        import torch
        self.buf.zero_()
        torch.amax(self.words)


def pipelined_e2e(dev, h_in, h_out, run, n_steps: int, n_sets: int = 2) -> float:
    """Milliseconds per end-to-end step over host-resident problems.

    Every step copies its inputs (pinned host tensors h_in) to the device, runs the computation and copies
    its outputs back (into the pinned host tensors h_out).  The copies of one step overlap the computation
    of its neighbours: one stream for host->device copies, one for the computation, one for device->host
    copies, and n_sets device buffer sets that the steps use in turn.  run(d_in, d_out, stream) enqueues
    the computation.  The timed region runs from before the first step's input copy to after the last
    step's output copy (CUDA events), so it holds every step's copies in full."""
    import torch

    s_in, s_comp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    sets = [([torch.empty(t.shape, dtype=t.dtype, device=dev) for t in h_in],
             [torch.empty(t.shape, dtype=t.dtype, device=dev) for t in h_out]) for _ in range(n_sets)]
    comp_done = [None] * n_sets  # the computation that last read a set's inputs
    out_done = [None] * n_sets   # the copy that last read a set's outputs

    def step(k):
        j = k % n_sets
        d_in, d_out = sets[j]
        if comp_done[j] is not None:
            s_in.wait_event(comp_done[j])
        with torch.cuda.stream(s_in):
            for d_, h_ in zip(d_in, h_in):
                d_.copy_(h_, non_blocking=True)
        e_in = torch.cuda.Event()
        e_in.record(s_in)
        s_comp.wait_event(e_in)
        if out_done[j] is not None:
            s_comp.wait_event(out_done[j])
        run(d_in, d_out, s_comp)
        e_c = torch.cuda.Event()
        e_c.record(s_comp)
        comp_done[j] = e_c
        s_out.wait_event(e_c)
        with torch.cuda.stream(s_out):
            for h_, d_ in zip(h_out, d_out):
                h_.copy_(d_, non_blocking=True)
        e_o = torch.cuda.Event()
        e_o.record(s_out)
        out_done[j] = e_o

    for k in range(n_sets):  # warm-up: every buffer set once
        step(k)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for k in range(n_steps):
        step(k)
    e1.record(s_out)
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) / n_steps


def run_ours(args, w):
    import torch
    import torch.distributed as dist

    import transformer_self_attention_gb300 as tsa
    from transformer_self_attention_gb300.shard import max_over_ranks

    world, rank, local = dist_setup()
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    if args.fp8:
        Qc, Kc, Vc, descales = wl.make_fp8_inputs(w)
        plan = tsa.Attention(w.B, w.Hq, w.Hkv, w.S, w.d, dtype="e4m3", scale=w.scale, kind=w.kind,
                             window=w.window, global_idx=list(w.globals_idx))
        plan.set_fp8_descale(*descales)
    else:
        Qc, Kc, Vc = wl.make_inputs(w)
        plan = tsa.Attention(w.B, w.Hq, w.Hkv, w.S, w.d, dtype=w.dtype, scale=w.scale, kind=w.kind,
                             window=w.window, global_idx=list(w.globals_idx))
    Q, K, V = Qc.to(dev), Kc.to(dev), Vc.to(dev)
    if args.alibi:
        plan.set_alibi(wl.alibi_slopes(w.Hq))
    if args.bias:  # a per-head bias matrix [1, Hq, S, S], bf16 N(0, 2^2), resident in HBM
        bias = make_bias_matrix(w).to(dev)
        plan.set_bias(bias)
    O = torch.empty(Q.shape, dtype=torch.bfloat16 if args.fp8 else Q.dtype, device=dev)
    LSE = torch.empty((w.B, w.Hq, w.S), dtype=torch.float32, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)
    launches_per_fwd = 1  # one launch of the tensor-core kernel (local + global included)

    def fwd():
        plan(Q, K, V, O=O, LSE=LSE, stream=stream)

    for _ in range(args.warmup):
        flush()
        fwd()
    torch.cuda.synchronize(dev)
    st, code = plan.poll_device_error()
    if st != 0:
        raise RuntimeError(f"device error during warm-up: {code}")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(local, dev) if rank == 0 else None
    if clocks:
        clocks.mark_start()
    wall0 = time.perf_counter()
    for s in range(args.steps):
        flush()
        starts[s].record(stream)
        fwd()
        ends[s].record(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    if clocks:
        clocks.mark_end()
    if world > 1:
        dist.barrier()
    clk = clocks.stop() if clocks else None
    step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    mean_ms = sum(step_ms) / len(step_ms)
    mean_ms = max_over_ranks(mean_ms, dev)  # the slowest rank
    st, code = plan.poll_device_error()
    if st != 0:
        raise RuntimeError(f"device error during the timed steps: {code}")

    useful = wl.useful_flops(w)
    value = world * useful / (mean_ms * 1e-3) / 1e12
    pk, pk_src = peaks()

    # end to end through the C ABI: pinned host inputs -> device, forward, O and LSE -> pinned host
    e2e = None
    if not args.no_e2e:
        h_in = [t.pin_memory() for t in (Qc, Kc, Vc)]
        h_out = [torch.empty(O.shape, dtype=O.dtype, pin_memory=True),
                 torch.empty(LSE.shape, dtype=LSE.dtype, pin_memory=True)]
        n_e2e = max(4, min(args.steps, 10))

        def e2e_run(d_in, d_out, st):
            plan(d_in[0], d_in[1], d_in[2], O=d_out[0], LSE=d_out[1], stream=st)

        e2e_ms = pipelined_e2e(dev, h_in, h_out, e2e_run, n_e2e)
        e2e_ms = max_over_ranks(e2e_ms, dev)  # the slowest rank
        bi = sum(t.numel() * t.element_size() for t in (Qc, Kc, Vc))
        bo = O.numel() * O.element_size() + LSE.numel() * LSE.element_size()
        e2e = {"value": world * useful / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": e2e_ms,
               "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
               "overlap": "copies of each step overlap the neighbouring steps' computation (3 streams, 2 buffer sets)"}

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    achieved = useful / (mean_ms * 1e-3) / 1e12
    peak = float(pk["bf16_tflops"]) * (2.0 if args.fp8 else 1.0)
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "traffic": None if args.fp8 else ncu_traffic(w.name),
                "peak_source": (f"{pk_src} bf16_tflops (burst, cuBLAS) x 2, the nominal E4M3:BF16 rate ratio"
                                if args.fp8 else f"{pk_src} bf16_tflops (burst, cuBLAS)"),
                "kernel": "attn_fwd_tc_kernel"}
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": mean_ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "e4m3" if args.fp8 else ("bf16" if w.dtype == "bf16" else "f32"),
            "data": "synthetic" + (" (E4M3, per-tensor scales)" if args.fp8 else ""),
            "config": fwd_config(args, w, world),
            "pct_of_peak": {"measured": 100.0 * achieved / peak, "nominal": 100.0 * achieved / NOMINAL_BF16_TFLOPS,
                            "peak_source": pk_src},
            "roofline": roofline, "gpu_launches": args.steps * launches_per_fwd,
            "wall_s_timed_region": wall}
    if e2e:
        line["e2e"] = e2e
    if clk:
        line["clocks"] = clk
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(w, sb=score_bias_host(args, w))
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


# ----------------------------------------------------------------------------- backward
BWD_METRIC = "attention bwd useful TFLOP/s and % of GB300 dense BF16 tensor peak"
BWD_KERNEL_SOURCES = ["transformer_self_attention_gb300/csrc/attn_bwd.cu",
                      "transformer_self_attention_gb300/csrc/sm103_ptx.h",
                      "transformer_self_attention_gb300/csrc/kernels.h"]


def cpu_baseline_backward(w: wl.Workload, target_s: float = 12.0, n_slices: int | None = None, sb=(None, None)):
    """The fp64 backward oracle, as it stands, on whole (batch, kv head) slices of the workload
    (every query head of the group, every row), with the score bias sb = (slopes, bias matrix)."""
    n_cores = len(os.sched_getaffinity(0))
    os.environ.setdefault("OMP_NUM_THREADS", str(n_cores))
    import oracle
    oracle.build()
    key = ("bwd", w.name)
    if key not in _INPUTS:
        Qc, Kc, Vc = wl.make_inputs(w)
        _INPUTS[key] = tuple(t.float().numpy() for t in (Qc, Kc, Vc, wl.make_grad_output(w)))
    Qf, Kf, Vf, dOf = _INPUTS[key]
    group = w.Hq // w.Hkv
    per_slice = wl.backward_flops(w) / (w.B * w.Hkv)

    def run(n):
        t0 = time.perf_counter()
        for k in range(n):
            b, g = divmod(k % (w.B * w.Hkv), w.Hkv)
            qs = slice(g * group, (g + 1) * group)
            oracle.backward(Qf[b:b + 1, qs], Kf[b:b + 1, g:g + 1], Vf[b:b + 1, g:g + 1], dOf[b:b + 1, qs], w.scale,
                            w.kind, w.window, globals_idx=list(w.globals_idx),
                            alibi=None if sb[0] is None else sb[0][qs],
                            bias=None if sb[1] is None else sb[1][:, qs])
        return time.perf_counter() - t0

    if n_slices is None:
        dt = run(1)
        n_slices = max(1, min(w.B * w.Hkv, int(target_s / max(dt, 1e-6))))
    dt = run(n_slices)
    fl = per_slice * n_slices
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": int(os.environ["OMP_NUM_THREADS"]),
            "kind": "oracle", "seconds": round(dt, 3), "n_slices": n_slices,
            "sample": f"{n_slices} of {w.B * w.Hkv} (batch, kv head) slices in full ({group} query heads each), "
                      f"{fl / 1e9:.1f} useful GFLOP, fp64 C oracle with OpenMP"}


def _bwd_config(w, useful, world: int = 1, alibi: bool = False, bias: bool = False):
    return {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "S": w.S, "d": w.d,
            "mask": wl.MASK_NAMES[w.kind], "window": w.window, "pass": "backward (dQ, dK, dV)",
            "useful_gflop_per_step": useful / 1e9, "flops_per_pair": f"10 d (2.5 x the forward's 4 d)",
            "score_bias": ("alibi, slopes 2^(-8(a+1)/H)" if alibi else
                           "matrix [1, Hq, S, S] bf16 N(0, 2^2)" if bias else "none"),
            "l2": L2Flush.NOTE,
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def run_reference_backward(args, w):
    world, rank, _ = dist_setup()
    if rank != 0:
        return 0
    sb = score_bias_host(args, w)
    cal = cpu_baseline_backward(w, target_s=max(2.0, 150.0 / max(1, args.steps + args.warmup)), sb=sb)
    times, r = [], None
    for s in range(args.warmup + args.steps):
        r = cpu_baseline_backward(w, n_slices=cal["n_slices"], sb=sb)
        if s >= args.warmup:
            times.append(r["seconds"])
    t = sum(times) / len(times)
    value = r["value"] * r["seconds"] / t
    line = {"impl": "reference", "metric": BWD_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": _bwd_config(w, wl.backward_flops(w), max(1, args.gpus), args.alibi, args.bias),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": r["cores"], "kind": "oracle",
                             "sample": r["sample"]},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_ours_backward(args, w):
    import torch
    import torch.distributed as dist

    import transformer_self_attention_gb300 as tsa
    from transformer_self_attention_gb300.shard import max_over_ranks

    world, rank, local = dist_setup()
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    Qc, Kc, Vc = wl.make_inputs(w)
    dOc = wl.make_grad_output(w)
    Q, K, V, dO = (t.to(dev) for t in (Qc, Kc, Vc, dOc))
    plan = tsa.Attention(w.B, w.Hq, w.Hkv, w.S, w.d, dtype=w.dtype, scale=w.scale, kind=w.kind, window=w.window,
                         global_idx=list(w.globals_idx))
    if args.alibi:
        plan.set_alibi(wl.alibi_slopes(w.Hq))
    if args.bias:  # the forward's per-head bias matrix, resident in HBM; both passes read it
        bias = make_bias_matrix(w).to(dev)
        plan.set_bias(bias)
    O, LSE = plan(Q, K, V)
    dQ, dK, dV = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        plan.backward(Q, K, V, O, LSE, dO, dQ, dK, dV, stream=stream)

    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize(dev)
    st, code = plan.poll_device_error()
    if st != 0:
        raise RuntimeError(f"device error during warm-up: {code}")
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(local, dev) if rank == 0 else None
    if clocks:
        clocks.mark_start()
    wall0 = time.perf_counter()
    for s in range(args.steps):
        flush()
        starts[s].record(stream)
        step()
        ends[s].record(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    if clocks:
        clocks.mark_end()
    if world > 1:
        dist.barrier()
    clk = clocks.stop() if clocks else None
    mean_ms = sum(a.elapsed_time(b) for a, b in zip(starts, ends)) / args.steps
    mean_ms = max_over_ranks(mean_ms, dev)  # the slowest rank
    st, code = plan.poll_device_error()
    if st != 0:
        raise RuntimeError(f"device error during the timed steps: {code}")
    useful = wl.backward_flops(w)
    value = world * useful / (mean_ms * 1e-3) / 1e12
    pk, pk_src = peaks()

    # end to end through the C ABI: Q, K, V, O, LSE and dO from pinned host memory, the
    # backward, dQ, dK and dV back to pinned host memory
    e2e = None
    if not args.no_e2e:
        hin = [t.pin_memory() for t in (Qc, Kc, Vc, O.cpu(), LSE.cpu(), dOc)]
        hout = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (dQ, dK, dV)]
        n_e2e = max(4, min(args.steps, 10))

        def e2e_run(d_in, d_out, st):
            plan.backward(*d_in[:5], d_in[5], d_out[0], d_out[1], d_out[2], stream=st)

        e2e_ms = pipelined_e2e(dev, hin, hout, e2e_run, n_e2e)
        e2e_ms = max_over_ranks(e2e_ms, dev)  # the slowest rank
        e2e = {"value": world * useful / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": e2e_ms,
               "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in hin),
               "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in hout),
               "overlap": "copies of each step overlap the neighbouring steps' computation (3 streams, 2 buffer sets)"}

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0
    achieved = useful / (mean_ms * 1e-3) / 1e12
    peak = float(pk["bf16_tflops"])
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "traffic": ncu_traffic(w.name, "attn_bwd", BWD_KERNEL_SOURCES),
                "peak_source": f"{pk_src} bf16_tflops (burst, cuBLAS)",
                "kernel": "the whole backward step (bwd_prep + attn_bwd_dq + attn_bwd_dkdv)"}
    line = {"metric": BWD_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": mean_ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": _bwd_config(w, useful, world, args.alibi, args.bias),
            "roofline": roofline, "gpu_launches": 3 * args.steps, "wall_s_timed_region": wall}
    if e2e:
        line["e2e"] = e2e
    if clk:
        line["clocks"] = clk
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline_backward(w, sb=score_bias_host(args, w))
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


# ----------------------------------------------------------------------------- decode
def _decode_oracle_inputs(w):
    key = ("decode", w.name)
    if key not in _INPUTS:
        Qc, Kc, Vc, lens = wl.make_decode_inputs(w)
        _INPUTS[key] = (Qc.float().numpy(), Kc.float().numpy(), Vc.float().numpy(), lens)
    return _INPUTS[key]


def cpu_baseline_decode(w, target_s: float = 12.0, n_seq: int | None = None, alibi=None):
    """The fp64 decode oracle, as it stands, on the first n_seq sequences of the batch (with the
    ALiBi slopes of the timed configuration, if any)."""
    n_cores = len(os.sched_getaffinity(0))
    os.environ.setdefault("OMP_NUM_THREADS", str(n_cores))
    import oracle
    oracle.build()
    Qf, Kf, Vf, lens = _decode_oracle_inputs(w)

    def run(nb):
        t0 = time.perf_counter()
        oracle.decode(Qf[:nb], Kf[:nb], Vf[:nb], lens[:nb], w.scale, w.kind, w.window, alibi=alibi)
        dt = time.perf_counter() - t0
        return dt, wl.decode_useful_flops(w, lens[:nb])

    if n_seq is None:
        dt, fl = run(1)
        per_seq = dt
        n_seq = max(1, min(w.B, int(target_s / max(per_seq, 1e-6))))
    dt, fl = run(n_seq)
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": int(os.environ["OMP_NUM_THREADS"]),
            "kind": "oracle", "seconds": round(dt, 3), "n_seq": n_seq,
            "sample": f"the first {n_seq} of {w.B} sequences (all heads and new rows), "
                      f"{fl / 1e9:.2f} useful GFLOP, fp64 C oracle with OpenMP"}


def _decode_config(args, w, lens, world: int = 1):
    return {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "S_q": w.S_q, "S_cap": w.S_cap, "d": w.d,
            "mask": wl.MASK_NAMES[w.kind], "window": w.window, "cache_len": list(lens),
            "cache": "resident in HBM (the step's inputs are the new query rows)",
            "useful_gflop_per_step": wl.decode_useful_flops(w, lens) / 1e9,
            "score_bias": "alibi, slopes 2^(-8(a+1)/H)" if args.alibi else "none",
            "l2": L2Flush.NOTE,
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def run_reference_decode(args, w):
    world, rank, _ = dist_setup()
    if rank != 0:
        return 0
    alibi = score_bias_host(args, w)[0] if args.alibi else None
    cal = cpu_baseline_decode(w, target_s=max(2.0, 150.0 / max(1, args.steps + args.warmup)), alibi=alibi)
    times, r = [], None
    for s in range(args.warmup + args.steps):
        r = cpu_baseline_decode(w, n_seq=cal["n_seq"], alibi=alibi)
        if s >= args.warmup:
            times.append(r["seconds"])
    t = sum(times) / len(times)
    value = r["value"] * r["seconds"] / t
    _, _, _, lens = _decode_oracle_inputs(w)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": _decode_config(args, w, lens, max(1, args.gpus)),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": r["cores"], "kind": "oracle",
                             "sample": r["sample"]},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_ours_decode(args, w):
    import torch
    import torch.distributed as dist

    import transformer_self_attention_gb300 as tsa
    from transformer_self_attention_gb300.shard import max_over_ranks

    world, rank, local = dist_setup()
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    Qc, Kc, Vc, lens = wl.make_decode_inputs(w)
    Q, K, V = Qc.to(dev), Kc.to(dev), Vc.to(dev)
    plan = tsa.DecodeAttention(w.B, w.Hq, w.Hkv, w.S_q, w.S_cap, w.d, scale=w.scale, kind=w.kind, window=w.window)
    if args.alibi:
        plan.set_alibi(wl.alibi_slopes(w.Hq))
    O = torch.empty_like(Q)
    LSE = torch.empty((w.B, w.Hq, w.S_q), dtype=torch.float32, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        plan(Q, K, V, lens, O=O, LSE=LSE, stream=stream)

    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize(dev)
    st, code = plan.poll_device_error()
    if st != 0:
        raise RuntimeError(f"device error during warm-up: {code}")
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(local, dev) if rank == 0 else None
    if clocks:
        clocks.mark_start()
    wall0 = time.perf_counter()
    for s in range(args.steps):
        flush()
        starts[s].record(stream)
        step()
        ends[s].record(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    if clocks:
        clocks.mark_end()
    if world > 1:
        dist.barrier()
    clk = clocks.stop() if clocks else None
    mean_ms = sum(a.elapsed_time(b) for a, b in zip(starts, ends)) / args.steps
    mean_ms = max_over_ranks(mean_ms, dev)  # the slowest rank
    st, code = plan.poll_device_error()
    if st != 0:
        raise RuntimeError(f"device error during the timed steps: {code}")
    launches_per_step = plan.launch_count()
    useful = wl.decode_useful_flops(w, lens)
    nbytes = wl.decode_bytes(w, lens)
    value = world * useful / (mean_ms * 1e-3) / 1e12
    pk, pk_src = peaks()

    # end to end through the C ABI: the new query rows from pinned host memory, the step, O and
    # LSE back to pinned host memory (the cache stays resident, as it does across decode steps)
    e2e = None
    if not args.no_e2e:
        hQ = Qc.pin_memory()
        hO = torch.empty(O.shape, dtype=O.dtype, pin_memory=True)
        hL = torch.empty(LSE.shape, dtype=LSE.dtype, pin_memory=True)
        dQ, dO, dL = torch.empty_like(Q), torch.empty_like(O), torch.empty_like(LSE)
        n_e2e = max(3, min(args.steps, 10))

        def e2e_step():
            dQ.copy_(hQ, non_blocking=True)
            plan(dQ, K, V, lens, O=dO, LSE=dL, stream=stream)
            hO.copy_(dO, non_blocking=True); hL.copy_(dL, non_blocking=True)

        e2e_step()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n_e2e):
            flush()
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = e0.elapsed_time(e1) / n_e2e
        e2e_ms = max_over_ranks(e2e_ms, dev)  # the slowest rank
        e2e = {"value": world * useful / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": e2e_ms,
               "h2d_bytes_per_step": Qc.numel() * Qc.element_size(),
               "d2h_bytes_per_step": O.numel() * O.element_size() + LSE.numel() * LSE.element_size(),
               "note": "includes the L2 flush of each step (256 MiB written, then read back)"}

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0
    achieved = nbytes / (mean_ms * 1e-3) / 1e9
    peak = float(pk["hbm_gbs"])
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": ncu_traffic(w.name, "attn_decode", DECODE_KERNEL_SOURCES),
                "algorithmic_bytes": nbytes, "peak_source": f"{pk_src} hbm_gbs (copy bandwidth)",
                "kernel": "attn_decode_kernel"}
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": mean_ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": _decode_config(args, w, lens, world),
            "roofline": roofline, "gpu_launches": args.steps * launches_per_step, "wall_s_timed_region": wall}
    if e2e:
        line["e2e"] = e2e
    if clk:
        line["clocks"] = clk
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline_decode(w, alibi=wl.alibi_slopes(w.Hq) if args.alibi else None)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=wl.CAUSAL_MHA_4K.name,
                    choices=sorted(wl.BY_NAME) + sorted(wl.DECODE_BY_NAME))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--fp8", action="store_true",
                    help="E4M3 Q, K, V with per-tensor scales (prefill workloads; same metric)")
    ap.add_argument("--alibi", action="store_true",
                    help="add the ALiBi score bias with slopes 2^(-8(a+1)/H) (same workload, same metric)")
    ap.add_argument("--bias", action="store_true",
                    help="add a per-head bias matrix [1, Hq, S, S] (bf16) to the scores (prefill, bf16)")
    ap.add_argument("--backward", action="store_true",
                    help="time the backward pass (dQ, dK, dV) of a prefill workload instead of the forward")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.bias and (args.fp8 or args.alibi or args.workload not in wl.BY_NAME):
        ap.error("--bias takes a bf16 prefill workload without --fp8 / --alibi")
    if args.backward:
        if args.workload not in wl.BY_NAME or args.fp8:
            ap.error("--backward takes a bf16 prefill workload without --fp8")
        w = wl.BY_NAME[args.workload]
        return run_reference_backward(args, w) if args.impl == "reference" else run_ours_backward(args, w)
    if args.workload in wl.DECODE_BY_NAME:
        w = wl.DECODE_BY_NAME[args.workload]
        return run_reference_decode(args, w) if args.impl == "reference" else run_ours_decode(args, w)
    w = wl.BY_NAME[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())

"""Benchmark of the GB300 dense GEMM library.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config 1..5] [--impl ours|reference]

One step is one call of the library on one batch of synthetic input (the
seeded workloads of workloads.py). The default workload is number 2, the BF16
GEMM M = N = K = 4096, on which the headline metric (TFLOPS and fraction of the
dense tensor-core peak) is quoted; --config picks another. Input sets are
rotated so that the operands of every timed call were evicted from L2 (their
total is several times the 129 MB L2). After the headline, the other four
workloads are timed the same way in the same process and reported under
"workloads" in the same JSON line (--no-extra skips them).

SM clocks, power and clock-event reasons are read in-process through NVML
while the timed region runs on the GPU (polled until its end event
completes), so even a region of a millisecond or two carries its own clock
record.

Rank 0 prints ONE JSON line. Under torchrun (N > 1) every rank runs the same
workload on its own GPU (independent replicas: GEMM problems shard without any
collective), the timed region is bracketed by barriers, and the time is the
maximum over ranks.

--impl reference times the oracle (oracle/, the float64 CPU restatement) on
the host cores on a bounded sample of the same workload, as the reference arm.
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOPS and % of GB300 dense BF16/FP8 peak (HBM % for skinny M)"
L2_BYTES = 129 * 2 ** 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
DESCRIPTIONS = {
    1: "BF16 GEMM M=N=K=512, B KxN, alpha 1.5, beta 0.5, FP32 C0 -> FP32 D",
    2: "BF16 GEMM M=N=K=4096, B KxN, N(0,1)/sqrt(K) entries -> BF16 D",
    3: "FP8 E4M3 GEMM M=4096 N=11008 K=4096, per-token x per-channel scales -> BF16 D",
    4: "decode BF16 GEMM M=16 N=18432 K=7168, weights NxK -> BF16 D",
    5: "FP8 E4M3 GEMM M=N=K=8192 + bias -> SiLU -> per-row E4M3 requant",
}
DEFAULT_STEPS = {1: 20000, 2: 10000, 3: 4000, 4: 20000, 5: 2000}


# ------------------------------------------------------------------ helpers

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value: float, device=None) -> float:
    """The largest of every rank's value (the job's time is its slowest rank's);
    the value itself when no process group is initialised."""
    import torch
    import torch.distributed as tdist
    if not (tdist.is_available() and tdist.is_initialized()) or tdist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank: float, world: int, seconds: float) -> float:
    """Whole-job throughput: the units every rank processed over the slowest
    rank's time (weak scaling: each rank runs the full workload)."""
    return world * units_per_rank / seconds


def parse_clock_rows(text: str) -> dict:
    """Median SM clock, max clock and power, and the throttle reasons seen in
    nvidia-smi rows of ClockSampler.FIELDS (csv, noheader, nounits)."""
    sm, smax, power, reasons = [], [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for line in text.strip().splitlines():
        r = [x.strip() for x in line.split(",")]
        if len(r) < 9:
            continue
        try:
            sm.append(float(r[1]))
            smax.append(float(r[2]))
            power.append(float(r[3]))
        except ValueError:
            continue
        for name, val in zip(names, r[5:9]):
            if val.lower() == "active":
                reasons.add(name)
    return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
            "power_w_max": max(power) if power else None, "reasons": sorted(reasons), "samples": len(sm)}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash() -> str:
    """sha256 prefix of the device code (kernel template, PTX wrappers, variant
    tables); host-side planning changes do not invalidate recorded counters."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "dense_gemm_persistent_gb300", "csrc")
    for p in sorted(glob.glob(os.path.join(csrc, "*"))):
        if os.path.basename(p) == "api.cu":
            continue
        with open(p, "rb") as f:
            h.update(os.path.basename(p).encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def plan_tile(plan):
    """The plan's tile as recorded beside a traffic figure: rows x columns x CTAs."""
    return f"{plan['tile_m']}x{plan['tile_n']}x{plan['cta_group']}"


def recorded_traffic(workload, plan=None, path=None):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the
    current kernel sources and, where the record names one, on the tile the
    current plan chooses (else None)."""
    path = path or os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    want = kernel_source_hash()
    for line in open(path):
        if line.startswith("#") or not line.strip():
            continue
        kv = dict(tok.split("=", 1) for tok in line.split() if "=" in tok)
        if plan is not None and "tile" in kv and kv["tile"] != plan_tile(plan):
            continue
        if kv.get("workload") == str(workload) and kv.get("kernel_src_sha") == want:
            return int(float(kv["dram_bytes_per_launch"]))
    return None


class NvmlClocks:
    """SM clock, power and clock-event reasons read in-process through NVML
    (the driver's libnvidia-ml.so.1, through ctypes; only reads). sample()
    returns (sm_mhz, power_w, reason_bits) or None."""
    # clock-event reason bits (nvml.h) that decide whether a timed region stands
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
    NVML_CLOCK_SM = 1

    def __init__(self, torch_index: int):
        import ctypes
        self.ok = False
        self.max_mhz = None
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
        except OSError:
            return
        self.c = ctypes
        self.lib = lib
        if lib.nvmlInit_v2() != 0:
            return
        self.h = ctypes.c_void_p()
        found = False
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(torch_index).uuid)
            if not uuid.startswith("GPU-"):
                uuid = "GPU-" + uuid
            found = lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.h)) == 0
        except Exception:
            found = False
        if not found:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            idx = torch_index
            parts = [x for x in vis.split(",") if x.strip()]
            if parts and parts[0].strip().isdigit() and torch_index < len(parts):
                idx = int(parts[torch_index])
            found = lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(idx), ctypes.byref(self.h)) == 0
        if not found:
            return
        self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons", None)
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(self.h, self.NVML_CLOCK_SM, ctypes.byref(mx)) == 0:
            self.max_mhz = float(mx.value)
        self.ok = True

    def sample(self):
        if not self.ok:
            return None
        c = self.c
        mhz, mw, bits = c.c_uint(), c.c_uint(), c.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.h, self.NVML_CLOCK_SM, c.byref(mhz)) != 0:
            return None
        power = float(mw.value) / 1000.0 if self.lib.nvmlDeviceGetPowerUsage(self.h, c.byref(mw)) == 0 else None
        reasons = int(bits.value) if (self.reasons_fn and self.reasons_fn(self.h, c.byref(bits)) == 0) else 0
        return float(mhz.value), power, reasons


def summarize_clock_samples(samples, max_mhz, before=None, after=None) -> dict:
    """Median SM clock, power and the clock-event reasons seen over the samples
    taken while the timed region ran (each (sm_mhz, power_w, reason_bits))."""
    sm = [x[0] for x in samples]
    power = [x[1] for x in samples if x[1] is not None]
    bits = 0
    for x in samples:
        bits |= x[2]
    reasons = sorted(name for b, name in NvmlClocks.REASONS.items() if bits & b)
    return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max_mhz,
            "sm_mhz_min": min(sm) if sm else None, "sm_mhz_max": max(sm) if sm else None,
            "power_w_max": max(power) if power else None, "reasons": reasons, "samples": len(sm),
            "sm_mhz_before": None if before is None else before[0],
            "sm_mhz_after": None if after is None else after[0],
            "source": "NVML in-process, polled while the timed region ran on the GPU"}


class RegionClocks:
    """Clock record of one timed region: one NVML sample right before it, then
    samples polled until its end event has completed, then one right after;
    nvidia-smi sampling (100 ms) where NVML cannot be loaded."""

    def __init__(self, torch_index: int):
        self.nvml = NvmlClocks(torch_index)
        self.smi = None if self.nvml.ok else ClockSampler(torch_index)

    def start(self):
        self.samples = []
        self.before = self.nvml.sample() if self.nvml.ok else None
        if self.smi:
            self.smi.start()

    def poll_until(self, event):
        """Samples while `event` (recorded after the timed launches) is pending."""
        import time as _t
        while not event.query():
            if self.nvml.ok:
                x = self.nvml.sample()
                if x is not None:
                    self.samples.append(x)
            else:
                _t.sleep(0.001)

    def stop(self) -> dict:
        if self.smi:
            return self.smi.stop()
        after = self.nvml.sample()
        return summarize_clock_samples(self.samples, self.nvml.max_mhz, self.before, after)


class ClockSampler:
    """nvidia-smi sampling of SM clock, power and throttle reasons (used when
    NVML cannot be loaded in-process)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = 100):
        self.gpu = gpu_index
        self.interval = interval_ms
        self.proc = None
        self.out = None

    def start(self):
        try:
            self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", str(self.interval)],
                                         stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.flush()
        self.out.seek(0)
        text = self.out.read()
        self.out.close()
        os.unlink(self.out.name)
        return parse_clock_rows(text)


def parse_shape(text: str):
    m, n, k = (int(x) for x in text.replace("x", ",").split(","))
    if min(m, n, k) <= 0:
        raise SystemExit("--shape wants positive M,N,K")
    return m, n, k


def make_workload(args):
    """The workload a run times: one of the five; with --k-group, workload 3's
    shape and recipe with per-K-group scales; with --shape M,N,K, workload 2's
    BF16 recipe at that size with B stored N x K (the weight layout)."""
    import workloads as wl
    if getattr(args, "shape", None):
        if args.config != 2 or getattr(args, "k_group", 0):
            raise SystemExit("--shape applies to workload 2's BF16 recipe")
        M, N, K = parse_shape(args.shape)
        w = wl.make(2, M=M, N=N, K=K)
        w.B = w.B.t().contiguous()
        w.b_layout = "nk"
        return w
    if getattr(args, "k_group", 0):
        if args.config != 3:
            raise SystemExit("--k-group applies to workload 3 (FP8 E4M3 4096 x 11008 x 4096)")
        return wl.fp8_grouped(k_group=args.k_group, b_block=getattr(args, "b_block", 1))
    if getattr(args, "b_block", 1) != 1:
        raise SystemExit("--b-block applies with --k-group")
    return wl.make(args.config)


def workload_key(args) -> str:
    if getattr(args, "shape", None):
        return "2s" + "x".join(str(v) for v in parse_shape(args.shape))
    if getattr(args, "k_group", 0):
        blk = getattr(args, "b_block", 1)
        return f"{args.config}g{args.k_group}" + (f"b{blk}" if blk != 1 else "")
    return str(args.config)


def describe(args) -> str:
    d = DESCRIPTIONS[args.config]
    if getattr(args, "shape", None):
        M, N, K = parse_shape(args.shape)
        return f"BF16 GEMM M={M} N={N} K={K}, entries N(0,1)/sqrt(K), B stored N x K -> BF16 D"
    if getattr(args, "k_group", 0):
        blk = getattr(args, "b_block", 1)
        wgt = f"per-({blk}-channel block, K group)" if blk != 1 else "per-(channel, K group)"
        d = d.replace("per-token x per-channel scales",
                      f"per-(token, {args.k_group}-element K group) x {wgt} scales")
    return d


def oracle_sample(w, seconds: float):
    """Time the oracle on whole rows of the workload until `seconds` have passed
    (at least one row); returns (flops, elapsed, rows, threads)."""
    import oracle
    import workloads as wl
    threads = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    C = None if w.C is None else w.C.numpy()
    if w.form == "bf16":
        A, B = wl.bits_u16(w.A), wl.bits_u16(w.B)
    else:
        A, B = wl.codes_u8(w.A), wl.codes_u8(w.B)
    done, chunk, t0 = 0, 1, time.perf_counter()
    while done < w.M:
        rows = (done, min(w.M, done + chunk))
        if w.form == "bf16":
            oracle.bf16_gemm_ref(A, B, w.b_layout, C, w.alpha, w.beta, rows=rows, nthreads=threads)
        else:
            y = oracle.fp8_gemm_ref(A, B, w.b_layout, w.a_scale.numpy(), w.b_scale.numpy(), C, w.alpha, w.beta,
                                    None if w.bias is None else w.bias.numpy(), w.act, rows=rows,
                                    nthreads=threads, k_group=w.k_group, b_block=w.b_block)
            if w.out_quant != "none":
                oracle.requant_rows(y)
        done = rows[1]
        el = time.perf_counter() - t0
        if el >= seconds:
            break
        chunk = min(2 * chunk, max(1, threads * 4))
    el = time.perf_counter() - t0
    return 2.0 * done * w.N * w.K, el, done, threads


# ------------------------------------------------------------------ our arm

class Rig:
    """Device-resident input sets of one workload, rotated so that every timed
    call finds its operands out of L2, and the library call on set i."""

    def __init__(self, w, dev, stream):
        import torch
        import dense_gemm_persistent_gb300 as dg
        self.w, self.dev, self.stream, self.dg = w, dev, stream, dg
        self.tdt = {"f32": torch.float32, "bf16": torch.bfloat16, "e4m3": torch.uint8}[w.d_dtype]
        self.ws_bytes = dg.dgemm_workspace_size(w.form == "fp8", w.M, w.N, w.K, w.b_layout, out_quant=w.out_quant)
        in_bytes = sum(t.numel() * t.element_size() for t in w.tensors().values())
        out_bytes = w.M * w.N * torch.tensor([], dtype=self.tdt).element_size()
        self.set_bytes = in_bytes + out_bytes + self.ws_bytes
        self.nsets = max(2, min(160, math.ceil(3 * L2_BYTES / max(self.set_bytes, 1))))
        self.sets = []
        for _ in range(self.nsets):
            g = w.to(dev)
            D = torch.empty(w.M, w.N, dtype=self.tdt, device=dev)
            s = torch.empty(w.M, dtype=torch.float32, device=dev) if w.out_quant != "none" else None
            ws = torch.empty(max(self.ws_bytes, 16), dtype=torch.uint8, device=dev) if self.ws_bytes else None
            self.sets.append((g, D, s, ws))

    def l2_note(self) -> str:
        return f"rotating {self.nsets} input sets of {self.set_bytes / 2**20:.0f} MiB (> L2 129 MiB)"

    def call(self, i, bufs=None):
        w, dg = self.w, self.dg
        g, D, s, ws = (bufs or self.sets)[i % (len(bufs) if bufs else self.nsets)]
        kw = dict(b_layout=w.b_layout, C=g.C, alpha=w.alpha, beta=w.beta, bias=g.bias, act=w.act,
                  out_quant=w.out_quant, out_row_scale=s, ws=ws, stream=self.stream)
        if w.form == "bf16":
            dg.dgemm_bf16(g.A, g.B, D, **kw)
        else:
            dg.dgemm_fp8_scaled(g.A, g.B, g.a_scale, g.b_scale, D, k_group=w.k_group, b_block=w.b_block, **kw)

    def status_ok(self) -> bool:
        """No bounded device wait gave up in any call so far (every set's
        workspace status word and the per-device word; each query clears)."""
        dg = self.dg
        ok = dg.dgemm_query_device_status(None, stream=self.stream) == 0
        for _, _, _, ws in self.sets:
            if ws is not None and dg.dgemm_query_device_status(ws, stream=self.stream) != 0:
                ok = False
        return ok

    def free(self):
        import torch
        self.sets = []
        torch.cuda.empty_cache()


def timed_region(rig, steps, warmup, dev, barrier, clocks):
    """W untimed calls, then exactly `steps` calls between CUDA events on the
    launching stream, bracketed by a barrier and a device synchronisation on
    both sides; the SM clocks are sampled while the region runs. Returns the
    milliseconds of the region (max over ranks) and its clock record."""
    import torch
    for i in range(warmup):
        rig.call(i)
    torch.cuda.synchronize(dev)
    if not rig.status_ok():
        raise RuntimeError("device status after warm-up")
    barrier()
    torch.cuda.synchronize(dev)
    clocks.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # A bounded GPU sleep ahead of the start event keeps the stream busy while
    # the host enqueues the first calls, so the region starts with calls
    # already queued instead of with the host's launch latency (the calls and
    # their work are unchanged; the sleep is outside the region).
    gate_s = min(2e-3, 1e-4 + 1.5e-5 * steps)
    torch.cuda._sleep(int(gate_s * 2.1e9))
    e0.record(rig.stream)
    for i in range(steps):
        rig.call(i)
    e1.record(rig.stream)
    clocks.poll_until(e1)
    torch.cuda.synchronize(dev)
    record = clocks.stop()
    barrier()
    ms_total = max_over_ranks(e0.elapsed_time(e1), dev)
    if not rig.status_ok():
        raise RuntimeError("device status after the timed region")
    return ms_total, record


def roofline_of(w, ms_step, clocks, peaks, peak_kind, n_sm, skinny, plan, traffic):
    """Achieved rate of the kernel (one launch per step) against its roofline:
    TFLOP/s against the tensor-core peak, or for skinny (HBM-bound) shapes the
    compulsory bytes against the measured copy bandwidth; beside it the tensor
    core's rate at the SM clock sampled during the region."""
    from dense_gemm_persistent_gb300 import roofline
    dsz = {"f32": 4, "bf16": 2, "e4m3": 1}[w.d_dtype]
    esz = 2 if w.form == "bf16" else 1
    c_in = 4 if (w.C is not None and w.beta != 0) else 0
    comp = roofline.compulsory_bytes(w.M, w.N, w.K, esz, esz, c_in, dsz)
    flops = w.flops
    if skinny:
        achieved = comp / (ms_step * 1e-3) / 1e9
        peak, unit, bound = peaks["hbm_gbs"], "GB/s", "hbm"
    else:
        achieved = flops / (ms_step * 1e-3) / 1e12
        base = peaks["bf16_tflops"]
        peak = base if w.form == "bf16" else 2.0 * base   # FP8:BF16 dense ratio 2
        unit, bound = "TFLOP/s", "tensor"
    # SMs x dense FLOP per clock per SM (128 x 256 x 16 BF16 or x 32 E4M3 MACs
    # per 128 cycles, measured at that rate) x the median sampled clock
    flop_per_clk = 8192 if w.form == "bf16" else 16384
    theo = (n_sm * flop_per_clk * clocks["sm_mhz"] * 1e6 / 1e12) if clocks.get("sm_mhz") else None
    tflops = flops / (ms_step * 1e-3) / 1e12
    return {"bound": bound, "achieved": round(achieved, 1), "peak": round(peak, 1), "unit": unit,
            "frac": round(achieved / peak, 4), "traffic": traffic,
            "peak_source": f"{peak_kind}" + ("" if w.form == "bf16" or skinny else " bf16 x 2 (FP8:BF16 ratio)"),
            "compulsory_bytes": int(comp),
            "tensor_peak_at_clock_tflops": None if theo is None else round(theo, 1),
            "frac_of_peak_at_clock": None if (theo is None or skinny) else round(tflops / theo, 4),
            "tiled_traffic_bytes_no_l2": int(roofline.tiled_read_elements(w.M, w.N, w.K, plan["tile_m"],
                                                                          plan["tile_n"]) * esz
                                             + w.M * w.N * (dsz + c_in))}


def plan_of(dg, w):
    return dg.dgemm_plan(w.form == "fp8", w.M, w.N, w.K, w.b_layout, w.d_dtype, out_quant=w.out_quant,
                         act=w.act, k_group=w.k_group, num_sms=0)


def is_skinny(w, number, shape, peaks):
    """HBM-bound: workload 4, or a --shape whose intensity is below the ridge point."""
    from dense_gemm_persistent_gb300 import roofline
    if number == 4:
        return True
    if not shape:
        return False
    esz = 2 if w.form == "bf16" else 1
    comp = roofline.compulsory_bytes(w.M, w.N, w.K, esz, esz, 0, 2)
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    return w.flops / comp < ridge


def config_of(args, w) -> dict:
    """The workload's identity: the same dict in both arms."""
    return {"workload": describe(args), "number": args.config, "M": w.M, "N": w.N, "K": w.K,
            "b_layout": w.b_layout, "k_group": w.k_group, "b_block": w.b_block}


def run_ours(args, rank, world, local):
    import torch

    import dense_gemm_persistent_gb300 as dg

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dg.load()
    w = make_workload(args)
    peaks, peak_kind = measured_peaks()
    stream = torch.cuda.current_stream(dev)
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    clocks = RegionClocks(local)

    dist = world > 1
    if dist:
        import torch.distributed as tdist

    def barrier():
        if dist:
            tdist.barrier()

    rig = Rig(w, dev, stream)
    ms_total, clock_rec = timed_region(rig, args.steps, args.warmup, dev, barrier, clocks)
    ms_step = ms_total / args.steps
    flops = w.flops
    tflops = job_rate(flops * args.steps, world, ms_total * 1e-3) / 1e12

    # ---- end to end: pinned host inputs -> device, call, result -> host.
    # Every step uploads its inputs from pinned host memory and reads its
    # result back; steps are double-buffered over two device input sets and
    # three streams (upload, GEMM, readback), so step i+1's upload overlaps
    # step i's GEMM and readback. Events order each buffer's reuse: an upload
    # into set b waits for the GEMM that last read it, a GEMM into set b waits
    # for the readback of that set's previous result.
    host = {k: t.pin_memory() for k, t in w.tensors().items()}
    nbuf = 2
    bufs = [rig.sets[b % rig.nsets] for b in range(nbuf)]
    Dh = [torch.empty(bufs[0][1].shape, dtype=bufs[0][1].dtype, pin_memory=True) for _ in range(nbuf)]
    sh = [torch.empty(w.M, dtype=torch.float32, pin_memory=True) if bufs[0][2] is not None else None
          for _ in range(nbuf)]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = Dh[0].numel() * Dh[0].element_size() + (sh[0].numel() * 4 if sh[0] is not None else 0)
    e2e_steps = max(4, min(args.steps, 50))
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()
    uploaded = [ev() for _ in range(nbuf)]
    computed = [None] * nbuf
    read_back = [None] * nbuf

    def e2e_step(i):
        b = i % nbuf
        g, D, sc, _ = bufs[b]
        with torch.cuda.stream(up):
            if computed[b] is not None:
                up.wait_event(computed[b])
            for k, t in host.items():
                getattr(g, k).copy_(t, non_blocking=True)
            uploaded[b].record(up)
        stream.wait_event(uploaded[b])
        if read_back[b] is not None:
            stream.wait_event(read_back[b])
        rig.call(b, bufs)
        computed[b] = ev()
        computed[b].record(stream)
        with torch.cuda.stream(down):
            down.wait_event(computed[b])
            Dh[b].copy_(D, non_blocking=True)
            if sh[b] is not None:
                sh[b].copy_(sc, non_blocking=True)
            read_back[b] = ev()
            read_back[b].record(down)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    barrier()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    up.wait_event(f0)
    for i in range(e2e_steps):
        e2e_step(i)
    for b in range(nbuf):
        stream.wait_event(read_back[b])
    f1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(f0.elapsed_time(f1) / e2e_steps, dev)
    if not rig.status_ok():
        raise RuntimeError("device status after the end-to-end steps")

    plan = plan_of(dg, w)
    skinny = is_skinny(w, args.config, args.shape, peaks)
    roof = roofline_of(w, ms_step, clock_rec, peaks, peak_kind, n_sm, skinny, plan,
                       recorded_traffic(workload_key(args), plan))
    l2_note = rig.l2_note()
    rig.free()
    del host, bufs, Dh, sh

    result = {
        "metric": METRIC, "value": round(tflops, 2), "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if w.form == "bf16" else "e4m3", "data": "synthetic",
        "config": config_of(args, w),
        "setup": {"parallelism": f"replicas x{world}", "l2": l2_note,
                  "plan": {k: plan[k] for k in ("swap_ab", "tile_m", "tile_n", "cta_group", "stages", "num_tiles",
                                                "grid", "cooperative", "tail_tiles", "tail_split", "tail_halves",
                                                "cluster_split")}},
        "clocks": clock_rec,
        "e2e": {"value": round(job_rate(flops, world, e2e_ms * 1e-3) / 1e12, 3), "unit": "TFLOPS",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
                "pipelining": "double-buffered: step i+1's upload overlaps step i's GEMM and readback"},
        "gpu_launches": args.steps,
        "roofline": roof,
    }
    if skinny:
        result["hbm_gbs"] = round(roof["achieved"], 1)

    # ---- the other workloads, timed the same way in the same process
    if not args.no_extra and not args.shape and not args.k_group:
        extra = {}
        launches = args.steps
        for number in sorted(DESCRIPTIONS):
            if number == args.config:
                continue
            steps = args.steps if args.steps_given else DEFAULT_STEPS[number]
            extra[str(number)] = time_other(number, steps, args.warmup, dev, stream, barrier, clocks, peaks,
                                            peak_kind, n_sm, world)
            launches += steps
        result["workloads"] = extra
        result["gpu_launches_all"] = launches
    return result, w


def time_other(number, steps, warmup, dev, stream, barrier, clocks, peaks, peak_kind, n_sm, world):
    """One more workload at its full size, timed like the headline (rotating
    input sets, CUDA events on the launching stream, clocks sampled during the
    region): microseconds per call, rate and roofline."""
    import dense_gemm_persistent_gb300 as dg

    class A:
        pass
    a = A()
    a.config, a.shape, a.k_group, a.b_block = number, None, 0, 1
    w = make_workload(a)
    rig = Rig(w, dev, stream)
    ms_total, rec = timed_region(rig, steps, warmup, dev, barrier, clocks)
    ms_step = ms_total / steps
    plan = plan_of(dg, w)
    skinny = number == 4
    roof = roofline_of(w, ms_step, rec, peaks, peak_kind, n_sm, skinny, plan, recorded_traffic(str(number), plan))
    out = {"workload": DESCRIPTIONS[number], "M": w.M, "N": w.N, "K": w.K, "steps": steps, "warmup": warmup,
           "us_per_call": round(ms_step * 1e3, 3),
           "value": round(job_rate(w.flops * steps, world, ms_total * 1e-3) / 1e12, 2), "unit": "TFLOPS",
           "dtype": "bf16" if w.form == "bf16" else "e4m3", "l2": rig.l2_note(),
           "plan": {k: plan[k] for k in ("swap_ab", "tile_m", "tile_n", "cta_group", "num_tiles", "grid",
                                         "cooperative", "tail_tiles", "tail_split", "tail_halves")},
           "roofline": roof, "clocks": rec}
    if skinny:
        out["hbm_gbs"] = roof["achieved"]
    rig.free()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", type=int, default=2, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="CPU time spent on the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--shape", default=None,
                    help="M,N,K: workload 2's BF16 recipe at this size, B stored N x K (e.g. 1024,1024,4096)")
    ap.add_argument("--k-group", type=int, default=0,
                    help="workload 3 with per-K-group FP8 scales of this group size (multiple of 128)")
    ap.add_argument("--b-block", type=int, default=1, choices=[1, 128],
                    help="with --k-group: output channels per weight scale (128: block-scaled weights)")
    ap.add_argument("--ref-seconds", type=float, default=120.0,
                    help="wall time the reference arm spends on warm-up + steps")
    ap.add_argument("--no-extra", action="store_true",
                    help="time only the selected workload (not the other four after it)")
    args = ap.parse_args()
    args.steps_given = args.steps is not None
    if args.steps is None:
        args.steps = 2000 if args.shape else DEFAULT_STEPS[args.config]
    args.warmup = max(args.warmup, 3)
    rank, world, local = dist_env()

    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args, world)), flush=True)
        return 0

    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(local)
        tdist.init_process_group("nccl", device_id=torch.device("cuda", local))
    result, w = run_ours(args, rank, world, local)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        fl, el, rows, threads = oracle_sample(w, args.cpu_seconds)
        result["cpu_baseline"] = {"value": round(fl / el / 1e12, 6), "unit": "TFLOPS", "cores": threads,
                                  "kind": "oracle", "seconds": round(el, 2),
                                  "sample": f"{rows} of {w.M} rows of the same workload "
                                            f"(2*rows*N*K = {fl:.3g} FLOP), float64 oracle, OpenMP"}
    if world > 1:
        import torch.distributed as tdist
        tdist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result), flush=True)
    return 0


def run_reference(args, world):
    """The reference arm: the oracle timed on the host cores, each step a bounded
    sample (whole rows) of the same workload, sized so warm-up + steps take about
    two minutes."""
    import workloads as wl
    w = make_workload(args)
    budget = args.ref_seconds / (args.steps + args.warmup)
    # calibrate rows per step on one row
    fl, el, rows, threads = oracle_sample(w, 0.0)
    per_row = el / max(rows, 1)
    rows_per_step = max(1, min(w.M, int(budget / max(per_row, 1e-9))))
    import oracle
    C = None if w.C is None else w.C.numpy()
    A = wl.bits_u16(w.A) if w.form == "bf16" else wl.codes_u8(w.A)
    B = wl.bits_u16(w.B) if w.form == "bf16" else wl.codes_u8(w.B)

    def step(i):
        r0 = (i * rows_per_step) % w.M
        rows = (r0, min(w.M, r0 + rows_per_step))
        if w.form == "bf16":
            oracle.bf16_gemm_ref(A, B, w.b_layout, C, w.alpha, w.beta, rows=rows, nthreads=threads)
        else:
            y = oracle.fp8_gemm_ref(A, B, w.b_layout, w.a_scale.numpy(), w.b_scale.numpy(), C, w.alpha, w.beta,
                                    None if w.bias is None else w.bias.numpy(), w.act, rows=rows,
                                    nthreads=threads, k_group=w.k_group, b_block=w.b_block)
            if w.out_quant != "none":
                oracle.requant_rows(y)
        return rows[1] - rows[0]

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    done = 0
    for i in range(args.steps):
        done += step(i)
    el = time.perf_counter() - t0
    value = 2.0 * done * w.N * w.K / el / 1e12
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOPS", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": config_of(args, w),
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOPS", "cores": threads, "kind": "oracle",
                         "sample": f"{rows_per_step} rows of {w.M} per step of the same workload, float64 "
                                   f"oracle, OpenMP"},
        "e2e": {"value": round(value, 6), "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


if __name__ == "__main__":
    sys.exit(main())

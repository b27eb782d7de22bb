"""Benchmark of the MoE layer forward pass (moe_forward through the C ABI).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference]

One step is one full forward pass (gate, dispatch, expert FFNs, combine) over
one batch of the workload (default: flat_n256_k4, T=16384 tokens, d=512,
h=1024, n=256 experts, k=4, bf16 FFN, fp32 gating, noisy).  Inputs are
synthetic and seeded; x/eps rotate over several device copies so that the
timed loop never re-reads them from L2 (the 537 MB of expert weights are
larger than the 126 MB L2 by themselves).  Rank 0 prints one JSON line.

Under torchrun every rank runs its own batch (weak scaling, no collective on
the data path); value = all ranks' tokens / the slowest rank's time.
`--impl reference` times the CPU oracle on the host cores instead (a bounded
sample of tokens per step), printing the same kind of line.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sparsely_gated_mixture_top_b300 import workloads as wl  # noqa: E402

METRIC = "MoE-layer tokens/sec (fused forward, 1xB300 per rank)"
UNIT = "tokens/s"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="flat_n256_k4", choices=sorted(wl.WORKLOADS))
    p.add_argument("--e2e-steps", type=int, default=50)
    p.add_argument("--cpu-seconds", type=float, default=15.0,
                   help="target CPU seconds of the oracle baseline sample")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-per-workload", action="store_true",
                   help="skip the other full-size workloads (per_workload field)")
    p.add_argument("--per-workload-steps", type=int, default=20)
    p.add_argument("--pass", dest="which", choices=["forward", "backward", "balanced", "ep"],
                   default="forward",
                   help="forward: moe_forward (the headline); backward: moe_backward with the "
                        "forward's selection; balanced: moe_forward_balanced with the batchwise "
                        "mask; ep: the expert-parallel layer (experts split over the ranks, "
                        "all-to-all over NCCL; one rank when run without torchrun)")
    p.add_argument("--traffic-summary", nargs=2, metavar=("NCU_CSV", "BENCH_JSON"),
                   help="print the DRAM-traffic record of one expert-FFN stage from an ncu "
                        "--csv log of the stage's launches (traffic_ncu) and the bench line "
                        "of the same command, then exit")
    return p.parse_args()


TRAFFIC_BENCH = "python bench.py --steps 3 --warmup 3 --e2e-steps 3 --no-cpu-baseline --no-per-workload"


def traffic_ncu(w: wl.Workload) -> str:
    """The ncu command (before TRAFFIC_BENCH) that counts the DRAM bytes of
    the launches of one moe_expert_ffn call (tile table, gather, then the
    fused kernel or the two grouped GEMMs).  TRAFFIC_BENCH runs six forward
    steps first, each launching the FFN kernels alone (their tables come from
    the dispatch); those launches are skipped."""
    per_step = 1 if fused_ffn(w) else 2
    return ("ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,gpu__time_duration.sum "
            f"--clock-control none -k regex:ffn_ -s {6 * per_step} -c {2 + per_step} --csv "
            "--log-file traffic.csv ")


def traffic_summary(csv_path: str, bench_json: str, w: wl.Workload) -> dict:
    """DRAM bytes of the launches of one expert-FFN stage (tile table, gather,
    the fused kernel or two grouped GEMMs) of the stage timing call, as ncu
    counted them."""
    import csv
    with open(csv_path) as f:
        lines = [ln for ln in f if ln.startswith('"')]
    rows = list(csv.DictReader(lines))
    launches = {}
    for r in rows:
        k = launches.setdefault(int(r["ID"]), {"kernel": r["Kernel Name"].split("(")[0]})
        v = float(r["Metric Value"].replace(",", ""))
        unit = r["Metric Unit"]
        scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "ns": 1, "us": 1e3, "usecond": 1e3,
                 "nsecond": 1, "ms": 1e6, "msecond": 1e6}[unit]
        key = {"dram__bytes_read.sum": "dram_read_bytes", "dram__bytes_write.sum": "dram_write_bytes",
               "gpu__time_duration.sum": "duration_ns_cold"}[r["Metric Name"]]
        k[key] = int(round(v * scale))
    kernels = [dict(launch=i, **launches[i]) for i in sorted(launches)]
    with open(bench_json) as f:
        line = json.loads(f.read().strip().splitlines()[-1])
    total = sum(k["dram_read_bytes"] + k["dram_write_bytes"] for k in kernels)
    return {
        "workload": w.name,
        "what": "DRAM bytes (read + write) of the launches of one expert-FFN stage "
                "(moe_expert_ffn: token-tile table, gather, "
                + ("both layers in one kernel" if fused_ffn(w) else "two pair GEMMs")
                + "), stage timing call",
        "command": f"{TRAFFIC_BENCH} (exit 0), then: {traffic_ncu(w)}{TRAFFIC_BENCH}",
        "source_sha256": source_digest(),
        "ffn_stage_dram_bytes_per_launch": total,
        "algorithmic_bytes_per_launch": line["roofline"]["algorithmic_per_launch"],
        "kernels": kernels,
    }


# ---------------------------------------------------------------------------
# Peaks and algorithmic work
# ---------------------------------------------------------------------------
def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            m = json.load(f)
        return dict(hbm=float(m["hbm_gbs"]), bf16=float(m["bf16_tflops"]),
                    bf16_sustained=float(m["bf16_tflops_sustained"]), source="measured")
    except (OSError, KeyError, ValueError):
        return dict(hbm=6400.0, bf16=1800.0, bf16_sustained=1400.0, source="fallback")


FFN_STAGE_SOURCES = ("ffn.cu", "ffn_tc.cu", "ffn_pair.cu", "ffn_fused.cu", "moe_device.cuh",
                     "moe_launch.h")


def source_digest() -> str:
    """sha256 of the sources the expert-FFN stage's kernels are built from
    (the kernels, their device helpers and the workspace layout)."""
    import hashlib
    h = hashlib.sha256()
    files = [os.path.join(ROOT, "sparsely_gated_mixture_top_b300", "csrc", f) for f in FFN_STAGE_SOURCES]
    for f in files:
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def stage_traffic(w: wl.Workload):
    """DRAM bytes (read + write) of one expert-FFN stage from the committed ncu
    summary of this workload, or None if there is none or the kernels changed
    since it was captured (its source digest no longer matches)."""
    path = os.path.join(ROOT, "profiles", f"traffic_{w.name}.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("source_sha256") != source_digest() or rec.get("workload") != w.name:
        return None
    return rec.get("ffn_stage_dram_bytes_per_launch")


def job_throughput(ms_local: float, tokens_per_rank: int, dist=None, device="cpu"):
    """Whole-job throughput of a weak-scaling run: every rank processes
    tokens_per_rank tokens; the job time is the slowest rank's time (MAX over
    ranks).  Returns (job ms, tokens per second over all ranks)."""
    ms = ms_local
    world = 1
    if dist is not None:
        t = torch.tensor([ms_local], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
        world = dist.get_world_size()
    return ms, tokens_per_rank * world / (ms / 1e3)


def algorithmic(w: wl.Workload, counts: np.ndarray) -> dict:
    """Algorithmic bytes and FLOPs of one forward pass, from the run's own counts."""
    eb = 2 if w.dtype == "bf16" else 4
    hit = int((counts > 0).sum())
    weights = hit * (2 * w.d * w.h * eb + 4 * (w.d + w.h))
    S = w.T * w.k
    x_b = w.T * w.d * eb
    y_b = w.T * w.d * eb
    if w.groups == 0:
        eps_b = w.T * w.n * 4 if w.noisy else 0
        gate_cols = w.n
    else:
        m = w.n // w.groups
        eps_b = w.T * (w.groups + w.k_groups * m) * 4 if w.noisy else 0
        gate_cols = w.groups + w.n
    wg_b = 2 * w.d * gate_cols * 4
    small = S * 8 + w.n * 8
    layer_bytes = weights + x_b + y_b + eps_b + wg_b + small
    # expert FFN stage: the hit experts' weights and x read once; the slot
    # buffer, hidden activations and gathered rows are not algorithmic
    ffn_bytes = weights + x_b
    flops = 4.0 * S * w.d * w.h
    # the gate's contraction: x against the score columns each token is
    # scored on (flat: n; hierarchical: the G group columns and the m columns
    # of each of its k_groups kept groups), clean and (noisy) noise matrices
    scored = w.n if w.groups == 0 else w.groups + w.k_groups * (w.n // w.groups)
    gate_flops = 2.0 * w.T * w.d * scored * (2 if w.noisy else 1)
    return dict(layer_bytes=layer_bytes, ffn_bytes=ffn_bytes, flops=flops,
                gate_flops=gate_flops, layer_flops=flops + gate_flops, experts_hit=hit)


# ---------------------------------------------------------------------------
# Clock sampling during the timed region
# ---------------------------------------------------------------------------
class _Nvml:
    """The few read-only NVML queries the clock sampler needs, through ctypes
    on the driver's libnvidia-ml (no Python binding required)."""
    CLOCK_SM = 1

    def __init__(self):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit_v2 failed")

    def handle(self, device_index):
        ct = self.ct
        h = ct.c_void_p()
        try:
            bus = torch.cuda.get_device_properties(device_index).pci_bus_id
            if self.lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ct.byref(h)) == 0:
                return h
        except Exception:
            pass
        if self.lib.nvmlDeviceGetHandleByIndex_v2(ct.c_uint(device_index), ct.byref(h)) != 0:
            raise RuntimeError("no NVML handle")
        return h

    def _uint(self, fn, h, *args):
        v = self.ct.c_uint()
        if fn(h, *args, self.ct.byref(v)) != 0:
            raise RuntimeError(fn.__name__)
        return v.value

    def sm_clock(self, h):
        return self._uint(self.lib.nvmlDeviceGetClockInfo, h, self.ct.c_int(self.CLOCK_SM))

    def max_sm_clock(self, h):
        return self._uint(self.lib.nvmlDeviceGetMaxClockInfo, h, self.ct.c_int(self.CLOCK_SM))

    def power_w(self, h):
        try:
            return self._uint(self.lib.nvmlDeviceGetPowerUsage, h) / 1000.0
        except RuntimeError:
            return None

    def reasons(self, h):
        v = self.ct.c_ulonglong()
        if self.lib.nvmlDeviceGetCurrentClocksEventReasons(h, self.ct.byref(v)) != 0:
            if self.lib.nvmlDeviceGetCurrentClocksThrottleReasons(h, self.ct.byref(v)) != 0:
                raise RuntimeError("clock event reasons")
        return int(v.value)


class ClockSampler:
    """Samples the SM clock, its maximum, the power draw and the active
    clock-event (throttle) reasons of one GPU every `period_s` seconds through
    NVML, read-only, from a background thread; falls back to `nvidia-smi -lms`
    when NVML is unavailable.  `stop()` summarises the samples taken between
    construction and the call."""
    REASONS = (("hw_slowdown", 0x8), ("sw_thermal_slowdown", 0x20),
               ("hw_thermal_slowdown", 0x40), ("hw_power_brake_slowdown", 0x80),
               ("sw_power_cap", 0x4))
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int, period_s: float = 0.001):
        self.samples = []          # (sm_mhz, max_mhz, power_w or None, reason bits)
        self.source = None
        self.proc = None
        self._stop = threading.Event()
        self.period = period_s
        try:
            self.nv = _Nvml()
            self.handle = self.nv.handle(device_index)
            self.max_mhz = float(self.nv.max_sm_clock(self.handle))
            self.source = "nvml"
            self._take()
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()
        except Exception as exc:  # NVML missing or refused: one nvidia-smi process instead
            self.nvml_error = repr(exc)
            self.source = None
            self._start_smi(device_index)

    def _take(self):
        nv = self.nv
        sm = float(nv.sm_clock(self.handle))
        pw = nv.power_w(self.handle)
        bits = nv.reasons(self.handle)
        self.samples.append((sm, self.max_mhz, pw, bits))

    def _poll(self):
        while not self._stop.wait(self.period):
            try:
                self._take()
            except Exception:
                return

    def _start_smi(self, gpu_index):
        self.lines = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi"
            self.thread = threading.Thread(target=self._read_smi, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read_smi(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != 7:
                continue
            try:
                sm, smax = float(parts[0]), float(parts[1])
                pw = float(parts[2])
            except ValueError:
                continue
            bits = 0
            for (name, bit), v in zip((self.REASONS[0], self.REASONS[2], self.REASONS[1],
                                       self.REASONS[4]), parts[3:]):
                if v.lower() == "active":
                    bits |= bit
            self.samples.append((sm, smax, pw, bits))

    def stop(self) -> dict:
        if self.source is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no clock source"],
                    "samples": 0}
        if self.source == "nvml":
            self._stop.set()
            self.thread.join(timeout=5)
            try:
                self._take()       # one more at the end of the region
            except Exception:
                pass
        else:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)
        sm = [x[0] for x in self.samples]
        smax = [x[1] for x in self.samples]
        power = [x[2] for x in self.samples if x[2] is not None]
        reasons = set()
        for x in self.samples:
            for name, bit in self.REASONS:
                if x[3] & bit:
                    reasons.add(name)
        extra = {"nvml_error": self.nvml_error} if getattr(self, "nvml_error", None) else {}
        return {**extra, "sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "sm_mhz_min": min(sm) if sm else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "source": self.source,
                "period_ms": self.period * 1e3 if self.source == "nvml" else 20.0,
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# CPU oracle timing (baseline leg and the reference arm)
# ---------------------------------------------------------------------------
def oracle_sample_rate(w: wl.Workload, seconds: float, max_tokens: int | None = None):
    """Time the oracle forward on the first tokens of the workload; returns
    (tokens/s, cores, tokens per sample, seconds).  Weight conversion to fp64
    happens before the clock starts."""
    import oracle
    inp = wl.make_inputs(w, tokens=slice(0, min(w.T, 64)))
    W1 = oracle._f64(inp["W1"])
    W2 = oracle._f64(inp["W2"])
    b1, b2 = oracle._f64(inp["b1"]), oracle._f64(inp["b2"])

    def run(ntok):
        part = wl.make_inputs(w, experts=False, tokens=slice(0, ntok))
        x, eps = oracle._f64(part["x"]), oracle._f64(part["eps"])
        t0 = time.perf_counter()
        oracle.forward(x, part["Wg"], part["Wn"], part["bg"], eps if w.noisy else None, W1, b1, W2,
                       b2, w.k, w.groups, w.k_groups)
        return time.perf_counter() - t0

    probe = min(w.T, 32)
    dt = run(probe)
    ntok = max(1, min(w.T, int(probe * seconds / max(dt, 1e-6))))
    if max_tokens:
        ntok = min(ntok, max_tokens)
    dt = run(ntok)
    return ntok / dt, oracle.num_threads(), ntok, dt


def reference_arm(args, w: wl.Workload):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    total_budget = 150.0
    per_step = total_budget / max(1, args.steps + args.warmup)
    rate, cores, ntok, dt = oracle_sample_rate(w, seconds=min(per_step, 20.0))
    import oracle
    inp = wl.make_inputs(w, tokens=slice(0, 64))
    W1, W2 = oracle._f64(inp["W1"]), oracle._f64(inp["W2"])
    b1, b2 = oracle._f64(inp["b1"]), oracle._f64(inp["b2"])
    part = wl.make_inputs(w, experts=False, tokens=slice(0, ntok))
    x = oracle._f64(part["x"])
    eps = oracle._f64(part["eps"]) if w.noisy else None
    Wg, Wn = oracle._f64(part["Wg"]), oracle._f64(part["Wn"])
    bg = oracle._f64(part["bg"])

    def step():
        oracle.forward(x, Wg, Wn, bg, eps, W1, b1, W2, b2, w.k, w.groups, w.k_groups)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    value = ntok * args.steps / el
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"first {ntok} tokens of the workload per step (fp64 C oracle, "
                                   f"OpenMP; weights converted to fp64 before timing)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_of(w: wl.Workload) -> dict:
    return {"workload": w.name, "T": w.T, "d": w.d, "h": w.h, "n": w.n, "k": w.k,
            "groups": w.groups, "k_groups": w.k_groups, "noisy": w.noisy,
            "ffn_dtype": w.dtype, "gate_dtype": "f32"}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def fused_ffn(w: wl.Workload) -> bool:
    """Whether the expert stage runs both layers in one kernel (bf16, model
    width 256 or 512, hidden width a multiple of 256, at most 128 rows per
    expert on average)."""
    return (w.dtype == "bf16" and w.d % 256 == 0 and w.d <= 512 and w.h % 256 == 0
            and w.T * w.k <= 128 * w.n)


def launches_per_step(w: wl.Workload) -> int:
    """Kernels moe_forward launches per step.  Flat gating: gate (weight pack,
    scores + KeepTopK) 2, dispatch (rank, column scan + tables, scatter with
    the x-row gather) 3, expert FFN (one kernel for both layers where the
    widths allow, else two grouped GEMMs; their tables come from the
    dispatch) 1 or 2, combine 1.  Hierarchical gating adds to the gate: the
    group pass (pack, scores + KeepTopK), a dispatch of the (token, group)
    pairs (3), their row tiles, the gather of their x rows, and the in-group
    pass (pack, scores + KeepTopK)."""
    gate = 2 if not w.groups else 2 + 3 + 1 + 1 + 2
    return gate + 3 + (1 if fused_ffn(w) else 2) + 1


def counted_launches(B, call, expected: int) -> dict:
    """Kernels of one step, counted: call() is recorded as a CUDA graph and
    its kernel nodes are counted.  Falls back to the expected count (and
    says why) if the capture fails."""
    try:
        g = B.capture(call)
        n = B.kernel_nodes(g)
        del g
        return {"per_step": n, "expected": expected, "source": "kernel nodes of one step "
                "recorded as a CUDA graph"}
    except Exception as exc:  # noqa: BLE001 - reported in the line
        return {"per_step": expected, "expected": expected,
                "source": f"expected count (graph capture failed: {exc})"}


def backward_launches(w: wl.Workload) -> int:
    """Kernels one moe_backward call launches (bf16 tensor-core path, output
    widths d and h multiples of 256): dispatch (3), recompute of the expert
    stage (tile table, x-row gather, two GEMMs: 4), dE
    rows, two row GEMMs (the weights read in their stored layout) and the
    ReLU mask, k-block table, four padded transposes, two weight-gradient GEMMs, Wg^T (and Wn^T), importance
    gradient, token kernel, chunk table and the chunked row sums (gate, db2,
    db1: 6)."""
    flat = 3 + 4 + 1 + 3 + 1 + 4 + 2 + (2 if w.noisy else 1) + 1 + 1 + 1 + 6
    # hierarchical: the pairs (token, kept group) built and routed by group
    # (1 + 3), and their chunk table and two-pass sums for the group columns (3)
    return flat + (7 if w.groups else 0)


def backward_arm(args, w: wl.Workload):
    """Times moe_backward on the workload: the forward runs once for idx, G
    and importance; each timed step is one backward call with the upstream
    gradient dy resident on the device."""
    from sparsely_gated_mixture_top_b300 import binding as B
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    host = wl.make_inputs(w)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in host.items()}
    s = B.shape_of(w)
    ws = B.workspace(s, dev)
    fwd = B.forward(s, d, ws=ws)
    bws = B.backward_workspace(s, dev)
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    gen = torch.Generator(device="cpu").manual_seed(w.seed + 31)
    dy = torch.randn((w.T, w.d), generator=gen).to(dt).to(dev)
    w_imp = 0.01

    def f32(*shape):
        return torch.empty(shape, dtype=torch.float32, device=dev)

    C = w.n + w.groups   # gate score columns (the group columns first)
    g = dict(dx=f32(w.T, w.d), dWg=f32(w.d, C), dWn=f32(w.d, C), dbg=f32(C),
             dW1=f32(w.n, w.h, w.d), db1=f32(w.n, w.h), dW2=f32(w.n, w.d, w.h), db2=f32(w.n, w.d))

    def step(st=stream):
        B.moe_backward(s, d["x"], d["Wg"], d["Wn"], d["eps"], d["W1"], d["b1"], d["W2"], d["b2"],
                       fwd["idx"], fwd["G"], fwd["importance"], dy, w_imp, g["dx"], g["dWg"],
                       g["dWn"], g["dbg"], g["dW1"], g["db1"], g["dW2"], g["db2"], bws, st)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if B.moe_check(bws, stream) != B.MOE_OK:
        raise RuntimeError("device error during warm-up")
    clocks = ClockSampler(0)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    status = B.moe_check(bws, stream)
    if status != B.MOE_OK:
        raise RuntimeError(f"device error in the timed region: {B.status_string(status)}")
    ms = e0.elapsed_time(e1) / args.steps
    launches = counted_launches(B, lambda: step(None), backward_launches(w))
    counts = fwd["counts"].cpu().numpy()
    hit = int((counts > 0).sum())
    eb = 2 if w.dtype == "bf16" else 4
    S = w.T * w.k
    # algorithmic: read the weights of the experts hit, x, dy, eps, the gate
    # matrices; write their gradients (fp32) and dx; contractions: the four
    # backward GEMMs (8 S d h) and the first layer recomputed for a (2 S d h)
    bytes_ = (hit * 2 * w.d * w.h * (eb + 4) + w.T * w.d * (2 * eb + 4) +
              (w.T * C * 4 if w.noisy else 0) + 4 * w.d * C * 4 + S * 8)
    flops = 10.0 * S * w.d * w.h
    pk = peaks()
    long_run = ms * args.steps > 1000.0
    tc_peak = pk["bf16_sustained"] if long_run else pk["bf16"]
    t_hbm, t_tc = bytes_ / (pk["hbm"] * 1e9), flops / (tc_peak * 1e12)
    if t_hbm >= t_tc:
        roof = {"bound": "hbm", "achieved": bytes_ / (ms / 1e3) / 1e9, "peak": pk["hbm"],
                "unit": "GB/s", "peak_source": pk["source"] + " copy bandwidth"}
    else:
        roof = {"bound": "tensor", "achieved": flops / (ms / 1e3) / 1e12, "peak": tc_peak,
                "unit": "TFLOP/s", "peak_source": pk["source"] + " bf16"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = None
    roof["kernel"] = "whole moe_backward call"
    roof["algorithmic_per_launch"] = bytes_ if t_hbm >= t_tc else flops
    roof["ms_per_launch"] = ms
    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        ntok = min(w.T, 64)
        t0 = time.time()
        eps_s = host["eps"][:ntok] if host["eps"] is not None else None
        if w.groups:
            oracle.backward_hier(host["x"][:ntok], host["Wg"], host["Wn"], host["bg"], eps_s,
                                 host["W1"], host["b1"], host["W2"], host["b2"], dy[:ntok].cpu(),
                                 w.k, w.groups, w.k_groups, w_imp)
        else:
            oracle.backward(host["x"][:ntok], host["Wg"], host["Wn"], host["bg"], eps_s,
                            host["W1"], host["b1"], host["W2"], host["b2"], dy[:ntok].cpu(), w.k,
                            w_imp)
        dt_cpu = time.time() - t0
        cpu = {"value": ntok / dt_cpu, "unit": "tokens/s", "cores": oracle.num_threads(),
               "kind": "oracle", "sample": f"first {ntok} tokens, one fp64 oracle backward "
                                            f"({dt_cpu:.1f} s, its forward gate included)"}
    line = {
        "metric": "MoE-layer backward tokens/sec (moe_backward, 1xB300)",
        "value": w.T / (ms / 1e3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "f32",
        "data": "synthetic (seeded counter-based normal)",
        "config": dict(config_of(w), w_importance=w_imp,
                       path="tensor cores" if (w.dtype == "bf16" and w.d % 128 == 0 and
                                               w.h % 128 == 0) else "CUDA cores"),
        "tflops": flops / (ms / 1e3) / 1e12,
        "roofline": roof, "cpu_baseline": cpu, "e2e": None,
        "gpu_launches": launches["per_step"] * args.steps, "gpu_launches_per_step": launches,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)


def ep_arm(args, w: wl.Workload):
    """Times the expert-parallel layer (ExpertParallelMoE.forward): every rank
    gates its own batch of the workload's T tokens against all n experts,
    holds n/P of the experts, and the rows travel by NCCL all-to-all.  Without
    torchrun it runs as a one-rank group (the exchange is then local).  The
    job time is the slowest rank's; value counts every rank's tokens."""
    import socket
    import torch.distributed as dist
    from sparsely_gated_mixture_top_b300 import binding as B
    from sparsely_gated_mixture_top_b300.expert_parallel import ExpertParallelMoE
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world == 1 and "MASTER_PORT" not in os.environ:
        with socket.socket() as so:
            so.bind(("127.0.0.1", 0))
            os.environ["MASTER_PORT"] = str(so.getsockname()[1])
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("nccl", rank=0, world_size=1, device_id=dev)
    else:
        dist.init_process_group("nccl", device_id=dev)
    try:
        host = wl.make_inputs(w.with_(seed=w.seed + rank))
        d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in host.items()}
        fields = dict(d=w.d, h=w.h, n=w.n, k=w.k, groups=w.groups, k_groups=w.k_groups,
                      dtype=w.dtype, noisy=w.noisy)
        layer = ExpertParallelMoE(fields, B.make_shape)
        sl = slice(layer.first_expert, layer.first_expert + layer.n_local)
        W1, W2 = d["W1"][sl].contiguous(), d["W2"][sl].contiguous()
        b1 = None if d["b1"] is None else d["b1"][sl].contiguous()
        b2 = None if d["b2"] is None else d["b2"][sl].contiguous()

        def step():
            return layer.forward(d["x"], d["Wg"], d["Wn"], d["bg"], d["eps"], W1, b1, W2, b2)

        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize(dev)
        layer.ops.check()
        dist.barrier()
        clocks = ClockSampler(local)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            out = step()
        e1.record()
        torch.cuda.synchronize(dev)
        clk = clocks.stop()
        dist.barrier()
        layer.ops.check()
        ms, value = job_throughput(e0.elapsed_time(e1), w.T * args.steps, dist, dev)
        if rank == 0:
            print(json.dumps({
                "metric": "MoE-layer tokens/sec, expert-parallel (ExpertParallelMoE.forward)",
                "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16" if w.dtype == "bf16" else "f32",
                "data": "synthetic (seeded counter-based normal)",
                "config": dict(config_of(w), experts_per_rank=layer.n_local,
                               exchange="NCCL all-to-all (counts, rows out, rows back), "
                                        "all-reduce of importance"),
                "rows_in_last_step": out["rows_in"], "e2e": None, "cpu_baseline": None,
                "clocks": clk}), flush=True)
    finally:
        dist.destroy_process_group()


def balanced_arm(args, w: wl.Workload):
    """Times moe_forward_balanced with the batchwise mask (every expert keeps
    floor(k*T/n) tokens) on the workload, inputs resident on the device."""
    from sparsely_gated_mixture_top_b300 import binding as B
    if w.groups:
        print(json.dumps({"metric": "MoE-layer balanced-routing tokens/sec", "unavailable":
                          "balanced routing covers flat gating only"}))
        return
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    host = wl.make_inputs(w)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in host.items()}
    s = B.shape_of(w)
    m = w.k * w.T // w.n
    cap = w.n * m
    ws = B.balanced_workspace(s, cap, dev)
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    y = torch.empty((w.T, w.d), dtype=dt, device=dev)
    counts = torch.empty((w.n,), dtype=torch.int32, device=dev)

    def step():
        B.moe_forward_balanced(s, d["x"], d["Wg"], d["Wn"], d["bg"], d["eps"], None, cap, d["W1"],
                               d["b1"], d["W2"], d["b2"], y, counts, None, ws, stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if B.moe_check(ws, stream) != B.MOE_OK:
        raise RuntimeError("device error during warm-up")
    clocks = ClockSampler(0)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    status = B.moe_check(ws, stream)
    if status != B.MOE_OK:
        raise RuntimeError(f"device error in the timed region: {B.status_string(status)}")
    ms = e0.elapsed_time(e1) / args.steps
    alg = algorithmic(w, counts.cpu().numpy())
    pk = peaks()
    t_roof = max(alg["layer_bytes"] / (pk["hbm"] * 1e9), alg["layer_flops"] / (pk["bf16"] * 1e12))
    line = {
        "metric": "MoE-layer tokens/sec with the batchwise mask (moe_forward_balanced, 1xB300)",
        "value": w.T / (ms / 1e3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "f32",
        "data": "synthetic (seeded counter-based normal)",
        "config": dict(config_of(w), rows_per_expert=m, gate_scores="fp32 CUDA cores"),
        "layer_roofline": {"t_roof_us": t_roof * 1e6, "t_meas_us": ms * 1e3,
                           "frac": t_roof / (ms / 1e3), "algorithmic_bytes": alg["layer_bytes"],
                           "flops": alg["layer_flops"]},
        "e2e": None, "cpu_baseline": None, "clocks": clk,
    }
    print(json.dumps(line), flush=True)


PER_WORKLOAD = ("hier_4096h_16x256", "skewed_zipf_n64", "sparse_n2048_T4096",
                "sparse_n2048_T32768", "sparse_n2048_T131072")


def device_inputs(w: wl.Workload, dev, rank: int = 0, max_sets: int = 8):
    """The workload's inputs on the device: weights shared by all ranks, x and
    eps per rank, plus rotating copies of (x, eps) so that, together with the
    weights, one step's inputs are out of L2 before they are read again."""
    wr = w.with_(seed=w.seed + 7919 * rank) if rank else w   # each rank its own batch
    host = wl.make_inputs(w)
    if rank:
        part = wl.make_inputs(wr, experts=False)
        host["x"], host["eps"] = part["x"], part["eps"]
    dinp = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in host.items()}
    per_set = host["x"].numel() * host["x"].element_size() + (
        host["eps"].numel() * 4 if host["eps"] is not None else 0)
    nsets = max(2, min(max_sets, math.ceil(256e6 / max(per_set, 1))))
    sets = [(dinp["x"], dinp["eps"])]
    for i in range(1, nsets):
        p = wl.make_inputs(wr.with_(seed=wr.seed + 104729 * i), experts=False)
        sets.append((p["x"].to(dev), p["eps"].to(dev) if p["eps"] is not None else None))
    return host, dinp, sets, per_set


def ffn_stage_ms(B, w, s, dinp, sets, out, ws, stream, dev, steps):
    """Mean CUDA-event time of the expert FFN stage (moe_expert_ffn) with the
    same inputs, between the component calls of the forward pass."""
    S = w.T * w.k
    comp = dict(idx=out["idx"], G=out["G"], counts=out["counts"],
                offsets=torch.empty(w.n + 1, dtype=torch.int32, device=dev),
                perm=torch.empty(S, dtype=torch.int32, device=dev),
                inv_perm=torch.empty(S, dtype=torch.int32, device=dev),
                Y=torch.empty((S, w.d), dtype=out["y"].dtype, device=dev))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    torch.cuda.synchronize(dev)
    for i in range(steps):
        x, eps = sets[i % len(sets)]
        B.moe_gate(s, x, dinp["Wg"], dinp["Wn"], dinp["bg"], eps, comp["idx"], comp["G"], ws,
                   stream)
        B.moe_dispatch(s, comp["idx"], comp["G"], comp["counts"], comp["offsets"], comp["perm"],
                       comp["inv_perm"], out["importance"], out["cv2"], ws, stream)
        ev[i][0].record(stream)
        B.moe_expert_ffn(s, x, comp["perm"], comp["offsets"], dinp["W1"], dinp["b1"], dinp["W2"],
                         dinp["b2"], comp["Y"], ws, stream)
        ev[i][1].record(stream)
        B.moe_combine(s, comp["Y"], comp["inv_perm"], comp["G"], out["y"], ws, stream)
    torch.cuda.synchronize(dev)
    status = B.moe_check(ws, stream)
    if status != B.MOE_OK:
        raise RuntimeError(f"device error in the stage timing: {B.status_string(status)}")
    return float(np.mean([a.elapsed_time(b) for a, b in ev]))


def rooflines(w, counts, ms_step, ffn_ms, long_run):
    """Layer roofline and the expert FFN stage's roofline record."""
    alg = algorithmic(w, counts)
    pk = peaks()
    # A contraction timed inside a loop of more than a second runs under the
    # power cap: its peak is the sustained one, else the burst one.
    tc_peak = pk["bf16_sustained"] if long_run else pk["bf16"]
    tc_label = "sustained" if long_run else "burst"
    ffn_bound_hbm = alg["ffn_bytes"] / (pk["hbm"] * 1e9) >= alg["flops"] / (tc_peak * 1e12)
    if ffn_bound_hbm:
        achieved = alg["ffn_bytes"] / (ffn_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm"], "unit": "GB/s"}
        roof["peak_source"] = pk["source"] + " copy bandwidth"
    else:
        achieved = alg["flops"] / (ffn_ms / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": tc_peak, "unit": "TFLOP/s"}
        roof["peak_source"] = f"{pk['source']} bf16 ({tc_label})"
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = stage_traffic(w)
    roof["kernel"] = "expert FFN stage (moe_expert_ffn)"
    roof["algorithmic_per_launch"] = alg["ffn_bytes"] if ffn_bound_hbm else alg["flops"]
    roof["algorithmic_accounting"] = ("weights of the experts hit + x read once (slot buffer, "
                                      "hidden activations and gathered rows excluded)"
                                      if ffn_bound_hbm else "4*S*d*h FLOPs")
    roof["ms_per_launch"] = ffn_ms
    t_hbm = alg["layer_bytes"] / (pk["hbm"] * 1e9)
    t_tc = alg["layer_flops"] / (tc_peak * 1e12)
    t_roof = max(t_hbm, t_tc)
    layer_roof = {"bound": "hbm" if t_hbm >= t_tc else "tensor",
                  "tensor_peak": f"{tc_label} {tc_peak} TFLOP/s",
                  "t_roof_us": t_roof * 1e6, "t_meas_us": ms_step * 1e3,
                  "frac": t_roof / (ms_step / 1e3), "algorithmic_bytes": alg["layer_bytes"],
                  "flops": alg["layer_flops"], "flops_accounting": "4*S*d*h (experts) + "
                  "2*T*d*(scored columns) per gate matrix", "experts_hit": alg["experts_hit"]}
    return alg, roof, layer_roof


def time_workload(B, w: wl.Workload, dev, stream, steps: int, warmup: int) -> dict:
    """One workload's forward pass, device-resident inputs: ms per step, its
    layer roofline fraction, the expert FFN stage's fraction and the clocks."""
    host, dinp, sets, per_set = device_inputs(w, dev, max_sets=3)
    del host
    s = B.shape_of(w)
    ws = B.workspace(s, dev)
    out = B.outputs(s, dev)

    def fwd(i):
        x, eps = sets[i % len(sets)]
        B.moe_forward(s, x, dinp["Wg"], dinp["Wn"], dinp["bg"], eps, dinp["W1"], dinp["b1"],
                      dinp["W2"], dinp["b2"], out["y"], out["G"], out["idx"], out["importance"],
                      out["cv2"], out["counts"], ws, stream)

    for i in range(warmup):
        fwd(i)
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(dev.index or 0)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        fwd(i)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    status = B.moe_check(ws, stream)
    if status != B.MOE_OK:
        raise RuntimeError(f"{w.name}: device error: {B.status_string(status)}")
    ms = e0.elapsed_time(e1)
    ms_step = ms / steps
    ffn_ms = ffn_stage_ms(B, w, s, dinp, sets, out, ws, stream, dev, max(3, steps // 2))
    alg, roof, layer_roof = rooflines(w, out["counts"].cpu().numpy(), ms_step, ffn_ms,
                                      ms > 1000.0)
    rec = {"config": config_of(w), "steps": steps, "warmup": warmup, "ms_per_step": ms_step,
           "tokens_per_s": w.T / (ms_step / 1e3),
           "tflops": alg["layer_flops"] / (ms_step / 1e3) / 1e12,
           "layer_roofline_frac": layer_roof["frac"], "layer_bound": layer_roof["bound"],
           "t_roof_us": layer_roof["t_roof_us"],
           "ffn_stage": {"ms": ffn_ms, "bound": roof["bound"], "achieved": roof["achieved"],
                         "unit": roof["unit"], "frac": roof["frac"]},
           "clocks": clk}
    del dinp, sets, ws, out
    torch.cuda.empty_cache()
    return rec


def main():
    args = parse()
    w = wl.WORKLOADS[args.workload]
    if args.traffic_summary:
        print(json.dumps(traffic_summary(*args.traffic_summary, w), indent=1))
        return
    if args.impl == "reference":
        reference_arm(args, w)
        return
    if args.which == "backward":
        backward_arm(args, w)
        return
    if args.which == "balanced":
        balanced_arm(args, w)
        return
    if args.which == "ep":
        ep_arm(args, w)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    from sparsely_gated_mixture_top_b300 import binding as B

    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    host, dinp, sets, per_set = device_inputs(w, dev, rank)
    nsets = len(sets)
    s = B.shape_of(w)
    ws = B.workspace(s, dev)
    out = B.outputs(s, dev)

    def fwd(i):
        x, eps = sets[i % nsets]
        B.moe_forward(s, x, dinp["Wg"], dinp["Wn"], dinp["bg"], eps, dinp["W1"], dinp["b1"],
                      dinp["W2"], dinp["b2"], out["y"], out["G"], out["idx"], out["importance"],
                      out["cv2"], out["counts"], ws, stream)

    for i in range(args.warmup):
        fwd(i)
    torch.cuda.synchronize(dev)
    status = B.moe_check(ws, stream)
    if status != B.MOE_OK:
        raise RuntimeError(f"device error during warm-up: {B.status_string(status)}")

    # ---- main timed region: K fused forward passes --------------------------
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(local)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        fwd(i)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    if dist:
        dist.barrier()
    ms = e0.elapsed_time(e1)
    status = B.moe_check(ws, stream)
    if status != B.MOE_OK:
        raise RuntimeError(f"device error in the timed region: {B.status_string(status)}")
    long_run = ms > 1000.0
    ms, value = job_throughput(ms, w.T * args.steps, dist, dev)
    ms_step = ms / args.steps

    # ---- launches: one step recorded as a CUDA graph, its kernel nodes ------
    launches = counted_launches(B, lambda: B.moe_forward(
        s, sets[0][0], dinp["Wg"], dinp["Wn"], dinp["bg"], sets[0][1], dinp["W1"], dinp["b1"],
        dinp["W2"], dinp["b2"], out["y"], out["G"], out["idx"], out["importance"], out["cv2"],
        out["counts"], ws, None), launches_per_step(w))

    # ---- stage timing: the expert FFN stage, same inputs, component calls ---
    ffn_ms = ffn_stage_ms(B, w, s, dinp, sets, out, ws, stream, dev, max(1, args.steps // 2))
    alg, roof, layer_roof = rooflines(w, out["counts"].cpu().numpy(), ms_step, ffn_ms, long_run)

    # ---- end to end: host buffers in, results out, through moe_forward ------
    # Every step copies its x and eps in from pinned host memory and its y, G,
    # idx, importance, cv2 and counts back.  As a serving loop would, the
    # copies of neighbouring steps overlap the forward pass: inputs go in on
    # one stream, the layer runs on another, results come back on a third,
    # with device buffers double-buffered and ordered by events.
    e2e = None
    if rank == 0 or world > 1:
        nb = 2
        pin_x = [st[0].cpu().pin_memory() for st in sets[:nb]]
        pin_e = [st[1].cpu().pin_memory() if st[1] is not None else None for st in sets[:nb]]
        dxs = [torch.empty_like(dinp["x"]) for _ in range(nb)]
        des = [torch.empty_like(dinp["eps"]) if dinp["eps"] is not None else None for _ in range(nb)]
        douts = [B.outputs(s, dev) for _ in range(nb)]
        keys = ("y", "G", "idx", "importance", "cv2", "counts")
        houts = [{k: torch.empty(douts[0][k].shape, dtype=douts[0][k].dtype, pin_memory=True)
                  for k in keys} for _ in range(nb)]
        h2d = pin_x[0].numel() * pin_x[0].element_size() + (
            pin_e[0].numel() * 4 if pin_e[0] is not None else 0)
        d2h = sum(t.numel() * t.element_size() for t in houts[0].values())
        # x and eps go in on two streams (two copy engines share the link)
        s_in, s_in2, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(nb)]
        ev_in2 = [torch.cuda.Event() for _ in range(nb)]
        ev_done = [torch.cuda.Event() for _ in range(nb)]
        ev_out = [torch.cuda.Event() for _ in range(nb)]
        for b in range(nb):  # all buffers start free
            ev_done[b].record(stream)
            ev_out[b].record(stream)

        def e2e_step(i):
            b = i % nb
            with torch.cuda.stream(s_in):
                s_in.wait_event(ev_done[b])      # step i-2 finished reading these inputs
                dxs[b].copy_(pin_x[i % nb], non_blocking=True)
                ev_in[b].record(s_in)
            if des[b] is not None:
                with torch.cuda.stream(s_in2):
                    s_in2.wait_event(ev_done[b])
                    des[b].copy_(pin_e[i % nb], non_blocking=True)
                    ev_in2[b].record(s_in2)
                stream.wait_event(ev_in2[b])
            stream.wait_event(ev_in[b])
            stream.wait_event(ev_out[b])         # step i-2's results are out of these buffers
            o = douts[b]
            B.moe_forward(s, dxs[b], dinp["Wg"], dinp["Wn"], dinp["bg"], des[b], dinp["W1"],
                          dinp["b1"], dinp["W2"], dinp["b2"], o["y"], o["G"], o["idx"],
                          o["importance"], o["cv2"], o["counts"], ws, stream)
            ev_done[b].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done[b])
                for k in keys:
                    houts[b][k].copy_(o[k], non_blocking=True)
                ev_out[b].record(s_out)

        for i in range(3):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s_in)
        s_in2.wait_event(a)   # no copy of the timed steps starts before the start mark
        for i in range(args.e2e_steps):
            e2e_step(i)
        b_.record(s_out)
        torch.cuda.synchronize(dev)
        status = B.moe_check(ws, stream)
        if status != B.MOE_OK:
            raise RuntimeError(f"device error in the end-to-end loop: {B.status_string(status)}")
        e_ms, e_value = job_throughput(a.elapsed_time(b_), w.T * args.e2e_steps, dist, dev)
        e2e = {"value": e_value, "unit": UNIT,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "steps": args.e2e_steps,
               "api": "moe_forward (pinned host x/eps in, y/G/idx/importance/cv2/counts out; "
                      "copies of neighbouring steps overlap the forward pass on separate streams)"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, cores, ntok, dt = oracle_sample_rate(w, args.cpu_seconds)
        cpu = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"first {ntok} tokens of the workload, one fp64 oracle forward "
                         f"({dt:.1f} s; weights converted to fp64 before timing)"}

    # ---- the other full-size workloads, one GPU (rank 0 of a 1-rank run) ----
    per_workload = None
    if rank == 0 and world == 1 and not args.no_per_workload:
        del dinp, sets, ws, out, host
        torch.cuda.empty_cache()
        per_workload = {}
        for name in PER_WORKLOAD:
            if name == w.name:
                continue
            per_workload[name] = time_workload(B, wl.WORKLOADS[name], dev, stream,
                                               steps=args.per_workload_steps, warmup=3)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16"
            if w.dtype == "bf16" else "f32", "data": "synthetic (seeded counter-based normal)",
            "config": dict(config_of(w), l2=f"{nsets} rotating x/eps sets ({nsets * per_set / 1e6:.0f} MB)"
                           f" + {alg['layer_bytes'] / 1e9:.2f} GB algorithmic bytes per step > 126 MB L2"),
            "tflops": alg["layer_flops"] / (ms_step / 1e3) / 1e12,
            "layer_roofline": layer_roof,
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches["per_step"] * args.steps,
            "gpu_launches_per_step": launches,
            "clocks": clk,
            "per_workload": per_workload,
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

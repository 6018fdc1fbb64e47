"""Benchmark of the online-softmax attention library on GB300.

One step = one attention forward (attn_fwd) over the prefill workload B=4, H=32,
N=4096, D=128, bf16, causal, inputs resident in HBM (Q, K and V are 402 MB together,
larger than L2).  Rank 0 prints one JSON line:
  value     whole-job attention TFLOP/s (algorithmic causal FLOPs 4*B*H*D*N(N+1)/2)
  e2e       the same metric through the public API with pinned host buffers and the
            host<->device copies inside the timed region
  roofline  the attention kernel against the measured dense BF16 peak, and against
            peaks that account for the SM clock sampled during the timed region
  clocks    SM clock and throttle reasons sampled in-process (NVML, ~1 ms) during it
  noncausal the same inputs without the causal rule
  combine   split-K LSE combine GB/s on 4096x32 row-heads, depth 128, P in {2,8,16,32,37}
  decode_splitk  split-K decode (64 x 32 heads, 32768 keys) + combine, GB/s; PDL
            against separate calls where the combine is a visible share (P = 37, 148)
  cpu_baseline   the FP64 oracle on the host cores, on a bounded sample (also inside
            the combine and decode objects, for those legs)
With --impl reference the FP64 oracle itself is timed (host cores) on samples of
the same workload.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attn fwd TFLOP/s & % BF16 peak (N=4096,D=128); split-K combine HBM GB/s"
B, H, N, D = 4, 32, 4096, 128
CAUSAL = True
SEED = 3
FLOPS = 4.0 * B * H * D * N * (N + 1) / 2  # algorithmic causal FLOPs per step
WORKLOAD = "prefill attention forward B=4 H=32 N=4096 D=128 bf16 causal"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# NVIDIA's published HBM3e bandwidth of one GB300 GPU (8 TB/s).  The measured peak
# (MEASURED_PEAKS.json) is a read+write copy, which read-dominated kernels can beat;
# fractions against this figure are reported beside it.
DATASHEET_HBM_GBS = 8000.0
PROFILE = os.path.join(ROOT, "profiles", "attn_fwd_prefill_b4h32n4096d128.md")
KERNEL_SOURCES = ["online_softmax_gb300/csrc/attn_fwd.cuh", "online_softmax_gb300/csrc/ptx.cuh",
                  "online_softmax_gb300/csrc/tmem_regs.cuh"]


# ---------------------------------------------------------------- host-side helpers
def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Maximum of a per-rank float over the process group (identity when world == 1)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash() -> str:
    """Hash of the prefill kernel's code: comments and runs of white space are dropped
    first, so that an edit to a comment does not retire the profiled DRAM counters."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        text = re.sub(r"\s+", " ", text).strip()
        h.update(text.encode("utf-8"))
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the
    current kernel source; otherwise None."""
    if not os.path.exists(PROFILE):
        return None
    vals = {}
    for line in open(PROFILE):
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_sha256_16") != kernel_source_hash():
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class _Nvml:
    """Read-only NVML queries through ctypes (clocks, clock-event reasons, power); None
    when the library or the device cannot be opened.  Nothing here sets anything."""
    SM_CLOCK = 1  # NVML_CLOCK_SM
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown"}

    def __init__(self, pci_bus_id: str | None, index: int):
        import ctypes
        self.ok = False
        try:
            self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        except OSError:
            return
        if self.lib.nvmlInit_v2() != 0:
            return
        self.h = ctypes.c_void_p()
        rc = -1
        if pci_bus_id:
            rc = self.lib.nvmlDeviceGetHandleByPciBusId_v2(pci_bus_id.encode(), ctypes.byref(self.h))
        if rc != 0:
            rc = self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.h))
        self.ok = rc == 0
        self.ctypes = ctypes

    def sm_mhz(self):
        v = self.ctypes.c_uint(0)
        return v.value if self.lib.nvmlDeviceGetClockInfo(self.h, self.SM_CLOCK, self.ctypes.byref(v)) == 0 else None

    def sm_max_mhz(self):
        v = self.ctypes.c_uint(0)
        return v.value if self.lib.nvmlDeviceGetMaxClockInfo(self.h, self.SM_CLOCK, self.ctypes.byref(v)) == 0 else None

    def reasons(self):
        v = self.ctypes.c_ulonglong(0)
        fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(self.lib, "nvmlDeviceGetCurrentClocksThrottleReasons", None)
        if fn is None or fn(self.h, self.ctypes.byref(v)) != 0:
            return None
        return [n for bit, n in self.REASONS.items() if v.value & bit]


class ClockSampler:
    """SM clock and throttle reasons sampled every ~1 ms while the timed region runs,
    with in-process NVML queries (read-only), so that a region of a few milliseconds
    still gets samples; falls back to nvidia-smi at 100 ms when NVML cannot be opened."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, pci_bus_id: str | None = None, period_s: float = 0.001):
        self.gpu = gpu_index
        self.pci = pci_bus_id
        self.period = period_s
        self.proc = None
        self.nvml = None
        self.lines = []
        self.stamped, self.smax = [], None
        self.t_start, self.t_end = None, None
        self._stop = threading.Event()

    def __enter__(self):
        self.nvml = _Nvml(self.pci, self.gpu)
        if self.nvml.ok:
            self.smax = self.nvml.sm_max_mhz()
            self.t = threading.Thread(target=self._poll, daemon=True)
            self.t.start()
            return self
        self.nvml = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def mark(self, start: bool):
        """Host time at which the timed region starts / ends: only samples taken
        between the two count (the poller starts a little before the region)."""
        if start:
            self.t_start = time.perf_counter()
        else:
            self.t_end = time.perf_counter()

    def _poll(self):
        while not self._stop.is_set():
            mhz = self.nvml.sm_mhz()
            r = self.nvml.reasons()
            self.stamped.append((time.perf_counter(), mhz, r))
            time.sleep(self.period)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        self._stop.set()
        if self.nvml is not None:
            self.t.join(timeout=5)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, smax, reasons = [], self.smax, set()
        for t, mhz, r in self.stamped:
            if (self.t_start is not None and t < self.t_start) or (self.t_end is not None and t > self.t_end):
                continue
            if mhz is not None:
                sm.append(float(mhz))
            if r:
                reasons.update(r)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm),
                "source": "nvml in-process, ~1 ms" if self.nvml is not None else "nvidia-smi, 100 ms"}


# ---------------------------------------------------------------- oracle baseline
def oracle_sample(budget_s: float, max_heads: int = B * H):
    """Time the FP64 oracle on whole heads of the prefill workload until `budget_s` of
    CPU work has run.  Returns (TFLOP/s, seconds, heads)."""
    import oracle
    import synth
    from tests import helpers as Hl
    done, t_total = 0, 0.0
    while done < max_heads and (t_total < budget_s or done == 0):
        bh = done
        qh = Hl.head_slice(SEED, synth.STREAM_Q, bh, N, D, "bf16")
        kh = Hl.head_slice(SEED, synth.STREAM_K, bh, N, D, "bf16")
        vh = Hl.head_slice(SEED, synth.STREAM_V, bh, N, D, "bf16")
        t0 = time.perf_counter()
        oracle.attention(qh, kh, vh, 1.0 / math.sqrt(D), CAUSAL)
        t_total += time.perf_counter() - t0
        done += 1
        del qh, kh, vh
    flops = 4.0 * D * N * (N + 1) / 2 * done
    return flops / t_total / 1e12, t_total, done


def run_reference(args):
    """The reference arm: the FP64 oracle on the host cores.  One step = the oracle on
    R query rows (the last R of one head, so each row sees ~N keys) with R chosen so the
    whole --warmup + --steps run stays near 90 s of CPU time."""
    import numpy as np
    import oracle
    import synth
    from tests import helpers as Hl
    rank, world, _ = dist_env()
    if rank != 0:
        return
    kh = Hl.head_slice(SEED, synth.STREAM_K, 0, N, D, "bf16")
    vh = Hl.head_slice(SEED, synth.STREAM_V, 0, N, D, "bf16")

    def run(rows):
        qr = Hl.head_slice(SEED, synth.STREAM_Q, 0, N, D, "bf16", rows)
        t0 = time.perf_counter()
        oracle.attention_rows(qr, rows, kh, vh, 1.0 / math.sqrt(D), CAUSAL)
        return time.perf_counter() - t0

    cal = np.arange(N - 256, N)
    t_row = min(run(cal) for _ in range(2)) / len(cal)
    R = int(min(N, max(16, 90.0 / (args.steps + args.warmup) / t_row)))
    rows = np.arange(N - R, N)
    flops_step = 4.0 * D * float(np.sum(rows + 1))  # causal: row i sees i+1 keys
    for _ in range(args.warmup):
        run(rows)
    times = [run(rows) for _ in range(args.steps)]
    per_step = sum(times) / len(times)
    value = flops_step / per_step / 1e12
    cores = os.cpu_count()
    sample = (f"last {R} query rows of one head of the workload per step (4096 keys, causal, D=128), "
              "FP64 numpy oracle")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_step * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "B": B, "H": H, "N": N, "D": D, "causal": CAUSAL, "sample": sample},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU measurements
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--part", default="all", choices=["all", "attn", "combine", "decode"],
                    help="all (default) or one measurement alone, e.g. for a profiler run")
    ap.add_argument("--combine-P", default="2,8,16,32,37")
    ap.add_argument("--combine-dtype", default="f32,bf16")
    ap.add_argument("--decode-batch", type=int, default=64)
    ap.add_argument("--decode-P", default="4,8,16,37")
    args = ap.parse_args()
    assert args.warmup >= 3, "at least 3 warm-up steps"
    if args.impl == "reference":
        return run_reference(args)

    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())

    import online_softmax_gb300 as ops
    import synth
    import synth.cuda as sc

    stream = torch.cuda.current_stream()
    pk, pk_kind = peaks()

    line = {"metric": METRIC, "unit": "TFLOP/s", "n_gpus": world, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic"}
    if args.part in ("all", "attn"):
        line.update(measure_attn(torch, ops, sc, synth, args, world, dev, pk, pk_kind, rank))
    cpu = rank == 0 and args.part == "all" and not args.no_cpu_baseline
    if args.part in ("all", "combine"):
        line["combine"] = measure_combine(torch, ops, sc, synth, pk, dev,
                                          [int(x) for x in args.combine_P.split(",")],
                                          args.combine_dtype.split(","), cpu)
    if args.part in ("all", "decode"):
        line["decode_splitk"] = measure_decode(torch, ops, sc, synth, pk, dev, args.decode_batch,
                                               [int(x) for x in args.decode_P.split(",")], cpu)
    torch.cuda.empty_cache()
    if rank == 0 and args.part == "all" and not args.no_cpu_baseline:
        tf, secs, heads = oracle_sample(12.0)
        line["cpu_baseline"] = {"value": tf, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
                                "sample": f"{heads} whole heads (4096x4096 causal, D=128) of the workload, "
                                          f"FP64 numpy oracle, {secs:.1f} s"}
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def measure_attn(torch, ops, sc, synth, args, world, dev, pk, pk_kind, rank):
    """Headline: K timed attention steps on resident inputs, then the end-to-end variant."""
    stream = torch.cuda.current_stream()

    # ---- inputs of the prefill workload, resident in HBM
    def rand(stream_id):
        t = torch.empty((B, H, N, D), dtype=torch.bfloat16, device=dev)
        return sc.fill_normal(t, SEED, stream_id, "bf16")
    q, k, v = rand(synth.STREAM_Q), rand(synth.STREAM_K), rand(synth.STREAM_V)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)

    def step():
        ops.attn_fwd(q, k, v, o, lse, causal=CAUSAL)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    barrier(world)
    with ClockSampler(dev.index, pci_bus_id(torch, dev)) as clk:
        torch.cuda.synchronize()
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        clk.mark(True)
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        clk.mark(False)
        barrier(world)
    ms = e0.elapsed_time(e1)
    ms_max = max_over_ranks(ms, world, dev)
    assert ops.device_error() == 0
    value = FLOPS * args.steps * world / (ms_max / 1e3) / 1e12
    per_launch_s = ms / 1e3 / args.steps
    achieved = FLOPS / per_launch_s / 1e12
    traffic = profiled_traffic()
    clocks = clk.summary()
    line = {
        "value": value, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max / args.steps,
        "config": {"workload": WORKLOAD, "B": B, "H": H, "N": N, "D": D, "causal": CAUSAL,
                   "flops_per_step": FLOPS, "l2": "inputs larger than L2 (Q, K, V = 402 MB per step)",
                   "parallelism": "replicas" if world == 1 else f"replicas x{world} (independent batches)"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": achieved / pk["bf16_tflops"], "traffic": traffic,
                     "peak_source": f"{pk_kind} (dense bf16 burst)", "kernel": "attn_fwd_persist_kernel<128,bf16>",
                     **clock_aware_roofline(achieved, pk, clocks,
                                             torch.cuda.get_device_properties(dev).multi_processor_count,
                                             peak_run_mhz())},
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    line["noncausal"] = measure_noncausal(torch, ops, q, k, v, pk)

    if args.part == "all":
        line["e2e"] = measure_e2e(torch, ops, q, k, v, args, world, dev)
        line["context"] = measure_sdpa(torch, q, k, v)
        line["masked"] = measure_masked(torch, ops, synth, q, k, v, dev)
    return line


def pci_bus_id(torch, dev):
    """NVML's PCI bus id string of a torch device (None if torch does not expose it)."""
    p = torch.cuda.get_device_properties(dev)
    try:
        return f"{p.pci_domain_id:08x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
    except AttributeError:
        return None


# Dense bf16 tensor-core work one SM retires per SM clock: one kind::f16 MMA of
# M=128, N=128, K=16 (2*128*128*16 FLOP) per 64 cycles, the back-to-back rate measured
# on this part with operands resident in shared memory.
FLOP_PER_SM_CLOCK = 2 * 128 * 128 * 16 / 64


def peak_run_mhz():
    """Median SM clock under load recorded beside the measured peaks (None if absent)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["clocks_under_load"]["sm_mhz_median"])
    except (OSError, KeyError, ValueError, TypeError):
        return None


def clock_aware_roofline(achieved, pk, clocks, sms, peak_mhz):
    """The attention rate against peaks that account for the SM clock.  The measured
    cuBLAS peak was taken at the power-capped clock recorded beside it (median under
    load), while this kernel runs at the clock sampled during its timed region:
      frac_clock_scaled = achieved * (peak run's MHz / kernel's MHz) / measured peak
      frac_of_clock_peak = achieved / (SMs * FLOP_PER_SM_CLOCK * kernel's MHz)."""
    out = {}
    mhz = clocks.get("sm_mhz")
    if mhz:
        at_clock = sms * FLOP_PER_SM_CLOCK * mhz * 1e6 / 1e12
        out["kernel_sm_mhz"] = mhz
        out["peak_at_kernel_clock"] = at_clock
        out["frac_of_clock_peak"] = achieved / at_clock
        if peak_mhz:
            out["peak_run_sm_mhz"] = peak_mhz
            out["frac_clock_scaled"] = achieved * (peak_mhz / mhz) / pk["bf16_tflops"]
    return out


def measure_noncausal(torch, ops, q, k, v, pk):
    """The same inputs without the causal rule (every query sees every key)."""
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    fn = lambda: ops.attn_fwd(q, k, v, o, lse, causal=False)
    for _ in range(3):
        fn()
    med, _ = time_launches(torch, fn, 20)
    flops = 4.0 * B * H * D * N * N
    assert ops.device_error() == 0
    return {"workload": "prefill attention forward B=4 H=32 N=4096 D=128 bf16 non-causal",
            "flops_per_step": flops, "tflops": flops / med / 1e12, "ms": med * 1e3,
            "frac": flops / med / 1e12 / pk["bf16_tflops"]}


def measure_masked(torch, ops, synth, q, k, v, dev):
    """The optional Boolean mask on the same prefill inputs (causal): one shared N x N
    mask per recipe, packed once and summarised once (attn_mask_blocks); the kernel
    still computes every tile the causal rule keeps, so the FLOP count is the unmasked
    one (dense-equivalent TFLOP/s).  `tflops` is attn_fwd_masked_blocks (persistent,
    walks the summary); `scan_tflops` is attn_fwd_masked (one CTA per query-tile pair,
    each scanning the mask)."""
    import numpy as np
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    plain = lambda: ops.attn_fwd(q, k, v, o, lse, causal=CAUSAL)
    for _ in range(3):
        plain()
    base, _ = time_launches(torch, plain, 20)
    masks = {"all visible": np.ones((N, N), dtype=bool),
             "sliding window 1024": synth.mask_band(N, N, 1024),
             "random 50%": synth.mask_random(SEED, (N, N), 0.5),
             "key padding [B,1,1,N], lengths >= N/2": synth.key_padding(SEED, B, N, N // 2)}
    out = {"workload": WORKLOAD + ", shared Boolean mask", "unit": "TFLOP/s (dense-equivalent)",
           "unmasked_tflops": FLOPS / base / 1e12, "results": []}
    for name, m in masks.items():
        mt = torch.from_numpy(np.array(m, dtype=bool, copy=True)).to(dev)
        pack = lambda: ops.attn_mask_pack(mt)
        pack_s, _ = time_launches(torch, pack, 5)
        bits = pack()
        summarise = lambda: ops.attn_mask_blocks(bits, B, H, N)
        summary_s, _ = time_launches(torch, summarise, 5)
        blocks = summarise()
        fn = lambda: ops.attn_fwd_masked_blocks(q, k, v, o, bits, blocks, lse, causal=CAUSAL)
        scan = lambda: ops.attn_fwd_masked(q, k, v, o, bits, lse, causal=CAUSAL)
        for _ in range(3):
            fn()
            scan()
        med, _ = time_launches(torch, fn, 20)
        med_scan, _ = time_launches(torch, scan, 20)
        out["results"].append({"mask": name, "tflops": FLOPS / med / 1e12, "vs_unmasked": base / med,
                               "scan_tflops": FLOPS / med_scan / 1e12, "scan_vs_unmasked": base / med_scan,
                               "pack_us": pack_s * 1e6, "summary_us": summary_s * 1e6})
    assert ops.device_error() == 0
    return out


def measure_sdpa(torch, q, k, v):
    """torch.nn.functional.scaled_dot_product_attention (PyTorch's own backend choice) on
    the same inputs: a comparison point reported beside the result, not a baseline."""
    import torch.nn.functional as F
    fn = lambda: F.scaled_dot_product_attention(q, k, v, is_causal=CAUSAL)
    try:
        for _ in range(3):
            fn()
        med, _ = time_launches(torch, fn, 20)
    except RuntimeError as e:  # a backend may be missing from this PyTorch
        return {"sdpa": f"unavailable: {str(e).splitlines()[0][:120]}"}
    return {"sdpa_tflops": FLOPS / med / 1e12, "sdpa_ms": med * 1e3,
            "note": "torch SDPA, default backend selection, same inputs; context only"}


def measure_e2e(torch, ops, q, k, v, args, world, dev):
    """Same metric through the public API with pinned host inputs and outputs
    (attn_fwd_host: per chunk of heads, copy in, attention and copy out on three streams)."""
    stream = torch.cuda.current_stream()
    hq, hk, hv = (x.cpu().pin_memory() for x in (q, k, v))
    dq, dk, dv = (torch.empty_like(x) for x in (q, k, v))
    do = torch.empty_like(q)
    dl = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    ho = torch.empty(do.shape, dtype=do.dtype, pin_memory=True)
    hl = torch.empty(dl.shape, dtype=dl.dtype, pin_memory=True)
    steps = max(10, min(args.steps, 200))

    def step():  # host buffers in and out; the library overlaps the copies with the attention
        ops.attn_fwd_host(hq, hk, hv, ho, hl, dq, dk, dv, do, dl, causal=CAUSAL)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv))
    d2h = ho.numel() * ho.element_size() + hl.numel() * hl.element_size()
    return {"value": FLOPS * steps * world / (ms / 1e3) / 1e12, "unit": "TFLOP/s", "steps": steps,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms / steps,
            "api": "attn_fwd_host (host buffers; copies overlapped with the attention of other heads)"}


def flush_l2(buf):
    """Evict the inputs from L2 by reading a buffer several times its size.  A read
    leaves clean lines, so the timed kernel does not pay for write-backs of the flush."""
    buf.sum(dtype=buf.dtype)


def time_launches(torch, fn, iters, flush=None):
    """Median and mean device time of `fn` over `iters` launches (L2 flushed before each)."""
    stream = torch.cuda.current_stream()
    ts = []
    for _ in range(iters):
        if flush is not None:
            flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        e1.synchronize()
        ts.append(e0.elapsed_time(e1) / 1e3)
    return statistics.median(ts), sum(ts) / len(ts)


def measure_combine(torch, ops, sc, synth, pk, dev, Ps, dtypes, cpu=False):
    rows, heads, depth = 4096, 32, 128
    RH = rows * heads
    l2buf = torch.ones(128 * 1024 * 1024, dtype=torch.float32, device=dev)  # 512 MB
    out = {"workload": "4096 tokens x 32 heads, depth 128, lse ~ N(10,2), 5% -inf, 0.1% rows all -inf",
           "unit": "GB/s", "l2": "flushed before every launch (512 MB read)", "results": []}
    best = None
    for dt, esz in (("f32", 4), ("bf16", 2)):
        if dt not in dtypes:
            continue
        for P in Ps:
            op = sc.fill_normal(torch.empty((P, RH, depth), dtype=getattr(torch, {"f32": "float32", "bf16": "bfloat16"}[dt]),
                                            device=dev), 21, synth.STREAM_OPART, dt)
            lp = sc.fill_lse(torch.empty((P, RH), dtype=torch.float32, device=dev), 21)
            o = torch.empty((RH, depth), dtype=op.dtype, device=dev)
            g = torch.empty(RH, dtype=torch.float32, device=dev)
            fn = lambda: ops.splitk_combine(op, lp, o, g, rows=rows, heads=heads)
            fn()
            med, mean = time_launches(torch, fn, 20, flush=lambda: flush_l2(l2buf))
            nbytes = P * RH * depth * esz + P * RH * 4 + RH * depth * esz + RH * 4
            gbs = nbytes / med / 1e9
            r = {"P": P, "dtype": dt, "bytes": nbytes, "us": med * 1e6, "GB/s": gbs,
                 "frac": gbs / pk["hbm_gbs"], "frac_datasheet": gbs / DATASHEET_HBM_GBS}
            out["results"].append(r)
            if best is None or r["frac"] > best["frac"]:
                best = r
            del op, lp, o, g
    assert ops.device_error() == 0
    del l2buf
    fr = [r["frac"] for r in out["results"]]
    fd = [r["frac_datasheet"] for r in out["results"]]
    out["roofline"] = {"bound": "hbm", "peak": pk["hbm_gbs"], "unit": "GB/s",
                       "frac_min": min(fr), "frac_median": statistics.median(fr), "frac_max": max(fr),
                       "datasheet_peak": DATASHEET_HBM_GBS, "frac_datasheet_min": min(fd),
                       "frac_datasheet_max": max(fd),
                       "below_0.70_of_datasheet": [f"{r['dtype']} P={r['P']}" for r in out["results"]
                                                   if r["frac_datasheet"] < 0.70]}
    if cpu:
        out["cpu_baseline"] = combine_cpu_baseline(6.0)
    return out


def combine_cpu_baseline(budget_s: float):
    """The FP64 oracle's combine on the host cores: the first 2048 row-heads of the f32
    P = 16 workload, combined again and again until `budget_s` of CPU work has run; GB/s
    of the same algorithmic bytes the GPU number counts."""
    import numpy as np
    import oracle
    import synth
    rows, heads, depth, P, n = 4096, 32, 128, 16, 2048
    RH = rows * heads
    lse = synth.lse_partials(21, P, RH, 0, n).astype(np.float64)
    # partition p's first n row-heads are one contiguous run of the generator's stream
    op = np.stack([synth.normal(21, synth.STREAM_OPART, p * RH * depth, n * depth).reshape(n, depth)
                   for p in range(P)]).astype(np.float64)
    reps, t_total = 0, 0.0
    while t_total < budget_s or reps == 0:
        t0 = time.perf_counter()
        oracle.combine(op, lse)
        t_total += time.perf_counter() - t0
        reps += 1
    done = reps * n
    nbytes = P * done * depth * 4 + P * done * 4 + done * depth * 4 + done * 4
    return {"value": nbytes / t_total / 1e9, "unit": "GB/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"the first {n} row-heads of the f32 P=16 workload, combined {reps} times by the FP64 "
                      f"numpy oracle, {t_total:.1f} s"}


def measure_decode(torch, ops, sc, synth, pk, dev, Bd, Ps, cpu=False):
    Hd, Nkv, Dd = 32, 32768, 128
    q = sc.fill_normal(torch.empty((Bd, Hd, 1, Dd), dtype=torch.bfloat16, device=dev), 5, synth.STREAM_Q, "bf16")
    k = sc.fill_normal(torch.empty((Bd, Hd, Nkv, Dd), dtype=torch.bfloat16, device=dev), 5, synth.STREAM_K, "bf16")
    v = sc.fill_normal(torch.empty((Bd, Hd, Nkv, Dd), dtype=torch.bfloat16, device=dev), 5, synth.STREAM_V, "bf16")
    RH = Bd * Hd
    out = {"workload": f"decode: {Bd} sequences x 1 query, 32 heads, 32768 keys, D=128, bf16; "
                       "fp32 partials, then combine",
           "unit": "GB/s", "l2": "K and V are far larger than L2", "results": []}
    for P in Ps:
        op = torch.empty((P, RH, Dd), dtype=torch.float32, device=dev)
        lp = torch.empty((P, RH), dtype=torch.float32, device=dev)
        o = torch.empty_like(q)
        # attn_fwd_splitk with an output: the combine is a programmatic dependent launch
        fn = lambda: ops.attn_fwd_splitk(q, k, v, P, op, lp, o, None)
        # the same two kernels as two separate calls (plain stream order)
        fn_sep = lambda: (ops.attn_fwd_splitk(q, k, v, P, op, lp, None, None),
                          ops.splitk_combine(op, lp, o.view(RH, Dd), rows=Bd, heads=Hd))
        # the merge inside the attention kernel (last CTA of each row-head)
        counters = torch.zeros(ops.attn_splitk_counters(Bd, Hd, 1), dtype=torch.int32, device=dev)
        fn_fused = lambda: ops.attn_fwd_splitk_fused(q, k, v, P, op, lp, counters, o, None)
        fn()
        fn_sep()
        fn_fused()
        med, _ = time_launches(torch, fn, 10)
        med_sep, _ = time_launches(torch, fn_sep, 10)
        med_fused, _ = time_launches(torch, fn_fused, 10)
        nbytes = 2 * Bd * Hd * Nkv * Dd * 2 + q.numel() * 2 + 2 * (P * RH * Dd * 4 + P * RH * 4) + o.numel() * 2
        gbs = nbytes / med / 1e9
        out["results"].append({"P": P, "bytes": nbytes, "us": med * 1e6, "GB/s": gbs, "frac": gbs / pk["hbm_gbs"],
                               "frac_datasheet": gbs / DATASHEET_HBM_GBS,
                               "us_separate_calls": med_sep * 1e6, "pdl_speedup": med_sep / med,
                               "us_fused_merge": med_fused * 1e6, "fused_speedup": med / med_fused})
    # one sequence: the merge is a larger share of a short step
    small = []
    for P in Ps:
        q1, k1, v1 = q[:1], k[:1], v[:1]
        op = torch.empty((P, Hd, Dd), dtype=torch.float32, device=dev)
        lp = torch.empty((P, Hd), dtype=torch.float32, device=dev)
        o1 = torch.empty_like(q1)
        counters = torch.zeros(ops.attn_splitk_counters(1, Hd, 1), dtype=torch.int32, device=dev)
        fn = lambda: ops.attn_fwd_splitk(q1, k1, v1, P, op, lp, o1, None)
        fn_fused = lambda: ops.attn_fwd_splitk_fused(q1, k1, v1, P, op, lp, counters, o1, None)
        fn()
        fn_fused()
        med, _ = time_launches(torch, fn, 20)
        med_fused, _ = time_launches(torch, fn_fused, 20)
        small.append({"P": P, "us": med * 1e6, "us_fused_merge": med_fused * 1e6, "fused_speedup": med / med_fused})
    out["one_sequence"] = {"workload": "1 sequence x 1 query, 32 heads, 32768 keys, D=128, bf16",
                           "results": small}
    # PDL where the combine is a visible share of the step ("fa4_splitk_combine", PDL
    # paragraph, measured 1.06-1.13x on P = 148 combine-heavy shapes on SM100): one
    # sequence, many partitions; the producer + PDL combine of attn_fwd_splitk against the
    # same two kernels as separate calls in plain stream order.
    heavy = []
    for P in (37, 148):
        q1, k1, v1 = q[:1], k[:1], v[:1]
        op = torch.empty((P, Hd, Dd), dtype=torch.float32, device=dev)
        lp = torch.empty((P, Hd), dtype=torch.float32, device=dev)
        o1 = torch.empty_like(q1)
        fn = lambda: ops.attn_fwd_splitk(q1, k1, v1, P, op, lp, o1, None)
        fn_sep = lambda: (ops.attn_fwd_splitk(q1, k1, v1, P, op, lp, None, None),
                          ops.splitk_combine(op, lp, o1.view(Hd, Dd), rows=1, heads=Hd))
        for _ in range(3):
            fn()
            fn_sep()
        meds, seps = [], []
        for _ in range(5):  # interleaved rounds, so that drifting clocks hit both alike
            meds.append(time_launches(torch, fn, 20)[0])
            seps.append(time_launches(torch, fn_sep, 20)[0])
        med, med_sep = statistics.median(meds), statistics.median(seps)
        heavy.append({"P": P, "us_pdl": med * 1e6, "us_separate_calls": med_sep * 1e6, "pdl_speedup": med_sep / med})
    out["pdl_combine_heavy"] = {"workload": "1 sequence x 1 query, 32 heads, 32768 keys, D=128, bf16, P in {37, 148}",
                                "results": heavy}
    out["multi_query"] = measure_splitk_prefill(torch, ops, sc, synth, dev)
    assert ops.device_error() == 0
    fr = [r["frac"] for r in out["results"]]
    fd = [r["frac_datasheet"] for r in out["results"]]
    out["roofline"] = {"bound": "hbm", "peak": pk["hbm_gbs"], "unit": "GB/s", "frac_min": min(fr),
                       "frac_max": max(fr), "datasheet_peak": DATASHEET_HBM_GBS,
                       "frac_datasheet_min": min(fd), "frac_datasheet_max": max(fd)}
    del q, k, v
    if cpu:
        out["cpu_baseline"] = decode_cpu_baseline(6.0, Ps)
    return out


def measure_splitk_prefill(torch, ops, sc, synth, dev):
    """Split-K over query tiles (the tensor-core split path): B=1, H=32, N=4096, D=128,
    bf16, causal, P = 4 and 8.  The PDL-launched combine of attn_fwd_splitk against the
    same two kernels as separate calls and against the in-kernel merge."""
    Bq, Hq, Nq, Dq = 1, 32, 4096, 128
    mk = lambda sid: sc.fill_normal(torch.empty((Bq, Hq, Nq, Dq), dtype=torch.bfloat16, device=dev), 7, sid, "bf16")
    q, k, v = mk(synth.STREAM_Q), mk(synth.STREAM_K), mk(synth.STREAM_V)
    o = torch.empty_like(q)
    res = []
    for P in (4, 8):
        op = torch.empty((P, Bq * Hq * Nq, Dq), dtype=torch.float32, device=dev)
        lp = torch.empty((P, Bq * Hq * Nq), dtype=torch.float32, device=dev)
        counters = torch.zeros(ops.attn_splitk_counters(Bq, Hq, Nq), dtype=torch.int32, device=dev)
        fn = lambda: ops.attn_fwd_splitk(q, k, v, P, op, lp, o, None, causal=True)
        fn_sep = lambda: (ops.attn_fwd_splitk(q, k, v, P, op, lp, None, None, causal=True),
                          ops.splitk_combine(op, lp, o.view(-1, Dq), rows=Nq, heads=Hq))
        fn_fused = lambda: ops.attn_fwd_splitk_fused(q, k, v, P, op, lp, counters, o, None, causal=True)
        for f in (fn, fn_sep, fn_fused):
            for _ in range(3):
                f()
        med = time_launches(torch, fn, 20)[0]
        med_sep = time_launches(torch, fn_sep, 20)[0]
        med_fused = time_launches(torch, fn_fused, 20)[0]
        res.append({"P": P, "us_pdl": med * 1e6, "us_separate_calls": med_sep * 1e6, "us_fused_merge": med_fused * 1e6,
                    "pdl_speedup": med_sep / med, "fused_speedup": med / med_fused})
    assert ops.device_error() == 0
    return {"workload": "split-K over query tiles: B=1, H=32, N=4096, D=128, bf16, causal", "results": res}


def decode_cpu_baseline(budget_s: float, Ps):
    """The FP64 oracle on decode row-heads of the workload (one query against 32768 keys,
    D=128): the split-K partials for the largest P of the run plus their combine, on the
    first two row-heads again and again until `budget_s` of CPU work has run; GB/s of the
    K/V bytes those row-heads read (bf16), the bytes the GPU number is dominated by."""
    import numpy as np
    import oracle
    import synth
    from tests import helpers as Hl
    Nkv, Dd, seed = 32768, 128, 5
    P = max(Ps)
    bounds = oracle.splitk_bounds(Nkv, P, 128)
    scale = 1.0 / math.sqrt(Dd)
    heads = [tuple(Hl.head_slice(seed, st, bh, n, Dd, "bf16") for st, n in
                   ((synth.STREAM_Q, 1), (synth.STREAM_K, Nkv), (synth.STREAM_V, Nkv))) for bh in (0, 1)]
    done, t_total = 0, 0.0
    while t_total < budget_s or done == 0:
        qr, kh, vh = heads[done % 2]
        t0 = time.perf_counter()
        Op, Lp = oracle.splitk_partials_rows(qr, np.array([0]), kh, vh, scale, False, bounds)
        oracle.combine(Op, Lp)
        t_total += time.perf_counter() - t0
        done += 1
    nbytes = done * 2 * Nkv * Dd * 2
    return {"value": nbytes / t_total / 1e9, "unit": "GB/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"row-heads 0 and 1 of the decode workload, {done} oracle runs (P={P} partials + combine), "
                      f"FP64 numpy oracle, {t_total:.1f} s"}


if __name__ == "__main__":
    main()

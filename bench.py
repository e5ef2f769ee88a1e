"""Benchmark: attention forward TFLOPS on GB300 through the C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

One step = one fa_fwd launch over one batch of the workload (default: the
non-causal B=2, H=16, N=4096, d=128 forward).  Prints one JSON line.
--path splitkv | bwd | paged | fp8 times fa_fwd_splitkv, fa_bwd,
fa_fwd_paged or fa_fwd_fp8 on the same workload instead.

* value: device-timed TFLOPS (4*B*H*Nq*Nk*d per step, halved when causal),
  inputs resident in HBM, K back-to-back steps bracketed by barrier + sync,
  rotating over enough input sets that every step's inputs exceed L2.
* e2e: the same metric through fa_fwd_host from pinned host memory, the
  host->device copies of Q, K, V and the device->host copies of O, LSE inside
  the timed region.
* roofline: the kernel's average launch time (CUDA events on its stream)
  against the measured dense-bf16 peak; traffic from the committed ncu
  summary when the kernel source still matches it.
* cpu_baseline: the fp64 oracle on the host cores, wall clock: a full run of
  the workload when it fits the --cpu-seconds budget, else a row sample.
* --impl reference: the oracle alone, each timed step a full run of the
  workload when all steps fit in about four minutes, else a row sample.
Under torchrun (N > 1) every rank runs its own batch (weak scaling, no
collective on the data path); rank 0 prints the max-over-ranks result.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from exact_attention_28_gb300 import inputs  # noqa: E402

METRIC = "attention fwd TFLOPS (bf16, 1 GB300) and % of dense BF16 tensor peak"
DEFAULT_WORKLOAD = "b2_h16_n4096_d128"
L2_BYTES = 126 * 1024 * 1024
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "fa_fwd_kernel_b2_h16_n4096_d128.txt")
KERNEL_SOURCES = ["fa_api.cu", "fa_fwd_kernel.cuh", "ptx_sm103.cuh"]


def env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "exact_attention_28_gb300", "csrc", name), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """dram bytes per launch from the committed ncu summary, if still valid."""
    try:
        fields = {}
        with open(PROFILE_SUMMARY, encoding="utf-8") as fh:
            for line in fh:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    fields[k.strip()] = v.strip()
        if fields.get("kernel_source_sha256") != kernel_source_hash():
            return None
        return float(fields["dram_bytes_per_full_launch"])
    except (OSError, KeyError, ValueError):
        return None


def reduce_max(values, world, device="cuda"):
    """Element-wise maximum of a list of floats over all ranks (the timing of
    a multi-GPU run is its slowest rank)."""
    if world <= 1:
        return list(values)
    import torch
    import torch.distributed as dist
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def aggregate_tflops(flops_per_rank, ms_per_step_max, world):
    """Whole-job throughput: every rank's work over the slowest rank's time."""
    return world * flops_per_rank / (ms_per_step_max * 1e-3) / 1e12


def shard_heads(num_heads, rank, world):
    """Contiguous [start, stop) slice of the B*H independent heads for one rank
    (heads are independent problems, so a strong-scaling split needs no
    communication on the data path)."""
    base, extra = divmod(num_heads, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def paged_cache(k, v, block_size, seed):
    """K, V [B, H, Nk, d] laid out as a paged cache: ([num_blocks, H, block_size, d]
    K and V caches, int32 block table [B, ceil(Nk / block_size)]).  Every
    sequence's logical blocks go to a seeded random permutation of the physical
    blocks (so consecutive key tiles come from scattered pages); the tail of
    the last block is zero and lies beyond the sequence length."""
    import torch
    B, H, Nk, d = k.shape
    nb = -(-Nk // block_size)
    perm = torch.from_numpy(np.random.default_rng(seed).permutation(B * nb).astype(np.int64)).to(k.device)
    caches = []
    for x in (k, v):
        padded = torch.zeros((B, H, nb * block_size, d), dtype=x.dtype, device=x.device)
        padded[:, :, :Nk] = x
        blocks = padded.view(B, H, nb, block_size, d).permute(0, 2, 1, 3, 4).reshape(B * nb, H, block_size, d)
        cache = torch.empty_like(blocks)
        cache[perm] = blocks
        caches.append(cache)
    table = perm.view(B, nb).to(torch.int32)
    return caches[0], caches[1], table


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json"), encoding="utf-8") as fh:
            return json.load(fh), "measured"
    except (OSError, ValueError):
        return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}, "fallback"


# ------------------------------------------------------------------ clocks

# Polls NVML in a child process (so the benchmark's own thread never waits for
# the interpreter lock): prints "time sm_mhz max_mhz reason_bits" every period.
# Read-only NVML queries; nothing is set.
_NVML_POLLER = r"""
import ctypes, sys, time
bus, index, period = sys.argv[1].encode(), int(sys.argv[2]), float(sys.argv[3])
lib = ctypes.CDLL("libnvidia-ml.so.1")
if lib.nvmlInit_v2() != 0:
    sys.exit(2)
h = ctypes.c_void_p()
if not bus or lib.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(h)) != 0:
    if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(h)) != 0:
        sys.exit(3)
reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or lib.nvmlDeviceGetCurrentClocksThrottleReasons
mx, mhz, bits = ctypes.c_uint(0), ctypes.c_uint(0), ctypes.c_ulonglong(0)
lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))
print("ready", flush=True)
while True:
    if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(mhz)) == 0 and reasons(h, ctypes.byref(bits)) == 0:
        sys.stdout.write(f"{time.time():.6f} {mhz.value} {mx.value} {bits.value}\n")
        sys.stdout.flush()
    time.sleep(period)
"""


class ClockSampler:
    """SM clock and clock-event (throttle) reasons of the benchmarked GPU during
    the timed region: NVML polled every `period` seconds by a child process,
    or nvidia-smi every 100 ms where NVML cannot be loaded."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, torch_index: int, period: float = 2.5e-4):
        self.samples = []          # (time, sm_mhz, max_mhz, reason bits)
        self.period = period
        self.source = "nvml"
        self.proc = None
        bus = ""
        try:   # the CUDA device's PCI address (NVML may number the GPUs differently)
            import torch
            pr = torch.cuda.get_device_properties(torch_index)
            bus = f"{pr.pci_domain_id:08x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0"
        except Exception:   # noqa: BLE001 -- older torch without the PCI fields
            bus = ""
        try:
            self.proc = subprocess.Popen([sys.executable, "-c", _NVML_POLLER, bus, str(torch_index), str(period)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            ready = self.proc.stdout.readline().strip() == "ready"
        except OSError:
            ready = False
        if not ready:
            self._kill()
            self.source = "nvidia-smi"
            self.period = 0.1
            self._start_smi(torch_index)
            return
        self.thread = threading.Thread(target=self._read_nvml, daemon=True)
        self.thread.start()

    def _read_nvml(self):
        for line in self.proc.stdout:
            parts = line.split()
            try:
                self.samples.append((float(parts[0]), float(parts[1]), float(parts[2]), int(parts[3])))
            except (IndexError, ValueError):
                continue

    def _start_smi(self, gpu_index):
        fields = ("timestamp,clocks.sm,clocks.max.sm,clocks_event_reasons.active,"
                  "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                  "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={fields}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.thread = threading.Thread(target=self._read_smi, daemon=True)
        self.thread.start()

    def _read_smi(self):
        bitmap = {4: 0x8, 5: 0x40, 6: 0x20, 7: 0x4}
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            try:
                bits = sum(b for i, b in bitmap.items() if parts[i].lower() == "active")
                self.samples.append((time.time(), float(parts[1]), float(parts[2]), bits))
            except (IndexError, ValueError):
                continue

    def _kill(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.proc = None

    def stop(self):
        self._kill()

    def summary(self, t0, t1):
        inside = [r for r in self.samples if t0 <= r[0] <= t1]
        window = "timed region"
        if len(inside) < 3:   # very short timed region: take the samples nearest to it
            inside = sorted(self.samples, key=lambda r: abs(r[0] - 0.5 * (t0 + t1)))[:5]
            window = "nearest samples (timed region shorter than the sampling period)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no clock samples"], "source": self.source}
        reasons = sorted({name for r in inside for bit, name in self.REASONS.items() if r[3] & bit})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside), "window": window, "source": self.source,
                "period_ms": round(self.period * 1e3, 3)}


# ---------------------------------------------------------------- CPU legs

def oracle_time(w, q, k, v, budget_s, nthreads):
    """Time the fp64 oracle on the workload with wall-clock time: one full run
    when a probe of 64 random rows predicts that it ends within budget_s, else
    a random row sample sized to about budget_s.
    Returns (TFLOPS, seconds, rows, threads, full_run)."""
    import oracle
    rng = np.random.default_rng(0)
    per_row = lambda rows: sum(4 * (min(w.Nk, (r % w.Nq) + 1) if w.causal else w.Nk) * w.d for r in rows)
    probe = rng.integers(0, w.B * w.H * w.Nq, 64)
    t = time.perf_counter()
    oracle.attention_rows(q, k, v, w.scale, w.causal, rows=probe, nthreads=nthreads)
    dt = max(time.perf_counter() - t, 1e-4)
    rate = per_row(probe) / dt                      # FLOP/s of the oracle on these cores
    if w.flops / rate <= budget_s:
        t = time.perf_counter()
        oracle.attention(q, k, v, w.scale, w.causal, nthreads=nthreads)
        dt = time.perf_counter() - t
        return w.flops / dt / 1e12, dt, w.B * w.H * w.Nq, nthreads, True
    n = int(min(w.B * w.H * w.Nq, max(64, 64 * budget_s / dt)))
    rows = rng.integers(0, w.B * w.H * w.Nq, n)
    t = time.perf_counter()
    oracle.attention_rows(q, k, v, w.scale, w.causal, rows=rows, nthreads=nthreads)
    dt = time.perf_counter() - t
    return per_row(rows) / dt / 1e12, dt, n, nthreads, False


def oracle_note(rows, dt, threads, full):
    what = f"full run of the workload ({rows} query rows)" if full else f"{rows} random query rows of the workload"
    return f"{what}, fp64 three-pass oracle, {dt:.1f} s wall clock, {threads} threads"


def run_reference(args, w):
    """The oracle as the reference arm: warm-up steps run short row samples,
    each timed step a full run of the workload when all of them fit in about
    four minutes, else a row sample per step sized to fit."""
    rank = env_int("RANK", 0)
    if rank != 0:
        return 0
    q, k, v, _ = inputs.make_inputs(w)
    cores = os.cpu_count() or 1
    per_step = max(0.5, 240.0 / max(1, args.steps))
    for _ in range(args.warmup):
        oracle_time(w, q, k, v, 0.0, cores)          # a short sample: threads and caches warm
    vals, secs, nrows, fulls = [], 0.0, 0, []
    for _ in range(args.steps):
        tf, dt, n, _, full = oracle_time(w, q, k, v, per_step, cores)
        vals.append(tf)
        secs += dt
        nrows += n
        fulls.append(full)
    value = statistics.median(vals)
    note = (f"{args.steps} full runs of the workload" if all(fulls) else
            f"{nrows} random query rows over {args.steps} steps (a full run would exceed the time budget)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(w, None),
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": cores, "kind": "oracle",
                         "sample": f"{note}, fp64 three-pass oracle, wall clock, {cores} threads"},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(w, l2_note, args=None):
    cfg = {"workload": w.name, "B": w.B, "H": w.H, "Nq": w.Nq, "Nk": w.Nk, "d": w.d, "causal": w.causal,
           "path": getattr(args, "path", "fwd") if args is not None else "fwd",
           "sigma_qkv": [w.sigma_q, w.sigma_k, w.sigma_v], "scale": "1/sqrt(d) as fp32",
           "global_batch": w.B, "seq_len": w.Nq, "parallelism": "independent replicas (weak)"}
    if l2_note:
        cfg["l2"] = l2_note
    return cfg


# -------------------------------------------------------------------- ours

def run_e2e(args, w, hq, hk, hv, dev_set, scale, stream):
    """ms per step of fa_fwd_host from pinned host buffers (copies included)."""
    import torch

    from exact_attention_28_gb300 import ops
    phq, phk, phv = hq.pin_memory(), hk.pin_memory(), hv.pin_memory()
    pho = torch.empty_like(hq).pin_memory()
    phl = torch.empty((w.B, w.H, w.Nq), dtype=torch.float32).pin_memory()
    e2e_steps = max(3, min(args.steps, 20))
    for _ in range(2):
        ops.fa_fwd_host(phq, phk, phv, pho, phl, *dev_set, scale, causal=w.causal, stream=stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        ops.fa_fwd_host(phq, phk, phv, pho, phl, *dev_set, scale, causal=w.causal, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    ops.check_device_status()
    return e0.elapsed_time(e1) / e2e_steps


def run_ours(args, w):
    import torch
    import torch.distributed as dist

    from exact_attention_28_gb300 import build, ops

    rank, world, local = env_int("RANK", 0), env_int("WORLD_SIZE", 1), env_int("LOCAL_RANK", 0)
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")
    build.build()
    ops.load_library()

    q, k, v, scale = inputs.make_inputs(w)
    as_t = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    hq, hk, hv = as_t(q), as_t(k), as_t(v)
    set_bytes = (2 * hq.numel() + 2 * hk.numel()) * 2 + w.B * w.H * w.Nq * 4
    n_sets = max(1, math.ceil(2 * L2_BYTES / set_bytes)) if set_bytes < 2 * L2_BYTES else 1
    sets = []
    for _ in range(n_sets):
        sets.append((hq.cuda(), hk.cuda(), hv.cuda(), torch.empty_like(hq, device="cuda"),
                     torch.empty((w.B, w.H, w.Nq), dtype=torch.float32, device="cuda")))
    l2_note = (f"rotating {n_sets} input sets, {n_sets * set_bytes / 2**20:.0f} MiB > 2x L2"
               if n_sets > 1 else f"inputs {set_bytes / 2**20:.0f} MiB > 2x L2")
    stream = torch.cuda.current_stream()

    workspace = None
    splits = 1
    if args.path == "bwd":
        # forward outputs and an upstream gradient for every input set
        import ctypes
        nb = ctypes.c_size_t(0)
        ops._check(ops.load_library().fa_bwd_workspace(w.B, w.H, w.Nq, w.Nk, w.d, ctypes.byref(nb)))
        workspace = torch.empty(nb.value, dtype=torch.uint8, device="cuda")
        bwd_bufs = []
        for si, s in enumerate(sets):
            ops.fa_fwd(s[0], s[1], s[2], s[3], s[4], scale=scale, causal=w.causal, stream=stream)
            do = as_t(inputs.normal_bf16(7000 + si, (w.B, w.H, w.Nq, w.d))).cuda()
            bwd_bufs.append((do, torch.empty_like(s[0]), torch.empty_like(s[1]), torch.empty_like(s[2])))
    if args.path == "splitkv":
        splits, nbytes = ops.splitkv_workspace(w.B, w.H, w.Nq, w.Nk, w.d, w.causal, 0)
        workspace = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    if args.path == "fp8":
        # E4M3 codes of the inputs (Q, K rotated by the same random signs, V
        # transposed), quantised once before timing; enough code sets that
        # every step's inputs exceed L2
        if w.d != 128:
            raise SystemExit("--path fp8 needs d = 128")
        signs = torch.from_numpy(np.random.default_rng(17).choice([-1.0, 1.0], size=w.d).astype(np.float32)).cuda()
        fp8_bytes = w.B * w.H * (w.Nq * w.d + 2 * (-(-w.Nk // 16) * 16) * w.d + 2 * w.Nq * w.d + 4 * w.Nq)
        n_fp8 = max(1, math.ceil(2 * L2_BYTES / fp8_bytes)) if fp8_bytes < 2 * L2_BYTES else 1
        fp8_sets = []
        for si in range(n_fp8):
            s = sets[si % n_sets]
            q8, dq = ops.quantize_fp8(s[0], signs)
            k8, dk = ops.quantize_fp8(s[1], signs)
            vt8, dv = ops.quantize_fp8(s[2], transpose=True)
            fp8_sets.append((q8, k8, vt8, dq, dk, dv, torch.empty_like(s[3]), torch.empty_like(s[4])))
        sets = sets[:1]
        n_sets = 1
        torch.cuda.synchronize()
        ops.check_device_status()
        l2_note = (f"rotating {n_fp8} E4M3 input sets, {n_fp8 * fp8_bytes / 2**20:.0f} MiB > 2x L2"
                   if n_fp8 > 1 else f"E4M3 inputs {fp8_bytes / 2**20:.0f} MiB > 2x L2")
    if args.path == "paged":
        # each input set's K/V as a paged cache (same keys, scattered pages)
        seq_lens = torch.full((w.B,), w.Nk, dtype=torch.int32, device="cuda")
        paged_bufs = [paged_cache(s[1], s[2], args.block_size, 9000 + si) for si, s in enumerate(sets)]
        sets = [(s[0], None, None, s[3], s[4]) for s in sets]   # the contiguous K/V are not used
        torch.cuda.empty_cache()
        # key slices as the library would choose them for this shape (1: no split, no merge)
        cap = paged_bufs[0][2].shape[1] * args.block_size
        splits, nbytes = ops.splitkv_workspace(w.B, w.H, w.Nq, cap, w.d, w.causal, 0)
        if splits > 1:
            workspace = torch.empty(nbytes, dtype=torch.uint8, device="cuda")

    def step(i):
        s = sets[i % n_sets]
        if args.path == "bwd":
            b = bwd_bufs[i % n_sets]
            ops.fa_bwd(s[0], s[1], s[2], s[3], s[4], b[0], b[1], b[2], b[3], scale=scale, causal=w.causal,
                       workspace=workspace, stream=stream)
        elif args.path == "fp8":
            f = fp8_sets[i % len(fp8_sets)]
            ops.fa_fwd_fp8(f[0], f[1], f[2], f[3], f[4], f[5], f[6], f[7], scale=scale, causal=w.causal,
                           stream=stream)
        elif args.path == "paged":
            kc, vc, table = paged_bufs[i % n_sets]
            ops.fa_fwd_paged(s[0], kc, vc, table, seq_lens, s[3], s[4], scale=scale, causal=w.causal, stream=stream,
                             num_splits=splits if splits > 1 else None, workspace=workspace)
        elif args.path == "splitkv":
            ops.fa_fwd_splitkv(s[0], s[1], s[2], s[3], s[4], scale=scale, causal=w.causal, num_splits=splits,
                               workspace=workspace, stream=stream)
        else:
            ops.fa_fwd(s[0], s[1], s[2], s[3], s[4], scale=scale, causal=w.causal, stream=stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    ops.check_device_status()

    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    for i in range(args.steps):
        starts[i].record(stream)
        step(i)
        ends[i].record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    if world > 1:
        dist.barrier()
    ops.check_device_status()
    total_ms = starts[0].elapsed_time(ends[-1])
    launch_ms = statistics.mean(s.elapsed_time(e) for s, e in zip(starts, ends))
    total_ms, launch_ms = reduce_max([total_ms, launch_ms], world)
    if sampler:
        time.sleep(0.25)
        sampler.stop()

    # end to end through the host-buffer entry point
    e2e_ms = float("nan")
    if not args.no_e2e and args.path == "fwd":
        e2e_ms = run_e2e(args, w, hq, hk, hv, sets[0], scale, stream)
    if not args.no_e2e and args.path == "fwd":
        e2e_ms = reduce_max([e2e_ms], world)[0]
    if rank == 0:
        peaks, peak_src = measured_peaks()
        ms_per_step = total_ms / args.steps
        # backward: five GEMMs of 2*Nq*Nk*d (dV, dP, dQ, dK and the recomputed S), 2.5x the forward
        flops = w.flops * 5 // 2 if args.path == "bwd" else w.flops
        value = aggregate_tflops(flops, ms_per_step, world)
        # E4M3 contractions: the measured bf16 peak times the nominal fp8/bf16 ratio (4.5 / 2.25)
        fp8 = args.path == "fp8"
        tensor_peak = float(peaks["bf16_tflops"]) * (2.0 if fp8 else 1.0)
        alg_bytes = (w.B * w.H * (w.Nq * w.d + 2 * w.Nk * w.d + 2 * w.Nq * w.d + 4 * w.Nq) if fp8
                     else w.algorithmic_bytes)
        ridge = tensor_peak * 1e12 / (float(peaks["hbm_gbs"]) * 1e9)
        tensor_bound = flops / alg_bytes >= ridge
        if tensor_bound:
            achieved, peak, unit, bound = flops / (launch_ms * 1e-3) / 1e12, tensor_peak, "TFLOP/s", "tensor"
        else:
            achieved, peak, unit, bound = alg_bytes / (launch_ms * 1e-3) / 1e9, float(peaks["hbm_gbs"]), \
                "GB/s", "hbm"
        traffic = profiled_traffic() if (w.name == DEFAULT_WORKLOAD and args.path == "fwd") else None
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "e4m3" if fp8 else "bf16", "data": "synthetic (seeded N(0, sigma^2) rounded to bf16)",
            "config": dict(workload_config(w, l2_note, args), kv_splits=splits,
                           **({"block_size": args.block_size} if args.path == "paged" else {})),
            "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                         "frac": achieved / peak, "traffic": traffic,
                         "peak_source": f"{peak_src} " + (("bf16_tflops (burst) x 2, the nominal fp8/bf16 ratio"
                                                            if fp8 else "bf16_tflops (burst)")
                                                           if tensor_bound else "hbm_gbs"),
                         "frac_of_sustained": (achieved / (float(peaks.get("bf16_tflops_sustained", peak))
                                                           * (2.0 if fp8 else 1.0))
                                               if tensor_bound else None),
                         "kernel": ("fa_bwd_dot + fa_bwd_dkdv + fa_bwd_dq <%d>" % w.d if args.path == "bwd" else
                                    "fa_fwd_kernel<128, 4> (E4M3)" if fp8 else
                                    "fa_fwd_kernel<%d, %d>" % (w.d, (2 if args.path == "paged" else 0) + (1 if splits > 1 else 0))
                                    + (" + fa_merge_kernel" if splits > 1 else "")),
                         "launch_ms": launch_ms},
            "e2e": None if (args.no_e2e or args.path != "fwd") else {
                "value": aggregate_tflops(w.flops, e2e_ms, world), "unit": "TFLOPS",
                "h2d_bytes_per_step": 2 * (hq.numel() + 2 * hk.numel()),
                "d2h_bytes_per_step": 2 * hq.numel() + 4 * w.B * w.H * w.Nq,
                "ms_per_step": e2e_ms},
            "gpu_launches": args.steps * (3 if args.path == "bwd" else (2 if splits > 1 else 1)),
            "clocks": sampler.summary(t0, t1) if sampler else None,
        }
        if world == 1 and not args.no_cpu_baseline:
            tf, dt, n, cores, full = oracle_time(w, q, k, v, args.cpu_seconds, os.cpu_count() or 1)
            line["cpu_baseline"] = {"value": tf, "unit": "TFLOPS", "cores": cores, "kind": "oracle",
                                    "sample": oracle_note(n, dt, cores, full)}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--cpu-seconds", type=float, default=30.0,
                    help="time budget of the oracle leg: a full run of the workload if it fits, else a row sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer leg (profiling runs)")
    ap.add_argument("--block-size", type=int, default=64, help="page size of --path paged")
    ap.add_argument("--path", choices=["fwd", "splitkv", "bwd", "paged", "fp8"], default="fwd",
                    help="fa_fwd, fa_fwd_splitkv with the library's slice count, fa_bwd, "
                         "fa_fwd_paged over the workload's K/V scattered into pages, or fa_fwd_fp8 on "
                         "E4M3 codes of the workload (quantised before timing)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = inputs.WORKLOADS[args.workload]
    return run_reference(args, w) if args.impl == "reference" else run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())

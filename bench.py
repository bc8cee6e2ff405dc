"""Benchmark: one step = build the topology CSR from K, then scheduled attention over it.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl {tsa,reference}]
                    [--workload NAME]
                    [--schedule topology|topology-content|segment:TOKENS|dense|density:P]

Metric: scheduled-attention forward TFLOP/s counted on visited blocks
(nnz * lanes * 4 * 64^2 * D per step) and ms per step.  Default workload: [B=2, H=32,
S=32768, D=128] bf16, block 64, sink 2, local_radius 4, topk 8, keys clustered over 32
means (the S 32768 configuration).  Inputs are synthetic, seeded and resident in HBM; the
default workload's are larger than L2 (no flush), smaller ones get L2 flushed before every step
(outside the step's events).  The roofline object names the bound that the kernel's arithmetic
intensity on compulsory bytes selects (tensor or HBM), against the burst peak when the timed
region is shorter than a second and the sustained peak otherwise.  Inputs are drawn with the CPU
generator (the same tensors the reference arm uses) and copied to the GPU before timing.

Under torchrun (--shard lanes, the default) one problem's lanes are spread over the ranks, the
workload's B*H lanes on each (weak scaling: B grows with the number of GPUs): every step each
rank sums its own lanes' key blocks, the block sums are all-gathered over NCCL in global lane
order, every rank builds the one shared CSR from them, and each rank runs the attention on its
own lanes.  The exchange is inside the timed step.  Before timing, rank 0 checks that the CSR
equals the one a single GPU builds from all lanes' keys.  --shard none runs an independent
problem per rank instead (no collective).

Schedules built on the GPU inside every step: "topology" (elder rule, index ties),
"topology-content" (content ties), "segment:TOKENS" (fixed segments).  "dense" and
"density:P" are built once before timing.

--pass bwd times the backward instead: one step = tsa_scheduled_attention_backward (the
transposed schedule, Delta = rowsum(dO * O), the dQ kernel and the dK/dV kernel) over a schedule
built once before timing, with O and the log-sum-exp from one forward call.  Its FLOPs count the
five 64 x 64 x D block products of the gradient on visited blocks (S recomputation excluded):
nnz * lanes * 10 * 64^2 * D per step.

--impl reference times the CPU oracle (oracle/, fp64) on the host cores on a bounded
sample of the same workload.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from topology_scheduled_gb300.workloads import WORKLOADS, make_qkv, random_density_csr  # noqa: E402

DEFAULT_WORKLOAD = "b2h32s32768"
# the attention kernel's sources: a traffic record applies only to the build it was taken on
ATTN_SOURCES = [os.path.join(ROOT, "topology_scheduled_gb300", "csrc", f)
                for f in ("attention.cu", "tsa_device.cuh", "tsa_internal.h")]


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["tsa", "reference"], default="tsa")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    p.add_argument("--schedule", default="topology")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--heads", type=int, default=0,
                   help="override H (a smaller case of the same workload, e.g. for ncu captures)")
    p.add_argument("--pass", dest="pass_", choices=["fwd", "bwd"], default="fwd",
                   help="time the forward step (default) or the backward call")
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="target CPU time of the oracle's attention sample")
    p.add_argument("--shard", choices=["lanes", "none"], default="lanes",
                   help="under torchrun: spread one problem's lanes over the ranks (lanes) or run an "
                        "independent problem per rank (none)")
    return p.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def visited_flops(nnz: int, lanes: int, D: int, block: int = 64) -> float:
    return float(nnz) * lanes * 4.0 * block * block * D


def aggregate_over_ranks(elapsed_ms: float, flops: float, device, world: int):
    """Whole-job timing: the slowest rank's time and the sum of all ranks' work."""
    if world <= 1:
        return elapsed_ms, flops
    import torch.distributed as dist
    t = torch.tensor([elapsed_ms], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    w = torch.tensor([flops], device=device, dtype=torch.float64)
    dist.all_reduce(w, op=dist.ReduceOp.SUM)
    return float(t.item()), float(w.item())


def launches_per_step(schedule: str) -> int:
    """Kernels of this library per step: the attention kernel, plus the builder's kernels when
    the schedule is built inside the step -- centroid_partial, centroid_final, pairwise_bounds and
    the cooperative graph kernel for a topology schedule (content_rank and permute_rows in
    addition under content ties), segment_rows and segment_fill for fixed segments."""
    return 1 + {"topology": 4, "topology-content": 6}.get(
        schedule, 2 if schedule.startswith("segment:") else 0)


def built_in_step(schedule: str) -> bool:
    return schedule in ("topology", "topology-content") or schedule.startswith("segment:")


def segment_tokens(schedule: str) -> int:
    return int(schedule.split(":")[1])


def dtype_name(dt) -> str:
    return {torch.float16: "f16", torch.bfloat16: "bf16"}[dt]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# A timed region shorter than this is compared with the burst tensor peak (a cuBLAS GEMM timed
# alone, clocks at their maximum); a longer one with the sustained peak (a seconds-long loop
# under the power cap).
BURST_REGION_MS = 1000.0


def tensor_peak(peaks: dict, kind: str, region_ms: float):
    """(peak TFLOP/s, description) for a timed region of region_ms milliseconds."""
    burst = float(peaks.get("bf16_tflops", peaks.get("bf16_tflops_sustained")))
    sustained = float(peaks.get("bf16_tflops_sustained", burst))
    if region_ms < BURST_REGION_MS:
        return burst, (f"{kind} bf16_tflops (cuBLAS bf16 burst; timed region {region_ms:.1f} ms "
                       f"< {BURST_REGION_MS:.0f} ms)")
    return sustained, (f"{kind} bf16_tflops_sustained (cuBLAS bf16, seconds-long loop; timed region "
                       f"{region_ms:.0f} ms)")


def attention_sources_sha1() -> str:
    """sha1 over the attention kernel's source files, concatenated in a fixed order."""
    h = hashlib.sha1()
    for path in ATTN_SOURCES:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def attention_traffic_per_launch(workload: str, schedule: str):
    """DRAM bytes per attention launch from the committed ncu summary, if it matches the source."""
    path = os.path.join(ROOT, "profiles", "attention_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    digest = attention_sources_sha1()
    entry = rec.get(f"{workload}/{schedule}")
    if not entry or entry.get("sources_sha1") != digest:
        return None
    return entry.get("dram_bytes_per_launch")


class ClockSampler:
    """SM clock and throttle-reason samples during the timed region, read-only.

    A thread polls NVML (libnvidia-ml, through ctypes) every 5 ms, so that even a region of a
    few tens of milliseconds gets samples; where NVML cannot be loaded it falls back to
    `nvidia-smi -lms 20`.  Nothing here changes a setting of the GPU."""

    PERIOD_S = 0.005
    # nvmlClocksEventReasons bits
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int):
        self.device = device
        self.proc = None
        self.thread = None
        self.rows = []  # (host time, sm MHz, max sm MHz, power W, reason names)
        self.source = None

    def _nvml(self):
        import ctypes
        nvml = ctypes.CDLL("libnvidia-ml.so.1")
        if nvml.nvmlInit_v2() != 0:
            raise OSError("nvmlInit")
        handle = ctypes.c_void_p()
        found = False
        try:  # the CUDA device's PCI address names the same GPU in NVML
            pr = torch.cuda.get_device_properties(self.device)
            bus = b"%08X:%02X:%02X.0" % (pr.pci_domain_id, pr.pci_bus_id, pr.pci_device_id)
            found = nvml.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(handle)) == 0
        except (AttributeError, RuntimeError):
            found = False
        if not found and nvml.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.device), ctypes.byref(handle)) != 0:
            raise OSError("nvmlDeviceGetHandle")
        reasons_fn = getattr(nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        return nvml, handle, reasons_fn

    def _poll(self, nvml, handle, reasons_fn):
        import ctypes
        clk, mx, mw, bits = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while not self.stop_flag:
            t = time.time()
            ok = nvml.nvmlDeviceGetClockInfo(handle, 1, ctypes.byref(clk)) == 0  # NVML_CLOCK_SM
            nvml.nvmlDeviceGetMaxClockInfo(handle, 1, ctypes.byref(mx))
            pw = nvml.nvmlDeviceGetPowerUsage(handle, ctypes.byref(mw)) == 0
            rs = reasons_fn(handle, ctypes.byref(bits)) == 0
            if ok:
                names = [n for b, n in self.REASONS.items() if rs and bits.value & b]
                self.rows.append((t, float(clk.value), float(mx.value), mw.value / 1e3 if pw else None, names))
            time.sleep(self.PERIOD_S)

    def start(self):
        import threading
        self.stop_flag = False
        try:
            nvml, handle, reasons_fn = self._nvml()
            self.thread = threading.Thread(target=self._poll, args=(nvml, handle, reasons_fn), daemon=True)
            self.thread.start()
            self.source = "NVML, 5 ms"
            return
        except (OSError, AttributeError):
            self.thread = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.device), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi, 20 ms"
        except OSError:
            self.proc = None

    def _smi_rows(self):
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        import datetime
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        num = lambda x: float(x) if x.replace(".", "").isdigit() else None  # noqa: E731
        for r in csv.reader(io.StringIO(out)):
            if len(r) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(r[0].strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                continue
            r = [x.strip() for x in r[1:]]
            if num(r[1]) is None:
                continue
            self.rows.append((ts, num(r[1]), num(r[2]), num(r[3]),
                              [names[i] for i in range(4) if r[5 + i] == "Active"]))

    def stop(self, t_begin: float, t_end: float):
        """Summary of the samples taken between host times t_begin and t_end (time.time())."""
        if self.thread is not None:
            self.stop_flag = True
            self.thread.join(timeout=5)
        elif self.proc is not None:
            self._smi_rows()
        else:
            return None
        inside = [r for r in self.rows if t_begin <= r[0] <= t_end]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "source": self.source}
        power = [r[3] for r in inside if r[3] is not None]
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside),
                "power_w_max": max(power) if power else None,
                "reasons": sorted({n for r in inside for n in r[4]}),
                "samples": len(inside), "source": self.source}


def workload(args):
    w = WORKLOADS[args.workload]
    if args.heads:
        from dataclasses import replace
        w = replace(w, H=args.heads, name=f"{w.name}-h{args.heads}")
    return w


def build_schedule_host(w, schedule: str):
    """CSR for non-topology schedules (host-built inputs, copied once before timing)."""
    if schedule == "dense":
        return None
    if schedule.startswith("density:"):
        return random_density_csr(w.nb, float(schedule.split(":")[1]), 0)
    raise ValueError(schedule)


def gpu_builder(schedule: str, w, tsa, k, ws):
    """The schedule build that runs inside every step, as a call writing (row_ptr, col_idx);
    called with no arguments it allocates them and returns them.  None for host-built CSRs."""
    if schedule in ("topology", "topology-content"):
        tie = "content" if schedule == "topology-content" else "index"
        cap = tsa.tsa_schedule_max_nnz(w.S, w.block, w.sink, w.local_radius, w.topk)

        def build(row_ptr=None, col_idx=None):
            if row_ptr is None:
                row_ptr = torch.empty(w.nb + 1, dtype=torch.int32, device=k.device)
                col_idx = torch.empty(cap, dtype=torch.int32, device=k.device)
            tsa.tsa_build_schedule(k, w.block, w.sink, w.local_radius, w.topk, tie_break=tie,
                                   workspace=ws, row_ptr=row_ptr, col_idx=col_idx)
            return row_ptr, col_idx
        return build
    if schedule.startswith("segment:"):
        seg = segment_tokens(schedule)
        nnz = tsa.tsa_fixed_segment_nnz(w.S, w.block, seg)
        L = tsa.lib()

        def build(row_ptr=None, col_idx=None):
            if row_ptr is None:
                row_ptr = torch.empty(w.nb + 1, dtype=torch.int32, device=k.device)
                col_idx = torch.empty(max(nnz, 1), dtype=torch.int32, device=k.device)
            st = L.tsa_fixed_segment_csr(w.S, w.block, seg, row_ptr.data_ptr(), col_idx.data_ptr(),
                                         col_idx.numel(), torch.cuda.current_stream().cuda_stream)
            if st != 0:
                raise tsa.TsaError(st, "tsa_fixed_segment_csr")
            return row_ptr, col_idx
        return build
    return None


def lane_sharded_builder(w, k_local, schedule: str, block_sums, from_sums, gather, world: int, rank: int):
    """The schedule build of a lane-sharded step, as a call writing (row_ptr, col_idx): this
    rank's block sums (block_sums(k, out)), the all-gather of every rank's sums in global lane
    order (gather(sums, counts)), and the CSR built from all of them (from_sums(sums, row_ptr,
    col_idx)).  Every rank holds the workload's B*H lanes.  The three operations are passed in
    so that the same driver runs on the GPU library (NCCL) and in CPU tests (gloo)."""
    counts = [w.lanes] * world

    def build(row_ptr, col_idx):
        local = block_sums(k_local)
        every = gather(local, counts)
        from_sums(every, row_ptr, col_idx)
        return row_ptr, col_idx
    return build


def check_csr_equal(row_ptr, col_idx, ref_row_ptr, ref_col_idx) -> bool:
    """True when two CSRs (torch or numpy, col_idx possibly longer than nnz) are identical."""
    a = np.asarray(row_ptr.cpu() if hasattr(row_ptr, "cpu") else row_ptr)
    b = np.asarray(ref_row_ptr.cpu() if hasattr(ref_row_ptr, "cpu") else ref_row_ptr)
    if a.shape != b.shape or not np.array_equal(a, b):
        return False
    n = int(a[-1])
    ca = np.asarray(col_idx.cpu() if hasattr(col_idx, "cpu") else col_idx)[:n]
    cb = np.asarray(ref_col_idx.cpu() if hasattr(ref_col_idx, "cpu") else ref_col_idx)[:n]
    return np.array_equal(ca, cb)


def run_gpu(args):
    import torch.distributed as dist

    import topology_scheduled_gb300 as tsa

    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = workload(args)
    stream = torch.cuda.current_stream()
    # the CPU generator, as the reference arm draws them; rank r draws shard / problem r
    q, k, v = (x.to(dev) for x in make_qkv(w, seed=rank, device="cpu"))
    torch.cuda.synchronize()
    out = torch.empty_like(q)
    topo = built_in_step(args.schedule)
    sharded = world > 1 and args.shard == "lanes" and args.schedule in ("topology", "topology-content")
    lanes_built = w.lanes * world if sharded else w.lanes
    ws = torch.empty(tsa.tsa_build_schedule_workspace_bytes(lanes_built, w.S, w.D, w.block),
                     dtype=torch.uint8, device=dev)
    if sharded:
        from topology_scheduled_gb300.distributed import gather_block_sums
        tie = "content" if args.schedule == "topology-content" else "index"
        sums_local = torch.empty((w.lanes, w.nb, w.D), dtype=torch.float64, device=dev)
        cap = tsa.tsa_schedule_max_nnz(w.S, w.block, w.sink, w.local_radius, w.topk)
        build_fn = lane_sharded_builder(
            w, k, args.schedule,
            block_sums=lambda kk: tsa.tsa_block_sums(kk, w.block, out=sums_local),
            from_sums=lambda sums, rp, ci: tsa.tsa_build_schedule_from_sums(
                sums, w.block, w.sink, w.local_radius, w.topk, S=w.S, tie_break=tie, workspace=ws,
                row_ptr=rp, col_idx=ci),
            gather=lambda sums, counts: gather_block_sums(sums, counts=counts),
            world=world, rank=rank)

        def build(row_ptr=None, col_idx=None):
            if row_ptr is None:
                row_ptr = torch.empty(w.nb + 1, dtype=torch.int32, device=dev)
                col_idx = torch.empty(cap, dtype=torch.int32, device=dev)
            return build_fn(row_ptr, col_idx)
    else:
        build = gpu_builder(args.schedule, w, tsa, k, ws)
    if topo:
        row_ptr, col_idx = build()
    elif args.schedule == "dense":
        row_ptr, col_idx = tsa.tsa_dense_causal_csr(w.S, w.block, device=dev)
    else:
        rp, ci = build_schedule_host(w, args.schedule)
        row_ptr, col_idx = torch.as_tensor(rp, device=dev), torch.as_tensor(ci, device=dev)

    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    def step(attn_events=None, build_events=None):
        if topo:
            if build_events:
                build_events[0].record(stream)
            build(row_ptr, col_idx)
            if build_events:
                build_events[1].record(stream)
        if attn_events:
            attn_events[0].record(stream)
        tsa.tsa_scheduled_attention(q, k, v, row_ptr, col_idx, w.scale, out=out)
        if attn_events:
            attn_events[1].record(stream)

    step()
    status = tsa.tsa_last_device_status()
    if status != 0:
        raise RuntimeError(f"device status {tsa.STATUS_NAMES.get(status, status)}")
    shard_check = None
    if sharded:
        shard_check = verify_lane_sharded_csr(w, tsa, k, row_ptr, col_idx, args.schedule, world, rank, dev)
    nnz = int(row_ptr[-1].item())
    flops = visited_flops(nnz, w.lanes, w.D, w.block)
    if args.pass_ == "bwd":
        return run_backward(args, w, tsa, q, k, v, row_ptr, col_idx, nnz, dev, world, rank, local)
    n_launch = launches_per_step(args.schedule)
    for _ in range(max(args.warmup, 0)):
        step()
    torch.cuda.synchronize()

    attn_ev = [(ev(), ev()) for _ in range(args.steps)]
    build_ev = [(ev(), ev()) for _ in range(args.steps)] if topo else [None] * args.steps
    # Inputs that L2 could hold get it flushed before every step (a write larger than L2, outside
    # the step's own events); the step time is then the sum of the per-step events.
    in_bytes = 4 * q.numel() * q.element_size()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev) if in_bytes < L2_FLUSH_BYTES else None
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.05)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0, t1 = ev(), ev()
    wall0 = time.perf_counter()
    host0 = time.time()
    t0.record(stream)
    for i in range(args.steps):
        if flush is not None:
            flush.fill_(i & 0xFF)
        step(attn_ev[i], build_ev[i])
    t1.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    host1 = time.time()
    if world > 1:
        dist.barrier()
    clk = clocks.stop(host0, host1)
    status = tsa.tsa_last_device_status()
    if status != 0:
        raise RuntimeError(f"device status after timing {tsa.STATUS_NAMES.get(status, status)}")
    elapsed_ms = t0.elapsed_time(t1)
    attn_ms = [a.elapsed_time(b) for a, b in attn_ev]
    build_ms = [a.elapsed_time(b) for a, b in build_ev] if topo else [0.0]
    if flush is not None:
        elapsed_ms = sum(attn_ms) + sum(build_ms)
    region_ms = elapsed_ms
    elapsed_ms, flops_all = aggregate_over_ranks(elapsed_ms, flops, dev, world)
    ms_per_step = elapsed_ms / args.steps
    value = flops_all * args.steps / (elapsed_ms * 1e-3) / 1e12

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, w, tsa, q, k, v, out, build, row_ptr, col_idx, topo, flops, stream, world,
                      sharded)

    peaks, peak_kind = measured_peaks()
    attn_mean = statistics.mean(attn_ms)
    achieved = flops / (attn_mean * 1e-3) / 1e12
    # the attention launches run inside a region of region_ms: that length picks the tensor peak
    peak, peak_desc = tensor_peak(peaks, peak_kind, region_ms)
    burst = float(peaks.get("bf16_tflops", peak))
    sustained = float(peaks.get("bf16_tflops_sustained", peak))
    if w.dtype == torch.float16:
        pass  # dense f16 and bf16 tensor rates are the same on this part
    traffic = attention_traffic_per_launch(args.workload, args.schedule) if not args.heads else None
    # Compulsory bytes of one attention launch: Q, K, V read and O written once per lane, plus the CSR.
    alg_bytes = 4 * q.numel() * q.element_size() + 4 * (w.nb + 1) + 4 * nnz
    hbm_peak = float(peaks["hbm_gbs"])
    achieved_gbs = alg_bytes / (attn_mean * 1e-3) / 1e9
    # The kernel is bound by whichever roof is lower at its arithmetic intensity.
    hbm_bound = flops / alg_bytes < peak * 1e12 / (hbm_peak * 1e9)
    if sharded:
        parallelism = (f"lane-sharded x{world}: {w.lanes} lanes per rank, block sums all-gathered over "
                       f"NCCL in lane order inside the step, one CSR built on every rank")
    else:
        parallelism = f"independent problem per rank x{world} (no collective)"
    line = {
        "metric": "scheduled-attn fwd TFLOP/s on visited blocks (% of GB300 bf16 peak); ms/call",
        "value": round(value, 3),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": dtype_name(w.dtype),
        "data": "synthetic (seeded N(0,1) Q/V, clustered K, drawn by the CPU generator; no dataset)",
        "config": {
            "workload": f"{w.name}: {w.describe()}",
            "schedule": args.schedule,
            "B": w.B * (world if sharded else 1), "H": w.H, "S": w.S, "D": w.D, "block": w.block,
            "lanes_per_rank": w.lanes,
            "nnz_blocks": nnz, "dense_blocks": w.nb * (w.nb + 1) // 2,
            "visited_flops_per_step": flops,
            "l2": ("inputs larger than L2 (Q,K,V,O %.2f GB per rank), no flush" % (in_bytes / 1e9)
                   if flush is None else
                   "L2 flushed before every step (%d MB written outside the step's events; Q,K,V,O %.1f MB)"
                   % (L2_FLUSH_BYTES >> 20, in_bytes / 1e6)),
            "parallelism": parallelism,
        },
        "breakdown": {
            "attention_ms": round(attn_mean, 4),
            "attention_tflops": round(achieved, 3),
            "build_ms": round(statistics.mean(build_ms), 4),
            "pct_of_bf16_peak_step": round(100.0 * value / world / peak, 2),
            "timed_region_ms": round(region_ms, 3),
            "wall_s_timed_region": round(wall, 3),
        },
        "roofline": {
            "kernel": "scheduled_attention_kernel",
            "bound": "hbm" if hbm_bound else "tensor",
            "achieved": round(achieved_gbs if hbm_bound else achieved, 3),
            "peak": hbm_peak if hbm_bound else peak,
            "unit": "GB/s" if hbm_bound else "TFLOP/s",
            "frac": round(achieved_gbs / hbm_peak if hbm_bound else achieved / peak, 4),
            "peak_source": (f"{peak_kind} hbm_gbs (copy, read + write bytes)" if hbm_bound else peak_desc),
            "traffic": traffic,
            "algorithmic_bytes": alg_bytes,
            "flop_per_byte": round(flops / alg_bytes, 1),
            "tensor_frac_burst": round(achieved / burst, 4),
            "tensor_frac_sustained": round(achieved / sustained, 4),
            "other_roof": ({"unit": "TFLOP/s", "achieved": round(achieved, 3), "frac": round(achieved / peak, 4)}
                           if hbm_bound else
                           {"unit": "GB/s", "achieved": round(achieved_gbs, 1),
                            "frac": round(achieved_gbs / hbm_peak, 4)}),
        },
        "gpu_launches": n_launch * args.steps,
        "clocks": clk,
        "e2e": e2e,
    }
    if shard_check is not None:
        line["config"]["csr_check"] = shard_check
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        bl = cpu_baseline(args, w, q.cpu(), k.cpu(), v.cpu(), row_ptr, col_idx, topo)
        bl.pop("_build")
        line["cpu_baseline"] = bl
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def verify_lane_sharded_csr(w, tsa, k, row_ptr, col_idx, schedule, world, rank, dev):
    """Before timing: every rank's CSR equals rank 0's, and rank 0's equals the CSR one GPU
    builds from all lanes' keys (gathered to rank 0).  Raises on a mismatch."""
    import torch.distributed as dist
    tie = "content" if schedule == "topology-content" else "index"
    ref_rp = row_ptr.clone()
    ref_ci = col_idx.clone()
    dist.broadcast(ref_rp, 0)
    dist.broadcast(ref_ci, 0)
    same = torch.tensor([1 if check_csr_equal(row_ptr, col_idx, ref_rp, ref_ci) else 0], device=dev)
    dist.all_reduce(same, op=dist.ReduceOp.MIN)
    if int(same.item()) != 1:
        raise RuntimeError("lane-sharded CSR differs between ranks")
    gathered = [torch.empty_like(k) for _ in range(world)] if rank == 0 else None
    dist.gather(k.contiguous(), gathered, dst=0)
    ok = True
    if rank == 0:
        every = torch.cat([g.reshape(-1, w.S, w.D) for g in gathered], dim=0)
        del gathered
        rp1, ci1 = tsa.tsa_build_schedule(every, w.block, w.sink, w.local_radius, w.topk, tie_break=tie)
        ok = check_csr_equal(row_ptr, col_idx, rp1, ci1)
        del every
    flag = torch.tensor([1 if ok else 0], device=dev)
    dist.broadcast(flag, 0)
    if int(flag.item()) != 1:
        raise RuntimeError("lane-sharded CSR differs from the single-GPU build over all lanes")
    torch.cuda.empty_cache()
    return f"identical on all {world} ranks and to the single-GPU build over all {w.lanes * world} lanes"


L2_FLUSH_BYTES = 256 << 20  # twice the 129 MB L2
BWD_LAUNCHES = 7  # bwd_rows, bwd_col_count, bwd_col_scan, bwd_col_fill, bwd_delta, bwd_dq, bwd_dkv


def run_backward(args, w, tsa, q, k, v, row_ptr, col_idx, nnz, dev, world, rank, local):
    """--pass bwd: time tsa_scheduled_attention_backward alone (schedule built once before)."""
    import torch.distributed as dist

    stream = torch.cuda.current_stream()
    O, lse = tsa.tsa_scheduled_attention_fwd(q, k, v, row_ptr, col_idx, w.scale)
    g = torch.Generator().manual_seed(1000 + rank)
    dO = torch.randn(q.shape, generator=g, dtype=torch.float32).to(q.dtype).to(dev)
    ws = torch.empty(tsa.tsa_attention_backward_workspace_bytes(w.lanes, w.S, w.block, col_idx.numel()),
                     dtype=torch.uint8, device=dev)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))

    def step():
        tsa.tsa_scheduled_attention_backward(q, k, v, O, dO, lse, row_ptr, col_idx, w.scale,
                                             dq=dq, dk=dk, dv=dv, workspace=ws)

    step()
    status = tsa.tsa_last_device_status()
    if status != 0:
        raise RuntimeError(f"device status {tsa.STATUS_NAMES.get(status, status)}")
    for _ in range(max(args.warmup, 0)):
        step()
    torch.cuda.synchronize()
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.05)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0, t1 = ev(), ev()
    host0 = time.time()
    t0.record(stream)
    for _ in range(args.steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    host1 = time.time()
    if world > 1:
        dist.barrier()
    clk = clocks.stop(host0, host1)
    status = tsa.tsa_last_device_status()
    if status != 0:
        raise RuntimeError(f"device status after timing {tsa.STATUS_NAMES.get(status, status)}")
    flops = 2.5 * visited_flops(nnz, w.lanes, w.D, w.block)
    region_ms = t0.elapsed_time(t1)
    elapsed_ms, flops_all = aggregate_over_ranks(region_ms, flops, dev, world)
    ms = elapsed_ms / args.steps
    value = flops_all * args.steps / (elapsed_ms * 1e-3) / 1e12
    peaks, peak_kind = measured_peaks()
    peak, peak_desc = tensor_peak(peaks, peak_kind, region_ms)
    achieved = flops / (ms * 1e-3) / 1e12
    line = {
        "metric": "scheduled-attn bwd TFLOP/s on visited blocks (5 block products); ms/call",
        "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": dtype_name(w.dtype),
        "data": "synthetic (seeded N(0,1) Q/V/dO, clustered K; no dataset)",
        "config": {
            "workload": f"{w.name}: {w.describe()}", "schedule": args.schedule, "pass": "bwd",
            "B": w.B, "H": w.H, "S": w.S, "D": w.D, "block": w.block, "nnz_blocks": nnz,
            "visited_flops_per_step": flops,
            "l2": "inputs larger than L2 (Q,K,V,O,dO %.2f GB per rank), no flush"
                  % (5 * q.numel() * q.element_size() / 1e9),
            "parallelism": f"independent problem per rank x{world} (no collective)",
        },
        "roofline": {
            "kernel": "tsa_scheduled_attention_backward (all launches of the call)",
            "bound": "tensor", "achieved": round(achieved, 3), "peak": peak, "unit": "TFLOP/s",
            "frac": round(achieved / peak, 4),
            "peak_source": peak_desc,
            "traffic": None,
        },
        "gpu_launches": BWD_LAUNCHES * args.steps,
        "clocks": clk,
        "e2e": None,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_backward(args, w, q, k, v, dO, row_ptr, col_idx, nnz)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def cpu_baseline_backward(args, w, q, k, v, dO, row_ptr, col_idx, nnz):
    """The fp64 CPU oracle's backward on whole lanes, one at a time until the time budget."""
    import oracle

    threads = os.cpu_count() or 1
    S, D = w.S, w.D
    rp = row_ptr.cpu().numpy()
    ci = col_idx.cpu().numpy()[: rp[-1]]
    sl = lambda t, i: t.reshape(-1, S, D)[i:i + 1].cpu()  # noqa: E731
    done, spent = 0, 0.0
    while done < w.lanes and spent < args.cpu_seconds:
        a = [sl(t, done) for t in (q, k, v, dO)]
        t0 = time.perf_counter()
        oracle.attention_backward(*a, rp, ci, w.block, w.scale, nthreads=threads)
        spent += time.perf_counter() - t0
        done += 1
    step_s = spent * w.lanes / done
    flops_all = 2.5 * visited_flops(nnz, w.lanes, D, w.block)
    return {"value": round(flops_all / step_s / 1e12, 6), "unit": "TFLOP/s", "cores": threads,
            "kind": "oracle",
            "sample": f"backward of {done} of {w.lanes} lanes ({spent:.1f} s), extrapolated by lanes; "
                      f"step estimate {step_s:.1f} s"}


def run_e2e(args, w, tsa, q, k, v, out, build, row_ptr, col_idx, topo, flops, stream, world, sharded=False):
    """Same step through the public API from pinned host buffers, copies inside the timing.
    Topology schedules go through tsa_topology_attention_host (the C-ABI call that takes host
    buffers and overlaps its copies with the build and the attention); the others copy with
    torch around the device-resident calls."""
    steps = max(1, min(args.steps, 5))
    hq, hk, hv = (x.cpu().pin_memory() for x in (q, k, v))
    ho = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    hnnz = torch.empty(1, dtype=torch.int32, pin_memory=True)
    # lane-sharded: the host buffers are this rank's lanes; the build needs every rank's block
    # sums, so the step is the torch copies around the device calls (exchange included)
    host_call = args.schedule in ("topology", "topology-content") and not sharded
    if host_call:
        ws = torch.empty(tsa.tsa_build_schedule_workspace_bytes(w.lanes, w.S, w.D, w.block),
                         dtype=torch.uint8, device=q.device)
        tie = "content" if args.schedule == "topology-content" else "index"

        def step():
            tsa.tsa_topology_attention_host(hq, hk, hv, w.block, w.sink, w.local_radius, w.topk, w.scale,
                                            tie_break=tie, out=ho, device_buffers=(q, k, v, out),
                                            row_ptr=row_ptr, col_idx=col_idx, workspace=ws)
    else:
        def step():
            q.copy_(hq, non_blocking=True)
            k.copy_(hk, non_blocking=True)
            v.copy_(hv, non_blocking=True)
            if topo:
                build(row_ptr, col_idx)
            tsa.tsa_scheduled_attention(q, k, v, row_ptr, col_idx, w.scale, out=out)
            ho.copy_(out, non_blocking=True)
            hnnz.copy_(row_ptr[-1:], non_blocking=True)

    step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    h2d = 3 * q.numel() * q.element_size()
    d2h = out.numel() * out.element_size() + (0 if host_call else 4)
    return {"value": round(flops * world / (ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
            "ms_per_step": round(ms, 3), "steps": steps,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "call": "tsa_topology_attention_host" if host_call else "torch copies + device calls"}


def cpu_baseline(args, w, q, k, v, row_ptr, col_idx, topo, reuse_build=None):
    """The fp64 CPU oracle on the host cores: full schedule build + a sample of attention rows.
    `reuse_build` = (seconds, row_ptr, col_idx) of a build already timed on this workload: the
    build is then not run again (it is deterministic) and its measured time is counted."""
    import oracle

    threads = os.cpu_count() or 1
    S, D = w.S, w.D
    kh = k.reshape(-1, S, D)
    t0 = time.perf_counter()
    if reuse_build is not None:
        _, rp, ci = reuse_build
    elif args.schedule.startswith("segment:"):
        rp, ci = oracle.fixed_segment_csr(S, w.block, segment_tokens(args.schedule))
    elif topo:
        tie = "content" if args.schedule == "topology-content" else "index"
        rp, ci, _ = oracle.build_schedule(kh, w.block, w.sink, w.local_radius, w.topk, tie=tie)
    else:
        rp = row_ptr.cpu().numpy()
        ci = col_idx.cpu().numpy()[: rp[-1]]
    t_build = reuse_build[0] if reuse_build is not None else time.perf_counter() - t0
    rng = np.random.default_rng(0)
    qh, vh = q.reshape(-1, S, D), v.reshape(-1, S, D)
    lens = np.diff(rp).astype(np.float64)
    n = 512
    done_rows, done_flops, t_attn = 0, 0.0, 0.0
    while t_attn < args.cpu_seconds:
        lanes = rng.integers(0, w.lanes, n).astype(np.int64)
        toks = rng.integers(0, S, n).astype(np.int64)
        t1 = time.perf_counter()
        oracle.attention(qh, kh, vh, rp, ci, w.block, w.scale, lanes=lanes, tokens=toks, nthreads=threads)
        t_attn += time.perf_counter() - t1
        done_rows += n
        done_flops += float(np.sum(lens[toks // w.block])) * 4.0 * w.block * D
        n = min(n * 2, 65536)
    total_rows = w.lanes * S
    flops_all = visited_flops(int(rp[-1]), w.lanes, D, w.block)
    attn_full_s = t_attn * (flops_all / done_flops)
    step_s = t_build + attn_full_s
    build_note = "timed on an earlier step, not rerun" if reuse_build is not None else "timed"
    return {"value": round(flops_all / step_s / 1e12, 6), "unit": "TFLOP/s", "cores": threads,
            "kind": "oracle",
            "sample": (f"full schedule build ({1e3 * t_build:.1f} ms, {build_note}) + {done_rows} attention "
                       f"rows drawn uniformly with replacement from the {total_rows} of the workload "
                       f"({t_attn:.1f} s), attention extrapolated by visited FLOPs; step estimate "
                       f"{1e3 * step_s:.1f} ms"),
            "_build": (t_build, rp, ci)}


def run_reference(args):
    """--impl reference: the CPU oracle on this workload (rank 0 only)."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    w = workload(args)
    topo = built_in_step(args.schedule)
    q, k, v = make_qkv(w, seed=0, device="cpu")
    if topo:
        rp = ci = None
    elif args.schedule == "dense":
        import oracle
        rp, ci = oracle.dense_causal_csr(w.nb)
    else:
        rp, ci = build_schedule_host(w, args.schedule)
    # each step is a bounded sample, so that warm-up + steps stay within a few minutes: the
    # attention rows get the per-step budget, and the schedule build (deterministic) is run
    # again only while it costs at most half of that budget, else its first timing is reused
    budget = 120.0 / max(1, args.warmup + args.steps)
    args.cpu_seconds = budget
    times, bl, reuse = [], None, None
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        bl = cpu_baseline(args, w, q, k, v, torch.as_tensor(rp) if rp is not None else None,
                          torch.as_tensor(ci) if ci is not None else None, topo, reuse_build=reuse)
        build = bl.pop("_build")
        if reuse is None and build[0] > 0.5 * budget:
            reuse = build
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    line = {
        "impl": "reference",
        "metric": "scheduled-attn fwd TFLOP/s on visited blocks (% of GB300 bf16 peak); ms/call",
        "value": bl["value"], "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded; the same CPU-generated tensors as the GPU arm)",
        "config": {"workload": f"{args.workload}: {w.describe()}", "schedule": args.schedule},
        "ms_per_step_sample": round(1e3 * statistics.mean(times), 1),
        "cpu_baseline": bl,
        "e2e": {"value": bl["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()

"""Benchmark of the fused NVFP4 linear-layer path on B300.

One step = one pass of the whole hot path over one batch of DiT-block activations at
M = 4608 tokens, with the weights already packed (offline) and resident in HBM:
    quantize X [4608, 3072]  -> QKV GEMM [x3072 -> 9216]   + per-head RMSNorm epilogue
    quantize X [4608, 3072]  -> up  GEMM [x3072 -> 24576]  + gated-SiLU epilogue (-> 12288)
    quantize X [4608, 12288] -> down GEMM [x12288 -> 3072] + bias epilogue
Every op is a kernel of libnvfp4.so called through the C ABI: 6 launches per step (each
activation quantized by one single-pass launch -- the down-projection input with a quarter
of its rows held in shared memory between the amax and the encode, the rest read twice --
and the three GEMMs).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0). `--impl reference` times the CPU oracle (test code, the
slow obviously-correct definition) on a bounded row sample of the same workload.
Multi-GPU (torchrun, N > 1) runs N independent replicas: the path has no exchange step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused NVFP4 GEMM+epilogue TFLOPS at M=4608 and % of B300 dense FP4 peak"
UNIT = "TFLOP/s"
NOMINAL_FP4_PF = 15.0          # B300 dense FP4 (NVIDIA's Blackwell Ultra figure)
FP4_OVER_BF16 = 13.5 / 2.25    # nominal dense FP4 : BF16 ratio used to scale the measured peak
FLUSH_BYTES = 256 << 20        # > 126 MB L2


class L2Flush:
    """Evicts L2 between timed steps: a 256 MiB write (every line of the step's inputs and
    outputs is evicted), then a read of a second 256 MiB buffer, which writes those dirty flush
    lines back to HBM outside the timed region and leaves L2 holding clean lines only, so no
    step pays for write-back traffic that is not its own."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(FLUSH_BYTES // 4, dtype=torch.int32, device=dev)

    def __call__(self):
        self.w.zero_()
        self.r.max()
WORKLOAD_NAME = ("dit_block_linears_m4608: qkv+head_rmsnorm [4608x3072x9216], "
                 "up+gated_silu [4608x3072x24576], down+bias [4608x12288x3072], "
                 "each with its bf16->nvfp4 activation quantize")


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-rows", type=int, default=16, help="oracle rows sampled per GEMM")
    p.add_argument("--only", choices=["qkv_rmsnorm", "gated_up", "down_bias"], default=None,
                   help="run one of the three layers only (for profiler captures)")
    p.add_argument("--chain", action="store_true",
                   help="up-projection -> down-projection at M=4608: fused NVFP4 output vs bf16 + quantize")
    p.add_argument("--fp8", action="store_true",
                   help="the three DiT GEMMs at M=4608 with FP8 (E4M3) operands: quantize + GEMM times")
    p.add_argument("--spin-up-ms", type=float, default=300.0,
                   help="--fp8, --attention: keep the GPU busy this long before timing (clocks settle)")
    p.add_argument("--attention", action="store_true",
                   help="attention at 4608 tokens x 12 heads x 256: this package's kernel vs torch's")
    p.add_argument("--attention-impl", choices=["kernel", "torch"], default="kernel",
                   help="--dit-block: which attention the block uses")
    p.add_argument("--dit-block", action="store_true",
                   help="one DiT block's linears chained at 4608 tokens: per-stage CUDA-event times")
    p.add_argument("--sweep", action="store_true",
                   help="batch sweep: one JSON line per (M, GEMM), M in 512..18432")
    p.add_argument("--mma-ceiling", action="store_true",
                   help="tensor-pipe rate of tcgen05.mma (NVFP4 / FP8 / BF16 kinds, cta_group 1/2, N 64..256): "
                        "cycles per instruction on one SM and on all SMs")
    p.add_argument("--probe-iters", type=int, default=20000)
    return p.parse_args(argv)


# ---------------------------------------------------------------------------------------
# Distributed plumbing (replicas only): max of the per-rank time, sum of the units.
# ---------------------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def aggregate(elapsed_s: float, units: float, dist=None):
    """(max elapsed over ranks, total units over ranks). Works on gloo and nccl groups."""
    if dist is None:
        return elapsed_s, units
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


# ---------------------------------------------------------------------------------------
# Clock sampling during the timed region (NVML, 10 ms period).
# ---------------------------------------------------------------------------------------

class _Nvml:
    """Minimal ctypes binding of the NVML calls the sampler needs (libnvidia-ml.so.1)."""
    CLOCK_SM = 1

    def __init__(self, index: int):
        import ctypes
        self.c = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        self._ok(self.lib.nvmlInit_v2())
        self.h = ctypes.c_void_p()
        self._ok(self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.h)))

    def _ok(self, rc):
        if rc != 0:
            raise RuntimeError(f"NVML error {rc}")

    def clock(self, max_clock=False) -> int:
        v = self.c.c_uint()
        f = self.lib.nvmlDeviceGetMaxClockInfo if max_clock else self.lib.nvmlDeviceGetClockInfo
        self._ok(f(self.h, self.c.c_int(self.CLOCK_SM), self.c.byref(v)))
        return int(v.value)

    def reasons(self) -> int:
        v = self.c.c_ulonglong()
        f = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self._ok(f(self.h, self.c.byref(v)))
        return int(v.value)


class ClockSampler:
    """Samples the SM clock and the clock-event (throttle) reasons every `period_s` during the
    timed region, through NVML (ctypes); falls back to nvidia-smi if NVML cannot be loaded."""
    REASONS = {
        "sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
        "hw_thermal_slowdown": 0x40, "hw_power_brake_slowdown": 0x80,
    }
    SMI_FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
                  "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                  "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, period_s: float = 0.002):
        self.samples, self.reasons, self.max_mhz = [], set(), None
        self.period = period_s
        self.error = None
        self.index = index
        self._stop = threading.Event()
        try:
            self.nv = _Nvml(index)
            self.max_mhz = self.nv.clock(max_clock=True)
        except Exception as e:
            self.nv = None
            self.error = f"nvml: {type(e).__name__}: {e}"

    def _run(self):
        while not self._stop.is_set():
            self._sample()
            time.sleep(self.period)

    def _sample(self):
        try:
            if self.nv is not None:
                self.samples.append(self.nv.clock())
                r = self.nv.reasons()
                for name, bit in self.REASONS.items():
                    if r & bit:
                        self.reasons.add(name)
            else:
                import subprocess
                out = subprocess.run(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.SMI_FIELDS,
                                      "--format=csv,noheader,nounits"], capture_output=True, text=True,
                                     timeout=5).stdout.strip().split(",")
                self.samples.append(float(out[0]))
                self.max_mhz = float(out[1])
                for name, v in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                                    "sw_power_cap"), out[2:]):
                    if v.strip() == "Active":
                        self.reasons.add(name)
        except Exception as e:
            self.error = f"{type(e).__name__}: {e}"

    def __enter__(self):
        self._sample()
        self.t = threading.Thread(target=self._run, daemon=True)
        self.t.start()
        return self

    def __exit__(self, *exc):
        self._stop.set()
        self.t.join()
        self._sample()

    def summary(self):
        s = {"sm_mhz": statistics.median(self.samples) if self.samples else None,
             "sm_min_mhz": min(self.samples) if self.samples else None,
             "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons),
             "samples": len(self.samples), "source": "nvml" if self.nv is not None else "nvidia-smi"}
        if self.error:
            s["error"] = self.error
        return s


# ---------------------------------------------------------------------------------------
# The GPU arm
# ---------------------------------------------------------------------------------------

KERNEL_SOURCES = {"gemm": ("gemm.cu", "nvfp4_device.cuh"), "quantize": ("quantize.cu", "nvfp4_device.cuh")}


def kernel_source_hash(op: str) -> str:
    """Hash of the CUDA sources that build `op`'s kernels ("gemm_*" or "quantize_*")."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES["gemm" if op.startswith("gemm") else "quantize"]:
        with open(os.path.join(ROOT, "nvfp4_gemm_act_b300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def read_traffic(op: str):
    """(DRAM bytes per launch of `op`, their provenance) from the committed ncu summary if it
    was taken on the current kernel sources (the file records the source hash); else
    (None, why)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    src = kernel_source_hash(op)
    if os.path.exists(path):
        for line in open(path):
            parts = line.split()
            if len(parts) >= 3 and not line.startswith("#") and parts[0] == op and parts[1] == src:
                return float(parts[2]), (f"ncu capture (dram__bytes_read.sum + dram__bytes_write.sum, one launch) "
                                         f"recorded in profiles/dram_traffic.txt for kernel-source hash {src}")
    return None, f"no ncu capture recorded for kernel-source hash {src}"


def spin_ahead(torch):
    """~1 ms of device spin ahead of a timed region: the host enqueues the region's launches
    (and its closing event) before the GPU reaches them, so an event pair times the device
    work only, not the host's launch overhead."""
    torch.cuda._sleep(2_000_000)


def instruction_ceiling(nv, torch, dev, iters=20000):
    """The NVFP4 MMA instruction ceiling measured now (nvfp4_debug_mma_rate): back-to-back
    tcgen05.mma kind::mxf4nvf4.block16 M256 N256 K64 on every SM pair; TFLOP/s = FLOPs of all
    pairs / the slowest pair's time."""
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    pairs = sms // 2
    nv.nvfp4_debug_mma_rate("nvfp4", 2, 256, iters, pairs)  # warm-up
    r = nv.nvfp4_debug_mma_rate("nvfp4", 2, 256, iters, pairs)
    torch.cuda.synchronize()
    r = r.cpu().numpy()
    flops = 2.0 * 256 * 256 * 64 * iters * pairs
    return flops / (float(r[:, 1].max()) * 1e-9) / 1e12


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            return json.load(fh), "measured"
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}, "fallback"


class Layer:
    """One DiT linear: resident packed weights + buffers for its activation and output."""

    def __init__(self, w, dev):
        import torch

        import nvfp4_gemm_act_b300 as nv
        from nvfp4_gemm_act_b300 import workloads as W
        self.w = w
        self.x = W.make_x(w).to(dev)
        self.qb = nv.nvfp4_pack_weights(W.make_w(w).to(dev), gated_interleave=w.epilogue == "gated_silu")
        b, g = W.make_bias(w), W.make_gamma(w)
        self.bias = None if b is None else b.to(dev)
        self.gamma = None if g is None else g.to(dev)
        self.qa = nv._alloc_nvfp4(w.M, w.K, dev)
        self.ws = torch.zeros(16, dtype=torch.uint8, device=dev)
        self.out = torch.empty((w.M, w.out_cols), dtype=torch.bfloat16, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)

    def quantize(self):
        import nvfp4_gemm_act_b300 as nv
        nv.nvfp4_quantize(self.x, out=self.qa, workspace=self.ws)

    def gemm(self):
        import nvfp4_gemm_act_b300 as nv
        w = self.w
        nv.nvfp4_gemm(self.qa, self.qb, w.epilogue, bias=self.bias, gamma=self.gamma,
                      head_dim=w.head_dim, norm_cols=w.norm_cols, eps=w.eps, out=self.out,
                      device_error=self.err)


def run_ours(args, world, rank, local):
    import torch

    import nvfp4_gemm_act_b300 as nv
    from nvfp4_gemm_act_b300 import workloads as W

    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    dist = init_dist(world, "nccl")
    nv.lib()
    layers = [Layer(w, dev) for w in (W.QKV_RMSNORM, W.GATED_UP, W.DOWN_BIAS)
              if args.only is None or w.name == args.only]
    flops_step = sum(l.w.flops for l in layers)
    flush = L2Flush(dev)
    ops = []  # (name, callable, flops, algorithmic bytes)
    for l in layers:
        w = l.w
        # algorithmic bytes: read X once (2 B/element), write codes (0.5) + scales (1/16)
        ops.append((f"quantize_{w.name}", l.quantize, 0, w.M * w.K * 2 + w.M * w.K // 2 + w.M * w.K // 16))
        gbytes = (w.M * w.K // 2 + w.M * w.K // 16 + w.N * w.K // 2 + w.N * w.K // 16
                  + w.M * w.out_cols * 2)
        ops.append((f"gemm_{w.name}", l.gemm, w.flops, gbytes))
    # launches per step: the GEMM, and the quantizer's one (single-pass: one CTA per SM, at
    # least a quarter of each CTA's rows held in 200 KB of shared memory) or two (amax, quantize)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count

    def quantize_launches(M, K):
        rows = -(-(-(-M // 128) * 128) // sms)
        resident = min(rows, (200 * 1024) // (K * 2))
        return 1 if resident >= 1 and resident * 4 >= rows else 2

    kernels_per_step = sum(1 + quantize_launches(l.w.M, l.w.K) for l in layers)

    def step(evs=None):
        for i, (_, fn, _, _) in enumerate(ops):
            if evs is not None:
                evs[i].record()
            fn()
        if evs is not None:
            evs[len(ops)].record()

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    for l in layers:
        assert nv.nvfp4_get_device_error(l.err) == 0

    K = args.steps
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(len(ops) + 1)] for _ in range(K)]
    barrier(dist)
    torch.cuda.synchronize()
    try:
        nvml_index = torch.cuda._get_nvml_device_index(local)
    except Exception:
        nvml_index = local
    # pass 1 (eager, an event before every launch): the per-kernel breakdown and the roofline.
    # A ~1 ms device spin ahead of each step lets the host enqueue the whole step before the
    # GPU reaches it, so the launches run back to back (as in the graph replay) and each event
    # difference is device time only, not host launch overhead.
    for k in range(K):
        flush()                    # evict L2 between steps (outside the timed events)
        spin_ahead(torch)
        step(events[k])
    torch.cuda.synchronize()
    per_op = np.array([[events[k][i].elapsed_time(events[k][i + 1]) for i in range(len(ops))]
                       for k in range(K)])  # ms
    eager_step_ms = per_op.sum(axis=1)
    # pass 2, the timed steps: the same step captured once as a CUDA graph and replayed, so no
    # host work sits between its launches; `value` comes from these K steps
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(max(args.warmup, 3)):
        flush()
        graph.replay()
    gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    barrier(dist)
    torch.cuda.synchronize()
    with ClockSampler(nvml_index) as clocks:
        for k in range(K):
            flush()                    # evict L2 between steps (outside the timed events)
            spin_ahead(torch)
            gev[k][0].record()
            graph.replay()
            gev[k][1].record()
        torch.cuda.synchronize()
    barrier(dist)
    step_ms = np.array([e0.elapsed_time(e1) for e0, e1 in gev])
    elapsed_s = float(step_ms.sum()) / 1e3
    for l in layers:
        assert nv.nvfp4_get_device_error(l.err) == 0
    t_max, units = aggregate(elapsed_s, flops_step * K, dist)
    value = units / t_max / 1e12

    peaks, peaks_src = measured_peaks()
    fp4_peak = peaks["bf16_tflops"] * FP4_OVER_BF16
    mean_op = per_op.mean(axis=0)
    dom = int(np.argmax(mean_op))
    dom_name, _, dom_flops, dom_bytes = ops[dom]
    achieved = dom_flops / (mean_op[dom] / 1e3) / 1e12
    breakdown = {}
    for i, (name, _, fl, by) in enumerate(ops):
        ms = float(mean_op[i])
        e = {"ms": round(ms, 5)}
        if fl:
            e["tflops"] = round(fl / (ms / 1e3) / 1e12, 1)
            e["frac_of_15pf"] = round(fl / (ms / 1e3) / 1e12 / (NOMINAL_FP4_PF * 1e3), 4)
        else:
            e["gbs"] = round(by / (ms / 1e3) / 1e9, 1)
            e["frac_of_hbm_measured"] = round(by / (ms / 1e3) / 1e9 / peaks["hbm_gbs"], 4)
        breakdown[name] = e
    gemm_ms = sum(mean_op[i] for i, o in enumerate(ops) if o[2])
    traffic, traffic_source = read_traffic(dom_name)
    ceiling = instruction_ceiling(nv, torch, dev)
    # the down-projection input's quantizer with a static tensor scale (one streaming pass; the
    # step uses the dynamic scale: one launch that reads x once for the amax and again, except
    # the rows it keeps in shared memory, to encode), timed alone, L2 flushed first
    down = [l for l in layers if l.w.name == "down_bias"]
    if down:
        l = down[0]
        ts_static = nv.nvfp4_quantize(l.x).ts.clone()  # the dynamic scale of this X, reused as a static one
        st_ms = []
        for it in range(max(args.warmup, 3) + K):
            flush()
            spin_ahead(torch)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            nv.nvfp4_quantize(l.x, tensor_scale_in=ts_static, out=l.qa)
            e1.record()
            torch.cuda.synchronize()
            if it >= max(args.warmup, 3):
                st_ms.append(e0.elapsed_time(e1))
        ms = float(np.median(st_ms))
        by = ops[[o[0] for o in ops].index("quantize_down_bias")][3]
        breakdown["quantize_down_bias_static_scale"] = {
            "ms": round(ms, 5), "gbs": round(by / (ms / 1e3) / 1e9, 1),
            "frac_of_hbm_measured": round(by / (ms / 1e3) / 1e9 / peaks["hbm_gbs"], 4),
            "note": "not part of the step: the same X with a static tensor scale (one pass), median of K"}

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(float(step_ms.mean()), 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "nvfp4",
        "data": "synthetic",
        "config": {"workload": WORKLOAD_NAME if args.only is None else f"{args.only} only (profiling)",
                   "M": 4608, "parallelism": "replicas" if world > 1 else "single",
                   "l2": "flushed between steps, outside the timed events: 256 MiB write, then a 256 MiB read of another buffer (L2 left holding clean lines)",
                   "timing": "each step replayed as one CUDA graph (events around the replay); the per-kernel breakdown and the roofline from an eager pass with an event before every launch",
                   "weights": "packed offline, resident in HBM",
                   "flops_per_step": flops_step},
        "roofline": {"bound": "tensor", "kernel": dom_name, "achieved": round(achieved, 1),
                     "peak": round(fp4_peak, 1), "unit": "TFLOP/s",
                     "frac": round(achieved / fp4_peak, 4),
                     "peak_basis": f"{peaks_src} bf16 burst {peaks['bf16_tflops']} x {FP4_OVER_BF16:g} (nominal fp4:bf16)",
                     "frac_of_15pf": round(achieved / (NOMINAL_FP4_PF * 1e3), 4),
                     "instruction_ceiling": round(ceiling, 1),
                     "frac_of_instruction_ceiling": round(achieved / ceiling, 4),
                     "instruction_ceiling_basis": "measured in this run: back-to-back tcgen05.mma kind::mxf4nvf4.block16 M256 N256 K64 on all SM pairs (nvfp4_debug_mma_rate), the fastest any NVFP4 GEMM here can go",
                     "traffic": traffic, "traffic_source": traffic_source, "algorithmic_bytes": dom_bytes},
        "gemm_only_tflops": round(flops_step / (gemm_ms / 1e3) / 1e12, 1),
        "step_ms_min_median": [round(float(step_ms.min()), 5), round(float(np.median(step_ms)), 5)],
        "eager_ms_per_step": round(float(eager_step_ms.mean()), 5),
        "breakdown": breakdown,
        "gpu_launches": kernels_per_step * K,
        "clocks": clocks.summary(),
    }
    if not args.no_e2e:
        result["e2e"] = run_e2e(args, layers, dev, dist)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(args.cpu_rows)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_e2e(args, layers, dev, dist):
    """Same metric through the public API with host inputs and outputs: every step copies the
    three activations from pinned host memory and the three outputs back to pinned host
    memory. Copies run on their own streams (host->device, device->host: PCIe is full
    duplex) and device buffers are double-buffered, so step k+1's inputs stream in and step
    k's outputs stream out while kernels run, as a serving loop would pipeline it."""
    import torch

    import nvfp4_gemm_act_b300 as nv
    hx = [l.x.cpu().pin_memory() for l in layers]
    hy = [[torch.empty(l.out.shape, dtype=l.out.dtype, pin_memory=True) for l in layers] for _ in range(2)]
    dx = [[torch.empty_like(l.x) for l in layers] for _ in range(2)]
    dy = [[torch.empty_like(l.out) for l in layers] for _ in range(2)]
    s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    x_free = [ev(), ev()]   # compute finished reading dx[b]
    x_ready = [ev(), ev()]  # dx[b] copied in
    y_ready = [ev(), ev()]  # dy[b] written
    y_free = [ev(), ev()]   # dy[b] copied out
    for b in range(2):
        for e_ in (x_free[b], y_free[b]):
            e_.record(s_comp)
    flops = sum(l.w.flops for l in layers)

    def step(k):
        b = k % 2
        with torch.cuda.stream(s_in):
            s_in.wait_event(x_free[b])
            for d, h in zip(dx[b], hx):
                d.copy_(h, non_blocking=True)
            x_ready[b].record(s_in)
        s_comp.wait_event(x_ready[b])
        s_comp.wait_event(y_free[b])
        for l, xin, yout in zip(layers, dx[b], dy[b]):
            w = l.w
            nv.nvfp4_quantize(xin, out=l.qa, workspace=l.ws, stream=s_comp)
            nv.nvfp4_gemm(l.qa, l.qb, w.epilogue, bias=l.bias, gamma=l.gamma, head_dim=w.head_dim,
                          norm_cols=w.norm_cols, eps=w.eps, out=yout, device_error=l.err, stream=s_comp)
        x_free[b].record(s_comp)
        y_ready[b].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(y_ready[b])
            for h, d in zip(hy[b], dy[b]):
                h.copy_(d, non_blocking=True)
            y_free[b].record(s_out)

    for k in range(max(args.warmup, 3)):
        step(k)
    torch.cuda.synchronize()
    K = max(3, min(args.steps, 20))
    barrier(dist)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for k in range(K):
        step(k)
    torch.cuda.synchronize()
    el = time.perf_counter() - t0
    for l in layers:
        assert nv.nvfp4_get_device_error(l.err) == 0
    t_max, units = aggregate(el, flops * K, dist)
    floor = copy_floor(hx, dx[0], hy[0], dy[0], s_in, s_out, K)
    step_ms = t_max / K * 1e3
    return {"value": round(units / t_max / 1e12, 2), "unit": UNIT,
            "h2d_bytes_per_step": int(sum(h.numel() * h.element_size() for h in hx)),
            "d2h_bytes_per_step": int(sum(h.numel() * h.element_size() for h in hy[0])),
            "steps": K, "pipelined": "H2D / compute / D2H streams, double-buffered",
            "ms_per_step": round(step_ms, 4),
            "copy_floor": dict(floor, frac=round(floor["both_ms"] / step_ms, 4))}


def copy_floor(hx, dx, hy, dy, s_in, s_out, reps):
    """The step's copies alone, as the e2e loop issues them (the three inputs host->device on
    one stream, the three outputs device->host on another), each direction alone and both at
    once: the time no pipelining can beat, measured in the same run."""
    import torch

    def run(h2d, d2h):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(reps):
            if h2d:
                with torch.cuda.stream(s_in):
                    for d, h in zip(dx, hx):
                        d.copy_(h, non_blocking=True)
            if d2h:
                with torch.cuda.stream(s_out):
                    for h, d in zip(hy, dy):
                        h.copy_(d, non_blocking=True)
        torch.cuda.synchronize()
        return (time.perf_counter() - t0) / reps * 1e3

    run(True, True)  # warm
    h2d_ms, d2h_ms, both_ms = run(True, False), run(False, True), run(True, True)
    nin = sum(h.numel() * h.element_size() for h in hx)
    nout = sum(h.numel() * h.element_size() for h in hy)
    return {"h2d_gbs": round(nin / h2d_ms / 1e6, 1), "d2h_gbs": round(nout / d2h_ms / 1e6, 1),
            "both_ms": round(both_ms, 4), "note": "pinned-host copies of the step alone; frac = both_ms / ms_per_step"}


# ---------------------------------------------------------------------------------------
# The CPU oracle (baseline leg and reference arm)
# ---------------------------------------------------------------------------------------

class OracleLayer:
    def __init__(self, w):
        from nvfp4_gemm_act_b300 import workloads as W
        from oracle import nvfp4_ref as R
        self.w, self.R = w, R
        self.x = W.make_x(w).float().numpy()
        self.b = R.pack_weights_ref(W.make_w(w).float().numpy(), w.epilogue == "gated_silu")
        bias, gamma = W.make_bias(w), W.make_gamma(w)
        self.bias = None if bias is None else bias.double().numpy()
        self.gamma = None if gamma is None else gamma.double().numpy()

    def run(self, rows):
        R, w = self.R, self.w
        a = R.quantize_ref(self.x[rows], R.tensor_scale_ref(self.x))
        return R.gemm_ref(*a, *self.b, w.epilogue, bias=self.bias, gamma=self.gamma,
                          head_dim=w.head_dim, norm_cols=w.norm_cols, eps=w.eps)


def cpu_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count()


def _oracle_layers():
    from nvfp4_gemm_act_b300 import workloads as W
    return [OracleLayer(w) for w in (W.QKV_RMSNORM, W.GATED_UP, W.DOWN_BIAS)]


def _cpu_cases(rows_per_gemm: int):
    """(config label, workload, sampled rows) for every config: C1 whole; C2-C4 on
    ``rows_per_gemm`` rows spread over M; the C5 batch sweep once per batch size: QKV at 512
    and 4608, down at 1024 and 9216, up (the costliest weight to dequantize) at 18432, so that
    every size and every GEMM is timed while the oracle's whole-weight dequantization, which
    does not depend on M, is not repeated fifteen times."""
    from nvfp4_gemm_act_b300 import workloads as W
    cases = [("C1", W.TINY_BIAS, np.arange(W.TINY_BIAS.M))]
    for label, w in (("C2", W.QKV_RMSNORM), ("C3", W.GATED_UP), ("C4", W.DOWN_BIAS)):
        cases.append((label, w, np.arange(rows_per_gemm) * (w.M // rows_per_gemm)))
    pick = {512: "qkv_rmsnorm", 1024: "down_bias", 4608: "qkv_rmsnorm", 9216: "down_bias", 18432: "gated_up"}
    for w in W.sweep_workloads():
        if w.name == f"{pick[w.M]}_m{w.M}":
            cases.append(("C5", w, np.arange(rows_per_gemm) * (w.M // rows_per_gemm)))
    return cases


def cpu_baseline(rows_per_gemm: int):
    """The oracle, as it stands, on the host cores: for each config, the quantize stage (the
    tensor amax over the whole X, then the block quantizer on the sampled rows) and the GEMM +
    epilogue stage (dequantize, fp64 matmul, epilogue) timed separately. Inputs are generated
    and the weights packed by the oracle before the clock starts (packing is offline in the
    method). ``value`` = the sampled GEMM FLOPs over both stages' total time."""
    from nvfp4_gemm_act_b300 import workloads as W
    from oracle import nvfp4_ref as R
    packed = {}
    per_config = {}
    flops = 0
    total_s = 0.0
    wall0 = time.perf_counter()
    for label, w, rows in _cpu_cases(rows_per_gemm):
        base = w.name.rsplit("_m", 1)[0]
        if base not in packed:
            packed[base] = R.pack_weights_ref(W.make_w(w).float().numpy(), w.epilogue == W.EPI_GATED_SILU)
        x = W.make_x(w).float().numpy()
        bias, gamma = W.make_bias(w), W.make_gamma(w)
        bias = None if bias is None else bias.double().numpy()
        gamma = None if gamma is None else gamma.double().numpy()
        t0 = time.perf_counter()
        a = R.quantize_ref(x[rows], R.tensor_scale_ref(x))
        t1 = time.perf_counter()
        R.gemm_ref(*a, *packed[base], w.epilogue, bias=bias, gamma=gamma, head_dim=w.head_dim,
                   norm_cols=w.norm_cols, eps=w.eps)
        t2 = time.perf_counter()
        del x
        f = 2 * len(rows) * w.N * w.K
        flops += f
        total_s += t2 - t0
        per_config[f"{label} {w.name}"] = {
            "M": w.M, "N": w.N, "K": w.K, "rows": int(len(rows)),
            "quantize_s": round(t1 - t0, 4),
            "quantize_gbs": round((w.M * w.K * 2 + len(rows) * w.K * 2.5625) / (t1 - t0) / 1e9, 3),
            "gemm_s": round(t2 - t1, 4), "gemm_tflops": round(f / (t2 - t1) / 1e12, 7)}
    return {"value": round(flops / total_s / 1e12, 7), "unit": UNIT, "cores": cpu_threads(),
            "kind": "oracle",
            "sample": (f"C1 whole; C2-C4, and the C5 sweep once per M (QKV at 512/4608, down at "
                       f"1024/9216, up at 18432), on "
                       f"{rows_per_gemm} rows spread over M. Quantize (full-X amax + block quantizer on the rows) and GEMM + "
                       f"epilogue (dequantize, fp64 matmul, epilogue) timed separately; inputs generated "
                       f"and weights packed by the oracle before timing; {total_s:.1f} s timed, "
                       f"{time.perf_counter() - wall0:.0f} s with set-up"),
            "per_config": per_config}


def run_reference(args, world, rank):
    """CPU oracle arm: each step is a bounded row sample of the same three GEMMs."""
    if rank != 0:
        return
    layers = _oracle_layers()
    rows_per_step = 4
    rng = np.random.default_rng(0)
    # step i runs 4 random rows through layer i % 3 (the three GEMMs in rotation), which
    # keeps one step to a few seconds of oracle time
    for i in range(args.warmup):
        layers[i % 3].run(rng.integers(0, 4608, rows_per_step))
    t0 = time.perf_counter()
    flops = 0
    for i in range(args.steps):
        l = layers[i % 3]
        l.run(rng.integers(0, 4608, rows_per_step))
        flops += 2 * rows_per_step * l.w.N * l.w.K
    el = time.perf_counter() - t0
    value = flops / el / 1e12
    res = {"metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(el / max(args.steps, 1) * 1e3, 3), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "impl": "reference",
           "config": {"workload": WORKLOAD_NAME if args.only is None else f"{args.only} only (profiling)",
                   "M": 4608,
                      "sample": f"{rows_per_step} random rows of one GEMM per step, the three GEMMs in rotation"},
           "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": cpu_threads(),
                            "kind": "oracle",
                            "sample": f"{rows_per_step} rows of one GEMM per step (rotating over the 3), {args.steps} steps"},
           "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)


def run_sweep(args):
    """The three DiT GEMMs at every batch size of the sweep (activations redrawn per size,
    weights fixed): CUDA-event time of the activation quantize and of the fused GEMM, L2
    flushed before each timed call; one JSON line per (M, GEMM)."""
    import torch

    import nvfp4_gemm_act_b300 as nv
    from nvfp4_gemm_act_b300 import workloads as W
    dev = "cuda:0"
    peaks, _ = measured_peaks()
    fp4_peak = peaks["bf16_tflops"] * FP4_OVER_BF16
    flush = L2Flush(dev)
    packed = {}
    for w in W.sweep_workloads():
        base = w.name.rsplit("_m", 1)[0]
        if base not in packed:
            packed[base] = nv.nvfp4_pack_weights(W.make_w(w).to(dev), gated_interleave=w.epilogue == "gated_silu")
        l = Layer.__new__(Layer)
        l.w, l.x, l.qb = w, W.make_x(w).to(dev), packed[base]
        b, g = W.make_bias(w), W.make_gamma(w)
        l.bias = None if b is None else b.to(dev)
        l.gamma = None if g is None else g.to(dev)
        l.qa = nv._alloc_nvfp4(w.M, w.K, dev)
        l.ws = torch.zeros(16, dtype=torch.uint8, device=dev)
        l.out = torch.empty((w.M, w.out_cols), dtype=torch.bfloat16, device=dev)
        l.err = torch.zeros(1, dtype=torch.int32, device=dev)
        times = {"quantize": [], "gemm": []}
        for it in range(max(args.warmup, 3) + args.steps):
            for name, fn in (("quantize", l.quantize), ("gemm", l.gemm)):
                flush()
                spin_ahead(torch)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                fn()
                e1.record()
                torch.cuda.synchronize()
                if it >= max(args.warmup, 3):
                    times[name].append(e0.elapsed_time(e1))
        assert nv.nvfp4_get_device_error(l.err) == 0
        qms, gms = float(np.median(times["quantize"])), float(np.median(times["gemm"]))
        qbytes = w.M * w.K * 2 + w.M * w.K // 2 + w.M * w.K // 16
        tf = w.flops / (gms / 1e3) / 1e12
        print(json.dumps({"sweep": w.name, "M": w.M, "epilogue": w.epilogue, "gemm_ms": round(gms, 5),
                          "gemm_tflops": round(tf, 1), "frac_of_measured_fp4": round(tf / fp4_peak, 4),
                          "frac_of_15pf": round(tf / (NOMINAL_FP4_PF * 1e3), 4),
                          "quantize_ms": round(qms, 5),
                          "quantize_gbs": round(qbytes / (qms / 1e3) / 1e9, 1)}), flush=True)


def run_chain(args):
    """The up-projection (gated SiLU) feeding the down-projection at M=4608, three ways: the up
    GEMM writing NVFP4 for the down GEMM (static scale); the up GEMM writing bf16, then the
    quantizer with the same static scale; bf16, then the quantizer with a dynamic scale. The
    static scale is calibrated once, before timing, from the bf16 output's amax. Each variant
    starts from the quantized up-projection input; L2 is flushed before every timed chain."""
    import torch

    import nvfp4_gemm_act_b300 as nv
    from nvfp4_gemm_act_b300 import workloads as W
    dev = "cuda:0"
    up, down = W.GATED_UP, W.DOWN_BIAS
    assert up.out_cols == down.K
    qa = nv.nvfp4_quantize(W.make_x(up).to(dev))
    qb_up = nv.nvfp4_pack_weights(W.make_w(up).to(dev), gated_interleave=True)
    qb_dn = nv.nvfp4_pack_weights(W.make_w(down).to(dev))
    bias_dn = W.make_bias(down).to(dev)
    y_mid = nv.nvfp4_gemm(qa, qb_up, up.epilogue)
    ts_mid = nv.nvfp4_quantize(y_mid).ts  # the library's dynamic tensor scale of the bf16 output
    q_mid = nv._alloc_nvfp4(up.M, up.out_cols, dev)
    ws = torch.zeros(16, dtype=torch.uint8, device=dev)
    out = torch.empty((down.M, down.out_cols), dtype=torch.bfloat16, device=dev)
    flush = L2Flush(dev)

    def fused():
        m = nv.nvfp4_gemm_nvfp4_out(qa, qb_up, up.epilogue, ts_mid, out=q_mid)
        nv.nvfp4_gemm(m, qb_dn, down.epilogue, bias=bias_dn, out=out)

    def unfused(static):
        nv.nvfp4_gemm(qa, qb_up, up.epilogue, out=y_mid)
        m = nv.nvfp4_quantize(y_mid, out=q_mid, tensor_scale_in=ts_mid if static else None, workspace=ws)
        nv.nvfp4_gemm(m, qb_dn, down.epilogue, bias=bias_dn, out=out)

    variants = {"fused_nvfp4_out": fused, "bf16_then_quantize_static": lambda: unfused(True),
                "bf16_then_quantize_dynamic": lambda: unfused(False)}
    res = {}
    for name, fn in variants.items():
        ts = []
        for it in range(max(args.warmup, 3) + args.steps):
            flush()
            spin_ahead(torch)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            if it >= max(args.warmup, 3):
                ts.append(e0.elapsed_time(e1))
        res[name] = round(float(np.median(ts)), 5)
    flops = up.flops + down.flops
    print(json.dumps({"chain": "up-projection (gated SiLU) -> down-projection, M=4608", "ms": res,
                      "tflops": {k: round(flops / (v / 1e3) / 1e12, 1) for k, v in res.items()},
                      "intermediate_bf16_mb": round(up.M * up.out_cols * 2 / 1e6, 1),
                      "intermediate_nvfp4_mb": round(up.M * up.out_cols * (0.5 + 1 / 16) / 1e6, 1),
                      "steps": args.steps}), flush=True)


def run_fp8(args):
    """The three DiT GEMMs at M=4608 in the FP8 variant (E4M3 operands, one scale per tensor, the
    same fused epilogues): CUDA-event time of the activation quantize and of the GEMM, L2 flushed
    before each timed call, against the FP8 dense peak (measured bf16 x 2); one JSON line per GEMM."""
    import torch

    import nvfp4_gemm_act_b300 as nv
    from nvfp4_gemm_act_b300 import workloads as W
    dev = "cuda:0"
    peaks, _ = measured_peaks()
    fp8_peak = peaks["bf16_tflops"] * 2.0
    flush = L2Flush(dev)
    spun = False
    for w in (W.QKV_RMSNORM, W.GATED_UP, W.DOWN_BIAS):
        if args.only is not None and w.name != args.only:
            continue
        x = W.make_x(w).to(dev)
        qb = nv.fp8_pack_weights(W.make_w(w).to(dev), gated_interleave=w.epilogue == "gated_silu")
        b, g = W.make_bias(w), W.make_gamma(w)
        bias = None if b is None else b.to(dev)
        gamma = None if g is None else g.to(dev)
        qa = nv._alloc_fp8(w.M, w.K, dev)
        ws = torch.zeros(16, dtype=torch.uint8, device=dev)
        out = torch.empty((w.M, w.out_cols), dtype=torch.bfloat16, device=dev)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        ops = {"quantize": lambda: nv.fp8_quantize(x, out=qa, workspace=ws),
               "gemm": lambda: nv.fp8_gemm(qa, qb, w.epilogue, bias=bias, gamma=gamma, head_dim=w.head_dim,
                                           norm_cols=w.norm_cols, eps=w.eps, out=out, device_error=err)}
        if not spun and args.spin_up_ms > 0:  # keep the GPU busy until its clocks have settled
            t0 = time.perf_counter()
            while (time.perf_counter() - t0) * 1e3 < args.spin_up_ms:
                for fn in ops.values():
                    fn()
                torch.cuda.synchronize()
            spun = True
        times = {"quantize": [], "gemm": []}
        for it in range(max(args.warmup, 3)):
            for fn in ops.values():
                fn()
        sampler = ClockSampler(0)
        with sampler:
            for it in range(args.steps):
                for name, fn in ops.items():
                    flush()
                    spin_ahead(torch)
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record()
                    fn()
                    e1.record()
                    torch.cuda.synchronize()
                    times[name].append(e0.elapsed_time(e1))
        assert nv.nvfp4_get_device_error(err) == 0
        qms, gms = float(np.median(times["quantize"])), float(np.median(times["gemm"]))
        tf = w.flops / (gms / 1e3) / 1e12
        print(json.dumps({"fp8": w.name, "M": w.M, "N": w.N, "K": w.K, "epilogue": w.epilogue,
                          "gemm_ms": round(gms, 5), "gemm_tflops": round(tf, 1),
                          "frac_of_measured_fp8": round(tf / fp8_peak, 4), "quantize_ms": round(qms, 5),
                          "quantize_gbs": round(w.M * w.K * 3 / (qms / 1e3) / 1e9, 1),
                          "clocks": sampler.summary()}), flush=True)


def run_attention(args):
    """Attention over a QKV projection output of 4608 tokens, 12 heads of 256 (Q, K, V ~ N(0,1)):
    CUDA-event time of this package's kernel (V transpose + attention) and of torch's
    scaled_dot_product_attention (its default choice, and the cuDNN backend where torch offers
    it), L2 flushed before each call; 4 * M^2 * hidden FLOPs; one JSON line."""
    import torch
    import torch.nn.functional as F

    import nvfp4_gemm_act_b300 as nv
    from nvfp4_gemm_act_b300 import workloads as W
    dev = "cuda:0"
    M, heads, hd = 4608, 12, 256
    H = heads * hd
    qkv = W.attention_qkv(M, heads, seed=9).to(dev)
    ws = torch.empty(nv.lib().attention_workspace_bytes(M, heads), dtype=torch.uint8, device=dev)
    out = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    q, k, v = qkv.view(M, 3, heads, hd).permute(1, 2, 0, 3).unsqueeze(1).unbind(0)
    flush = L2Flush(dev)
    impls = {"kernel": lambda: nv.attention(qkv, heads, out=out, workspace=ws, device_error=err),
             "torch_default": lambda: F.scaled_dot_product_attention(q, k, v)}
    try:
        from torch.nn.attention import SDPBackend, sdpa_kernel

        def cudnn():
            with sdpa_kernel([SDPBackend.CUDNN_ATTENTION]):
                return F.scaled_dot_product_attention(q, k, v)
        cudnn()
        torch.cuda.synchronize()
        impls["torch_cudnn"] = cudnn
    except Exception as e:  # not offered for this shape / build
        print(json.dumps({"note": f"cudnn backend unavailable: {type(e).__name__}"}), flush=True)
    t0 = time.perf_counter()
    while (time.perf_counter() - t0) * 1e3 < args.spin_up_ms:  # clocks settle
        impls["kernel"]()
        torch.cuda.synchronize()
    res = {}
    sampler = ClockSampler(0)
    for name, fn in impls.items():
        for _ in range(max(args.warmup, 3)):
            fn()
        ts = []
        with sampler if name == "kernel" else _nullctx():
            for _ in range(args.steps):
                flush()
                spin_ahead(torch)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                fn()
                e1.record()
                torch.cuda.synchronize()
                ts.append(e0.elapsed_time(e1))
        res[name] = float(np.median(ts))
    assert nv.nvfp4_get_device_error(err) == 0
    flops = 4 * M * M * H
    peaks, _ = measured_peaks()
    print(json.dumps({"attention": f"M={M} heads={heads}x{hd}, no mask, bf16",
                      "ms": {k: round(v, 5) for k, v in res.items()},
                      "tflops": {k: round(flops / (v / 1e3) / 1e12, 1) for k, v in res.items()},
                      "kernel_frac_of_measured_bf16": round(flops / (res["kernel"] / 1e3) / 1e12 / peaks["bf16_tflops"], 4),
                      "steps": args.steps, "clocks": sampler.summary()}), flush=True)


class _nullctx:
    def __enter__(self):
        return self

    def __exit__(self, *exc):
        return False


def run_dit_block(args):
    """One DiT block at 4608 tokens (hidden 3072, 12 heads of 256, MLP 12288): the up-projection's
    static output scale calibrated once from its bf16 output, then per step (L2 flushed first)
    the whole block with a CUDA-event pair around each stage. One JSON line: median ms per stage
    (a stage's time includes its activation quantize), its share, and the GEMM rate."""
    import torch

    from nvfp4_gemm_act_b300.dit_block import STAGES, seeded_dit_block
    dev = "cuda:0"
    M = 4608
    blk, x = seeded_dit_block(M, dev, attention_impl=args.attention_impl)
    blk.calibrate(x)
    flush = L2Flush(dev)
    times = {}
    total = []
    sampler = ClockSampler(0)

    def one(t):
        flush()
        spin_ahead(torch)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        y = blk(x, timings=t)
        e1.record()
        torch.cuda.synchronize()
        return y, e0.elapsed_time(e1)

    for _ in range(max(args.warmup, 3)):
        one(None)
    with sampler:
        for _ in range(args.steps):
            t = {}
            y, ms_total = one(t)
            for k, v in t.items():
                times.setdefault(k, []).extend(v)
            total.append(ms_total)
    assert bool(torch.isfinite(y.float()).all())
    # the same block replayed as one CUDA graph (no per-launch host work between stages)
    replay, _ = blk.graph(x)
    graph_ms = []
    for it in range(max(args.warmup, 3) + args.steps):
        flush()
        spin_ahead(torch)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        replay()
        e1.record()
        torch.cuda.synchronize()
        if it >= max(args.warmup, 3):
            graph_ms.append(e0.elapsed_time(e1))
    h, m = blk.hidden, blk.mlp
    flops = {"qkv_rmsnorm": 2 * M * h * 3 * h, "attention": 4 * M * M * h, "out_proj": 2 * M * h * h,
             "up_gated_silu": 2 * M * h * 2 * m, "down": 2 * M * m * h}
    ms = {k: round(float(np.median(times[k])), 5) for k in STAGES}
    tot = float(np.median(total))
    print(json.dumps({"dit_block": f"M={M} hidden={h} heads={blk.heads}x{blk.head_dim} mlp={m}",
                      "total_ms": round(tot, 5), "graph_total_ms": round(float(np.median(graph_ms)), 5), "ms": ms,
                      "share": {k: round(v / sum(ms.values()), 4) for k, v in ms.items()},
                      "tflops": {k: round(flops[k] / (ms[k] / 1e3) / 1e12, 1) for k in STAGES},
                      "nvfp4_gemm_tflops_block": round(blk.gemm_flops(M) / ((tot - ms["attention"]) / 1e3) / 1e12, 1),
                      "attention": ("this package's attention kernel" if args.attention_impl == "kernel"
                                    else "torch scaled_dot_product_attention") + ", bf16",
                      "steps": args.steps, "l2": "flushed before each block",
                      "clocks": sampler.summary()}), flush=True)


def run_mma_ceiling(args):
    """The tensor pipe's instruction rate (nvfp4_debug_mma_rate): for each kind, cta_group and N,
    `--probe-iters` back-to-back instructions per CTA (pair) on one SM (pair) and on every SM;
    one JSON line each with the median cycles per instruction, FLOP per cycle per SM, and the
    whole-GPU rate from the per-CTA nanoseconds (sum of FLOPs over the slowest CTA's time)."""
    import torch

    import nvfp4_gemm_act_b300 as nv
    dev = "cuda:0"
    torch.cuda.set_device(0)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    iters = args.probe_iters
    nv.nvfp4_debug_mma_rate("nvfp4", 2, 256, iters, sms // 2, device_error=err)  # warm-up, clocks settle
    torch.cuda.synchronize()
    sampler = ClockSampler(0)
    with sampler:
        for kind in ("nvfp4", "fp8", "bf16"):
            for cg in (1, 2):
                for n in (64, 128, 256):
                    for ctas in (1, sms // cg):
                        nv.nvfp4_debug_mma_rate(kind, cg, n, iters, ctas, device_error=err)  # warm
                        r = nv.nvfp4_debug_mma_rate(kind, cg, n, iters, ctas, device_error=err)
                        torch.cuda.synchronize()
                        r = r.cpu().numpy()
                        assert (r > 0).all(), f"probe wait ran out: {kind} cta_group {cg} n {n}"
                        cyc = float(np.median(r[:, 0])) / iters
                        m = 128 * cg
                        flop = 2 * m * n * nv.PROBE_K[kind]
                        print(json.dumps({
                            "mma_ceiling": kind, "cta_group": cg, "M": m, "N": n, "K": nv.PROBE_K[kind],
                            "ctas": ctas, "sms": ctas * cg, "iters": iters,
                            "cycles_per_instr": round(cyc, 2),
                            "flop_per_clk_per_sm": round(flop / cyc / cg, 1),
                            "tflops_all_ctas": round(flop * iters * ctas / (float(r[:, 1].max()) * 1e-9) / 1e12, 1),
                            "sm_mhz_implied": round(float(np.median(r[:, 0] / r[:, 1])) * 1e3, 0)}), flush=True)
    assert nv.nvfp4_get_device_error(err) == 0
    print(json.dumps({"mma_ceiling_clocks": sampler.summary()}), flush=True)


def main(argv=None):
    args = parse_args(argv)
    world, rank, local = dist_env()
    if args.dit_block:
        run_dit_block(args)
        return
    if args.fp8:
        run_fp8(args)
        return
    if args.attention:
        run_attention(args)
        return
    if args.chain:
        run_chain(args)
        return
    if args.sweep:
        run_sweep(args)
        return
    if args.mma_ceiling:
        run_mma_ceiling(args)
        return
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()

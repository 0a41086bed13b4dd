"""Benchmark of the NVFP4 MoE expert FFN on GB300.

One step = one pass of the whole path over one batch: moe_route_permute
(top-k routing, padded permutation, NVFP4 staging of x) -> L1 grouped GEMM with
the fused SwiGLU + NVFP4 epilogue -> L2 grouped GEMM -> the routing-weighted
combine.  By default the steps form a serving pipeline (batches alternate
between two buffer sets): step i routes batch i, runs the L2 GEMM of batch i-1
with batch i's activation staging on two spare warps per CTA, then the L1 GEMM
of batch i with batch i-1's combine on two spare warps per CTA.  The timed
region starts the pipeline empty (its first step routes, stages and runs L1
only) and ends with the last batch's L2 GEMM and combine, so it holds exactly
the steps' batches.  `--no-overlap-combine` runs each batch's whole path in
its own step, every stage its own launch.  The default workload is the prefill batch: T=16384 tokens,
H=7168, I=2048, E=256 experts, top-8, Zipf-skewed routing (seeded synthetic
data).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  `value` is whole-job TFLOP/s of the FFN
(algorithmic FLOPs 6*k*H*I per token, padding rows not credited) with inputs
resident in HBM; `e2e` repeats the measurement through the library's
host-buffer calls (nvfp4_moe_step_host / nvfp4_moe_finish_host, which run the
same pipeline, or nvfp4_moe_forward_host without it), with the inputs copied from
pinned host memory and the output copied back inside the timed region.
Under torchrun each rank runs its own batch (weak scaling, no data-path
collective); the timed region is bracketed by barriers and the max over ranks
is taken.  `--impl reference` times the CPU oracle on the host cores on a
bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import inputs  # noqa: E402

METRIC = "NVFP4 MoE FFN TFLOPS & tokens/s (frac of FP4 peak); quantize GB/s vs HBM"

# DRAM bytes (read + write) of one L1 launch per workload, from an ncu capture
# of that launch (dram__bytes_read.sum + dram__bytes_write.sum; on the prefill
# batch the CTA-pair launch plus the single-CTA launch beside it, captured one
# after the other), and the hash of the kernel sources' code it was taken on
# (comments and blank lines left out: kernel_code).  Reported as
# roofline.traffic only while the code still hashes the same (a changed kernel
# reports null).
L1_TRAFFIC_RECORD = {"sources_sha256": "e58cf74a9954716401cccb58b8e3a5e620e555dac638d5193b94021efbdf2121",
                     "bytes": {"prefill": (1064234240 + 153088000) + (664541184 + 498176),
                               "prefill_overlap": (2945267968 + 384792320) + (664382208 + 409344),
                               "decode": 4351559168 + 3329792}}
KERNEL_SOURCES = ("nvfp4_block_scaled_moe_gb300/csrc/gemm.cu", "nvfp4_block_scaled_moe_gb300/csrc/gemm_pair.cu",
                  "nvfp4_block_scaled_moe_gb300/csrc/common.cuh", "nvfp4_block_scaled_moe_gb300/csrc/internal.h",
                  "nvfp4_block_scaled_moe_gb300/csrc/stage.cuh")


def kernel_code(text: str) -> str:
    """A CUDA source without its comments and blank lines: what the hash of the
    traffic record covers (a comment edit leaves the kernels, and the record,
    as they were; any code edit changes the hash)."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(ln.rstrip() for ln in text.splitlines() if ln.strip())


def kernel_sources_sha256() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), encoding="utf-8") as fh:
            h.update(kernel_code(fh.read()).encode())
    return h.hexdigest()


def l1_traffic(key: str = "prefill"):
    """The recorded traffic of one L1 launch: key is the workload, with
    "_overlap" when the launch also runs the previous batch's combine."""
    rec = L1_TRAFFIC_RECORD
    if rec["sources_sha256"] == kernel_sources_sha256():
        return rec["bytes"].get(key)
    return None


WORKLOAD = "prefill"
FP4_OVER_BF16 = 13.5 / 2.25          # nominal dense ratio (FP4 / BF16 tensor peak)


# ------------------------------------------------------------------ helpers --
def peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return dict(hbm_gbs=p["hbm_gbs"], bf16=p["bf16_tflops"], bf16_sustained=p["bf16_tflops_sustained"],
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


def ffn_flops(T: int, H: int, I: int, k: int) -> tuple:
    l1 = 2.0 * T * k * (2 * I) * H
    l2 = 2.0 * T * k * I * H
    return l1, l2


class ClockSampler:
    """SM clock and clock-event reasons sampled during the timed region.

    A background thread polls NVML (read-only queries through ctypes) every
    2 ms and stamps each sample with the host clock; stop(t0, t1) keeps the
    samples taken inside the timed region [t0, t1], so even a 50 ms region
    gets a few dozen.  Without NVML it falls back to `nvidia-smi -lms 100`,
    whose samples cover the sampler's whole lifetime (it needs a few hundred
    ms to start)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    # NVML clock-event reason bits that mark a throttled run (power capping is kept and noted)
    REASON_BITS = ((0x8, "hw_slowdown"), (0x40, "hw_thermal_slowdown"), (0x20, "sw_thermal_slowdown"),
                   (0x80, "hw_power_brake_slowdown"), (0x4, "sw_power_cap"))
    PERIOD_S = 0.002

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.tmp = None
        self.nvml = None
        self.thread = None
        self.samples = []           # (host time, sm MHz, max sm MHz, reason bits)

    def _nvml_open(self):
        import ctypes

        import torch
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        handle = ctypes.c_void_p()
        props = torch.cuda.get_device_properties(self.gpu)
        bus = getattr(props, "pci_bus_id", None)
        ok = -1
        if bus is not None:
            pci = "%08x:%02x:%02x.0" % (getattr(props, "pci_domain_id", 0), bus, getattr(props, "pci_device_id", 0))
            ok = lib.nvmlDeviceGetHandleByPciBusId_v2(pci.encode(), ctypes.byref(handle))
        if ok != 0:
            ok = lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.gpu), ctypes.byref(handle))
        if ok != 0:
            raise OSError("no NVML handle for the device")
        reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        return ctypes, lib, handle, reasons

    def _poll(self):
        ctypes, lib, handle, reasons_fn = self.nvml
        mhz, mx, bits = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while not self.stopping.is_set():
            t = time.time()
            if (lib.nvmlDeviceGetClockInfo(handle, 1, ctypes.byref(mhz)) == 0 and           # NVML_CLOCK_SM
                    lib.nvmlDeviceGetMaxClockInfo(handle, 1, ctypes.byref(mx)) == 0 and
                    reasons_fn(handle, ctypes.byref(bits)) == 0):
                self.samples.append((t, mhz.value, mx.value, bits.value))
            self.stopping.wait(self.PERIOD_S)

    def start(self):
        import threading
        try:
            self.nvml = self._nvml_open()
            self.stopping = threading.Event()
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()
            return
        except Exception:                  # no NVML: fall back to nvidia-smi
            self.nvml = None
        try:
            self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.tmp, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def window(self, t0=None, t1=None, what="timed region") -> dict:
        """Summary of the NVML samples taken in [t0, t1] (host clock); the sampler keeps running."""
        samples = list(self.samples)
        inside = [x for x in samples if t0 is None or t0 <= x[0] <= t1]
        window = what
        if not inside:                           # a region shorter than the poll period
            inside = sorted(samples, key=lambda x: abs(x[0] - (t0 + t1) / 2))[:1] if t0 else samples
            window = f"nearest sample to the {what}"
        reasons = sorted({name for bit, name in self.REASON_BITS for x in inside if x[3] & bit})
        return {"sm_mhz": statistics.median(x[1] for x in inside) if inside else None,
                "sm_max_mhz": max(x[2] for x in inside) if inside else None,
                "samples": len(inside), "reasons": reasons,
                "source": f"NVML every {self.PERIOD_S * 1e3:g} ms, {window}"}

    def stop(self, t0=None, t1=None) -> dict:
        if self.nvml is not None:
            self.stopping.set()
            self.thread.join(timeout=5)
            self.nvml[1].nvmlShutdown()
            return self.window(t0, t1)
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.tmp.flush()
        with open(self.tmp.name) as f:
            lines = [ln.strip() for ln in f if ln.strip()]
        os.unlink(self.tmp.name)
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "samples": len(sm), "reasons": sorted(reasons), "source": "nvidia-smi -lms 100, sampler lifetime"}


def dist_setup():
    import torch
    import torch.distributed as dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return world, rank, local


def max_over_ranks(x: float, world: int) -> float:
    """Max of a host scalar over ranks (the only collective: timing, never data)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# --------------------------------------------------------- the oracle arm --
class OracleArm:
    """The CPU oracle, as it stands, on sampled tokens of the workload (inputs drawn
    once, outside any timing; expert dequantisations cached as the oracle allows)."""

    def __init__(self, spec: dict, seed: int = 1234):
        self.spec = spec
        _, self.x = inputs.moe_x(spec)
        self.logits = inputs.moe_logits(spec)
        self.order = np.random.default_rng(seed).permutation(spec["T"])
        self.next = 0
        self.cache: dict = {}

    def run(self, budget_s: float, max_tokens: int) -> dict:
        from oracle import moe as omoe
        spec = self.spec
        done, t0 = 0, time.perf_counter()
        while done < max_tokens:
            t = self.order[self.next % len(self.order)]
            self.next += 1
            omoe.moe_ffn_tokens(self.x[[t]], self.logits[[t]], lambda e: inputs.moe_w1(spec, e),
                                lambda e: inputs.moe_w2(spec, e), spec["top_k"], cache=self.cache)
            done += 1
            if time.perf_counter() - t0 >= budget_s:
                break
        dt = time.perf_counter() - t0
        l1, l2 = ffn_flops(done, spec["H"], spec["I"], spec["top_k"])
        return dict(tokens=done, seconds=dt, tflops=(l1 + l2) / dt / 1e12, tokens_per_s=done / dt)


def run_reference(args, world: int, rank: int) -> None:
    if rank != 0:
        return
    name = args.workload if args.workload in ("prefill", "decode") else WORKLOAD
    spec = dict(inputs.CONFIGS[name])
    arm = OracleArm(spec)
    tok, sec = 0, 0.0
    for i in range(args.warmup + args.steps):
        r = arm.run(budget_s=0.0, max_tokens=1)
        if i >= args.warmup:
            tok += r["tokens"]
            sec += r["seconds"]
    l1, l2 = ffn_flops(tok, spec["H"], spec["I"], spec["top_k"])
    value = (l1 + l2) / sec / 1e12
    cores = os.cpu_count()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sec / max(args.steps, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": _workload_name(spec, name), "step": "oracle on one sampled token per step"},
        "tokens_per_s": tok / sec,
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"{tok} sampled tokens of the {name} batch, one per step, expert "
                                   "dequantisation cached across steps"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def mma_ceiling(nv) -> dict:
    """The measured issue ceiling of the GEMMs' FP4 MMA (nvfp4_mma_peak_probe: the
    CTA-pair instruction stream with resident operands on every SM pair), run once
    before the timed region; the roofline objects add the achieved fraction of it."""
    tf, mhz = nv.nvfp4_mma_peak_probe(20000)
    return {"value": tf, "unit": "TFLOP/s", "sm_mhz": mhz,
            "what": "tcgen05.mma.cta_group::2.kind::mxf4nvf4 M=256 N=256 K=64 with the GEMM's scale-factor "
                    "copies and commits, operands resident in shared memory, every SM pair"}


def _workload_name(spec: dict, name: str = WORKLOAD) -> str:
    routing = "Zipf(1.2)-skewed routing" if spec.get("zipf") else "N(0,1) routing logits"
    return (f"{name} NVFP4 MoE FFN T={spec['T']} H={spec['H']} I={spec['I']} E={spec['E']} "
            f"top-{spec['top_k']} {routing}")


# ------------------------------------------------------------ our GPU arm --
def e2e_host_call(nv, pipeline, s, w, b, x_h, logits_h, k, steps, world, y_ref):
    """Each step is one nvfp4_moe_forward_host call: host x and logits copied in,
    route, FFN, combine, y copied out to host, all on one stream.  Steps alternate
    between two device buffer sets on two streams, so one step's copies run beside
    its neighbour's kernels.  The last step's y must equal the resident run's."""
    import torch
    sets = [b.enable_host_io(), pipeline.MoeBuffers(s).enable_host_io()]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    y_h = [torch.empty((s.T, s.H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    main = torch.cuda.current_stream()
    nv.nvfp4_moe_forward_host(x_h, logits_h, y_h[0], k, w, sets[1], stream=streams[1])    # warm the second set
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(main)
    for st in streams:
        st.wait_event(s0)
    for i in range(steps):
        j = i & 1
        nv.nvfp4_moe_forward_host(x_h, logits_h, y_h[j], k, w, sets[j], stream=streams[j])
    for st in streams:
        main.wait_stream(st)
    s1.record(main)
    torch.cuda.synchronize()
    nv.nvfp4_device_status()
    if not (torch.equal(y_h[(steps - 1) & 1], y_ref) and torch.equal(y_h[steps & 1], y_ref)):
        raise RuntimeError("end-to-end: the copied-out y differs from the resident run's")
    barrier(world)
    del sets[1]
    return (max_over_ranks(s0.elapsed_time(s1), world),
            "one nvfp4_moe_forward_host C-ABI call per step: pinned host x and logits copied in, route, L1, L2, "
            "combine, y copied out to pinned host memory, on one stream; steps alternate between two device "
            "buffer sets on two streams, so one step's copies overlap its neighbour's kernels")


def e2e_step_host(nv, pipeline, s, w, b, x_h, logits_h, k, steps, world, y_ref):
    """Each step is one nvfp4_moe_step_host C-ABI call: host x and logits copied in,
    routing, the previous batch's L2 (also staging this batch on spare warps),
    this batch's L1 (also running the previous batch's combine on spare warps),
    and the previous batch's y copied out to host; one nvfp4_moe_finish_host
    call after the last step runs the last batch's L2 and combine and copies its
    y out, so the region holds exactly the steps' batches.  Steps
    rotate over three device buffer sets on three streams, each step's kernels
    waiting for the previous step's.  On one stream a step's copy-in queues
    behind the copy-out of the step three back, so each copy pair has two steps'
    kernels to hide behind.  Every batch's y must equal the resident run's."""
    import torch
    n_sets = 3
    sets = [b.enable_host_io()] + [pipeline.MoeBuffers(s).enable_host_io() for _ in range(n_sets - 1)]
    streams = [torch.cuda.Stream() for _ in range(n_sets)]
    done = [torch.cuda.Event() for _ in range(n_sets)]
    for ev, st in zip(done, streams):
        ev.record(st)                              # the events exist from here on
    y_h = [torch.zeros((s.T, s.H), dtype=torch.bfloat16).pin_memory() for _ in range(n_sets)]
    main = torch.cuda.current_stream()

    def run(n):
        for i in range(n):
            j, p = i % n_sets, (i - 1) % n_sets
            nv.nvfp4_moe_step_host(x_h, logits_h, k, w, sets[j], prev=sets[p] if i else None,
                                   prev_y_host=y_h[p] if i else None, compute_after=done[p] if i else None,
                                   compute_done=done[j], stream=streams[j])
        last = (n - 1) % n_sets
        nv.nvfp4_moe_finish_host(w, sets[last], k, y_h[last], stream=streams[last])

    run(n_sets)                                    # warm every set (untimed)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(main)
    for st in streams:
        st.wait_event(s0)
    run(steps)
    for st in streams:
        main.wait_stream(st)
    s1.record(main)
    torch.cuda.synchronize()
    nv.nvfp4_device_status()
    if not all(torch.equal(y, y_ref) for y in y_h):
        raise RuntimeError("end-to-end: a copied-out y differs from the resident run's")
    barrier(world)
    del sets[1:]
    return (max_over_ranks(s0.elapsed_time(s1), world),
            "one nvfp4_moe_step_host C-ABI call per step: pinned host x and logits copied in, routing, the previous "
            "batch's L2 (staging this batch on spare warps), this batch's L1 (combining the previous batch on spare "
            "warps), the previous batch's y copied out to pinned host memory; one nvfp4_moe_finish_host call for "
            "the last batch's L2, combine and copy-out; steps rotate over three device buffer sets on three streams "
            "(each step's kernels wait for the previous step's), so copies overlap kernels")


def e2e_copy_streams(step, x_d, logits_d, b, x_h, logits_h, T, H, stream, steps, world):
    """The variant workloads (gathering L1, two-level scale, shared expert): host
    copies on two copy streams around the device-pointer calls, double-buffered
    device x, logits and y; the last y must equal the resident run's."""
    import torch
    y_h = torch.empty((T, H), dtype=torch.bfloat16).pin_memory()
    xs, lgs, ys = [x_d, torch.empty_like(x_d)], [logits_d, torch.empty_like(logits_d)], [b.y, torch.empty_like(b.y)]
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]      # inputs of buffer j have landed
    ev_done = [torch.cuda.Event() for _ in range(2)]    # step on buffer j finished (inputs free, y ready)
    ev_out = [torch.cuda.Event() for _ in range(2)]     # y of buffer j has left
    barrier(world)
    torch.cuda.synchronize()
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    fetched = [False, False]

    def fetch(j):
        h2d.wait_event(ev_done[j]) if fetched[j] else h2d.wait_event(s0)
        with torch.cuda.stream(h2d):
            xs[j].copy_(x_h, non_blocking=True)
            lgs[j].copy_(logits_h, non_blocking=True)
        ev_in[j].record(h2d)
        fetched[j] = True

    fetch(0)
    for i in range(steps):
        j = i & 1
        if i + 1 < steps:
            fetch(1 - j)
        stream.wait_event(ev_in[j])
        if i >= 2:
            stream.wait_event(ev_out[j])                 # y buffer j: its previous copy-out is done
        step(x_in=xs[j], logits_in=lgs[j], y_out=ys[j])
        ev_done[j].record(stream)
        d2h.wait_event(ev_done[j])
        with torch.cuda.stream(d2h):
            y_h.copy_(ys[j], non_blocking=True)
        ev_out[j].record(d2h)
    stream.wait_stream(d2h)
    s1.record(stream)
    torch.cuda.synchronize()
    if not torch.equal(y_h, ys[0].cpu()):
        raise RuntimeError("end-to-end pipeline: the copied-out y differs from the resident run's")
    barrier(world)
    return (max_over_ranks(s0.elapsed_time(s1), world),
            "pinned host x and logits in, y out, every step; H2D and D2H on two copy streams overlapping the "
            "neighbouring steps' compute (double-buffered device x, logits, y)")


def run_ours(args, world: int, rank: int, local: int) -> None:
    import torch

    import nvfp4_block_scaled_moe_gb300 as nv
    from nvfp4_block_scaled_moe_gb300 import build as nvbuild
    from nvfp4_block_scaled_moe_gb300 import pipeline

    nvbuild.build()
    nv.load()
    torch.cuda.set_device(local)
    spec = dict(inputs.CONFIGS[args.workload])
    spec["seed"] = spec["seed"] + 1000 * rank if rank else spec["seed"]     # each rank its own batch
    T, H, I, E, k = spec["T"], spec["H"], spec["I"], spec["E"], spec["top_k"]
    s = pipeline.MoeShape(T=T, H=H, I=I, E=E, top_k=k)
    two = args.two_level
    w = pipeline.MoeWeights(s, two_level=two)
    pool, o1, o2 = inputs.moe_weight_pool(spec)
    w.set_from_pool(torch.from_numpy(pool).cuda(), o1, o2, float(inputs.WEIGHT_STD))
    b = pipeline.MoeBuffers(s, gather=args.gather)
    x_t, _ = inputs.moe_x(spec)
    logits_np = inputs.moe_logits(spec)
    x_d = x_t.cuda()
    logits_d = torch.from_numpy(logits_np).cuda()
    if two:
        # the L1 output's encode scale, calibrated once on this batch (setup, untimed)
        pipeline.calibrate_a2_scale(x_d, logits_d, w, b)
        b.h_debug = None
    sh = None
    if args.shared_expert:
        sh = pipeline.SharedExpert(s, I)
        w1s, w2s = inputs.moe_shared_weights(spec, I)
        sh.set_weights(torch.from_numpy(w1s).cuda(), torch.from_numpy(w2s).cuda())
        del w1s, w2s
    torch.cuda.synchronize()

    stream = torch.cuda.current_stream()
    R = b.rows_max
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]

    gs1 = dict(a_global_scale=b.x_gs, b_global_scale=w.w1_gs, out_global_scale=b.a2_gs) if two else {}
    gs2 = dict(a_global_scale=b.a2_gs, b_global_scale=w.w2_gs) if two else {}
    gather1 = dict(a_gather=b.perm_token, a_gather_rows=T) if b.gather else {}

    def step(events=None, x_in=None, logits_in=None, y_out=None):
        x_in = x_d if x_in is None else x_in
        logits_in = logits_d if logits_in is None else logits_in
        y_out = b.y if y_out is None else y_out
        if events:
            events[0].record(stream)
        if two:                                  # x's encode scale, per batch (timed with routing)
            nv.nvfp4_global_scale(x_in, b.x_gs)
        nv.moe_route_permute(logits_in, x_in, k, b.topk_ids, b.topk_w, b.counts, b.offsets, b.perm_token,
                             b.inv_perm, b.a1_q, b.a1_sf, b.workspace, x_global_scale=b.x_gs if two else None,
                             x_q=b.x_q)
        if events:
            events[1].record(stream)
        nv.nvfp4_grouped_gemm(b.x_q if b.gather else b.a1_q, b.a1_sf, R, b.offsets, b.counts, E, 2 * I, H,
                              w.w1_q, w.w1_sf, 1.0, nv.EPI_SWIGLU_NVFP4, out_q=b.a2_q, out_sf=b.a2_sf, **gs1,
                              **gather1)
        if events:
            events[2].record(stream)
        nv.nvfp4_grouped_gemm(b.a2_q, b.a2_sf, R, b.offsets, b.counts, E, H, I, w.w2_q, w.w2_sf, 1.0,
                              nv.EPI_BF16, out_bf16=b.rows_out, **gs2)
        if events:
            events[3].record(stream)
        shared_rows = None if sh is None else sh.forward(x_in)
        if events:
            events[4].record(stream)
        nv.moe_combine(b.rows_out, b.inv_perm, b.topk_w, y_out, shared=shared_rows)
        if events:
            events[5].record(stream)

    # --overlap-combine (the serving pipeline): batches alternate between two
    # buffer sets; step i routes batch i, runs batch i-1's L2 GEMM with batch i's
    # staging on its side warps, then batch i's L1 GEMM with batch i-1's combine
    # on its side warps; finish_ov runs the last batch's L2 GEMM and combine
    ov = args.overlap_combine
    sets = [b, pipeline.MoeBuffers(s)] if ov else [b]
    n_done = [0]                       # batches stepped since the pipeline was empty

    def l1_call(cur, job=None):
        nv.nvfp4_grouped_gemm(cur.a1_q, cur.a1_sf, R, cur.offsets, cur.counts, E, 2 * I, H, w.w1_q, w.w1_sf, 1.0,
                              nv.EPI_SWIGLU_NVFP4, out_q=cur.a2_q, out_sf=cur.a2_sf, side_combine=job)

    def l2_call(cur, stage=None):
        nv.nvfp4_grouped_gemm(cur.a2_q, cur.a2_sf, R, cur.offsets, cur.counts, E, H, I, w.w2_q, w.w2_sf, 1.0,
                              nv.EPI_BF16, out_bf16=cur.rows_out, side_stage=stage)

    def step_ov(events=None):
        i = n_done[0]
        cur, prev = sets[i & 1], (sets[(i - 1) & 1] if i > 0 else None)
        if events:
            events[0].record(stream)
        nv.moe_route_permute(logits_d, x_d, k, cur.topk_ids, cur.topk_w, cur.counts, cur.offsets, cur.perm_token,
                             cur.inv_perm, cur.a1_q if prev is None else None,
                             cur.a1_sf if prev is None else None, cur.workspace)
        if events:
            events[1].record(stream)
        if prev is not None:
            l2_call(prev, dict(x=x_d, inv_perm=cur.inv_perm, counts=cur.counts, offsets=cur.offsets,
                               a1_q=cur.a1_q, a1_sf=cur.a1_sf))
        if events:
            events[2].record(stream)
        l1_call(cur, None if prev is None else (prev.rows_out, prev.inv_perm, prev.topk_w, prev.y))
        if events:
            events[3].record(stream)
        n_done[0] += 1

    def finish_ov():
        last = sets[(n_done[0] - 1) & 1]
        l2_call(last)
        nv.moe_combine(last.rows_out, last.inv_perm, last.topk_w, last.y)
        n_done[0] = 0

    if ov:
        step = step_ov                 # noqa: F811 (the overlapped step replaces the plain one)

    ceiling = mma_ceiling(nv)
    # the clock sampler starts before the warm-up so that no idle gap (in which the
    # GPU drops its clocks) separates the warm-up from the timed region
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    for _ in range(args.warmup):
        step()
    if ov:
        finish_ov()                    # the timed region starts with the pipeline empty
    nv.nvfp4_device_status()
    torch.cuda.synchronize()

    # ---- timed region: inputs resident in HBM
    barrier(world)
    torch.cuda.synchronize()
    t_region = time.time()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(args.steps):
        step(ev[i])
    if ov:
        tail0 = torch.cuda.Event(enable_timing=True)
        tail0.record(stream)
        finish_ov()
    end.record(stream)
    torch.cuda.synchronize()
    t_region_end = time.time()
    # in the pipeline the sampler keeps running for the GEMMs timed alone below (NVML only)
    keep = ov and clocks.nvml is not None
    clk = clocks.window(t_region, t_region_end) if keep else clocks.stop(t_region, t_region_end)
    # the SM clock the MMA probe sees right after the region (clock64 over
    # globaltimer), beside its reading before the warm-up: NVML's reading can stay
    # at the maximum while the clock under load is lower
    clk = dict(clk, probe_sm_mhz_before=ceiling["sm_mhz"], probe_sm_mhz_after=nv.nvfp4_mma_peak_probe(2000)[1])
    barrier(world)
    nv.nvfp4_device_status()
    ms_local = start.elapsed_time(end)
    ms = max_over_ranks(ms_local, world)
    if ov:
        # steps 1.. (the first has no previous batch): routing without staging, the
        # previous batch's L2 with this batch's staging, this batch's L1 with the
        # previous batch's combine
        full = range(1, args.steps) if args.steps > 1 else range(args.steps)
        per = {name: statistics.mean(ev[i][j].elapsed_time(ev[i][j + 1]) for i in full)
               for j, name in enumerate(("route_permute", "l2_gemm_bf16", "l1_gemm_swiglu_nvfp4"))}
        per["combine"] = 0.0           # inside each step's L1 (the previous batch's)
        per["first_step_route_with_staging"] = ev[0][0].elapsed_time(ev[0][1])
        per["last_batch_l2_and_combine_once"] = tail0.elapsed_time(end)
    else:
        names = ("route_permute", "l1_gemm_swiglu_nvfp4", "l2_gemm_bf16", "shared_expert", "combine")
        per = {name: statistics.mean(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(args.steps))
               for j, name in enumerate(names) if name != "shared_expert" or sh is not None}


    # in the pipeline each L1 launch also streams the previous batch's combine and
    # each L2 launch stages the next batch: time both GEMMs alone and with their
    # side jobs in one block after the timed region (3 untimed rounds, then 10
    # rounds of the four launches, interleaved so that all four see the same state
    # of the GPU), with its own clock samples. The block starts after a second's
    # rest: at the end of the region the GPU's power limit has already lowered the
    # clock (probe_sm_mhz_after), and the block is to see the state the region
    # started in.
    alone = None
    if ov:
        time.sleep(1.0)
        cur, other = sets[0], sets[1]
        comb = (other.rows_out, other.inv_perm, other.topk_w, other.y)
        stage = dict(x=x_d, inv_perm=other.inv_perm, counts=other.counts, offsets=other.offsets,
                     a1_q=other.a1_q, a1_sf=other.a1_sf)
        calls = (lambda: l1_call(cur), lambda: l2_call(cur), lambda: l1_call(cur, comb),
                 lambda: l2_call(cur, stage))
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(13)]
        t_alone = time.time()
        for e in evs:
            e[0].record(stream)
            for j, fn in enumerate(calls):
                fn()
                e[j + 1].record(stream)
        torch.cuda.synchronize()
        alone_clk = clocks.stop(t_alone, time.time()) if keep else None
        med = [statistics.median(e[j].elapsed_time(e[j + 1]) for e in evs[3:]) for j in range(4)]
        alone = {"l1_ms": med[0], "l2_ms": med[1], "l1_with_combine_ms": med[2], "l2_with_staging_ms": med[3],
                 "clocks": alone_clk}

    l1, l2 = ffn_flops(T, H, I, k)
    step_flops = l1 + l2
    if sh is not None:                      # the shared expert: one dense L1 + L2 per token
        shared_l1, shared_l2 = ffn_flops(T, H, I, 1)
        step_flops += shared_l1 + shared_l2
    value = world * args.steps * step_flops / (ms * 1e-3) / 1e12
    tokens_per_s = world * args.steps * T / (ms * 1e-3)

    # ---- end to end: every step copies its inputs in from pinned host memory and
    # its y out to pinned host memory, inside the timed region.
    x_h = x_t.pin_memory()
    logits_h = torch.from_numpy(logits_np).pin_memory()
    plain = not (args.gather or args.two_level or args.shared_expert)
    time.sleep(1.0)                            # from the state the timed region started in, as above
    e2e_steps = max(args.steps, 2)             # both buffer sets take part
    if plain:
        y_ref = b.y.cpu()                      # the resident run's y (the same inputs every step)
        if ov and not torch.equal(sets[1].y.cpu(), y_ref):
            raise RuntimeError("pipeline: the two buffer sets' y differ")
        e2e = e2e_step_host if ov else e2e_host_call
        e2e_ms, e2e_how = e2e(nv, pipeline, s, w, b, x_h, logits_h, k, e2e_steps, world, y_ref)
    else:
        e2e_ms, e2e_how = e2e_copy_streams(step, x_d, logits_d, b, x_h, logits_h, T, H, stream, e2e_steps, world)
    e2e_value = world * e2e_steps * step_flops / (e2e_ms * 1e-3) / 1e12

    # the metric's second half: the standalone SwiGLU + NVFP4 quantiser on its own
    # workload (BF16 gate/up 32768 x 2x2048), timed after the FFN step with its own
    # clock samples, against the HBM copy bandwidth
    del x_h, logits_h
    torch.cuda.empty_cache()
    q_ms, q_bytes, q_clk = time_quantizer(nv, local, steps=50, warmup=5)

    # sustained: the serving pipeline run without a break for about a second. The
    # timed region above is a burst of tens of ms; held for longer, the GPU's power
    # limit lowers its clocks and each step takes longer. Reported beside value.
    sustained = None
    if ov:
        n_sus = max(args.steps, int(1000.0 / (ms / args.steps)))
        sampler = ClockSampler(local)
        sampler.start()
        time.sleep(0.3)
        for _ in range(args.warmup):
            step()
        finish_ov()
        barrier(world)
        torch.cuda.synchronize()
        t_sus = time.time()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        for _ in range(n_sus):
            step()
        finish_ov()
        s1.record(stream)
        torch.cuda.synchronize()
        sus_clk = sampler.stop(t_sus, time.time())
        nv.nvfp4_device_status()
        sus_ms = max_over_ranks(s0.elapsed_time(s1), world)
        sustained = {"steps": n_sus, "ms_per_step": sus_ms / n_sus,
                     "value": world * n_sus * step_flops / (sus_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                     "what": "the same pipeline and inputs, about one second without a break", "clocks": sus_clk}

    if rank != 0:
        return
    # launches per grouped GEMM: the prefill batch's are split (CTA pairs beside a
    # single-CTA launch), a gathering L1 is not
    l2_n = 2 if args.workload == WORKLOAD else 1
    l1_n = 2 if args.workload == WORKLOAD and not args.gather else 1
    pk = peaks()
    # a sub-second region at the maximum SM clock: the burst BF16 figure x the
    # nominal FP4 / BF16 dense ratio
    fp4_peak = pk["bf16"] * FP4_OVER_BF16
    l1_ms = per["l1_gemm_swiglu_nvfp4"]
    achieved = l1 / (l1_ms * 1e-3) / 1e12
    # the probe runs outside the timed region, at whatever clock it met: its rate
    # scaled to the timed region's median SM clock is the ceiling the kernel faced
    ceiling = dict(ceiling)
    if clk.get("sm_mhz") and ceiling.get("sm_mhz"):
        ceiling["value_at_region_clock"] = ceiling["value"] * clk["sm_mhz"] / ceiling["sm_mhz"]
        ceiling["region_sm_mhz"] = clk["sm_mhz"]
    ceil_tf = ceiling.get("value_at_region_clock", ceiling["value"])
    q_gbs = q_bytes / (q_ms * 1e-3) / 1e9
    quantize = {"workload": "SwiGLU+NVFP4 quantiser, BF16 gate/up (32768, 2x2048), Student-t(3)x0.5 with planted "
                            "tiny, saturating and tie blocks",
                "kernel": "quantize_kernel<SWIGLU_GU8>", "value": q_gbs, "unit": "GB/s", "ms_per_launch": q_ms,
                "bound": "hbm", "peak": pk["hbm_gbs"], "frac": q_gbs / pk["hbm_gbs"],
                "peak_source": f"{pk['source']} copy bandwidth",
                "algorithmic": f"{q_bytes} bytes per launch (BF16 gate/up read, nibbles + swizzled SF written)",
                "launch": "50 launches replayed from one CUDA graph after 5 eager ones; inputs larger than L2",
                "gpu_launches": 50, "clocks": q_clk}
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        r = OracleArm(dict(inputs.CONFIGS[args.workload])).run(budget_s=args.cpu_budget, max_tokens=4096)
        cpu = {"value": r["tflops"], "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"{r['tokens']} sampled tokens of the {args.workload} batch in {r['seconds']:.1f} s "
                         "(float64 numpy; BLAS threads = cores, elementwise single-threaded)"}
    # the traffic records were taken on the plain prefill and decode steps
    tensor_view = {"achieved": achieved, "peak": fp4_peak, "unit": "TFLOP/s", "frac": achieved / fp4_peak,
                   "peak_source": f"{pk['source']} bf16 burst {pk['bf16']} x {FP4_OVER_BF16:g} "
                                  "(nominal FP4/BF16 dense ratio)",
                   "algorithmic": "2*T*k*(2I)*H FLOP per launch (real rows only)"}
    l2_ms = per["l2_gemm_bf16"]
    gemms = {"l2_achieved": l2 / (l2_ms * 1e-3) / 1e12, "l2_frac": l2 / (l2_ms * 1e-3) / 1e12 / fp4_peak,
             "l1_l2_achieved": (l1 + l2) / ((l1_ms + l2_ms) * 1e-3) / 1e12,
             "l1_l2_frac": (l1 + l2) / ((l1_ms + l2_ms) * 1e-3) / 1e12 / fp4_peak}
    if args.workload == "decode":
        # a few rows per expert: the L1 GEMM streams the touched experts' weights
        touched = int((b.counts > 0).sum().item())
        rows = T * k
        l1_bytes = touched * (2 * I) * (H // 2 + H // 16) + rows * (H // 2 + H // 16) + rows * (I // 2 + I // 16)
        gbs = l1_bytes / (l1_ms * 1e-3) / 1e9
        traffic = l1_traffic("decode") if plain else None
        roofline = {"kernel": "L1 GEMM + SwiGLU + NVFP4 epilogue: nvf4_gemm_kernel<0, 256> (single CTAs)",
                    "bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                    "frac": gbs / pk["hbm_gbs"], "peak_source": f"{pk['source']} copy bandwidth",
                    "peak_note": ("the copy peak moves half its bytes each way; this kernel almost only reads, "
                                  "and DRAM reads alone stream a little faster than a copy, so frac can pass 1"),
                    "algorithmic": (f"W1 and its scales of the {touched} experts the batch touches, plus A1 read "
                                    f"and A2 written for the T*k real rows: {l1_bytes} bytes per launch"),
                    "traffic": traffic,
                    "traffic_unit": "bytes per launch (dram read + write)",
                    "traffic_gbs": traffic / (l1_ms * 1e-3) / 1e9 if traffic else None,
                    "tensor_view": dict(tensor_view, instruction_ceiling=ceil_tf)}
    else:
        side = None
        if ov and args.workload == WORKLOAD:
            comb_bytes = T * k * H * 2 + T * H * 2 + T * k * 8
            n_real = int(b.counts.sum().item())
            stage_bytes = T * H * 2 + n_real * (H // 2 + H // 16) + T * k * 4
            a = alone
            side = {"l1": {"what": "each L1 launch also runs the previous batch's combine on two spare warps per CTA",
                           "bytes": comb_bytes, "gbs_over_launch": comb_bytes / (l1_ms * 1e-3) / 1e9,
                           "l1_alone_ms": a["l1_ms"], "l1_with_combine_ms": a["l1_with_combine_ms"],
                           "l1_alone_achieved": l1 / (a["l1_ms"] * 1e-3) / 1e12,
                           "l1_alone_frac": l1 / (a["l1_ms"] * 1e-3) / 1e12 / fp4_peak},
                    "l2": {"what": "each L2 launch also stages the next batch's activation (x quantised once per "
                                   "token, written into its k permuted rows) on two spare warps per CTA",
                           "bytes": stage_bytes, "gbs_over_launch": stage_bytes / (l2_ms * 1e-3) / 1e9,
                           "l2_alone_ms": a["l2_ms"], "l2_with_staging_ms": a["l2_with_staging_ms"],
                           "l2_alone_achieved": l2 / (a["l2_ms"] * 1e-3) / 1e12,
                           "l2_alone_frac": l2 / (a["l2_ms"] * 1e-3) / 1e12 / fp4_peak},
                    "measured": ("after the timed region: 3 untimed rounds, then the median of 10 rounds of L1 "
                                 "alone, L2 alone, L1 with a combine, L2 with a staging (interleaved)"),
                    "clocks": a["clocks"]}
        roofline = dict({"kernel": ("L1 GEMM + SwiGLU + NVFP4 epilogue: nvf4_gemm_pair_kernel<0> (CTA pairs, all but "
                                    "8 SMs) with nvf4_gemm_kernel<0, 256> beside it on 8 SMs (the last block of the "
                                    "thinnest odd groups)"
                                    if args.workload == WORKLOAD else
                                    "L1 GEMM + SwiGLU + NVFP4 epilogue: nvf4_gemm_kernel<0, 256> (single CTAs)"),
                         "bound": "tensor"}, **tensor_view, side_job=side,
                        traffic=(l1_traffic("prefill_overlap" if ov else "prefill")
                                 if plain and args.workload == WORKLOAD else None),
                        traffic_unit="bytes per launch (dram read + write)",
                        gemms=gemms,
                        instruction_ceiling=dict(ceiling, frac=achieved / ceil_tf))
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "nvfp4 (e2m1 x e4m3/16) -> fp32 accum", "data": "synthetic",
        "config": {"workload": _workload_name(spec, args.workload), "tokens_per_rank": T, "rows_padded_max": R,
                   "l2_policy": "inputs larger than L2 (5.7 GB of expert weights, 0.6 GB staged activations)",
                   "parallelism": f"replicas x{world} (independent batches)",
                   "scales": ("two-level: per-tensor encode scales for x (computed each step), W1/W2 "
                              "(per expert) and the L1 output (calibrated once), plus the per-16 E4M3 scales"
                              if args.two_level else "per-16 E4M3 block scales (global scale 1)"),
                   "shared_expert": (f"one shared expert (I={I}) on every token, FLOPs credited"
                                     if args.shared_expert else "none"),
                   "combine": ("serving pipeline: each batch's staging runs inside the previous batch's L2 GEMM and "
                               "its combine inside the next batch's L1 GEMM (two spare warps per CTA each); the "
                               "region starts with the pipeline empty and ends with the last batch's L2 and combine"
                               if ov else "every stage its own launch, each batch's whole path in its own step")},
        "tokens_per_s": tokens_per_s,
        "kernel_ms": per,
        "roofline": roofline,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": T * H * 2 + T * E * 4,
                "d2h_bytes_per_step": T * H * 2, "steps": e2e_steps, "ms_per_step": e2e_ms / e2e_steps,
                "copies": e2e_how},
        # per step: top-k, offsets, assign, scatter, L1, L2, combine (+ x's amax and
        # its finalisation with --two-level; + the shared expert's quantise, L1, L2);
        # the pipeline: top-k, offsets, assign, L2 (+ staging), L1 (+ combine) per
        # step (the first: scatter in place of L2), then the last L2 and combine.
        # On the prefill batch each grouped GEMM is two launches (CTA pairs, and
        # the single-CTA launch beside it over the thinnest odd groups' last
        # blocks), except a gathering L1
        "gpu_launches": (4 + l1_n + (args.steps - 1) * (3 + l1_n + l2_n) + l2_n + 1 if ov else
                         (5 + l1_n + l2_n + (2 if args.two_level else 0) + (3 if args.shared_expert else 0))
                         * args.steps),
        "clocks": clk,
        "quantize": quantize,
        "sustained": sustained,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line))


def _flush_l2(buf):
    buf.add_(1)                         # writes 256 MiB: evicts the 129 MB L2


def run_dense(args, world: int, rank: int, local: int) -> None:
    """One dense NVFP4 GEMM: the single-expert L1 (A 8192 x 7168 x B 4096 x 7168 with
    the fused SwiGLU + NVFP4 epilogue -> 8192 x 2048 NVFP4), or with --workload
    dense_l2 the prefill batch's L2 shape as one group (A 16384 x 2048 x B 7168 x 2048
    -> 16384 x 7168 BF16).  Inputs fit in L2, so L2 is flushed between steps and each
    step is timed by its own CUDA events."""
    import torch

    import nvfp4_block_scaled_moe_gb300 as nv
    from nvfp4_block_scaled_moe_gb300 import build as nvbuild

    nvbuild.build()
    torch.cuda.set_device(local)
    spec = dict(inputs.CONFIGS["dense" if args.workload == "dense_swiglu_bf16" else args.workload])
    M, N, K = spec["M"], spec["N"], spec["K"]
    bf16_out = spec.get("epilogue") == "bf16"
    compact = args.workload == "dense_swiglu_bf16"     # the compact BF16 SwiGLU output (compatibility path)
    a, bw = inputs.dense_inputs(spec)
    a_d, b_d = torch.from_numpy(a).cuda(), torch.from_numpy(bw).cuda()
    a_q = torch.empty((M, K // 2), dtype=torch.uint8, device="cuda")
    a_sf = torch.empty(nv.sf_bytes(M, K), dtype=torch.uint8, device="cuda")
    b_q = torch.empty((N, K // 2), dtype=torch.uint8, device="cuda")
    b_sf = torch.empty(nv.sf_bytes(N, K), dtype=torch.uint8, device="cuda")
    nv.nvfp4_quantize(a_d, K, nv.MODE_PLAIN, a_q, a_sf)
    nv.nvfp4_quantize(b_d, K, nv.MODE_PLAIN, b_q, b_sf)
    del a_d, b_d
    out_q = torch.empty((M, N // 4), dtype=torch.uint8, device="cuda")
    out_sf = torch.empty(nv.sf_bytes(M, N // 2), dtype=torch.uint8, device="cuda")
    out_bf16 = (torch.empty((M, N), dtype=torch.bfloat16, device="cuda") if bf16_out else
                torch.empty((M, N // 2), dtype=torch.bfloat16, device="cuda") if compact else None)
    flush = torch.zeros(64 << 20, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        if bf16_out:
            nv.nvfp4_grouped_gemm(a_q, a_sf, M, None, None, 1, N, K, b_q, b_sf[None], 1.0, nv.EPI_BF16,
                                  out_bf16=out_bf16)
        elif compact:
            nv.nvfp4_grouped_gemm(a_q, a_sf, M, None, None, 1, N, K, b_q, b_sf[None], 1.0, nv.EPI_SWIGLU_BF16,
                                  out_bf16=out_bf16)
        else:
            nv.nvfp4_grouped_gemm(a_q, a_sf, M, None, None, 1, N, K, b_q, b_sf[None], 1.0, nv.EPI_SWIGLU_NVFP4,
                                  out_q=out_q, out_sf=out_sf)

    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    ceiling = mma_ceiling(nv)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    for _ in range(args.warmup):
        _flush_l2(flush)
        step()
    nv.nvfp4_device_status()
    torch.cuda.synchronize()
    # each timed step replays a one-launch CUDA graph right after the L2 flush, so
    # the host-side launch path (tensor-map encoding included) overlaps the flush
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    t_region = time.time()
    for e0, e1 in evs:
        _flush_l2(flush)
        e0.record(stream)
        graph.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop(t_region, time.time())
    nv.nvfp4_device_status()
    ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in evs)
    flops = 2.0 * M * N * K
    tflops = flops / (ms * 1e-3) / 1e12
    pk = peaks()
    if clk.get("sm_mhz") and ceiling.get("sm_mhz"):
        ceiling = dict(ceiling, value_at_region_clock=ceiling["value"] * clk["sm_mhz"] / ceiling["sm_mhz"],
                       region_sm_mhz=clk["sm_mhz"])
    fp4_peak = pk["bf16"] * FP4_OVER_BF16
    print(json.dumps({
        "metric": METRIC, "value": tflops, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "nvfp4 (e2m1 x e4m3/16) -> fp32 accum", "data": "synthetic",
        "config": {"workload": f"dense NVFP4 GEMM M={M} N={N} K={K} + "
                               + ("BF16 output" if bf16_out else "SwiGLU -> compact BF16 output" if compact
                                  else "SwiGLU + NVFP4 requant"),
                   "l2_policy": "L2 flushed (256 MiB write) before every step; per-step CUDA events",
                   "launch": "each step a one-launch CUDA graph replayed after the flush"},
        "roofline": {"kernel": ("nvf4_gemm_pair_kernel<1> (BF16 epilogue, CTA pairs)" if bf16_out else
                                "nvf4_gemm_pair_kernel<2> (compact BF16 SwiGLU epilogue, CTA pairs)" if compact else
                                "nvf4_gemm_pair_kernel<0> (SwiGLU + NVFP4 epilogue, CTA pairs)"), "bound": "tensor",
                     "achieved": tflops,
                     "peak": fp4_peak, "unit": "TFLOP/s", "frac": tflops / fp4_peak,
                     "peak_source": f"{pk['source']} bf16 burst {pk['bf16']} x {FP4_OVER_BF16:g}",
                     "algorithmic": "2*M*N*K FLOP per launch", "traffic": None,
                     "instruction_ceiling": dict(ceiling, frac=tflops / ceiling.get("value_at_region_clock",
                                                                                     ceiling["value"]))},
        "gpu_launches": args.steps, "clocks": clk}))


def run_hbm_stage(args, world: int, rank: int, local: int) -> None:
    """One HBM-bound stage of the prefill step on its own: --workload route times
    moe_route_permute (top-k, offsets, ranks, x quantised into its k permuted
    rows, padding zeroed) on the prefill batch's logits and x; --workload combine
    times moe_combine on that batch's routing with seeded random BF16 rows in
    place of the L2 output.  Inputs are larger than L2; the K timed launches are
    replayed from one CUDA graph."""
    import torch

    import nvfp4_block_scaled_moe_gb300 as nv
    from nvfp4_block_scaled_moe_gb300 import build as nvbuild
    from nvfp4_block_scaled_moe_gb300 import pipeline

    nvbuild.build()
    torch.cuda.set_device(local)
    spec = dict(inputs.CONFIGS["prefill"])
    T, H, I, E, k = spec["T"], spec["H"], spec["I"], spec["E"], spec["top_k"]
    s = pipeline.MoeShape(T=T, H=H, I=I, E=E, top_k=k)
    b = pipeline.MoeBuffers(s)
    x_t, _ = inputs.moe_x(spec)
    x_d = x_t.cuda()
    logits_d = torch.from_numpy(inputs.moe_logits(spec)).cuda()

    def route():
        nv.moe_route_permute(logits_d, x_d, k, b.topk_ids, b.topk_w, b.counts, b.offsets, b.perm_token,
                             b.inv_perm, b.a1_q, b.a1_sf, b.workspace)

    route()
    nv.nvfp4_device_status()
    R_pad = int(b.offsets[-1].item())
    if args.workload == "route":
        step = route
        nbytes = (T * E * 4 + T * H * 2 + R_pad * (H // 2 + H // 16) + T * k * 12 + R_pad * 4)
        kernel = "route_scatter_kernel (with top-k, offsets and rank kernels)"
        what = ("logits + x read, the permuted NVFP4 rows and scale words (padding rows included), "
                "ids, weights, inv_perm and perm_token written")
    else:
        g = torch.Generator(device="cuda").manual_seed(spec["seed"] + 7)
        b.rows_out.copy_(torch.randn(b.rows_out.shape, generator=g, device="cuda", dtype=torch.bfloat16))
        del x_d
        torch.cuda.empty_cache()

        def step():
            nv.moe_combine(b.rows_out, b.inv_perm, b.topk_w, b.y)
        nbytes = T * k * H * 2 + T * H * 2 + T * k * 8
        kernel = "combine_kernel"
        what = "the k BF16 rows of every token read, y written, inv_perm and weights read"
    stream = torch.cuda.current_stream()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    for _ in range(args.warmup):
        step()
    nv.nvfp4_device_status()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(args.steps):
            step()
    graph.replay()                      # untimed
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_region = time.time()
    e0.record(stream)
    graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop(t_region, time.time())
    nv.nvfp4_device_status()
    ms = e0.elapsed_time(e1) / args.steps
    gbs = nbytes / (ms * 1e-3) / 1e9
    pk = peaks()
    print(json.dumps({
        "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 -> nvfp4" if args.workload == "route" else "bf16 (fp32 accumulate)", "data": "synthetic",
        "config": {"workload": f"{args.workload} stage of the prefill MoE FFN (T={T}, H={H}, E={E}, top-{k})",
                   "l2_policy": "inputs larger than L2", "launch": "the K steps replayed from one CUDA graph"},
        "roofline": {"kernel": kernel, "bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / pk["hbm_gbs"], "algorithmic": f"{nbytes} bytes per step ({what})",
                     "traffic": None},
        "gpu_launches": args.steps * (4 if args.workload == "route" else 1), "clocks": clk}))


def time_quantizer(nv, local: int, steps: int, warmup: int, deinterleave: bool = False, clocks: bool = True):
    """The standalone SwiGLU + NVFP4 quantiser on the BF16 gate/up workload
    (32768, 2 x 2048): the K launches replayed from one CUDA graph after `warmup`
    eager ones.  Returns (ms per launch, algorithmic bytes per launch, clocks)."""
    import torch

    spec = dict(inputs.CONFIGS["quantizer"])
    rows, cols = spec["rows"], spec["cols"]
    gu, _ = inputs.quantizer_input(spec)
    gu_d = gu.cuda()
    del gu
    q = torch.empty((rows, cols // 2), dtype=torch.uint8, device="cuda")
    sf = torch.empty(nv.sf_bytes(rows, cols), dtype=torch.uint8, device="cuda")
    mode = nv.MODE_DEINTERLEAVE_GU8 if deinterleave else nv.MODE_SWIGLU_GU8

    def step():
        nv.nvfp4_quantize(gu_d, cols, mode, q, sf)

    sampler = ClockSampler(local) if clocks else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    for _ in range(warmup):
        step()
    nv.nvfp4_device_status()
    torch.cuda.synchronize()
    # the K timed launches are replayed from one CUDA graph, so that the host-side
    # launch path (Python, ctypes, argument checks) cannot leave the GPU idle
    # between 50-microsecond kernels
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(steps):
            step()
    graph.replay()                      # untimed
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_region = time.time()
    e0.record(stream)
    graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    clk = sampler.stop(t_region, time.time()) if sampler else None
    nv.nvfp4_device_status()
    ms = e0.elapsed_time(e1) / steps
    nbytes = rows * 2 * cols * 2 + rows * cols // 2 + nv.sf_bytes(rows, cols)
    del graph, gu_d, q, sf
    torch.cuda.empty_cache()
    return ms, nbytes, clk


def run_quantizer(args, world: int, rank: int, local: int) -> None:
    """The standalone SwiGLU + NVFP4 quantiser on BF16 gate/up (32768, 2 x 2048):
    HBM-bound, 306 MB moved per launch (inputs larger than L2).  With --workload
    quantizer_deinterleave, the compatibility mode that quantises the kept 8 of
    every 16 interleaved slots of the same buffer (an L1 output whose up slots
    already hold SwiGLU values): the kept and dropped halves alternate every 16
    bytes, below the 32-byte DRAM sector, so the whole buffer is read."""
    import torch

    import nvfp4_block_scaled_moe_gb300 as nv
    from nvfp4_block_scaled_moe_gb300 import build as nvbuild

    nvbuild.build()
    torch.cuda.set_device(local)
    spec = dict(inputs.CONFIGS["quantizer"])
    rows, cols = spec["rows"], spec["cols"]
    deinterleave = args.workload == "quantizer_deinterleave"
    kernel = "quantize_kernel<DEINTERLEAVE_GU8>" if deinterleave else "quantize_kernel<SWIGLU_GU8>"
    ms, nbytes, clk = time_quantizer(nv, local, args.steps, args.warmup, deinterleave)
    gbs = nbytes / (ms * 1e-3) / 1e9
    pk = peaks()
    print(json.dumps({
        "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16 -> nvfp4",
        "data": "synthetic",
        "config": {"workload": (f"deinterleave + NVFP4 quantiser of the kept slots, BF16 ({rows}, 2x{cols})"
                                if deinterleave else f"SwiGLU+NVFP4 quantiser BF16 gate/up ({rows}, 2x{cols})"),
                   "l2_policy": "inputs larger than L2 (268 MB read per step)",
                   "launch": "the K steps replayed from one CUDA graph"},
        "roofline": {"kernel": kernel, "bound": "hbm", "achieved": gbs,
                     "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": gbs / pk["hbm_gbs"],
                     "algorithmic": f"{nbytes} bytes per launch (input read + nibbles + SF written)",
                     "traffic": None},
        "gpu_launches": args.steps, "clocks": clk}))


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--gather", action=argparse.BooleanOptionalAction, default=False,
                    help="L1 gathers its A rows from x quantised once in token order (TMA gather4) instead of a "
                         "permuted copy written by the routing call")
    ap.add_argument("--shared-expert", action="store_true",
                    help="prefill/decode plus one shared expert (a dense NVFP4 FFN of every token, I = the "
                         "routed experts' I) added in the combine")
    ap.add_argument("--overlap-combine", action=argparse.BooleanOptionalAction, default=None,
                    help="prefill/decode: each step's L1 GEMM also runs the previous batch's combine on spare warps "
                         "(batches alternate between two buffer sets; the last batch's combine runs after the last "
                         "step, inside the timed region). On by default for the plain prefill step")
    ap.add_argument("--two-level", action="store_true",
                    help="prefill/decode with the two-level scale (per-tensor encode scales next to the per-16 "
                         "ones); the CPU baseline stays the one-level oracle")
    ap.add_argument("--workload", choices=("prefill", "decode", "dense", "dense_l2", "dense_swiglu_bf16", "quantizer",
                                           "quantizer_deinterleave", "route", "combine"), default=WORKLOAD,
                    help="prefill (default) and decode time the whole MoE FFN step; dense times the L1 GEMM of "
                         "one 8192-row expert, dense_l2 the prefill L2 GEMM shape as one group; quantizer the "
                         "standalone SwiGLU + NVFP4 quantiser; dense_swiglu_bf16 and quantizer_deinterleave the "
                         "compatibility paths (the compact BF16 SwiGLU output; deinterleave + quantise); route and "
                         "combine the prefill step's HBM-bound stages on their own")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    variant = args.gather or args.two_level or args.shared_expert
    if args.overlap_combine and variant:
        ap.error("--overlap-combine runs the plain path (no --gather, --two-level or --shared-expert)")
    if args.overlap_combine is None:
        # on by default where L1 runs on CTA pairs (prefill); a decode batch's L1
        # runs on single CTAs, where the combine would be its own launch anyway
        args.overlap_combine = not variant and args.workload == "prefill"
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    elif args.workload in ("dense", "dense_l2", "dense_swiglu_bf16"):
        run_dense(args, world, rank, local)
    elif args.workload in ("quantizer", "quantizer_deinterleave"):
        run_quantizer(args, world, rank, local)
    elif args.workload in ("route", "combine"):
        run_hbm_stage(args, world, rank, local)
    else:
        run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()

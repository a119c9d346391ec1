"""Benchmark: dense tensor-core GEMM C = A * B^T on GB300, through the library's C ABI.

Default workload: BF16 M = N = K = 8192 (the headline configuration), entries uniform in
[-1, 1] from seed 2, FP32 accumulation, BF16 output. One step = one GEMM call on the
next of R rotating input sets whose total footprint exceeds 2x L2, so no step reads
operands left in L2 by the previous one.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config c1..c5] [--impl ours|reference]

Prints ONE JSON line (rank 0). --impl reference times the CPU oracle (FP64, OpenMP over the
host cores) on a bounded sample of the same workload instead.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

CONFIGS = {
    "c1": dict(kind="bf16", M=256, N=256, K=256, seed=0, workload="bf16_gemm_256x256x256"),
    "c2": dict(kind="bf16", M=4096, N=4096, K=4096, seed=1, workload="bf16_gemm_4096x4096x4096"),
    "c3": dict(kind="bf16", M=8192, N=8192, K=8192, seed=2, workload="bf16_gemm_8192x8192x8192"),
    "c4": dict(kind="bf16", M=4000, N=14336, K=4096, seed=3, workload="bf16_gemm_4000x14336x4096_ragged"),
    "c5": dict(kind="nvfp4", M=8192, N=8192, K=8192, seed=4, workload="nvfp4_gemm_8192x8192x8192"),
}
# The page's own number for this metric and workload: "Achieve cuBLAS Performance on NVIDIA
# GB300 for HGEMM", Performance table, v7 at M = N = K = 8192 on GB300.
PAGE_TFLOPS = {"c3": 1980.925}
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "hbm_gbs": 6800.0}
CLC_MODES = {"auto": 0, "on": 1, "off": 2}   # gemm_options_t.clc
NOMINAL_FP4_OVER_BF16 = 13.5 / 2.25   # nominal dense FP4 / BF16 tensor rates (6x)
KERNEL_SOURCES = {
    "bf16": ["csrc/ptx.cuh", "csrc/common.cuh", "csrc/schedule.h", "csrc/gemm_bf16.cu", "csrc/gemm_bf16_wide.cu"],
    "nvfp4": ["csrc/ptx.cuh", "csrc/common.cuh", "csrc/schedule.h", "csrc/gemm_nvfp4.cu"],
}


def kernel_source_hash(kind: str) -> str:
    """Hash of the sources the GEMM kernel of this precision is built from."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, "dense_tensor_core_persistent_gb300", rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def recorded_traffic(workload: str, kind: str):
    """DRAM bytes per launch from the committed ncu summary, if taken on the current kernel sources."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    cur = kernel_source_hash(kind)
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 3 and not line.startswith("#") and parts[0] == workload and parts[1] == cur:
                return int(parts[2])
    return None


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while the timed region runs."""

    MIN_REGION_S = 0.5

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None, start: bool = True):
        self.rows = []
        self.proc = None
        self.t0 = self.t1 = None
        if not start:  # rows supplied by the caller (tests)
            return
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        if uuid:
            cmd += ["-i", uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), line.strip()))

    def wait_first_sample(self, timeout=5.0):
        t = time.time()
        while self.proc and not self.rows and time.time() - t < timeout:
            time.sleep(0.05)

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()

    def window(self, t0, t1):
        """Median SM clock, power and the throttle reasons seen in samples taken in [t0, t1]."""
        rows = [r for (t, r) in self.rows if t0 is not None and t1 is not None and t0 <= t <= t1]
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            f = [x.strip() for x in r.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {
            "sm_mhz": statistics.median(sm) if sm else None,
            "sm_max_mhz": max(smax) if smax else None,
            "power_w_median": statistics.median(power) if power else None,
            "samples": len(sm),
            "reasons": sorted(reasons),
        }

    def summary(self, after=None):
        """Clocks of the timed region. Only samples taken inside it count: when the region is
        shorter than the sampling period and none falls inside, sm_mhz is null and says so
        (`after`, if given, is the window of a continuation of the same launches after the
        timed region, reported separately and labelled as such)."""
        if self.proc is None and not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.stop()
        out = self.window(self.t0, self.t1)
        region_s = (self.t1 - self.t0) if self.t0 and self.t1 else 0.0
        if region_s < self.MIN_REGION_S:
            # nvidia-smi reports values averaged over its last period: in a region this short
            # its few samples (if any) describe the load before the region, not the region
            out = {"sm_mhz": None, "power_w_median": None, "samples": out["samples"], "reasons": [],
                   "note": f"the {region_s * 1e3:.1f} ms timed region is shorter than {self.MIN_REGION_S:.1f} s "
                           "(5 sampling periods of 100 ms): no clock is claimed for it"}
            # the sampler's maximum clock does not depend on load
            out["sm_max_mhz"] = self.window(float("-inf"), float("inf"))["sm_max_mhz"]
        if after is not None:
            cont = self.window(*after)
            cont["what"] = (f"untimed continuation of the same launches for {(after[1] - after[0]):.2f} s "
                            "right after the timed region")
            out["after_region"] = cont
        return out


# ------------------------------------------------------------------ distributed plumbing

def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("nccl" if n_gpus > 0 else "gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ workloads

def make_inputs(cfg, r, device, scales="rowmajor"):
    """Rotation set r on the device. NVFP4 scales are drawn row-major; for the blocked path
    they are rearranged once here by the library's pack kernel (input preparation, like
    packing two E2M1 codes per byte), outside the timed region."""
    import synthetic_inputs as si
    seed = si.rotation_seed(cfg["seed"], r)
    if cfg["kind"] == "bf16":
        return si.bf16_problem(seed, cfg["M"], cfg["N"], cfg["K"], device=device)
    a, sfa, b, sfb = si.nvfp4_problem(seed, cfg["M"], cfg["N"], cfg["K"], device=device)
    if scales == "blocked":
        import dense_tensor_core_persistent_gb300 as g
        sfa, sfb = g.pack_scales(sfa), g.pack_scales(sfb)
    return a, sfa, b, sfb


def set_bytes(cfg):
    M, N, K = cfg["M"], cfg["N"], cfg["K"]
    if cfg["kind"] == "bf16":
        return 2 * (M * K + N * K) + 2 * M * N
    return (M * K + N * K) // 2 + (M * K + N * K) // 16 + 2 * M * N


# Fused epilogues selectable with --epilogue: (alpha, beta, with bias, activation name).
EPILOGUES = {
    "none": None,
    "relu_bias": (1.0, 0.0, True, "relu"),
    "gelu_beta_bias": (0.5, 1.0, True, "gelu_tanh"),
}


def make_epilogue(g, name, N, device):
    import torch
    spec = EPILOGUES[name]
    if spec is None:
        return None
    alpha, beta, with_bias, act = spec
    gen = torch.Generator().manual_seed(7)
    bias = torch.empty(N).uniform_(-1, 1, generator=gen).to(torch.bfloat16).to(device) if with_bias else None
    code = {"relu": g.GEMM_ACT_RELU, "gelu_tanh": g.GEMM_ACT_GELU_TANH}[act]
    ep = g.epilogue(alpha, beta, bias, code)
    ep._bias_keepalive = bias
    return ep


def launch(g, cfg, ins, C, stream, opts, scales="rowmajor", epi=None):
    M, N, K = cfg["M"], cfg["N"], cfg["K"]
    if epi is not None:
        if cfg["kind"] == "bf16":
            g.gemm_bf16_fused(ins[0], ins[1], C, M, N, K, epi, stream, opts)
        elif scales == "blocked":
            g.gemm_nvfp4_blocked_fused(ins[0], ins[1], ins[2], ins[3], C, M, N, K, epi, stream, opts)
        else:
            g.gemm_nvfp4_fused(ins[0], ins[1], ins[2], ins[3], C, M, N, K, epi, stream, opts)
        return
    if cfg["kind"] == "bf16":
        g.gemm_bf16(ins[0], ins[1], C, M, N, K, stream, opts)
    elif scales == "blocked":
        g.gemm_nvfp4_blocked(ins[0], ins[1], ins[2], ins[3], C, M, N, K, stream, opts)
    else:
        g.gemm_nvfp4(ins[0], ins[1], ins[2], ins[3], C, M, N, K, stream, opts)


PROBE_CTAS = 4096  # clock-probe records per launch (the persistent grids use at most 152 CTAs)


def summarize_probes(g, probes):
    """Median over the probed launches of each launch's median CTA clock (MHz)."""
    per = [g.clock_probe_mhz(p) for p in probes]
    per = [r for r in per if r.get("ctas")]
    if not per:
        return None
    mhz = sorted(r["sm_mhz"] for r in per)
    return {"sm_mhz": mhz[len(mhz) // 2], "sm_mhz_min": mhz[0], "sm_mhz_max": mhz[-1], "launches_probed": len(per),
            "ctas_per_launch": per[0]["ctas"],
            "what": ("SM clock inside the GEMM: each CTA's clock64 over %globaltimer from the start to the end of "
                     "its work (median over the CTAs), on every launch of the timed region that carried a probe "
                     "(gemm_options_t.clock_probe; median over those launches)")}


def cpu_model() -> str:
    """The host CPU's model, from /proc/cpuinfo (x86: "model name"; Arm: implementer and part codes)."""
    try:
        fields = {}
        with open("/proc/cpuinfo") as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    fields.setdefault(k.strip(), v.strip())
        if "model name" in fields:
            return fields["model name"]
        arm_parts = {"0xd4f": "Neoverse V2", "0xd40": "Neoverse V1", "0xd0c": "Neoverse N1", "0xd49": "Neoverse N2"}
        part = fields.get("CPU part", "?")
        return f"Arm implementer {fields.get('CPU implementer', '?')} part {part} ({arm_parts.get(part, 'unknown part')})"
    except OSError:
        return "unknown"


def oracle_rows(cfg, ins_cpu, rows):
    import oracle
    if cfg["kind"] == "bf16":
        return oracle.gemm_bf16(ins_cpu[0], ins_cpu[1], 0, rows)
    return oracle.gemm_nvfp4(*ins_cpu, 0, rows)


def cpu_baseline(cfg, target_s=10.0):
    """The oracle as it stands on the host cores, on a bounded sample: the first `rows` rows
    of C (all N columns, full K). Rows are sized from a short calibration run."""
    import oracle
    import synthetic_inputs as si
    M, N, K = cfg["M"], cfg["N"], cfg["K"]
    oracle.build()
    cal = min(M, 4 * oracle.num_threads())
    ins_cpu = make_sample_inputs(cfg, cal)
    t = time.perf_counter()
    oracle_rows(cfg, ins_cpu, cal)
    t_cal = max(time.perf_counter() - t, 1e-4)
    rows = int(max(1, min(M, cal * target_s / t_cal)))
    ins_cpu = make_sample_inputs(cfg, rows)
    t = time.perf_counter()
    oracle_rows(cfg, ins_cpu, rows)
    dt = time.perf_counter() - t
    flops = 2.0 * rows * N * K
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(), "cpu": cpu_model(),
            "kind": "oracle",
            "sample": f"first {rows} of {M} rows of C (all {N} columns, K={K}), FP64, {dt:.1f} s",
            "seconds": dt, "rows": rows}


def make_sample_inputs(cfg, rows):
    """Rows 0..rows-1 of A (and SFA) plus all of B (and SFB) of rotation set 0, on the host."""
    import synthetic_inputs as si
    M, N, K = cfg["M"], cfg["N"], cfg["K"]
    seed = cfg["seed"]
    if cfg["kind"] == "bf16":
        A = si.uniform_bf16(seed, si.TENSOR_A, rows, K)
        B = si.uniform_bf16(seed, si.TENSOR_B, N, K)
        return (A, B)
    a = si.e2m1_codes_packed(seed, si.TENSOR_A, rows, K)
    b = si.e2m1_codes_packed(seed, si.TENSOR_B, N, K)
    sfa = si.e4m3_scales(seed, si.TENSOR_SFA, rows, K // 16)
    sfb = si.e4m3_scales(seed, si.TENSOR_SFB, N, K // 16)
    return (a, sfa, b, sfb)


# ------------------------------------------------------------------ arms

def oracle_at(cfg, ins_cpu, rows, cols):
    import oracle
    if cfg["kind"] == "bf16":
        return oracle.gemm_bf16_at(ins_cpu[0], ins_cpu[1], rows, cols)
    return oracle.gemm_nvfp4_at(*ins_cpu, rows, cols)


def run_reference(args, cfg, world, rank):
    """The oracle as it stands, on the host cores: each step computes a fixed bounded sample
    of output elements of the workload (sized so warm-up + timed steps take about 2 minutes)."""
    if rank != 0:
        return
    import numpy as np

    import oracle
    M, N, K = cfg["M"], cfg["N"], cfg["K"]
    oracle.build()
    sample_rows = min(M, 64)
    ins_cpu = make_sample_inputs(cfg, sample_rows)
    rng = np.random.default_rng(cfg["seed"])
    total = args.steps + args.warmup
    budget = args.ref_seconds
    cal = 256
    rows, cols = rng.integers(0, sample_rows, cal), rng.integers(0, N, cal)
    oracle_at(cfg, ins_cpu, rows, cols)
    t = time.perf_counter()
    oracle_at(cfg, ins_cpu, rows, cols)
    per_elem = max((time.perf_counter() - t) / cal, 1e-8)
    n = int(max(16, min(M * N, budget / total / per_elem)))
    rows, cols = rng.integers(0, sample_rows, n), rng.integers(0, N, n)
    for _ in range(args.warmup):
        oracle_at(cfg, ins_cpu, rows, cols)
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle_at(cfg, ins_cpu, rows, cols)
    dt = time.perf_counter() - t
    value = 2.0 * n * K * args.steps / dt / 1e12
    sample = f"each step: {n} output elements of C (K={K} each) at fixed random coordinates, FP64"
    line = {
        "impl": "reference",
        "metric": metric_name(cfg), "value": value, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": cfg["workload"], "M": M, "N": N, "K": K, "sample_per_step": sample},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.num_threads(), "cpu": cpu_model(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def metric_name(cfg):
    if cfg["kind"] == "bf16":
        return f"BF16 GEMM TFLOP/s @ M={cfg['M']} N={cfg['N']} K={cfg['K']} on 1 GB300"
    return f"NVFP4 GEMM TFLOP/s @ M={cfg['M']} N={cfg['N']} K={cfg['K']} on 1 GB300"


def default_kernel(g, cfg, props, args):
    """What the library's default kernel choice is for this workload."""
    M, N, K = cfg["M"], cfg["N"], cfg["K"]
    if cfg["kind"] == "nvfp4":
        return "2-CTA, 256 x 256 tile, 6 stages of 256 K"
    if g.bf16_plan(M, N, K)[0]:
        return "C^T = B A^T (few rows)"
    wide = (args.clc != "on" and not args.no_persistent and not args.max_clusters
            and g.bf16_wide_rule(M, N, K, props.multi_processor_count // 2))
    return ("2-CTA, 512 x 256 tile (two 128-row M-waves per CTA), 64-K stages" if wide
            else "2-CTA, 256 x 256 tile, 128-K stages")


def run_ours(args, cfg, world, rank, local):
    import torch

    import dense_tensor_core_persistent_gb300 as g
    from dense_tensor_core_persistent_gb300 import build as gbuild

    gbuild.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2 ** 20))
    M, N, K = cfg["M"], cfg["N"], cfg["K"]
    sb = set_bytes(cfg)
    R = max(3, math.ceil(2 * l2 / sb) + 1)
    sets = [make_inputs(cfg, r, dev, args.scales) for r in range(R)]
    outs = [torch.zeros(M, N, dtype=torch.bfloat16, device=dev) for _ in range(R)]
    stream = torch.cuda.Stream(device=dev)
    epi = make_epilogue(g, args.epilogue, N, dev)
    opts = g.options(kernel=args.kernel, group_m=args.group_m, max_clusters=args.max_clusters,
                     persistent=0 if args.no_persistent else 1, no_tail_split=1 if args.no_tail_split else 0,
                     no_pdl=1 if args.no_pdl else 0, clc=CLC_MODES[args.clc])
    flops = 2.0 * M * N * K
    torch.cuda.synchronize()

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            launch(g, cfg, sets[i % R], outs[i % R], stream, opts, args.scales, epi)
    stream.synchronize()
    st, detail = g.get_device_status(stream)
    if st != 0:
        raise RuntimeError(f"kernel status {st} ({detail:#x}) during warm-up")

    uuid = None
    try:
        uuid = "GPU-" + str(props.uuid)
    except Exception:
        pass
    clocks = ClockSampler(uuid if rank == 0 else None) if rank == 0 else None
    if clocks:
        clocks.wait_first_sample()

    graph, graph_launches = None, 0
    if args.graph:
        # the K timed steps captured once into a CUDA graph (the library's launches become
        # kernel nodes, with programmatic dependencies where the launches ask for them), then
        # replayed once untimed before the timed replay
        launches_c0 = g.launch_count()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream, capture_error_mode="thread_local"):
            for i in range(args.steps):
                launch(g, cfg, sets[i % R], outs[i % R], stream, opts, args.scales, epi)
        graph_launches = g.launch_count() - launches_c0
        with torch.cuda.stream(stream):
            graph.replay()
        stream.synchronize()

    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    launches0 = g.launch_count()
    # The SM clock inside the GEMM, from its own CTAs: every `stride`-th launch of the timed
    # region (at most 64 of them) carries a clock probe (gemm_options_t.clock_probe: each
    # CTA stores clock64 and %globaltimer at the start and end of its work, 4 stores per
    # CTA). nvidia-smi samples about every 100 ms and sees nothing of a burst of launches.
    probes, probe_opts = [], {}
    if graph is None:
        stride = max(1, -(-args.steps // 64))
        for i in range(0, args.steps, stride):
            buf = torch.zeros(4 * PROBE_CTAS, dtype=torch.int64, device=dev)
            probes.append(buf)
            probe_opts[i] = g.options(kernel=args.kernel, group_m=args.group_m, max_clusters=args.max_clusters,
                                      persistent=0 if args.no_persistent else 1,
                                      no_tail_split=1 if args.no_tail_split else 0, no_pdl=1 if args.no_pdl else 0,
                                      clc=CLC_MODES[args.clc], clock_probe=buf)
        torch.cuda.synchronize()
    if clocks:
        clocks.mark_start()
    ev0.record(stream)
    if graph is not None:
        with torch.cuda.stream(stream):
            graph.replay()
    else:
        for i in range(args.steps):
            launch(g, cfg, sets[i % R], outs[i % R], stream, probe_opts.get(i, opts), args.scales, epi)
    ev1.record(stream)
    stream.synchronize()
    if clocks:
        clocks.mark_end()
    torch.cuda.synchronize()
    barrier(world)
    launches = graph_launches if graph is not None else g.launch_count() - launches0
    ms = ev0.elapsed_time(ev1)
    ms = max_over_ranks(ms, world)
    st, detail = g.get_device_status(stream)
    if st != 0:
        raise RuntimeError(f"kernel status {st} ({detail:#x}) in the timed region")
    kernel_clock = summarize_probes(g, probes) if probes else None
    after = None
    if clocks and (clocks.t1 - clocks.t0) < ClockSampler.MIN_REGION_S:
        # A timed region too short for the sampler: the same launches continue, untimed, for
        # about a second, so that the clocks under this load are still on record (labelled
        # apart from the timed region's own samples).
        a0 = time.time()
        i = 0
        with torch.cuda.stream(stream):
            while time.time() - a0 < 1.0:
                for _ in range(8):
                    launch(g, cfg, sets[i % R], outs[i % R], stream, opts, args.scales, epi)
                    i += 1
                stream.synchronize()
        after = (a0, time.time())
    clock_info = clocks.summary(after) if clocks else None

    per_launch_s = ms / 1e3 / args.steps
    value = flops * args.steps * world / (ms / 1e3) / 1e12

    # ---- end to end through the C ABI with host buffers: every step copies its inputs from
    # pinned host memory, runs the GEMM and copies C back. Steps are pipelined over three
    # streams and two device buffer sets: the copy-in of step i+1 and the copy-out of step
    # i-1 overlap the GEMM of step i, as a host-fed application would run them.
    e2e_steps = max(3, min(args.steps, args.e2e_steps))
    host_in = [t.cpu().pin_memory() for t in sets[0]]
    host_out = [torch.empty(M, N, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    dev_in = [[torch.empty_like(t) for t in sets[0]] for _ in range(2)]
    dev_out = [torch.empty(M, N, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = host_out[0].numel() * host_out[0].element_size()
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_gemm = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    used = [False, False]

    def e2e_step(i):
        b = i % 2
        if used[b]:
            s_in.wait_event(ev_gemm[b])       # the GEMM of step i-2 has read dev_in[b]
        with torch.cuda.stream(s_in):
            for d, h in zip(dev_in[b], host_in):
                d.copy_(h, non_blocking=True)
        ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        if used[b]:
            stream.wait_event(ev_out[b])      # the copy-out of step i-2 has read dev_out[b]
        launch(g, cfg, dev_in[b], dev_out[b], stream, opts, args.scales, epi)
        ev_gemm[b].record(stream)
        s_out.wait_event(ev_gemm[b])
        with torch.cuda.stream(s_out):
            host_out[b].copy_(dev_out[b], non_blocking=True)
        ev_out[b].record(s_out)
        used[b] = True

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(e2e_steps):
        e2e_step(i)
    s_out.wait_event(ev_out[(e2e_steps - 1) % 2])
    e1.record(s_out)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    e2e_value = flops * e2e_steps * world / (e2e_ms / 1e3) / 1e12

    if rank != 0:
        return

    peaks, peak_src = load_peaks()
    if cfg["kind"] == "bf16":
        peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
        peak_note = f"{peak_src} cuBLAS BF16 8192^3 burst (MEASURED_PEAKS bf16_tflops)"
    else:
        peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])) * NOMINAL_FP4_OVER_BF16
        peak_note = f"{peak_src} BF16 burst x nominal FP4/BF16 ratio 6"
    achieved = flops / per_launch_s / 1e12
    # The MMA instruction's own rate on this GPU (FLOP per SM clock), and what it gives at the
    # SM clock sampled during the timed region: the ceiling for a kernel built from it.
    rate = None
    try:
        fpc = g.measure_mma_rate(g.GEMM_MMA_BF16 if cfg["kind"] == "bf16" else g.GEMM_MMA_NVFP4)
        mhz = clock_info.get("sm_mhz") if clock_info else None
        clock_src = "timed region"
        if not mhz and clock_info and clock_info.get("after_region"):
            mhz = clock_info["after_region"].get("sm_mhz")
            clock_src = "untimed continuation after the timed region"
        rate = {"flop_per_clk_per_sm": fpc, "sms": props.multi_processor_count}
        if mhz:
            ceiling = fpc * props.multi_processor_count * mhz * 1e6 / 1e12
            rate.update({"ceiling_at_sampled_clock": ceiling, "frac_of_ceiling": achieved / ceiling,
                         "clock_mhz": mhz, "clock_from": clock_src})
        if kernel_clock and kernel_clock.get("sm_mhz"):
            kc = kernel_clock["sm_mhz"]
            ceiling = fpc * props.multi_processor_count * kc * 1e6 / 1e12
            rate.update({"ceiling_at_kernel_clock": ceiling, "frac_of_ceiling_at_kernel_clock": achieved / ceiling,
                         "kernel_clock_mhz": kc})
    except Exception as e:  # report, do not fail the benchmark line
        rate = {"error": str(e)}
    # the recorded counters are those of the plain kernel
    traffic = (recorded_traffic(cfg["workload"] + ("" if cfg["kind"] == "bf16" else f"_{args.scales}"), cfg["kind"])
               if args.epilogue == "none" else None)
    cpu = cpu_baseline(cfg, args.cpu_seconds) if not args.no_cpu_baseline else None
    if cpu:
        cpu.pop("seconds", None)
        cpu.pop("rows", None)
    baseline = PAGE_TFLOPS.get(args.config)
    line = {
        "metric": metric_name(cfg),
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": (value / world / baseline) if baseline else None,
        "dtype": "bf16" if cfg["kind"] == "bf16" else "nvfp4",
        "data": "synthetic: seeded SplitMix64 operands with the workload's value distribution",
        "config": {
            "workload": cfg["workload"], "M": M, "N": N, "K": K,
            "l2_flush": f"rotation over {R} input sets of {sb / 2**20:.0f} MiB (> 2x L2 = {2 * l2 / 2**20:.0f} MiB)",
            "kernel": {0: "default: " + default_kernel(g, cfg, props, args), 1: "1-CTA",
                       2: "2-CTA, 256 x 256 tile, 128-K stages",
                       3: "2-CTA, 256 x 256 tile, 64-K stages",
                       4: "2-CTA, 512 x 256 tile (two 128-row M-waves per CTA), 64-K stages"}[args.kernel]
            + ("" if not args.no_persistent else ", one tile per cluster")
            + (", no tail split" if args.no_tail_split else "")
            + (", plain launches (no programmatic dependent launch)" if args.no_pdl else ""),
            "scales": (None if cfg["kind"] == "bf16" else
                       "blocked tensor-core layout (packed once at input setup)" if args.scales == "blocked"
                       else "row-major [rows][K/16], packed to the tensor-core layout inside each call"),
            "group_m": args.group_m or "auto",
            "launch": "one CUDA graph replay of the timed steps" if args.graph else "one library call per step from the host",
            "scheduler": {"auto": "default (gemm_clc_rule: cluster launch control only for BF16 beyond one wave "
                                  "with K >= 16384)", "on": "cluster launch control",
                          "off": "static grid stride"}[args.clc],
            "epilogue": ("plain BF16 rounding" if args.epilogue == "none" else
                         f"fused {args.epilogue}: alpha, beta, bias, activation = {EPILOGUES[args.epilogue]}"
                         + (" (e2e: the prior C is the device buffer's previous contents)"
                            if EPILOGUES[args.epilogue][1] != 0.0 else "")),
            "baseline": "HGEMM v7 on GB300, 1980.925 TFLOP/s (page 1 Performance table)" if baseline else None,
        },
        "roofline": {
            "bound": "tensor",
            "achieved": achieved,
            "peak": peak,
            "unit": "TFLOP/s",
            "frac": achieved / peak,
            "traffic": traffic,
            "peak_source": peak_note,
            "algorithmic_flops_per_launch": flops,
            "achieved_over": ("one step = the scale-packing launch and the GEMM launch of one gemm_nvfp4 call "
                              "(the GEMM launch alone is shorter)"
                              if cfg["kind"] == "nvfp4" and args.scales == "rowmajor" else
                              "one step = one GEMM launch"),
            "instruction_rate": rate,
        },
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps,
                "pipelining": "copy-in of step i+1 and copy-out of step i-1 overlap the GEMM of step i "
                              "(3 streams, 2 device buffer sets, pinned host memory)"},
        "gpu_launches": int(launches),
        "clocks": dict(clock_info or {}, kernel=kernel_clock) if kernel_clock else clock_info,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=300)
    ap.add_argument("--config", default="c3", choices=sorted(CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--kernel", type=int, default=0)
    ap.add_argument("--no-pdl", action="store_true", help="launch without programmatic stream serialization")
    ap.add_argument("--group-m", type=int, default=0)
    ap.add_argument("--max-clusters", type=int, default=0)
    ap.add_argument("--no-persistent", action="store_true")
    ap.add_argument("--no-tail-split", action="store_true")
    ap.add_argument("--graph", action="store_true",
                    help="time one replay of a CUDA graph holding the K steps instead of K launches from the host")
    ap.add_argument("--clc", default="auto", choices=sorted(CLC_MODES),
                    help="tile scheduler: the default rule, cluster launch control, or the static grid stride")
    ap.add_argument("--scales", default="rowmajor", choices=["blocked", "rowmajor"],
                    help="NVFP4 scales: row-major, packed inside each gemm_nvfp4 call (the boundary call, "
                         "default), or pre-packed once outside the timed region (gemm_nvfp4_blocked)")
    ap.add_argument("--epilogue", default="none", choices=sorted(EPILOGUES),
                    help="fused epilogue of the *_fused calls (default: the plain GEMM)")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-seconds", type=float, default=120.0,
                    help="--impl reference: host seconds for warm-up + timed steps together")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    cfg = CONFIGS[args.config]
    world, rank, local = dist_setup(args.gpus if args.impl == "ours" else 0)
    if args.impl == "reference":
        run_reference(args, cfg, world, rank)
    else:
        run_ours(args, cfg, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

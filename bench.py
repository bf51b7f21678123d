#!/usr/bin/env python
"""Throughput of the VLA forward recurrence on GB300.

One step = one vla_forward call over the whole workload (every head, every
token: eq. 9-11 of "Variational Linear Attention", §3.3). The default workload
is the d_h = 96 configuration (B=8, H=16, T=4096, bf16 q/k/v/u drawn N(0,1)
with ||v_t|| <= 4, fp32 state); its inputs (403 MB) are larger than L2, so no
L2 flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0). With N > 1 (torchrun, one rank per GPU) every
rank runs its own copy of the workload (heads are independent: weak scaling,
no collective on the data path); the time is the max over ranks.
``--impl reference`` times the fp64 CPU oracle on the host cores instead, on
a bounded sample of the same workload.

``--pass backward`` times the reverse-mode gradient instead (one step = one
vla_backward call over the whole workload with a seeded upstream gradient
dL/do; the forward recurrence is recomputed inside the call).
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "VLA head-tokens/sec at d_h=96,T=4096; % of FP32-FMA roofline"
METRIC_BW = "VLA backward head-tokens/sec at d_h=96,T=4096; % of FP32-FMA roofline"
METRIC_DEC = "VLA decode head-tokens/sec at d_h=96, T=1, carried state; % of HBM roofline"
UNIT = "head-tokens/s"
# algorithmic FP32 work per head-token, in units of d^2 FLOP: the forward is 6 matrix-vector
# products / rank-1 updates of d x d matrices (2 d^2 FLOP each); the backward recomputes 5 of
# them (A u^, A k^, S k^ and the rank-1 updates of A and S) and then runs 8 matrix-vector
# products and 6 rank-1 updates on S, A and their adjoints (19 x 2 d^2)
# (the fixed-A variant skips A u^ and the A update: 8 d^2)
FLOP_D2 = {"forward": 12, "backward": 38, "fixed_a": 8}
FP32_LANES_PER_SM = 128          # FP32 FMA lanes per SM (sm_103)
FALLBACK_SM_MAX_MHZ = 2070.0
FALLBACK_HBM_GBS = 6800.0

# The source files each kernel is compiled from (besides the launch code).
KERNEL_FILES = {
    "vla_tc_kernel": ("vla_tc.cuh", "vla_device.cuh"),
    "vla_fused_kernel": ("vla_fused.cuh", "vla_device.cuh"),
    "vla_backward_kernel": ("vla_backward.cuh", "vla_device.cuh"),
    # the split reverse sweep (d = 128): its S side and A side as a cluster of two CTAs per head
    "vla_backward_pair_kernel": ("vla_backward_split.cuh", "vla_backward.cuh", "vla_device.cuh"),
    "vla_decode_kernel": ("vla_decode.cuh", "vla_backward.cuh", "vla_device.cuh"),
    "vla_tc2_kernel": ("vla_tc2.cuh", "vla_tc.cuh", "vla_device.cuh"),
    "vla_tc3_kernel": ("vla_tc3.cuh", "vla_tc2.cuh", "vla_tc.cuh", "vla_device.cuh"),
}

# DRAM bytes per launch of a bench line's kernel (dram__bytes_read.sum +
# dram__bytes_write.sum) from one ncu capture, valid only for the workload it
# was taken on (B, H, T, d, input dtype) and while that kernel's own sources
# hash to source_sha; otherwise reported as null.
NCU_TRAFFIC = {
    "vla_tc_kernel": {"source_sha": "a42f512597716e3c", "workload": (8, 16, 4096, 96, "bf16"),
                      "bytes_per_launch": 403375360 + 175656448},
    # from a capture at T = 8192 (the full launch holds about 3.2 GB on the device), the per-token part
    # scaled by 8; the final S, A, z^key writes (32 x (2 d^2 + d) x 4 bytes) are per head
    "vla_tc3_kernel": {"source_sha": "dfea88a0086d207e", "workload": (1, 32, 65536, 128, "bf16"),
                       "bytes_per_launch": 8 * (268556544 + 108200448 - 4227072) + 4227072},
    # the reverse sweep (the step's dominant kernel, after the taped chunked forward), from a capture of
    # the same workload at B=2 (32 heads; a full step holds about 2.8 GB on the device) scaled by 4:
    # every byte it moves is per head-token or per head
    "vla_backward_kernel": {"source_sha": "5315436c0f21b084", "workload": (8, 16, 4096, 96, "bf16"),
                            "bytes_per_launch": 4 * (436128256 + 176882432)},
    # the split reverse sweep (d = 128) on the long-context workload cut to 4096 tokens
    "vla_backward_pair_kernel": {"source_sha": "5df2099d1b2bece4", "workload": (1, 32, 4096, 128, "bf16"),
                                 "bytes_per_launch": 648319488 + 307634432},
    "vla_decode_kernel": {"source_sha": "46994107829e6084", "workload": (128, 16, 1, 96, "bf16"),
                          "bytes_per_launch": 153393408 + 98091264},
    "vla_fused_kernel": {"source_sha": "565a71784acabc88", "workload": (8, 16, 4096, 96, "bf16"),
                         "bytes_per_launch": 403125248 + 175399936},
}


def kernel_source_sha(kernel: str = None) -> str:
    """Hash of the CUDA sources: of one kernel's own files, or of all of them."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sherman_morrison_memory_gb300", "csrc")
    names = sorted(KERNEL_FILES[kernel]) if kernel else sorted(os.listdir(csrc))
    for name in names:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload=None):
    """Captured DRAM bytes per launch of `kernel` on `workload` = (B, H, T, d, dtype), or None."""
    t = NCU_TRAFFIC.get(kernel)
    if not t or t["source_sha"] != kernel_source_sha(kernel):
        return None
    if workload is not None and tuple(workload) != t["workload"]:
        return None
    return t["bytes_per_launch"]


def kernel_for(algo: int, T: int, d: int, heads: int = 1 << 30, n_sm: int = 152) -> str:
    """The kernel one vla_forward call launches (the choice VLA_ALGO_AUTO makes
    for `heads` = B * H heads on `n_sm` SMs); for the segmented path, the
    chunked kernel that its three side-by-side runs use."""
    if algo == 3 or (algo == 0 and T <= 4):
        return "vla_decode_kernel"
    if algo == 6 or (algo == 0 and d <= 96 and T >= 1024 and 3 * heads <= n_sm):
        return "vla_tc_kernel"
    if algo == 5 or (algo == 0 and d >= 96 and 3 * heads <= n_sm):
        return "vla_tc3_kernel"
    if algo == 4 or (algo == 0 and d == 128):
        return "vla_tc2_kernel"
    if algo == 2 or (algo == 0 and d <= 96):
        return "vla_tc_kernel"
    return "vla_fused_kernel"


def measure_ffma_peak(dev, n_sm: int, iters: int = 100000, reps: int = 3) -> dict:
    """FP32 FMA throughput of this GPU, measured now: the library's probe
    (include/vla_probe.h: 8 independent FMA chains per thread, 4 CTAs x 256
    threads per SM), scalar and packed, best of `reps` timed launches each,
    CUDA events on the launching stream. The roofline's denominator."""
    import torch

    from sherman_morrison_memory_gb300 import _binding

    blocks, threads = 4 * n_sm, 256
    sink = torch.empty(blocks * threads, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    out = {"blocks": blocks, "threads": threads, "iters": iters}
    for packed in (False, True):
        flop = _binding.vla_probe_ffma(blocks, threads, iters, packed, sink)  # warm-up
        best = None
        for _ in range(reps):
            torch.cuda.synchronize(dev)
            e0.record(stream)
            _binding.vla_probe_ffma(blocks, threads, iters, packed, sink)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            ms = e0.elapsed_time(e1)
            best = ms if best is None else min(best, ms)
        out["packed_tflops" if packed else "scalar_tflops"] = flop / (best / 1e3) / 1e12
        out["packed_ms" if packed else "scalar_ms"] = best
    out["tflops"] = max(out["scalar_tflops"], out["packed_tflops"])
    return out


def load_peaks() -> dict:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except (OSError, ValueError):
        return {}


# ---------------------------------------------------------------------------
# distributed plumbing (host logic is exercised on CPU with gloo in the tests)
# ---------------------------------------------------------------------------

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def rank_seed(base_seed: int, rank: int) -> int:
    """Each rank draws its own copy of the workload (weak scaling)."""
    return base_seed + 1000 * rank


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int, device=None):
    if world <= 1:
        return
    import torch.distributed as dist

    if device is not None and device.type == "cuda":
        dist.barrier(device_ids=[device.index])
    else:
        dist.barrier()


def aggregate_value(units_per_rank: int, world: int, max_seconds: float) -> float:
    """Whole-job throughput: units all ranks processed / max-over-ranks time."""
    return units_per_rank * world / max_seconds


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------

CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="vla_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader",
                 "-lms", "100"], stdout=self.out, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.out.close()

    def summary(self) -> dict:
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) < 9:
                        continue
                    try:
                        sm = float(parts[1].split()[0])
                        smax = float(parts[2].split()[0])
                    except ValueError:
                        continue
                    rows.append((sm, smax, parts))
            os.unlink(self.path)
        except OSError:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, p in rows for i in range(4) if p[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# the fp64 oracle on the host cores (CPU baseline / reference arm)
# ---------------------------------------------------------------------------

def oracle_time(arrs, w, tokens: int, heads: int):
    import oracle

    orc = oracle.load()
    sub = [a.reshape(-1, w.T, w.d)[:heads, :tokens] for a in arrs]
    t0 = time.perf_counter()
    r = orc.forward(*sub, lambda0=w.lambda0, eps=w.eps, want_o=True)
    dt = time.perf_counter() - t0
    return heads * tokens / dt, r.threads, dt


def oracle_time_bw(arrs, gO, w, tokens: int, heads: int):
    import oracle

    orc = oracle.load()
    sub = [a.reshape(-1, w.T, w.d)[:heads, :tokens].astype("float64") for a in arrs]
    g = gO.reshape(-1, w.T, w.d)[:heads, :tokens].astype("float64")
    t0 = time.perf_counter()
    r = orc.backward(*sub, w.lambda0, w.eps, gO=g)
    dt = time.perf_counter() - t0
    return heads * tokens / dt, r["threads"], dt


def run_reference_decode(args, w):
    """The oracle on the decode step: all heads, one token, from the state the
    oracle reached over the same earlier tokens."""
    import oracle
    from sherman_morrison_memory_gb300 import workloads as W

    B, H, T, warm = DECODE_WORKLOAD["B"], DECODE_WORKLOAD["H"], DECODE_WORKLOAD["T"], DECODE_WORKLOAD["warm"]
    wr = W.Workload("decode", B, H, warm + T, w.d, w.dtype, w.structure, w.lambda0, w.eps, seed=w.seed)
    arrs = W.make(wr)
    orc = oracle.load()
    r0 = orc.forward(*[a[:, :, :warm] for a in arrs], lambda0=w.lambda0, eps=w.eps, want_o=False)
    sq = [a[:, :, -T:] for a in arrs]
    total, steps = 0.0, 0
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        r = orc.forward(*sq, lambda0=w.lambda0, eps=w.eps, S0=r0.S, A0=r0.A, zk0=r0.zk)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            total += dt
            steps += 1
    value = B * H * T * steps / total
    line = {
        "impl": "reference", "metric": METRIC_DEC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"decode: B={B},H={H},T={T},d_h={w.d}, carried state from {warm} earlier tokens"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": r.threads, "kind": "oracle",
                         "sample": f"one decode step of all {B * H} heads per step (fp64 oracle, OpenMP over heads)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_reference(args, w):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from sherman_morrison_memory_gb300 import workloads as W

    if args.pass_ == "decode":
        run_reference_decode(args, w)
        return
    arrs = W.make(w)
    heads = w.heads
    bw = args.pass_ == "backward"
    if bw:
        gO = W.upstream_grad(w)
        timer = lambda tok: oracle_time_bw(arrs, gO, w, tok, heads)
    else:
        timer = lambda tok: oracle_time(arrs, w, tok, heads)
    # size each step's sample so that warmup + steps end within about 2.5 minutes
    probe_tokens = min(w.T, 16)
    rate, threads, dt = timer(probe_tokens)
    budget = 150.0 / max(1, args.steps + args.warmup)
    tokens = int(max(1, min(w.T, probe_tokens * budget / max(dt, 1e-6))))
    for _ in range(args.warmup):
        timer(tokens)
    total_units, total_time = 0, 0.0
    for _ in range(args.steps):
        rate, threads, dt = timer(tokens)
        total_units += heads * tokens
        total_time += dt
    value = total_units / total_time
    what = "fp64 oracle backward" if bw else "fp64 oracle"
    sample = f"all {heads} heads x first {tokens} of {w.T} tokens per step ({what}, OpenMP over heads)"
    line = {
        "impl": "reference", "metric": METRIC_BW if bw else METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_time / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": w.describe()},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# the CUDA path
# ---------------------------------------------------------------------------

def run_ours(args, w):
    import torch
    import torch.distributed as dist

    from sherman_morrison_memory_gb300 import (VLA_OK, vla_forward, vla_get_last_device_status,
                                               vla_linear_attention_state)
    from sherman_morrison_memory_gb300 import workloads as W

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    wr = W.Workload(w.name, w.B, w.H, w.T, w.d, w.dtype, w.structure, w.lambda0, w.eps,
                    seed=rank_seed(w.seed, rank))
    arrs = W.make(wr)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    q, k, v, u = (torch.from_numpy(a).to(dev).to(tdt) for a in arrs)
    B, H, T, d = w.B, w.H, w.T, w.d
    o = torch.empty((B, H, T, d), dtype=torch.float32, device=dev)
    S = torch.empty((B, H, d, d), dtype=torch.float32, device=dev)
    A = torch.empty_like(S)
    zk = torch.empty((B, H, d), dtype=torch.float32, device=dev)
    out = (o, S, A, zk)
    stream = torch.cuda.current_stream(dev)

    fa = bool(args.fixed_a)
    if fa:
        u = None  # not read by the fixed-A variant
    for _ in range(args.warmup):
        vla_forward(q, k, v, u, w.lambda0, w.eps, out=out, algo=args.algo, fixed_a=fa)
    st, detail = vla_get_last_device_status(dev)
    if st != VLA_OK:
        raise RuntimeError(f"device status {st} {detail} after warm-up")

    props = torch.cuda.get_device_properties(dev)
    gpu_id = str(getattr(props, "uuid", "") or "")
    gpu_id = ("GPU-" + gpu_id) if gpu_id and not gpu_id.startswith("GPU-") else (gpu_id or str(local))
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(gpu_id) as clk:
        barrier(world, dev)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(args.steps):
            vla_forward(q, k, v, u, w.lambda0, w.eps, out=out, algo=args.algo, fixed_a=fa)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world, dev)
    ms = e0.elapsed_time(e1) / args.steps
    st, detail = vla_get_last_device_status(dev)
    if st != VLA_OK:
        raise RuntimeError(f"device status {st} {detail} in the timed region")
    ms_max = max_over_ranks(ms, world, dev)
    units = w.head_tokens
    value = aggregate_value(units, world, ms_max / 1e3)

    # roofline of the one kernel that a step launches, against the FP32 FMA
    # peak measured by the probe in this run (the nominal figure beside it)
    kernel = kernel_for(args.algo, T, d, w.heads, props.multi_processor_count)
    peaks = load_peaks()
    sm_max = float(peaks.get("sm_max_mhz", FALLBACK_SM_MAX_MHZ))
    n_sm = props.multi_processor_count
    nominal_tflops = n_sm * FP32_LANES_PER_SM * 2 * sm_max * 1e6 / 1e12
    probe = measure_ffma_peak(dev, n_sm)
    peak_tflops = probe["tflops"]
    flop_d2 = FLOP_D2["fixed_a" if fa else "forward"]
    flops = flop_d2 * d * d * units
    achieved = flops / (ms / 1e3) / 1e12
    in_bytes = (3 if fa else 4) * units * d * (2 if w.dtype == "bf16" else 4)
    out_bytes = units * d * 4 + w.heads * (2 * d * d + d) * 4
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    hbm_gbs = (in_bytes + out_bytes) / (ms / 1e3) / 1e9
    sha = kernel_source_sha(kernel)
    traffic = ncu_traffic(kernel, (B, H, T, d, w.dtype))

    # the same metric end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        hq, hk, hv = (x.cpu().pin_memory() for x in (q, k, v))
        hu = None if u is None else u.cpu().pin_memory()
        hout = tuple(torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in out)
        ksteps = max(3, min(args.steps, args.e2e_steps))
        for _ in range(2):
            vla_forward(hq, hk, hv, hu, w.lambda0, w.eps, out=hout, algo=args.algo, fixed_a=fa)
        torch.cuda.synchronize(dev)
        barrier(world, dev)
        e0.record(stream)
        for _ in range(ksteps):
            vla_forward(hq, hk, hv, hu, w.lambda0, w.eps, out=hout, algo=args.algo, fixed_a=fa)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world, dev)
        e2e_ms = max_over_ranks(e0.elapsed_time(e1) / ksteps, world, dev)
        e2e = {"value": aggregate_value(units, world, e2e_ms / 1e3), "unit": UNIT,
               "h2d_bytes_per_step": sum(x.numel() * x.element_size() for x in (hq, hk, hv, hu) if x is not None),
               "d2h_bytes_per_step": sum(x.numel() * x.element_size() for x in hout),
               "ms_per_step": e2e_ms, "steps": ksteps,
               "path": "vla_forward_host: automatic chunks (about T/4 tokens), H2D on two streams, kernels, D2H overlapped"}

    # ||S_T||_F of VLA next to plain cumulative linear attention on the same inputs
    vla_fro = torch.linalg.matrix_norm(S).mean().item()
    S_la = vla_linear_attention_state(k, v)
    la_fro = torch.linalg.matrix_norm(S_la).mean().item()
    torch.cuda.synchronize(dev)

    # the other workloads, each timed in this run (the headline stays the one above)
    configs = None
    if world == 1 and not args.no_configs and not fa and args.algo == 0 and args.batch == 0 and args.tokens == 0:
        configs = time_workloads([i for i in sorted(W.WORKLOADS) if i != args.workload], dev, peak_tflops)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        carr = arrs if not fa else (arrs[0], arrs[1], arrs[2], arrs[3] * 0)
        rate, threads, dt = oracle_time(carr, w, w.T, w.heads)
        cpu = {"value": rate, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"the full workload once ({w.heads} heads x {w.T} tokens, fp64"
                         f"{', u = 0 for fixed A' if fa else ''}, {dt:.1f} s)"}

    if rank == 0:
        line = {
            "metric": METRIC + ("; fixed-A variant" if fa else ""), "value": value, "unit": UNIT,
            "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.describe(), "B": B, "H": H, "T": T, "d_h": d, "input_dtype": w.dtype,
                       "variant": "fixed A (A = I/lambda0, eq. 9 skipped, u not read)" if fa else "full",
                       "per_rank_heads": w.heads,
                       "l2": f"inputs larger than L2 ({in_bytes / 1e6:.0f} MB per step), no flush"},
            "roofline": {"bound": "alu", "achieved": achieved, "peak": peak_tflops, "unit": "TFLOP/s",
                         "frac": achieved / peak_tflops, "traffic": traffic,
                         "peak_basis": "measured in this run: FFMA probe (include/vla_probe.h), best of scalar "
                                       f"{probe['scalar_tflops']:.1f} and packed {probe['packed_tflops']:.1f} TFLOP/s "
                                       f"on {probe['blocks']} CTAs x {probe['threads']} threads",
                         "peak_nominal": nominal_tflops,
                         "peak_nominal_basis": f"{n_sm} SMs x {FP32_LANES_PER_SM} FP32 FMA lanes x 2 x {sm_max:.0f} MHz",
                         "frac_of_nominal": achieved / nominal_tflops,
                         "achieved_basis": "nominal FLOP (12 d^2 per head-token, the FP32 FMA work of the "
                                           "recurrence) / kernel time; the kernel runs its d x d products on the "
                                           "tensor cores in 3-term tf32",
                         "flop_per_head_token": flop_d2 * d * d, "kernel": kernel},
            "fp32_roofline_pct": 100.0 * achieved / peak_tflops,
            "ffma_probe": probe,
            "configs": configs,
            "hbm": {"achieved_gbs": hbm_gbs, "peak_gbs": hbm_peak, "frac": hbm_gbs / hbm_peak,
                    "algorithmic_bytes_per_launch": in_bytes + out_bytes},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": args.steps,
            "clocks": clk.summary(),
            "state_norm_fro_mean": {"vla": vla_fro, "linear_attention": la_fro},
            "kernel_source_sha": sha,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def time_workloads(ids, dev, peak_tflops: float, steps: int = 20, warmup: int = 3) -> dict:
    """Each workload in `ids` timed in this run with the default kernel
    choice: `warmup` untimed calls, then `steps` calls between CUDA events on
    the launching stream. Inputs of workloads up to 1 GB are the seeded numpy
    draws of workloads.make (the ones the parity tests use); larger ones are
    drawn on the device (torch generator, seed 0, the same N(0,1) bf16
    distribution) to keep the run short. The kernels' timing does not depend
    on the values."""
    import torch

    from sherman_morrison_memory_gb300 import VLA_OK, vla_forward, vla_get_last_device_status
    from sherman_morrison_memory_gb300 import workloads as W

    out = {}
    stream = torch.cuda.current_stream(dev)
    for wid in ids:
        w = W.WORKLOADS[wid]
        B, H, T, d = w.B, w.H, w.T, w.d
        tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
        in_bytes = 4 * w.head_tokens * d * (2 if w.dtype == "bf16" else 4)
        if in_bytes <= (1 << 30):
            src = "workloads.make (numpy, seeded)"
            q, k, v, u = (torch.from_numpy(a).to(dev).to(tdt) for a in W.make(w))
        else:
            src = "device draw (torch generator, seed 0)"
            g = torch.Generator(device=dev)
            g.manual_seed(0)
            q, k, v, u = (torch.randn((B, H, T, d), generator=g, device=dev, dtype=torch.float32).to(tdt)
                          for _ in range(4))
        o = torch.empty((B, H, T, d), dtype=torch.float32, device=dev)
        S = torch.empty((B, H, d, d), dtype=torch.float32, device=dev)
        res = (o, S, torch.empty_like(S), torch.empty((B, H, d), dtype=torch.float32, device=dev))
        for _ in range(warmup):
            vla_forward(q, k, v, u, w.lambda0, w.eps, out=res)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(steps):
            vla_forward(q, k, v, u, w.lambda0, w.eps, out=res)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        st, detail = vla_get_last_device_status(dev)
        if st != VLA_OK:
            raise RuntimeError(f"workload {wid}: device status {st} {detail}")
        ms = e0.elapsed_time(e1) / steps
        tflops = FLOP_D2["forward"] * d * d * w.head_tokens / (ms / 1e3) / 1e12
        n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
        out[str(wid)] = {"workload": w.describe(), "kernel": kernel_for(0, T, d, w.heads, n_sm), "ms_per_step": ms,
                         "head_tokens_per_s": w.head_tokens / (ms / 1e3), "achieved_tflops": tflops,
                         "fp32_roofline_frac": tflops / peak_tflops, "steps": steps, "warmup": warmup,
                         "inputs": src}
        del q, k, v, u, o, S, res
        torch.cuda.empty_cache()
    return out


DECODE_WORKLOAD = dict(B=128, H=16, T=1, warm=16)


def run_ours_decode(args, w):
    """One decode step for B*H heads (T = 1) from a carried state that a
    previous call produced: the state is read and written once per step."""
    import torch
    import torch.distributed as dist

    from sherman_morrison_memory_gb300 import VLA_OK, vla_forward, vla_get_last_device_status
    from sherman_morrison_memory_gb300 import workloads as W

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    B, H, T = DECODE_WORKLOAD["B"], DECODE_WORKLOAD["H"], DECODE_WORKLOAD["T"]
    d = w.d
    wr = W.Workload("decode", B, H, DECODE_WORKLOAD["warm"] + T, d, w.dtype, w.structure, w.lambda0, w.eps,
                    seed=rank_seed(w.seed, rank))
    arrs = W.make(wr)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    warm_in = [torch.from_numpy(a[:, :, :-T].copy()).to(dev).to(tdt) for a in arrs]
    q, k, v, u = (torch.from_numpy(a[:, :, -T:].copy()).to(dev).to(tdt) for a in arrs)
    _, state = vla_forward(*warm_in, w.lambda0, w.eps, check=True)  # the carried state
    o = torch.empty((B, H, T, d), dtype=torch.float32, device=dev)
    out = (o, torch.empty_like(state[0]), torch.empty_like(state[1]), torch.empty_like(state[2]))
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        vla_forward(q, k, v, u, w.lambda0, w.eps, state, out=out)
    st, detail = vla_get_last_device_status(dev)
    if st != VLA_OK:
        raise RuntimeError(f"device status {st} {detail} after warm-up")

    props = torch.cuda.get_device_properties(dev)
    gpu_id = str(getattr(props, "uuid", "") or "")
    gpu_id = ("GPU-" + gpu_id) if gpu_id and not gpu_id.startswith("GPU-") else (gpu_id or str(local))
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(gpu_id) as clk:
        barrier(world, dev)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(args.steps):
            vla_forward(q, k, v, u, w.lambda0, w.eps, state, out=out)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world, dev)
    ms = e0.elapsed_time(e1) / args.steps
    st, detail = vla_get_last_device_status(dev)
    if st != VLA_OK:
        raise RuntimeError(f"device status {st} {detail} in the timed region")
    ms_max = max_over_ranks(ms, world, dev)
    units = B * H * T
    value = aggregate_value(units, world, ms_max / 1e3)
    esz = 2 if w.dtype == "bf16" else 4
    state_bytes = B * H * (2 * d * d + d) * 4
    step_bytes = 2 * state_bytes + units * d * (4 * esz + 4)
    peaks = load_peaks()
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    gbs = step_bytes / (ms / 1e3) / 1e9

    e2e = None
    if not args.no_e2e:
        hin = [x.cpu().pin_memory() for x in (q, k, v, u)]
        hst = tuple(x.cpu().pin_memory() for x in state)
        hout = tuple(torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in out)
        ksteps = max(3, min(args.steps, args.e2e_steps))
        for _ in range(2):
            vla_forward(*hin, w.lambda0, w.eps, hst, out=hout)
        torch.cuda.synchronize(dev)
        barrier(world, dev)
        e0.record(stream)
        for _ in range(ksteps):
            vla_forward(*hin, w.lambda0, w.eps, hst, out=hout)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world, dev)
        e2e_ms = max_over_ranks(e0.elapsed_time(e1) / ksteps, world, dev)
        e2e = {"value": aggregate_value(units, world, e2e_ms / 1e3), "unit": UNIT,
               "h2d_bytes_per_step": sum(x.numel() * x.element_size() for x in hin + list(hst)),
               "d2h_bytes_per_step": sum(x.numel() * x.element_size() for x in hout),
               "ms_per_step": e2e_ms, "steps": ksteps}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle

        orc = oracle.load()
        sq = [a[:, :, -T:] for a in arrs]
        hs = [x.cpu().numpy().astype("float64") for x in state]
        t0 = time.perf_counter()
        r = orc.forward(*sq, lambda0=w.lambda0, eps=w.eps, S0=hs[0], A0=hs[1], zk0=hs[2])
        dt = time.perf_counter() - t0
        cpu = {"value": units / dt, "unit": UNIT, "cores": r.threads, "kind": "oracle",
               "sample": f"one decode step of all {B * H} heads from the same state (fp64, {dt:.2f} s)"}

    if rank == 0:
        line = {
            "metric": METRIC_DEC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": f"decode: B={B},H={H},T={T},d_h={d}, {w.dtype} q,k,v,u N(0,1), "
                                   f"carried fp32 state from {DECODE_WORKLOAD['warm']} earlier tokens",
                       "pass": "decode", "B": B, "H": H, "T": T, "d_h": d,
                       "l2": f"state larger than L2 ({state_bytes / 1e6:.0f} MB read and written per step), no flush"},
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s",
                         "frac": gbs / hbm_peak, "traffic": ncu_traffic("vla_decode_kernel", (B, H, T, d, w.dtype)),
                         "bytes_per_head_token": step_bytes // units, "kernel": "vla_decode_kernel"},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": args.steps,
            "clocks": clk.summary(),
            "kernel_source_sha": kernel_source_sha("vla_decode_kernel"),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_ours_backward(args, w):
    import torch
    import torch.distributed as dist

    from sherman_morrison_memory_gb300 import vla_backward
    from sherman_morrison_memory_gb300 import workloads as W

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    wr = W.Workload(w.name, w.B, w.H, w.T, w.d, w.dtype, w.structure, w.lambda0, w.eps,
                    seed=rank_seed(w.seed, rank))
    arrs = W.make(wr)
    gO_np = W.upstream_grad(wr)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    q, k, v, u = (torch.from_numpy(a).to(dev).to(tdt) for a in arrs)
    gO = torch.from_numpy(gO_np).to(dev)
    B, H, T, d = w.B, w.H, w.T, w.d
    shapes = [(B, H, T, d)] * 4 + [(B, H, d, d), (B, H, d, d), (B, H, d)]
    out = tuple(torch.empty(sh, dtype=torch.float32, device=dev) for sh in shapes)
    stream = torch.cuda.current_stream(dev)

    for i in range(args.warmup):
        vla_backward(q, k, v, u, w.lambda0, w.eps, None, gO, out=out, check=(i == args.warmup - 1))

    props = torch.cuda.get_device_properties(dev)
    gpu_id = str(getattr(props, "uuid", "") or "")
    gpu_id = ("GPU-" + gpu_id) if gpu_id and not gpu_id.startswith("GPU-") else (gpu_id or str(local))
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(gpu_id) as clk:
        barrier(world, dev)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(args.steps):
            vla_backward(q, k, v, u, w.lambda0, w.eps, None, gO, out=out)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world, dev)
    ms = e0.elapsed_time(e1) / args.steps
    # the status record is sticky: a failure in any timed call is reported here
    vla_backward(q, k, v, u, w.lambda0, w.eps, None, gO, out=out, check=True)
    ms_max = max_over_ranks(ms, world, dev)
    units = w.head_tokens
    value = aggregate_value(units, world, ms_max / 1e3)

    peaks = load_peaks()
    sm_max = float(peaks.get("sm_max_mhz", FALLBACK_SM_MAX_MHZ))
    n_sm = props.multi_processor_count
    nominal_tflops = n_sm * FP32_LANES_PER_SM * 2 * sm_max * 1e6 / 1e12
    probe = measure_ffma_peak(dev, n_sm)
    peak_tflops = probe["tflops"]
    flops = FLOP_D2["backward"] * d * d * units
    achieved = flops / (ms / 1e3) / 1e12
    esz = 2 if w.dtype == "bf16" else 4
    in_bytes = 4 * units * d * esz + units * d * 4
    out_bytes = 4 * units * d * 4 + w.heads * (2 * d * d + d) * 4
    tape_bytes = 2 * units * (3 * d + 8) * 4
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    hbm_gbs = (in_bytes + out_bytes) / (ms / 1e3) / 1e9
    # d <= 96: the taped chunked forward and the single-kernel reverse sweep;
    # d = 128: the taped cluster-pair chunked forward and the split sweep (one cluster of two CTAs per head)
    kernel = "vla_backward_kernel" if d <= 96 else "vla_backward_pair_kernel"
    launches_per_step = 2
    sha = kernel_source_sha(kernel)
    traffic = ncu_traffic(kernel, (w.B, w.H, w.T, w.d, w.dtype))

    e2e = None
    if not args.no_e2e:
        hq, hk, hv, hu = (x.cpu().pin_memory() for x in (q, k, v, u))
        hg = gO.cpu().pin_memory()
        hout = tuple(torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in out)
        ksteps = max(3, min(args.steps, args.e2e_steps))
        for _ in range(2):
            vla_backward(hq, hk, hv, hu, w.lambda0, w.eps, None, hg, out=hout)
        torch.cuda.synchronize(dev)
        barrier(world, dev)
        e0.record(stream)
        for _ in range(ksteps):
            vla_backward(hq, hk, hv, hu, w.lambda0, w.eps, None, hg, out=hout)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world, dev)
        e2e_ms = max_over_ranks(e0.elapsed_time(e1) / ksteps, world, dev)
        e2e = {"value": aggregate_value(units, world, e2e_ms / 1e3), "unit": UNIT,
               "h2d_bytes_per_step": sum(x.numel() * x.element_size() for x in (hq, hk, hv, hu, hg)),
               "d2h_bytes_per_step": sum(x.numel() * x.element_size() for x in hout),
               "ms_per_step": e2e_ms, "steps": ksteps}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        probe = min(w.T, 16)
        _, _, dt = oracle_time_bw(arrs, gO_np, w, probe, w.heads)
        tokens = int(max(1, min(w.T, probe * 15.0 / max(dt, 1e-6))))
        rate, threads, dt = oracle_time_bw(arrs, gO_np, w, tokens, w.heads)
        cpu = {"value": rate, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"all {w.heads} heads x first {tokens} of {w.T} tokens (fp64 oracle backward, {dt:.1f} s)"}

    if rank == 0:
        line = {
            "metric": METRIC_BW, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.describe(), "pass": "backward", "B": B, "H": H, "T": T, "d_h": d,
                       "input_dtype": w.dtype, "upstream": "dL/do ~ N(0,1) fp32, no state gradients",
                       "per_rank_heads": w.heads,
                       "l2": f"inputs larger than L2 ({in_bytes / 1e6:.0f} MB per step), no flush"},
            "roofline": {"bound": "alu", "achieved": achieved, "peak": peak_tflops, "unit": "TFLOP/s",
                         "frac": achieved / peak_tflops, "traffic": traffic,
                         "peak_basis": "measured: the FFMA probe in this run (packed FP32 FMA), of measured",
                         "peak_nominal": nominal_tflops, "frac_of_nominal": achieved / nominal_tflops,
                         "ffma_probe": probe,
                         "flop_per_head_token": FLOP_D2["backward"] * d * d, "kernel": kernel},
            "fp32_roofline_pct": 100.0 * achieved / peak_tflops,
            "hbm": {"achieved_gbs": hbm_gbs, "peak_gbs": hbm_peak, "frac": hbm_gbs / hbm_peak,
                    "algorithmic_bytes_per_launch": in_bytes + out_bytes,
                    "tape_bytes_per_launch": tape_bytes},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk.summary(),
            "kernel_source_sha": sha,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=3, help="workload id (1-5); 3 is d_h=96, T=4096")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip timing the other workloads (the `configs` object of the forward line)")
    ap.add_argument("--algo", type=int, default=0,
                    help="kernel: 0 automatic (chunked tensor-core kernel for d_h <= 96, its cluster forms "
                         "for d_h = 128, the segmented path for few heads of long sequences), 1 per-token, "
                         "2 chunked, 3 decode, 4 chunked on a cluster pair, 5 chunked on a cluster with S's "
                         "rows split, 6 the sequence's two halves side by side")
    ap.add_argument("--pass", dest="pass_", choices=["forward", "backward", "decode"], default="forward",
                    help="time the forward recurrence (default), its reverse-mode gradient, or one "
                         "decode step (T = 1) of 2048 heads from a carried state")
    ap.add_argument("--fixed-a", action="store_true",
                    help="forward pass: the fixed-A variant (A held at I/lambda0, eq. 9 skipped)")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's batch size B (smaller cases for profiler captures)")
    ap.add_argument("--tokens", type=int, default=0,
                    help="override the workload's sequence length T (smaller cases for profiler captures)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    from sherman_morrison_memory_gb300 import workloads as W

    w = W.WORKLOADS[args.workload]
    if args.batch > 0:
        w = dataclasses.replace(w, B=args.batch)
    if args.tokens > 0:
        w = dataclasses.replace(w, T=args.tokens)
    if args.impl == "reference":
        run_reference(args, w)
    elif args.pass_ == "backward":
        run_ours_backward(args, w)
    elif args.pass_ == "decode":
        run_ours_decode(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()

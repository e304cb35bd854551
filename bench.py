#!/usr/bin/env python3
"""TriMul forward benchmark on GB300: B=1, N=4096, D=C=256, outgoing, bf16 in/out.

One step = one trimul_forward (LN_in + gated in-projection, triangle GEMM,
LN_out + out-projection + gate) over inputs resident in HBM.  Prints ONE JSON
line (rank 0):
  value         TFLOP/s of algorithmic GEMM FLOPs, device-timed (CUDA events)
  e2e           same metric through trimul_forward_host with pinned host
                buffers: host->device of z and mask and device->host of out of
                every call inside the timed region.  value: calls made with
                FLAG_DEFER_OUTPUT (each call's output copy overlaps the next
                call's kernels), joined by trimul_host_join before the timer
                stops; sync_ms_per_step: the same calls without the flag.
  roofline      the dominant kernel (the triangle GEMM) against the measured
                burst dense bf16 peak (the stage runs inside a 35 ms step),
                with the fractions of the sustained and nominal peaks beside it
  cpu_baseline  the fp64 CPU oracle on a bounded sample of the same workload
``--impl reference`` times the CPU oracle alone (the reference arm).
``--oracle-table`` times the oracle's full evaluation of the two small
workloads on all host cores and on one core (no GPU needed).

Multi-GPU (torchrun): every rank runs an independent replica of the workload
(the path has no exchange step); value = FLOPs of all ranks / max time.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "TriMul fwd TFLOP/s & ms/call at N=4096 D=C=256 bf16; % of BF16 roofline"
WORKLOAD = "n4096_d256_c256"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Nominal dense bf16 (and fp16) tensor peak of one GB300, for context beside
# the measured peaks.
NOMINAL_BF16_TFLOPS = 2250.0
FP8_OVER_BF16 = 4500.0 / 2250.0  # nominal dense e4m3 / bf16 tensor rates

# DRAM bytes (read + write) of the triangle GEMM per channel plane at
# N = 4096, from a one-pass ncu capture (dram__bytes_read.sum +
# dram__bytes_write.sum) of this benchmark on B=1 N=4096 D=32 C=56, whose
# two launches of 28 planes match the 29-plane launches of the B=1 N=4096
# C=256 forward; scaled by its planes.  Valid only for the kernel and launch
# code it was taken on: the digest covers k2_triangle.cu and the triangle's
# launch code in trimul_api.cu.
K2_TRAFFIC_BYTES_PER_PLANE = 6751819520 / 56
K2_TRAFFIC_SOURCE_SHA256_16 = "038c1ed38d0b92f6"


def gemm_flops(B, N, D, C):
    """Algorithmic GEMM FLOPs: four D->C projections, the per-channel N^3
    contraction, the two output projections."""
    return B * (2 * N * N * D * 4 * C + 2 * C * N ** 3 + 2 * N * N * (D * D + C * D))


def backward_flops(B, N, D, C):
    """Algorithmic GEMM FLOPs of one backward, which recomputes the forward:
    the forward's, plus dy = dv W_o and dg W_g, the two triangle gradients,
    dz' through the four input projections, and the six weight gradients
    (sums over all pairs of outer products)."""
    P = B * N * N
    return (gemm_flops(B, N, D, C) + 2 * P * (D * C + D * D) + 4 * B * C * N ** 3
            + 2 * P * 4 * C * D + 2 * P * (D * C + D * D) + 2 * P * 4 * C * D)


def min_bytes(B, N, D, C):
    """Compulsory HBM bytes: read z (bf16) and the mask, write out (bf16), plus weights."""
    weights = 2 * (4 * C * D + D * C + D * D) + 4 * 2 * (D + C)
    return B * N * N * (2 * D + 2 + 2 * D) + weights


def sampled_flops(B, N, D, C, n_rows, n_cols):
    """GEMM FLOPs the sampled oracle evaluates: the token lines it needs (value
    and gate projections of N pairs each) and, per sampled pair, its
    contraction over k and its two output projections."""
    lines = n_rows + n_cols
    return B * (lines * 2 * 2 * N * D * C + n_rows * n_cols * (2 * C * N + 2 * D * (D + C)))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def peak_value(peaks, *keys):
    for k in keys:
        v = peaks.get(k)
        if isinstance(v, (int, float)):
            return float(v)
        if isinstance(v, dict):
            for kk in ("value", "tflops", "gbs"):
                if isinstance(v.get(kk), (int, float)):
                    return float(v[kk])
    return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (FileNotFoundError, OSError):
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

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        # the samples taken while the GPU ran at load (upper half of the clocks)
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if os.environ.get("BENCH_BACKEND", "nccl") == "nccl" else "gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def allreduce_max(x, world, device):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def oracle_sample(z_host, mask, params, w, n_rows, n_cols):
    """Time the fp64 CPU oracle on a rows x cols grid of pairs of the workload."""
    from co_folding_pair_gb300 import synthetic as S
    from oracle import trimul_oracle as O

    rows, cols = S.sample_grid(w, n_rows, n_cols)
    pn = {k: v.double().numpy() for k, v in params.items()}
    m = mask.float().cpu().numpy()
    zv = S.Bf16HostView.of(z_host)
    t0 = time.perf_counter()
    O.trimul_forward_sampled(zv, m, pn, w.directions[0], rows, cols)
    dt = time.perf_counter() - t0
    fl = sampled_flops(w.B, w.N, w.D, w.C, len(rows[0]), len(cols[0]))
    return dt, fl


def k2_traffic_digest():
    """sha256 (first 16 hex digits) of k2_triangle.cu and of trimul_api.cu's
    triangle launch code (from the launch grouping to the end of run_triangle)."""
    import hashlib
    csrc = os.path.join(ROOT, "co_folding_pair_gb300", "csrc")
    h = hashlib.sha256()
    with open(os.path.join(csrc, "k2_triangle.cu"), "rb") as f:
        h.update(f.read())
    with open(os.path.join(csrc, "trimul_api.cu"), "rb") as f:
        api = f.read()
    i0 = api.find(b"constexpr long long kTriTilesPerPair")
    i1 = api.find(b"trimul_status run_outproj(")
    if i0 < 0 or i1 < i0:
        return None
    h.update(api[i0:i1])
    return h.hexdigest()[:16]


def k2_traffic(w):
    """DRAM bytes of the triangle GEMM of one forward (all its launches) at
    B=1 N=4096 C=256, scaled from the per-plane capture, or None when the
    kernel or its launch code has changed since the capture or the workload
    is another (other launch sizes re-read the operands at other rates)."""
    if K2_TRAFFIC_BYTES_PER_PLANE is None or (w.B, w.N, w.C) != (1, 4096, 256):
        return None
    if k2_traffic_digest() != K2_TRAFFIC_SOURCE_SHA256_16:
        return None
    return K2_TRAFFIC_BYTES_PER_PLANE * w.B * w.C


def cores_used():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def run_reference(args, world, rank):
    """The reference arm: the fp64 CPU oracle as it stands, on a bounded sample
    of the workload per step (rank 0 only)."""
    if rank != 0:
        return
    import torch
    from co_folding_pair_gb300 import synthetic as S

    w = S.WORKLOADS[args.workload]
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    z, mask, params = S.make_case(w, device=dev)
    z_host = z.cpu()
    del z
    times, flops = [], 0
    for i in range(args.warmup + args.steps):
        dt, fl = oracle_sample(z_host, mask, params, w, args.cpu_rows, args.cpu_cols)
        if i >= args.warmup:
            times.append(dt)
            flops = fl
    total = sum(times)
    value = flops * len(times) / total / 1e12
    sample = (f"{args.cpu_rows}x{args.cpu_cols} grid of (i,j) pairs per step "
              f"({args.cpu_rows + args.cpu_cols} token lines of N={w.N}); value = GEMM FLOPs of the sampled "
              f"evaluation / its time")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores_used(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


ORACLE_TABLE_WORKLOADS = ("n64_d32_c32", "n256_d128_c128_tailmask")


def oracle_table_child(name, reps):
    """Time the oracle's full evaluation of one small workload (a child process,
    so that its BLAS thread count is fixed before numpy loads)."""
    import torch
    from co_folding_pair_gb300 import synthetic as S
    from oracle import trimul_oracle as O

    w = S.WORKLOADS[name]
    z, mask, params = S.make_case(w, device="cpu")
    pn = {k: v.double().numpy() for k, v in params.items()}
    zn, mn = z.double().numpy(), mask.double().numpy()
    O.trimul_forward(zn, mn, pn, w.directions[0])
    times = []
    for _ in range(reps):
        t0 = time.perf_counter()
        O.trimul_forward(zn, mn, pn, w.directions[0])
        times.append(time.perf_counter() - t0)
    dt = statistics.median(times)
    print(json.dumps({"workload": name, "cores": cores_used(), "median_s": dt, "reps": reps,
                      "tflops": gemm_flops(w.B, w.N, w.D, w.C) / dt / 1e12,
                      "torch_threads": torch.get_num_threads()}), flush=True)


def run_oracle_table():
    """The oracle's full evaluation of the small workloads, timed on all host
    cores and on one core (thread-count variables set and the process pinned
    to one CPU)."""
    rows = []
    all_cores = sorted(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else None
    for name in ORACLE_TABLE_WORKLOADS:
        for one in (False, True):
            env = dict(os.environ)
            if one:
                for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
                    env[k] = "1"
            code = ("import os, sys; sys.path.insert(0, %r); " % ROOT +
                    ("os.sched_setaffinity(0, {%d}); " % all_cores[0] if one and all_cores else "") +
                    "import bench; bench.oracle_table_child(%r, 5)" % name)
            r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, cwd=ROOT)
            if r.returncode != 0:
                raise RuntimeError(r.stderr)
            rows.append(json.loads(r.stdout.strip().splitlines()[-1]))
    print(json.dumps({"oracle_table": rows}), flush=True)


def workload_config(w, direction=None):
    direction = direction or w.directions[0]
    return {"workload": f"{w.name}: TriMul {direction} forward, B={w.B} N={w.N} D={w.D} C={w.C}, "
                        f"z ~ N(0,1) bf16, mask all ones, seed {w.seed}",
            "B": w.B, "N": w.N, "D": w.D, "C": w.C, "direction": direction,
            "io_dtype": "bf16", "mma_dtype": "fp16", "accumulate": "fp32",
            "l2": "inputs larger than L2 (z alone is %.1f GB); no flush" % (w.B * w.N * w.N * w.D * 2 / 1e9)}


def bench_backward(T, torch, w, z, mask, params, direction, local, dev, world, args, tensor_peak, hbm_peak,
                   peak_src):
    """trimul_backward on the same workload with a seeded dout: device time per
    call, whole-job TFLOP/s of its algorithmic FLOPs, and its roofline."""
    hb = T.trimul_create(params, device=local)
    stream = torch.cuda.current_stream(dev)
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed + 7)
    dout = torch.randn(z.shape, generator=g, device=dev).to(torch.bfloat16)
    dz = torch.empty_like(z)
    _, grads = T.trimul_backward(hb, z, mask, dout, direction, dz=dz, flags=T.FLAG_CHECK)
    for _ in range(2):
        T.trimul_backward(hb, z, mask, dout, direction, dz=dz, grads=grads)
    torch.cuda.synchronize()
    steps = args.backward_steps
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    barrier(world)
    with ClockSampler(local) as clk:
        torch.cuda.synchronize()
        start.record(stream)
        ev[0].record(stream)
        for i in range(steps):
            T.trimul_backward(hb, z, mask, dout, direction, dz=dz, grads=grads)
            ev[i + 1].record(stream)
        end.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    ms = allreduce_max(start.elapsed_time(end), world, dev)
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
    fl = backward_flops(w.B, w.N, w.D, w.C)
    achieved = fl * steps / (ms * 1e-3) / 1e12
    io_bytes = w.B * w.N * w.N * (3 * 2 * w.D + 2)  # z, dout in; dz out; mask
    t_roof = max(fl / (tensor_peak * 1e12), io_bytes / (hbm_peak * 1e9)) * 1e3
    res = {
        "metric": "TriMul bwd (gradients of z and every parameter, forward recomputed) TFLOP/s & ms/call",
        "value": fl * steps * world / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": ms / steps,
        "step_ms": {"median": statistics.median(per), "min": min(per)}, "steps": steps, "warmup": 3,
        "flops_per_step": fl, "dtype": "bf16 gradient planes, fp32 accumulation",
        "workspace_bytes": T.trimul_backward_workspace_bytes(hb, w.B, w.N),
        "gpu_launches": T.trimul_kernels_per_backward(hb, w.B, w.N) * steps,
        "roofline": {"kernel": "whole backward", "bound": "tensor", "achieved": achieved, "peak": tensor_peak,
                     "unit": "TFLOP/s", "frac": achieved / tensor_peak, "peak_kind": "burst",
                     "roofline_ms": t_roof, "path_frac": t_roof / (ms / steps), "source": peak_src},
        "clocks": clk.summary(),
    }
    T.trimul_destroy(hb)
    del dout, dz, grads
    torch.cuda.empty_cache()
    return res


def bench_fp8(T, torch, h, w, z, mask, out, direction, stream, world, dev, args, tensor_peak):
    """trimul_forward with FLAG_FP8 (e4m3 a and b, 8-bit triangle contraction):
    the same workload, step count and per-stage events as the main line.  The
    triangle kernel's roofline takes the dense e4m3 peak as the measured bf16
    burst peak times the nominal ratio of the two (4.5 / 2.25 PFLOP/s)."""
    for _ in range(args.warmup):
        T.trimul_forward(h, z, mask, direction, out=out, flags=T.FLAG_FP8)
    T.trimul_forward(h, z, mask, direction, out=out, flags=T.FLAG_FP8 | T.FLAG_CHECK)
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    for e4 in ev:  # created (recorded once) before the library records them
        for e in e4:
            e.record(stream)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier(world)
    with ClockSampler(dev.index) as clk:
        torch.cuda.synchronize()
        start.record(stream)
        for i in range(args.steps):
            T.trimul_set_stage_events(h, ev[i])
            T.trimul_forward(h, z, mask, direction, out=out, flags=T.FLAG_FP8)
        end.record(stream)
        torch.cuda.synchronize()
    T.trimul_set_stage_events(h, None)
    barrier(world)
    ms_max = allreduce_max(start.elapsed_time(end), world, dev)
    stage_ms = [statistics.mean(e4[k].elapsed_time(e4[k + 1]) for e4 in ev) for k in range(3)]
    fp8_peak = tensor_peak * FP8_OVER_BF16
    tri_achieved = 2 * w.B * w.C * w.N ** 3 / (stage_ms[1] * 1e-3) / 1e12
    return {
        "value": gemm_flops(w.B, w.N, w.D, w.C) * args.steps * world / (ms_max * 1e-3) / 1e12, "unit": "TFLOP/s",
        "ms_per_step": ms_max / args.steps, "steps": args.steps, "dtype": "e4m3 triangle operands, fp16 elsewhere",
        "accuracy": "opt-in: about 4e-2 relative Frobenius error against the exact result (default path 2e-3)",
        "stages_ms": {"k1_inproj": stage_ms[0], "k2_triangle": stage_ms[1], "k3_outproj": stage_ms[2]},
        "gpu_launches": T.trimul_kernels_per_forward(h, w.B, w.N) * args.steps,
        "roofline": {"kernel": "k2_triangle (e4m3)", "bound": "tensor", "achieved": tri_achieved, "peak": fp8_peak,
                     "unit": "TFLOP/s", "frac": tri_achieved / fp8_peak, "traffic": None,
                     "peak_source": "measured dense bf16 burst x 2 (nominal e4m3 / bf16 ratio)"},
        "clocks": clk.summary(),
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--direction", choices=["outgoing", "incoming"], default=None,
                    help="override the workload's direction (profiling runs)")
    ap.add_argument("--e2e-steps", type=int, default=None, help="timed host-buffer calls (default: --steps)")
    ap.add_argument("--cpu-rows", type=int, default=None,
                    help="rows of the oracle's sample grid (default 192 for cpu_baseline, 32 per reference step)")
    ap.add_argument("--cpu-cols", type=int, default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-backward", action="store_true", help="skip the backward-pass measurement")
    ap.add_argument("--backward-steps", type=int, default=10)
    ap.add_argument("--no-fp8", action="store_true", help="skip the opt-in e4m3 triangle path's measurement")
    ap.add_argument("--oracle-table", action="store_true",
                    help="time the oracle's full evaluation of the small workloads on all cores and on one core")
    args = ap.parse_args()
    if args.oracle_table:
        run_oracle_table()
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world, rank, local = dist_setup()
    default_grid = 32 if args.impl == "reference" else 192
    args.cpu_rows = args.cpu_rows or default_grid
    args.cpu_cols = args.cpu_cols or default_grid
    if args.impl == "reference":
        run_reference(args, world, rank)
        return

    import torch
    from co_folding_pair_gb300 import synthetic as S
    from co_folding_pair_gb300 import trimul as T

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = S.WORKLOADS[args.workload]
    direction = args.direction or w.directions[0]
    z, mask, params = S.make_case(w, device=dev)
    h = T.trimul_create(params, device=local)
    T.trimul_prepare(h, w.B, w.N)
    out = torch.empty_like(z)
    stream = torch.cuda.current_stream(dev)

    # ---------------- warm-up
    for _ in range(args.warmup):
        T.trimul_forward(h, z, mask, direction, out=out)
    T.trimul_forward(h, z, mask, direction, out=out, flags=T.FLAG_CHECK)  # surfaces any kernel timeout
    torch.cuda.synchronize()

    # ---------------- device-timed region with per-stage events
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    for e4 in ev:
        for e in e4:
            e.record(stream)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier(world)
    with ClockSampler(local) as clk:
        torch.cuda.synchronize()
        start.record(stream)
        for i in range(args.steps):
            T.trimul_set_stage_events(h, ev[i])
            T.trimul_forward(h, z, mask, direction, out=out)
        end.record(stream)
        torch.cuda.synchronize()
    T.trimul_set_stage_events(h, None)
    barrier(world)
    ms = start.elapsed_time(end)
    ms_max = allreduce_max(ms, world, dev)
    flops = gemm_flops(w.B, w.N, w.D, w.C)
    value = flops * args.steps * world / (ms_max * 1e-3) / 1e12
    stage_ms = [statistics.mean(e4[k].elapsed_time(e4[k + 1]) for e4 in ev) for k in range(3)]
    clocks = clk.summary()

    # ---------------- roofline of the dominant kernel (triangle GEMM) and of the path
    # The burst peak is the denominator: each step is a ~35 ms forward and
    # the whole timed region well under a second, not a seconds-long loop.
    # The sustained and nominal fractions are reported beside it.
    peaks, peak_src = load_peaks()
    tensor_peak = peak_value(peaks, "bf16_tflops") or FALLBACK_PEAKS["bf16_tflops"]
    sustained_peak = peak_value(peaks, "bf16_tflops_sustained") or FALLBACK_PEAKS["bf16_tflops_sustained"]
    hbm_peak = peak_value(peaks, "hbm_gbs") or FALLBACK_PEAKS["hbm_gbs"]
    tri_flops = 2 * w.B * w.C * w.N ** 3
    tri_achieved = tri_flops / (stage_ms[1] * 1e-3) / 1e12
    roofline = {"kernel": "k2_triangle", "bound": "tensor", "achieved": tri_achieved, "peak": tensor_peak,
                "unit": "TFLOP/s", "frac": tri_achieved / tensor_peak, "traffic": k2_traffic(w),
                "peak_kind": "burst", "peak_source": f"{peak_src} dense bf16 burst (fp16 runs at the bf16 rate)",
                "frac_of_sustained": tri_achieved / sustained_peak,
                "frac_of_nominal": tri_achieved / NOMINAL_BF16_TFLOPS}
    bytes_min = min_bytes(w.B, w.N, w.D, w.C)
    t_roof_ms = max(flops / (tensor_peak * 1e12), bytes_min / (hbm_peak * 1e9)) * 1e3
    t_roof_nominal_ms = max(flops / (NOMINAL_BF16_TFLOPS * 1e12), bytes_min / (hbm_peak * 1e9)) * 1e3
    ms_step = ms_max / args.steps
    step_ms = [e4[0].elapsed_time(e4[3]) for e4 in ev]

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp16", "data": "synthetic", "config": workload_config(w, direction),
        "parallelism": "replicas" if world > 1 else "single",
        "gpu_launches": T.trimul_kernels_per_forward(h, w.B, w.N) * args.steps,
        "step_ms": {"mean": ms_step, "median": statistics.median(step_ms), "min": min(step_ms),
                    "note": "median and min of the per-step stage-event spans; mean = timed region / steps"},
        "path_roofline": {"roofline_ms": t_roof_ms, "frac": t_roof_ms / ms_step, "peak_kind": "burst",
                          "tensor_peak_tflops": tensor_peak, "hbm_peak_gbs": hbm_peak, "source": peak_src,
                          "nominal_roofline_ms": t_roof_nominal_ms, "frac_of_nominal": t_roof_nominal_ms / ms_step,
                          "nominal_tensor_tflops": NOMINAL_BF16_TFLOPS},
        "stages_ms": {"k1_inproj": stage_ms[0], "k2_triangle": stage_ms[1], "k3_outproj": stage_ms[2]},
        "roofline": roofline, "clocks": clocks,
    }

    # ---------------- end to end through the host-buffer entry point
    if not args.no_e2e:
        z_host = z.cpu().pin_memory()
        m_host = mask.cpu().pin_memory()
        o_host = torch.empty_like(z_host).pin_memory()
        T.trimul_forward_host(h, z_host, m_host, direction, out_host=o_host, flags=T.FLAG_CHECK)
        torch.cuda.synchronize()
        barrier(world)
        e2e_steps = args.e2e_steps or args.steps

        def timed_host_calls(flags):
            """e2e_steps host-buffer calls back to back: every call copies its
            inputs in and its output out inside the timed region."""
            torch.cuda.synchronize()
            barrier(world)
            s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s2.record(stream)
            for _ in range(e2e_steps):
                T.trimul_forward_host(h, z_host, m_host, direction, out_host=o_host, flags=flags)
            T.trimul_host_join(h)  # every output copy is done before the timer stops
            e2.record(stream)
            torch.cuda.synchronize()
            barrier(world)
            return allreduce_max(s2.elapsed_time(e2), world, dev)

        ms_sync = timed_host_calls(0)  # stream waits for each call's output copy
        ms_e2e = timed_host_calls(T.FLAG_DEFER_OUTPUT)  # output copy of call i overlaps call i+1
        line["e2e"] = {"value": flops * e2e_steps * world / (ms_e2e * 1e-3) / 1e12, "unit": "TFLOP/s",
                       "ms_per_step": ms_e2e / e2e_steps, "steps": e2e_steps,
                       "mode": "pipelined: each call's output copy overlaps the next call (FLAG_DEFER_OUTPUT), "
                               "joined before the timer stops",
                       "sync_ms_per_step": ms_sync / e2e_steps,
                       "h2d_bytes_per_step": z_host.numel() * 2 + m_host.numel() * 2,
                       "d2h_bytes_per_step": o_host.numel() * 2}
        line["gpu_launches"] += 2 * T.trimul_kernels_per_forward_host(h, w.B, w.N) * e2e_steps
    else:
        z_host = None

    # ---------------- the opt-in 8-bit triangle path (its own timed region)
    if not args.no_fp8 and direction == "outgoing" and w.N % 16 == 0:
        line["fp8"] = bench_fp8(T, torch, h, w, z, mask, out, direction, stream, world, dev, args, tensor_peak)

    # ---------------- backward pass (its own handle and timed region)
    if not args.no_backward:
        T.trimul_destroy(h)
        h = None
        if z_host is not None:
            del z_host, m_host, o_host
            z_host = None
        del out
        torch.cuda.empty_cache()
        line["backward"] = bench_backward(T, torch, w, z, mask, params, direction, local, dev, world, args,
                                          tensor_peak, hbm_peak, peak_src)

    # ---------------- CPU oracle on a bounded sample (rank 0, single GPU only)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        if z_host is None:
            z_host = z.cpu()
        dt, fl = oracle_sample(z_host, mask, params, w, args.cpu_rows, args.cpu_cols)
        line["cpu_baseline"] = {
            "value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": cores_used(), "kind": "oracle",
            "sample": f"{args.cpu_rows}x{args.cpu_cols} grid of (i,j) pairs of the workload "
                      f"({args.cpu_rows + args.cpu_cols} token lines of N={w.N}), {dt:.1f} s; "
                      f"value = GEMM FLOPs of the sampled evaluation / its time"}
    if h is not None:
        T.trimul_destroy(h)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

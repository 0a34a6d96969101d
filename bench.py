#!/usr/bin/env python3
"""Benchmark of mamba_mimo_bwd_fwd on the pages' timed shape
(B=1, S=8192, H=16, G=1, R=4, N=P=64, C=16, rotary_dim_divisor=4, reduced
dout, D and Z on; synthetic inputs).  Prints one JSON line.

A step is one call of the C ABI entry point (all kernels of the op) on one
input set already resident in HBM.  Four input/output sets rotate between
steps (together larger than the 129 MB L2), so no step reuses the previous
step's data from L2.  Time is taken with CUDA events on the launching stream,
with a barrier and synchronize on both sides; under torchrun every rank runs
its own replica and the slowest rank's time counts.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl cuda|reference]

``--op bwd_bwd`` instead times the second backward stage (mamba_mimo_bwd_bwd)
on the same shape and prints its own line (metric, tensor roofline of its
gradient kernel, CPU-oracle baseline on a sample of heads).
"""

from __future__ import annotations

import argparse
import ctypes
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import synthetic_inputs as si  # noqa: E402

METRIC = "MIMO bwd_fwd tokens/s at B1 S8192 H16 N=P=64 R4 C16; HBM GB/s % of peak"
WORKLOAD_INDEX = 2
# The pages' own median for this shape (Ascend910, 53.849475 ms per call).
PAGES_TOKENS_PER_S = 8192 / 0.053849475
DOMINANT = "chunk_output"
KERNEL_DIR = os.path.join(ROOT, "mamba_mimo_chunked_gb300", "csrc")


# The sources of the first stage's kernels (the dominant kernel's traffic in
# profiles/ is valid while these are unchanged; the second stage's kernels
# live in mmbb.cuh).
FIRST_STAGE_SOURCES = ("mmbf_fast.cuh", "mmbf_tc.cuh", "mmbf_kernels.cu")


def kernel_source_sha256():
    """sha256 over the first stage's CUDA sources (in the order listed, concatenated)."""
    h = hashlib.sha256()
    for name in FIRST_STAGE_SOURCES:
        h.update(open(os.path.join(KERNEL_DIR, name), "rb").read())
    return h.hexdigest()
# Tensor instructions of each first-stage kernel family (by its variant number)
TENSOR_PATHS = {
    3: "tcgen05.mma kind::f16 M=64 N=64 K=16, TMEM accumulators (inter, intra); "
       "mma.sync m16n8k16 bf16 (causal scores, state fold, same-token qk_dot)",
    0: "mma.sync m16n8k16 bf16 (inter, scores, intra, qk_dot); tcgen05.mma state sums",
    4: "mma.sync m16n8k16 bf16 (inter, scores, intra, qk_dot, state sums and updates)",
}
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["cuda", "reference"], default="cuda")
    ap.add_argument("--sets", type=int, default=4)
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--with-y", action="store_true",
                    help="time mamba_mimo_bwd_fwd_y (the op plus the layer's forward output y)")
    ap.add_argument("--workload", type=int, default=None,
                    help="index into synthetic_inputs.WORKLOADS (default: the timed shape, 2); other "
                         "shapes print their own line (no pages' number to compare, no profile traffic)")
    ap.add_argument("--quick", action="store_true",
                    help="warm-up and timed steps only (no clock-load stretch, per-kernel event pass, "
                         "end-to-end pass or CPU baseline): the short command ncu captures run")
    ap.add_argument("--heads", type=int, default=None,
                    help="with --quick: the workload with H heads (G capped at H) instead of its own "
                         "count, the same per-head shape; a smaller case of the same kernels for ncu")
    ap.add_argument("--op", choices=["bwd_fwd", "bwd_bwd"], default="bwd_fwd",
                    help="bwd_bwd: time the second backward stage instead (its own JSON line)")
    return ap.parse_args()


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, dev) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def measured_bf16_tflops():
    """Sustained dense bf16 tensor throughput of this machine's GPUs (the
    output kernel runs inside a long step), or the fallback figure."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"])), "measured sustained"
    except Exception:
        return 1700.0, "fallback sustained"


def algorithmic_flop(wl):
    """Dense contraction FLOP per call, masked upper triangle not counted:
    per chunk and (b,h), 4*CR*N*P (state GEMM + inter) + R^2*C*(C-1)*(N+P)
    (strictly causal Q K^T and A PsiV) + 2*C*R^2*(N+P) (qk_dot + diagonal)."""
    nc = -(-wl.S // wl.C)
    CR = wl.C * wl.R
    per = 4 * CR * wl.N * wl.P + wl.R ** 2 * wl.C * (wl.C - 1) * (wl.N + wl.P) \
        + 2 * wl.C * wl.R ** 2 * (wl.N + wl.P)
    return per * nc * wl.B * wl.H


def profile_traffic():
    """Per-launch DRAM bytes of the dominant kernel from the committed ncu
    summary, if it was taken on the current kernel source (else None)."""
    sha = kernel_source_sha256()
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None
    for name in sorted(os.listdir(pdir)):
        if not name.startswith(DOMINANT) or not name.endswith(".md"):
            continue
        vals = {}
        for line in open(os.path.join(pdir, name)):
            if ":" in line and line.strip().startswith(("traffic_bytes_per_launch", "source_sha256")):
                k, v = line.strip().split(":", 1)
                vals[k.strip()] = v.strip().strip("`")
        if vals.get("source_sha256") == sha and "traffic_bytes_per_launch" in vals:
            return float(vals["traffic_bytes_per_launch"])
    return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""

    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, dev):
        try:
            self.uuid = str(torch.cuda.get_device_properties(dev).uuid)
        except Exception:
            self.uuid = None
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        rows = [r.split(", ") for r in out.strip().splitlines() if r.count(",") >= 7]
        if self.uuid:
            mine = [r for r in rows if self.uuid.replace("GPU-", "") in r[0]]
            rows = mine or rows
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({n for r in rows for n, v in zip(names, r[4:8]) if v.strip() == "Active"})
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(sm)}


def nbytes(t):
    return 0 if t is None else t.numel() * t.element_size()


def cpu_baseline(inp_cpu, wl):
    """The oracle as it stands, timed on this host's cores on the whole
    workload (every (b,h) head of one input set, BF16-boundary mode)."""
    cores = os.cpu_count() or 1
    os.environ.setdefault("OMP_NUM_THREADS", str(cores))
    import oracle
    oracle.build()
    t0 = time.perf_counter()
    oracle.bwd_fwd(*si.args_of(inp_cpu))
    dt = time.perf_counter() - t0
    used = min(cores, int(os.environ.get("OMP_NUM_THREADS", cores)), wl.B * wl.H)  # OpenMP over heads
    return {"value": wl.B * wl.S / dt, "unit": "tokens/s", "cores": used, "kind": "oracle",
            "sample": f"one full pass over all B*H={wl.B * wl.H} heads of {wl.name} "
                      f"(BF16-boundary oracle, OpenMP over heads), {dt:.2f} s"}


def run_reference(args, world, rank):
    """Reference arm: the CPU oracle, timed on host cores.  Each step is a
    bounded sample of the workload: every (b,h) head (OpenMP over heads) over
    a prefix of the sequence, sized so the whole run takes about two minutes."""
    if rank != 0:
        return
    cores = os.cpu_count() or 1
    os.environ.setdefault("OMP_NUM_THREADS", str(cores))
    import oracle
    oracle.build()
    wl = si.WORKLOADS[WORKLOAD_INDEX]
    inp = si.workload_inputs(WORKLOAD_INDEX)
    used = min(cores, int(os.environ.get("OMP_NUM_THREADS", cores)), wl.B * wl.H)
    # Calibrate: seconds per chunk of all heads.
    probe = _prefix(inp, wl.C * 4, wl.C)
    t0 = time.perf_counter()
    oracle.bwd_fwd(*si.args_of(probe))
    per_chunk = max((time.perf_counter() - t0) / 4, 1e-6)
    budget = 120.0 / max(args.steps + args.warmup, 1)
    chunks = int(min(wl.nchunks, max(1, budget / per_chunk)))
    tokens = chunks * wl.C
    sample_inp = _prefix(inp, tokens, wl.C)
    for i in range(args.warmup):
        oracle.bwd_fwd(*si.args_of(sample_inp))
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle.bwd_fwd(*si.args_of(sample_inp))
    dt = time.perf_counter() - t0
    value = tokens * wl.B * args.steps / dt
    sample = f"per step: all {wl.B * wl.H} heads of {wl.name}, first {tokens} tokens ({chunks} chunks)"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": value / PAGES_TOKENS_PER_S, "dtype": "f64+bf16-rounding",
            "data": "synthetic", "config": {"workload": wl.name},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": used, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def _prefix(inp, tokens, C):
    """The first `tokens` tokens (a multiple of C) of a problem (every head)."""
    out = dict(inp)
    nc = tokens // C
    for n in ("dout", "q", "k", "v", "z", "angles"):
        if inp[n] is not None:
            out[n] = inp[n][:, :tokens].contiguous()
    for n in ("da_cs", "da_cs_rev", "dt", "trap"):
        out[n] = inp[n][:, :, :tokens].contiguous()
    out["segsum"] = inp["segsum"][:, :, :nc].contiguous()
    return out


BB_METRIC = "MIMO bwd_bwd tokens/s at B1 S8192 H16 N=P=64 R4 C16"
TF32_PER_BF16 = 1.1 / 2.25  # nominal dense TF32 / BF16 tensor throughput of a GB300


def bb_grad_flop(wl):
    """Algorithmic FLOP of the second stage's gradient kernel per call:
    per chunk and (b,h), the five strictly causal products (Q Ks^T, A^T dPhiO,
    dPhiO PsiV^T, dS Ks, dS^T Q: R^2 C(C-1)/2 x (3N + 2P) multiply-adds) and
    the four state products (dPhiO Hc^T, k_state D, PsiV D^T, Q Hc: 4 CR N P)."""
    nc = -(-wl.S // wl.C)
    CR = wl.C * wl.R
    macs = wl.R ** 2 * wl.C * (wl.C - 1) // 2 * (3 * wl.N + 2 * wl.P) + 4 * CR * wl.N * wl.P
    return 2 * macs * nc * wl.B * wl.H


def _bb_inputs(wl, seed, device):
    inp = si.make_inputs(B=wl.B, S=wl.S, H=wl.H, G=wl.G, R=wl.R, N=wl.N, P=wl.P, C=wl.C, div=wl.div,
                         reduced=True, has_z=False, has_d=True, seed=seed, device=device)
    states, qk = si.make_stage1_caches(B=wl.B, S=wl.S, H=wl.H, R=wl.R, N=wl.N, P=wl.P, C=wl.C, seed=seed + 1,
                                       device=device)
    args = [inp["dout"], inp["q"], inp["k"], inp["v"], inp["q_bias"], inp["k_bias"], inp["mimo_v"], states, qk,
            inp["da_cs"], inp["da_cs_rev"], inp["dt"], inp["trap"], inp["segsum"], inp["angles"],
            inp["mimo_o"], inp["d"]]
    return args


def run_bwd_bwd(args, world, rank, local):
    """Second backward stage: C-ABI calls on resident input/output sets."""
    import mamba_mimo_chunked_gb300 as mm

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    mm.build()
    lib = mm.load_library()
    wl = si.WORKLOADS[WORKLOAD_INDEX if args.workload is None else args.workload]
    stream = torch.cuda.current_stream(dev)
    steps = args.steps if args.steps != 20000 else 300   # the default count is the first stage's
    nsets = 2                                            # each set ~0.45 GB, over the L2
    sets = []
    for s in range(nsets):
        a = _bb_inputs(wl, si.WORKLOAD_SEED_BASE + 31 * s + 104729 * rank, dev)
        outs = mm.mamba_mimo_bwd_bwd(*a[:15], mimo_o=a[15], d=a[16], chunk_size=wl.C, rotary_dim_divisor=wl.div,
                                     output_dtype=torch.float32)  # the pages' example call
        sets.append((a, outs))
    torch.cuda.synchronize(dev)
    in_bytes = sum(nbytes(t) for t in sets[0][0])
    out_bytes = sum(nbytes(t) for t in sets[0][1].values())
    ws_bytes = mm.bwd_bwd_workspace_size(wl.B, wl.S, wl.H, wl.G, wl.R, wl.N, wl.P, wl.C, wl.div)
    workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    dims = mm._Dims(wl.B, wl.S, wl.H, wl.G, wl.R, wl.N, wl.P)
    sh = ctypes.c_void_p(stream.cuda_stream)
    call_args = [[ctypes.byref(dims)] + [mm._ptr(t) for t in a] + [wl.C, wl.div, 1, 0]
                 + [mm._ptr(o[n]) for n in mm.BWD_BWD_OUTPUTS] + [mm._ptr(workspace), ws_bytes, sh]
                 for a, o in sets]
    for i in range(args.warmup):
        st = lib.mamba_mimo_bwd_bwd(*call_args[i % nsets])
        if st:
            mm._raise(lib, st)
    launches = lib.mamba_mimo_last_launch_count()
    every = max(1, steps // 100)
    n_samples = (steps + every - 1) // every
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(8)] for _ in range(n_samples)]
    for row in ev:
        for e in row:
            e.record(stream)
    torch.cuda.synchronize(dev)
    ev_arrays = [(ctypes.c_void_p * 8)(*[ctypes.c_void_p(e.cuda_event) for e in row]) for row in ev]
    sampler = ClockSampler(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    sampler.start()
    time.sleep(0.3)
    start.record(stream)
    bad = 0
    for i in range(steps):
        if i % every == 0:
            lib.mamba_mimo_set_stage_events(ev_arrays[i // every], 8)
            bad |= lib.mamba_mimo_bwd_bwd(*call_args[i % nsets])
            lib.mamba_mimo_set_stage_events(None, 0)
        else:
            bad |= lib.mamba_mimo_bwd_bwd(*call_args[i % nsets])
    end.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    barrier(world)
    if bad:
        raise RuntimeError("a timed call failed")
    elapsed_s = max_over_ranks(start.elapsed_time(end) / 1e3, world, dev)
    stage_ms = {}
    for k in range(launches):
        name = lib.mamba_mimo_stage_name(k)
        if name:
            stage_ms[name.decode()] = statistics.mean(row[2 * k].elapsed_time(row[2 * k + 1]) for row in ev)
    grad_ms = stage_ms["bb_grad"]
    # the products run on the tensor cores in TF32 (three passes per FP32
    # product): the peak is TF32's, the measured BF16 figure times the
    # nominal TF32 / BF16 ratio
    bf16_peak, bf16_kind = measured_bf16_tflops()
    tc_peak = bf16_peak * TF32_PER_BF16
    flop = bb_grad_flop(wl)
    achieved = flop / (grad_ms * 1e-3) / 1e12
    hbm, hbm_kind = measured_peaks()
    ms_per_step = elapsed_s * 1e3 / steps
    value = wl.B * wl.S * steps * world / elapsed_s
    line = {
        "metric": BB_METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": wl.name + "_bwd_bwd", "B": wl.B, "S": wl.S, "H": wl.H, "G": wl.G, "R": wl.R,
                   "N": wl.N, "P": wl.P, "chunk_size": wl.C, "rotary_dim_divisor": wl.div, "reduced_dout": True,
                   "d": True, "caches": "seeded stand-ins for states / qk_dot",
                   "parallelism": f"replicas{world}",
                   "l2": f"{nsets} rotating input+output sets, {nsets * (in_bytes + out_bytes) / 1e6:.0f} MB > 129 MB L2"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": tc_peak, "unit": "TFLOP/s",
                     "frac": achieved / tc_peak, "traffic": None, "kernel": "bb_grad",
                     "algorithmic_flop_per_launch": flop,
                     "peak_source": f"{bf16_kind} bf16 x nominal tf32/bf16 {TF32_PER_BF16:.3f}",
                     "path": "mma.sync m16n8k8 tf32, three passes per FP32 product (hi.hi + hi.lo + lo.hi)"},
        "op_hbm_frac": (in_bytes + out_bytes) / (ms_per_step * 1e-3) / 1e9 / hbm,
        "algorithmic_bytes_per_call": in_bytes + out_bytes,
        "stage_ms": stage_ms, "gpu_launches": launches * steps, "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = bb_cpu_baseline(sets[0][0], wl)
    if rank == 0:
        print(json.dumps(line), flush=True)


def bb_cpu_baseline(a, wl, heads=2):
    """The second-stage oracle as it stands (numpy, float64), timed on a
    sample of `heads` heads of the workload and scaled to tokens/s of the
    whole problem."""
    from oracle import bwd_bwd as bb
    cpu = [None if t is None else t.cpu() for t in a]
    hs = slice(0, heads)
    dout, q, k, v, qb, kb, mv, st, qk, dcs, dcr, dt, tr, seg, ang, mo, d = cpu
    t0 = time.perf_counter()
    bb.bwd_bwd(dout[:, :, hs], q, k, v[:, :, hs], qb[hs], kb[hs], mv[hs], st[:, hs], qk[:, hs], dcs[:, hs],
               dcr[:, hs], dt[:, hs], tr[:, hs], seg[:, hs], ang[:, :, hs], mimo_o=mo[hs], d=d[hs],
               chunk_size=wl.C, rotary_dim_divisor=wl.div)
    dt_s = time.perf_counter() - t0
    return {"value": wl.B * wl.S / (dt_s * wl.H / heads), "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{heads} of {wl.H} heads of {wl.name} (numpy float64, one thread), {dt_s:.2f} s"}


def main():
    args = parse_args()
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    if args.op == "bwd_bwd":
        run_bwd_bwd(args, world, rank, local)
        return
    import mamba_mimo_chunked_gb300 as mm

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    mm.build()
    lib = mm.load_library()
    wi = WORKLOAD_INDEX if args.workload is None else args.workload
    wl = si.WORKLOADS[wi]
    timed_shape = wi == WORKLOAD_INDEX
    if args.heads is not None:
        if not args.quick:
            raise SystemExit("--heads is for the short capture runs (--quick) only")
        g = min(wl.G, args.heads)
        if args.heads < 1 or args.heads % g:
            raise SystemExit(f"--heads {args.heads}: H must be a positive multiple of G = {g}")
        wl = dataclasses.replace(wl, name=f"{wl.name}_h{args.heads}", H=args.heads, G=g)
        timed_shape = False
    stream = torch.cuda.current_stream(dev)

    # Input/output sets, resident in HBM before timing starts.
    sets = []
    for s in range(args.sets):
        inp = si.make_inputs(**wl.shape_kwargs(), seed=si.WORKLOAD_SEED_BASE + wi + 7919 * s
                             + 104729 * rank, device=dev)
        if args.with_y:  # y travels with the outputs (last field)
            out, y = mm.mamba_mimo_bwd_fwd_with_y(*si.args_of(inp))
            out = tuple(out) + (y,)
        else:
            out = mm.mamba_mimo_bwd_fwd(*si.args_of(inp))  # allocates outputs, validates once
        sets.append((inp, out))
    torch.cuda.synchronize(dev)
    in_bytes = sum(nbytes(sets[0][0][n]) for n in si.ARG_NAMES)
    out_bytes = sum(nbytes(t) for t in sets[0][1])
    alg_bytes = in_bytes + out_bytes
    ws_bytes = mm.workspace_size(wl.B, wl.S, wl.H, wl.G, wl.R, wl.N, wl.P, wl.C, wl.div,
                                 wl.reduced, wl.has_z)
    workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    dims = mm._Dims(wl.B, wl.S, wl.H, wl.G, wl.R, wl.N, wl.P)
    sh = ctypes.c_void_p(stream.cuda_stream)

    def cargs(inp, out):
        ptr = mm._ptr
        return ([ctypes.byref(dims)] + [ptr(inp[n]) for n in si.ARG_NAMES] + [wl.C, wl.div]
                + [ptr(o) for o in out] + [ptr(workspace), ws_bytes, sh])

    call_args = [cargs(i, o) for i, o in sets]
    call = lib.mamba_mimo_bwd_fwd_y if args.with_y else lib.mamba_mimo_bwd_fwd

    for i in range(args.warmup):
        st = call(*call_args[i % len(call_args)])
        if st:
            mm._raise(lib, st)
    launches_per_call = lib.mamba_mimo_last_launch_count()
    variant = lib.mamba_mimo_last_kernel_variant()

    # Per-kernel CUDA events are taken in a separate, untimed pass after the
    # timed region: an event recorded between two kernels of a call keeps the
    # next kernel from launching early (programmatic dependent launch), so
    # timed steps carry no events.
    n_samples = 200
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(8)] for _ in range(n_samples)]
    for row in ev:                      # torch creates the CUDA event on first record
        for e in row:
            e.record(stream)
    torch.cuda.synchronize(dev)
    ev_arrays = [(ctypes.c_void_p * 8)(*[ctypes.c_void_p(e.cuda_event) for e in row]) for row in ev]
    assert all(e.cuda_event for row in ev for e in row)

    # The clock sampler runs across a stretch of untimed steps (about half a
    # second) directly before the timed region and across the timed region
    # itself, so a short timed region still has samples under load.
    sampler = ClockSampler(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    sampler.start()
    t_load = time.perf_counter()
    i = 0
    while not args.quick and time.perf_counter() - t_load < 0.6:
        for _ in range(64):
            bad = call(*call_args[i % len(call_args)])
            i += 1
            if bad:
                mm._raise(lib, bad)
        torch.cuda.synchronize(dev)
    barrier(world)
    torch.cuda.synchronize(dev)
    start.record(stream)
    bad = 0
    for i in range(args.steps):
        bad |= call(*call_args[i % len(call_args)])
    end.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    barrier(world)
    if bad:
        raise RuntimeError("a timed call failed")
    elapsed_s = max_over_ranks(start.elapsed_time(end) / 1e3, world, dev)

    for i in range(0 if args.quick else n_samples):  # untimed: per-kernel durations
        lib.mamba_mimo_set_stage_events(ev_arrays[i], 8)
        st = call(*call_args[i % len(call_args)])
        lib.mamba_mimo_set_stage_events(None, 0)
        if st:
            mm._raise(lib, st)
    torch.cuda.synchronize(dev)

    if args.quick:  # the short run ncu captures: timing only
        if rank == 0:
            print(json.dumps({"metric": METRIC if timed_shape else f"MIMO bwd_fwd tokens/s at {wl.name}",
                              "quick": True, "ms_per_step": elapsed_s * 1e3 / args.steps,
                              "value": wl.B * wl.S * args.steps * world / elapsed_s, "unit": "tokens/s",
                              "config": {"workload": wl.name}}), flush=True)
        return
    stage_ms = {}
    for k in range(min(4, launches_per_call)):
        name = lib.mamba_mimo_stage_name(k)
        if not name:
            continue
        name = name.decode() if isinstance(name, bytes) else ctypes.string_at(name).decode()
        stage_ms[name] = statistics.mean(row[2 * k].elapsed_time(row[2 * k + 1]) for row in ev)
    dom_ms = stage_ms[DOMINANT]
    peak, peak_kind = measured_peaks()
    achieved = alg_bytes / (dom_ms * 1e-3) / 1e9
    alg_flop = algorithmic_flop(wl)
    tpeak, tpeak_kind = measured_bf16_tflops()
    tflops = alg_flop / (dom_ms * 1e-3) / 1e12
    ms_per_step = elapsed_s * 1e3 / args.steps
    value = wl.B * wl.S * args.steps * world / elapsed_s

    # End to end through the public API with host buffers: every step uploads
    # its inputs from pinned host memory, runs the op and downloads its
    # outputs.  Steps are pipelined the way a data path would run them: an
    # upload stream, the compute stream and a download stream, two device
    # buffer sets and two host output sets, ordered by events, so step i+1's
    # upload and step i-1's download overlap step i's compute.
    # Each step's inputs and outputs sit in one contiguous buffer each (views
    # at 256-byte aligned offsets), so a step is one upload and one download.
    src_inp, src_out = sets[0]
    in_names = [n for n in si.ARG_NAMES if isinstance(src_inp[n], torch.Tensor)]

    def packed(tensors, **alloc):
        offs, off = [], 0
        for t in tensors:
            offs.append(off)
            off += (t.numel() * t.element_size() + 255) // 256 * 256
        buf = torch.empty(off, dtype=torch.uint8, **alloc)
        views = [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
                 for o, t in zip(offs, tensors)]
        return buf, views

    host_in_buf, host_in_views = packed([src_inp[n] for n in in_names], pin_memory=True)
    for v, n in zip(host_in_views, in_names):
        v.copy_(src_inp[n])
    out_list = [t for t in src_out if t is not None]
    bufs = []
    for _ in range(2):
        dbuf, dviews = packed([src_inp[n] for n in in_names], device=dev)
        inp = dict(src_inp)
        inp.update(dict(zip(in_names, dviews)))
        obuf, oviews = packed(out_list, device=dev)
        it = iter(oviews)
        out = tuple(None if t is None else next(it) for t in src_out)
        bufs.append((dbuf, inp, obuf, out))
    host_out = [packed(out_list, pin_memory=True)[0] for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    for e in ev_comp + ev_out:
        e.record(stream)
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def e2e_step(i):
        k = i % 2
        dbuf, inp, obuf, out = bufs[k]
        with torch.cuda.stream(s_in):
            s_in.wait_event(ev_comp[k])          # step i-2 has consumed this input set
            dbuf.copy_(host_in_buf, non_blocking=True)
            ev_in[k].record(s_in)
        stream.wait_event(ev_in[k])
        stream.wait_event(ev_out[k])             # step i-2's outputs have been downloaded
        if args.with_y:
            mm.mamba_mimo_bwd_fwd_with_y(*si.args_of(inp), out=mm.MambaMimoBwdFwdOutputs(*out[:5]),
                                         workspace=workspace, y=out[5])
        else:
            mm.mamba_mimo_bwd_fwd(*si.args_of(inp), out=mm.MambaMimoBwdFwdOutputs(*out),
                                  workspace=workspace)
        ev_comp[k].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[k])
            host_out[k].copy_(obuf, non_blocking=True)
            ev_out[k].record(s_out)

    for i in range(4):
        e2e_step(i)
    barrier(world)
    torch.cuda.synchronize(dev)
    e_start.record(s_in)
    for i in range(args.e2e_steps):
        e2e_step(i)
    e_end.record(s_out)
    torch.cuda.synchronize(dev)
    e2e_s = max_over_ranks(e_start.elapsed_time(e_end) / 1e3, world, dev)
    e2e = {"value": wl.B * wl.S * args.e2e_steps * world / e2e_s, "unit": "tokens/s",
           "h2d_bytes_per_step": host_in_buf.numel(), "d2h_bytes_per_step": host_out[0].numel(),
           "ms_per_step": e2e_s * 1e3 / args.e2e_steps,
           "pipelining": "upload / compute / download streams, two buffer sets, "
                         "one packed buffer each way per step"}

    line = {
        "metric": METRIC if timed_shape else f"MIMO bwd_fwd tokens/s at {wl.name}",
        "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": value / (PAGES_TOKENS_PER_S * world) if timed_shape else None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl.name, "B": wl.B, "S": wl.S, "H": wl.H, "G": wl.G, "R": wl.R,
                   "N": wl.N, "P": wl.P, "chunk_size": wl.C, "rotary_dim_divisor": wl.div,
                   "reduced_dout": wl.reduced, "z": wl.has_z, "d": wl.has_d,
                   "parallelism": f"replicas{world}", "with_y": bool(args.with_y),
                   "l2": f"{args.sets} rotating input+output sets, "
                         f"{args.sets * alg_bytes / 1e6:.0f} MB > 129 MB L2"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": profile_traffic() if timed_shape else None,
                     "kernel": DOMINANT, "algorithmic_bytes_per_launch": alg_bytes,
                     "peak_source": peak_kind},
        "op_hbm_frac": alg_bytes / (ms_per_step * 1e-3) / 1e9 / peak,
        "tensor": {"achieved": tflops, "peak": tpeak, "unit": "TFLOP/s", "frac": tflops / tpeak,
                   "kernel": DOMINANT, "algorithmic_flop_per_launch": alg_flop,
                   "peak_source": tpeak_kind, "path": TENSOR_PATHS.get(variant, "mma.sync m16n8k16 bf16")},
        "stage_ms": stage_ms,
        "gpu_launches": launches_per_call * args.steps,
        "e2e": e2e,
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        inp_cpu = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in sets[0][0].items()}
        line["cpu_baseline"] = cpu_baseline(inp_cpu, wl)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

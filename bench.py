"""Benchmark of the NVFP4 MoE decode hot path on GB300.

One step = one MoE decode pass over a batch of 256 tokens with 128 experts
and top-8 routing: route, quantise the BF16 activations on the fly into
route order, gate_up grouped GEMM (K=6144, N=4096), quantise the
route-ordered intermediate, down grouped GEMM (K=2048, N=6144) with the
weighted scatter-combine back to token order.  The metric is the grouped
GEMM throughput at ~16 tokens per expert, in TFLOPS, with HBM GB/s and the
roofline fraction alongside.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun every rank runs its own replica (independent batches, no
data-path collective): weak scaling.  Weights are NVFP4, resident in HBM
(2.72 GB per step, far larger than L2, so every step streams them from
HBM).  `--impl reference` times the CPU oracle on a bounded sample of the
same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from moe_grouped_gemm_nvfp4_gb300 import attention, inputs, moe  # noqa: E402
from moe_grouped_gemm_nvfp4_gb300 import nvfp4 as F  # noqa: E402

METRIC = "NVFP4 grouped-GEMM TFLOPS & HBM GB/s (frac. of roofline) at 16-64 tok/expert"
UNIT = "TFLOPS"
E, TOPK, T = 128, 8, 256    # T = 2 * E keeps 16 routes per expert (see --experts)
K1, N1 = 6144, 4096        # gate_up
K2, N2 = 2048, 6144        # down
FALLBACK_HBM_GBS = 6800.0


def _set_experts(n):
    global E, T
    E, T = n, 2 * n


def workload_config():
    return {
        "workload": f"moe_decode_layer E{E} top{TOPK} T{T}: gate_up K{K1} N{N1} + down K{K2} N{N2}",
        "tokens_per_expert_mean": T * TOPK / E,
        "global_batch": T,
        "weights": "NVFP4 E2M1 + E4M3/16 + FP32 per expert, ~N(0,0.02) before quantisation",
        "activations": "BF16 ~N(0,1), quantised on the fly each step",
        "l2": f"inputs larger than L2 ({E * (N1 * K1 + N2 * K2) * 0.5625 / 1e9:.2f} GB of "
              f"expert weights streamed per step)",
        "parallelism": "replicas",
    }


def flops_per_step():
    R = T * TOPK
    return 2.0 * R * N1 * K1 + 2.0 * R * N2 * K2


def gemm_bytes(K, N, n_active, R, out_rows):
    """Algorithmic bytes of one grouped-GEMM launch: NVFP4 weights of the
    active experts (0.5 + 1/16 B per element), the quantised activations
    read once (same rate), BF16 output written once."""
    w = n_active * N * K * (0.5 + 1.0 / 16)
    a = R * K * (0.5 + 1.0 / 16)
    o = out_rows * N * 2.0
    return w + a + o


def sparse_gemm_bytes(K, N, n_active, R, out_rows):
    """gemm_bytes with 2:4-sparse weights: per weight element 0.25 B of kept
    codes, 0.0625 B of combination indices (4 bits per 8 elements) and the
    0.0625 B of scales."""
    w = n_active * N * K * (0.25 + 0.0625 + 0.0625)
    a = R * K * (0.5 + 1.0 / 16)
    o = out_rows * N * 2.0
    return w + a + o


def step_bytes(n_active, sparse=False):
    """Algorithmic HBM bytes of a step: weights of the active experts, BF16
    activations in (x, h) and BF16 outputs (gate_up, down) once each."""
    R = T * TOPK
    w = n_active * (N1 * K1 + N2 * K2) * ((0.375 if sparse else 0.5 + 1.0 / 16))
    io = 2.0 * (T * K1 + R * K2 + R * N1 + T * N2)
    return w + io


def max_over_ranks(values, world, device):
    """Elementwise max of per-rank timings (every rank gets the result)."""
    local = torch.tensor(values, dtype=torch.float64)
    if world > 1:
        t = local.to(device)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        local = t.cpu()
    return local.tolist()


def aggregate_tflops(flops_per_rank_step, steps, ms_max, world):
    """Whole-job throughput: every rank's work over the slowest rank's time."""
    return world * flops_per_rank_step * steps / (ms_max * 1e-3) / 1e12


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d.get("hbm_gbs", FALLBACK_HBM_GBS)), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def normalised_source(src):
    """C++ source without comments, runs of blank space as one space."""
    import re
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return " ".join(src.split())


def kernel_source_hash():
    """Hash of the GEMM kernel's sources with comments and blank space taken
    out, so that edits to comments keep the recorded counters valid."""
    h = hashlib.sha256()
    for f in ("gemm.cu", "common.cuh", "kernels.h"):
        with open(os.path.join(ROOT, "moe_grouped_gemm_nvfp4_gb300", "csrc", f)) as fh:
            h.update(normalised_source(fh.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic():
    """DRAM bytes per gate_up launch from the committed ncu summary, or None
    when the kernel source changed since the counters were taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("kernel_source_hash") != kernel_source_hash():
        return None
    return d.get("dram_bytes_per_gate_up_launch")


class ClockSampler:
    """nvidia-smi clock/throttle sampling during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.5)

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [r.split(", ") for r in out.strip().splitlines() if r.count(",") >= 8]
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip() == "Active"})
        # samples taken while the GPU was loaded (clock within 60% of max or the
        # middle of the sequence when the timed region was shorter than a sample)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


def build_problem(device, seed_base=2, tokens=None, sparse=False):
    """Resident NVFP4 weights and one batch of per-step inputs (seeded);
    sparse: the same weights pruned to 2:4 and held as sparse tiles."""
    T = globals()["T"] if tokens is None else tokens
    t0 = time.time()
    w1 = torch.empty((E, N1, K1), dtype=torch.bfloat16, device=device)
    w2 = torch.empty((E, N2, K2), dtype=torch.bfloat16, device=device)
    for e in range(E):
        w1[e] = inputs.device_normal_bf16((N1, K1), 0.02, seed_base * 100003 + e, device)
        w2[e] = inputs.device_normal_bf16((N2, K2), 0.02, (seed_base + 1) * 100003 + e, device)
    prep = moe.quantize_experts_sparse if sparse else moe.quantize_experts
    W1 = prep(w1)
    W2 = prep(w2)
    g = inputs.rng(seed_base)
    x = inputs.normal_bf16(g, (T, K1))
    ids = inputs.uniform_topk(g, T, E, TOPK)
    h = inputs.normal_bf16(inputs.rng(seed_base + 1), (T * TOPK, K2))
    wts = inputs.dirichlet_weights(inputs.rng(seed_base + 1), T, TOPK)
    torch.cuda.synchronize()
    setup_s = time.time() - t0
    host = dict(x=x, ids=torch.from_numpy(ids), h=h, wts=torch.from_numpy(wts))
    return W1, W2, w1, w2, host, setup_s


def run_ours(args, rank, world, local_rank):
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    W1, W2, w1, w2, host, setup_s = build_problem(device, sparse=args.sparse)
    ids_np = host["ids"].numpy()
    n_active = int(np.count_nonzero(np.bincount(ids_np.reshape(-1), minlength=E)))
    del w1, w2
    torch.cuda.empty_cache()
    layer = moe.DecodeLayer(W1, W2, T, TOPK, device)
    dev_in = {k: v.to(device) for k, v in host.items()}
    stream = torch.cuda.current_stream()

    def step(timing=None):
        return layer.step(dev_in["x"], dev_in["ids"], dev_in["h"], dev_in["wts"], timing=timing)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    F.nvfp4_device_status(reset=True)
    # soak ~0.5 s so the clocks under load are representative, then time K steps
    soak_end = time.time() + 0.5
    while time.time() < soak_end:
        step()
    torch.cuda.synchronize()

    sampler = ClockSampler(local_rank)
    sampler.start()
    ev = [[[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(2)]
          for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("timed")
    start.record()
    for i in range(args.steps):
        step(timing=ev[i])
    end.record()
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    status = F.nvfp4_device_status(reset=True)
    if status != F.NVFP4_OK:
        raise RuntimeError(f"device status {F.nvfp4_status_string(status)} during the timed run")
    eager_ms_total = start.elapsed_time(end)
    gu_ms = statistics.mean(e[0][0].elapsed_time(e[0][1]) for e in ev)
    dn_ms = statistics.mean(e[1][0].elapsed_time(e[1][1]) for e in ev)

    # The same step recorded in a CUDA graph (one launch per step): the way a
    # server runs a fixed-shape decode step.  This is the headline figure.
    captured = moe.CapturedStep(layer, dev_in["x"], dev_in["ids"], dev_in["h"], dev_in["wts"])
    for _ in range(args.warmup):
        captured.replay()
    torch.cuda.synchronize()
    sampler2 = ClockSampler(local_rank)
    sampler2.start()
    gs, ge = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("timed_graph")
    gs.record()
    for _ in range(args.steps):
        captured.replay()
    ge.record()
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    if world > 1:
        torch.distributed.barrier()
    clocks_graph = sampler2.stop()
    status = F.nvfp4_device_status(reset=True)
    if status != F.NVFP4_OK:
        raise RuntimeError(f"device status {F.nvfp4_status_string(status)} during the graph run")
    ms_total = gs.elapsed_time(ge)

    # end to end through the public API with host buffers: every step copies
    # its inputs from pinned host memory, runs, and reads both outputs back.
    # As a serving loop does, the copies of one step overlap the compute of
    # its neighbours: two device input/output sets (two captured steps over
    # the same weights) alternate, with H2D and D2H on their own streams.
    pinned = {k: v.pin_memory() for k, v in host.items()}
    out_gu = [torch.empty((T * TOPK, N1), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    out_dn = [torch.empty((T, N2), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in pinned.values())
    d2h = out_gu[0].numel() * 2 + out_dn[0].numel() * 2
    layer2 = moe.DecodeLayer(W1, W2, T, TOPK, device)
    dev_in2 = {k: v.to(device) for k, v in host.items()}
    layer2.step(dev_in2["x"], dev_in2["ids"], dev_in2["h"], dev_in2["wts"])
    sets = [(dev_in, captured),
            (dev_in2, moe.CapturedStep(layer2, dev_in2["x"], dev_in2["ids"], dev_in2["h"],
                                       dev_in2["wts"]))]
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    compute = torch.cuda.current_stream(device)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_run = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    for b in range(2):                   # start with every buffer free
        ev_run[b].record(compute)
        ev_out[b].record(compute)

    def e2e_step(i):
        b = i & 1
        din, cap = sets[b]
        with torch.cuda.stream(s_in):    # inputs of step i once step i-2 is done with them
            s_in.wait_event(ev_run[b])
            for k in din:
                din[k].copy_(pinned[k], non_blocking=True)
            ev_in[b].record(s_in)
        compute.wait_event(ev_in[b])
        compute.wait_event(ev_out[b])    # step i-2's outputs have been read back
        gu, dn = cap.replay()
        ev_run[b].record(compute)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_run[b])
            out_gu[b].copy_(gu[: T * TOPK], non_blocking=True)
            out_dn[b].copy_(dn[:T], non_blocking=True)
            ev_out[b].record(s_out)

    for i in range(max(3, args.warmup)):
        e2e_step(i)
    torch.cuda.synchronize()
    s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    s2.record(compute)
    for b in range(2):                   # the timed region starts with idle copy streams
        s_in.wait_event(ev_in[b])
    for i in range(args.steps):
        e2e_step(i)
    for b in range(2):                   # and ends when the last read-back landed
        compute.wait_event(ev_out[b])
    e2.record(compute)
    torch.cuda.synchronize()
    e2e_ms = s2.elapsed_time(e2)
    del layer2, sets, dev_in2

    ms_total, eager_ms_total, e2e_ms, gu_ms, dn_ms = max_over_ranks(
        [ms_total, eager_ms_total, e2e_ms, gu_ms, dn_ms], world, device)
    if rank != 0:
        return None

    ms_step = ms_total / args.steps
    fl = flops_per_step()
    value = aggregate_tflops(fl, args.steps, ms_total, world)
    e2e_value = aggregate_tflops(fl, args.steps, e2e_ms, world)
    peak, peak_kind = measured_peaks()
    R = T * TOPK
    launch_bytes = sparse_gemm_bytes if args.sparse else gemm_bytes
    gu_bytes = launch_bytes(K1, N1, n_active, R, R)
    dn_bytes = launch_bytes(K2, N2, n_active, R, T)
    achieved = gu_bytes / (gu_ms * 1e-3) / 1e9
    # the recorded DRAM counters belong to the dense gate_up launch
    traffic = None if args.sparse else recorded_traffic()
    sbytes = step_bytes(n_active, sparse=args.sparse)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "nvfp4",
        "data": "synthetic", "config": workload_config(),
        "hbm_gbs": round(world * sbytes / (ms_step * 1e-3) / 1e9, 1),
        "frac_of_hbm_roofline": round(sbytes / (ms_step * 1e-3) / 1e9 / peak, 4),
        "roofline": {
            "kernel": "nvfp4_gemm_kernel (gate_up grouped launch)", "bound": "hbm",
            "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "traffic": traffic,
            "algorithmic_bytes_per_launch": int(gu_bytes), "launch_ms": round(gu_ms, 4),
            "peak_source": f"{peak_kind} hbm_gbs",
        },
        "down_launch": {"achieved_gbs": round(dn_bytes / (dn_ms * 1e-3) / 1e9, 1),
                        "launch_ms": round(dn_ms, 4), "algorithmic_bytes": int(dn_bytes)},
        "e2e": {"value": round(e2e_value, 2), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "ms_per_step": round(e2e_ms / args.steps, 4),
                "note": "pinned H2D of every step's inputs and D2H of both outputs, overlapped "
                        "with the neighbouring steps' compute (two buffer sets, copy streams)"},
        "gpu_launches": 8 * args.steps,
        "step_mode": "CUDA graph replay of the whole step (one graph launch per step)",
        "eager": {"ms_per_step": round(eager_ms_total / args.steps, 4),
                  "value": round(aggregate_tflops(fl, args.steps, eager_ms_total, world), 2),
                  "note": "same step launched kernel by kernel; the per-launch CUDA events of "
                          "this pass give roofline.launch_ms and down_launch"},
        "clocks": clocks_graph or clocks,
        "clocks_eager": clocks,
        "setup_s": round(setup_s, 1),
    }
    if args.sparse:
        line["config"]["workload"] += " (2:4-sparse weights)"
        line["config"]["weights"] = ("the same weights pruned to 2:4 over element pairs, NVFP4, "
                                     "streamed as sparse tiles (2/3 of the dense bytes)")
        line["note"] = ("TFLOPS count the dense GEMMs' FLOPs; not the headline (different "
                        "weights); cpu_baseline is reported on the dense line")
    elif world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(W_host_seed=2, budget_s=args.cpu_budget)
    return line


# --------------------------------------------------------------- CPU oracle

def _oracle_batch(seed_base=2):
    """The per-batch part of the decode pass run by the CPU oracle: routing
    and the activation quantisation of x and h.  Returns its results and its
    wall time."""
    import oracle
    g = inputs.rng(seed_base)
    x = inputs.normal_bf16(g, (T, K1)).float().numpy()
    ids = inputs.uniform_topk(g, T, E, TOPK)
    h = inputs.normal_bf16(inputs.rng(seed_base + 1), (T * TOPK, K2)).float().numpy()
    wts = inputs.dirichlet_weights(inputs.rng(seed_base + 1), T, TOPK)
    t0 = time.perf_counter()
    off, tok, slot = oracle.route(ids, E)
    xh = oracle.dequantize(*oracle.quantize(x))
    hh = oracle.dequantize(*oracle.quantize(h))
    return dict(off=off, tok=tok, slot=slot, xh=xh, hh=hh, wts=wts), time.perf_counter() - t0


def _oracle_expert(batch, e, seed_base=2):
    """One expert of the pass in the CPU oracle: its weight quantisation
    (offline on the GPU side, timed apart), then its routes' gate_up and down
    GEMMs and their combine.  Returns (GEMM FLOPs, weight-quantise s, GEMM s)."""
    import oracle
    w1 = _host_weight(seed_base * 100003 + e, (N1, K1))
    w2 = _host_weight((seed_base + 1) * 100003 + e, (N2, K2))
    t0 = time.perf_counter()
    w1h = oracle.dequantize(*oracle.quantize(w1))
    w2h = oracle.dequantize(*oracle.quantize(w2))
    t1 = time.perf_counter()
    off, tok = batch["off"], batch["tok"]
    lo, hi = int(off[e]), int(off[e + 1])
    y1 = batch["xh"][tok[lo:hi]] @ w1h.T
    y2 = batch["hh"][lo:hi] @ w2h.T
    oracle.combine(y2, tok[lo:hi], batch["slot"][lo:hi], batch["wts"], T)
    t2 = time.perf_counter()
    del y1
    return 2.0 * (hi - lo) * (N1 * K1 + N2 * K2), t1 - t0, t2 - t1


def _host_weight(seed, shape):
    """The expert weight the device generator draws for `seed`, on the host.

    torch's CPU and CUDA generators differ, so the oracle sample draws its
    own N(0, 0.02) weights with the host generator: the work is the same
    size and kind, which is what the baseline times."""
    return inputs.normal_bf16(inputs.rng(seed), shape, 0.02).float().numpy()


def cpu_baseline(W_host_seed=2, budget_s=20.0):
    """The oracle on the host cores over a bounded sample of the decode pass:
    the whole batch's routing and activation quantisation, then whole experts
    until about budget_s seconds have gone.  The value is the sampled GEMM
    FLOPs over the GEMM time plus the sampled experts' share of the batch
    quantisation; the weight quantisation (offline on the GPU side) is timed
    but left out of it."""
    batch, t_batch = _oracle_batch(W_host_seed)
    experts = []
    flops, t_wq, t_gemm = 0.0, 0.0, 0.0
    e = 0
    while t_batch + t_wq + t_gemm < budget_s and e < E:
        f, wq, gm = _oracle_expert(batch, e, W_host_seed)
        flops += f
        t_wq += wq
        t_gemm += gm
        experts.append(e)
        e += 1
    share = t_batch * len(experts) / E
    cores = _blas_threads()
    return {"value": round(flops / (t_gemm + share) / 1e12, 6), "unit": UNIT, "cores": cores,
            "kind": "oracle",
            "activation_quantize_s": round(t_batch, 3), "gemm_s": round(t_gemm, 3),
            "weight_quantize_s": round(t_wq, 3),
            "sample": f"experts {experts[0]}..{experts[-1]} of the gate_up+down pass "
                      f"({len(experts)} of {E}): their GEMMs and combine ({t_gemm:.1f} s) plus "
                      f"{len(experts)}/{E} of the batch's routing and activation quantisation "
                      f"({t_batch:.1f} s for the batch); their weight quantisation "
                      f"({t_wq:.1f} s) is offline on the GPU side and left out"}


def _blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def run_reference(args, rank, world):
    """The oracle as the reference arm: each step one expert's GEMMs and
    combine plus 1/E of the batch's routing and activation quantisation."""
    if rank != 0:
        return None
    batch, t_batch = _oracle_batch()
    for i in range(args.warmup):
        _oracle_expert(batch, i % E)
    times, flops, t_wq = [], 0.0, 0.0
    for i in range(args.steps):
        f, wq, gm = _oracle_expert(batch, (args.warmup + i) % E)
        times.append(gm + t_batch / E)
        flops += f
        t_wq += wq
    total = sum(times)
    value = flops / total / 1e12
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * total / args.steps, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(),
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": _blas_threads(),
                         "kind": "oracle", "activation_quantize_s": round(t_batch, 3),
                         "weight_quantize_s": round(t_wq, 3),
                         "sample": "each step: one expert's gate_up + down GEMMs and combine, "
                                   "plus 1/E of the batch's routing and activation "
                                   "quantisation; the expert's weight quantisation is timed "
                                   "apart and left out (offline on the GPU side)"},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# ------------------------------------------------------ per-configuration table

def _timed(fn, iters, flush):
    """Mean device time of fn over `iters` runs, L2 flushed before each run."""
    fn()
    torch.cuda.synchronize()
    total = 0.0
    for _ in range(iters):
        flush.zero_()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        fn()
        e.record()
        torch.cuda.synchronize()
        total += s.elapsed_time(e)
    return total / iters


def _peaks():
    """(HBM GB/s, dense FP4 TFLOPS, source): the measured HBM copy rate, and
    the FP4 peak as 6 x the measured BF16 burst (the nominal dense ratio
    13.5 / 2.25 PFLOPS)."""
    hbm, kind = measured_peaks()
    bf16 = None
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            bf16 = json.load(f).get("bf16_tflops")
    return hbm, (bf16 or 1900.0) * 6.0, f"{kind} hbm_gbs; fp4 = 6 x {kind} bf16_tflops"


def _entry(ms, flops, byts, hbm, fp4, **extra):
    """One configuration's figures: time, TFLOPS, GB/s and the achieved
    fraction of the slower of its two rooflines (max(t_hbm, t_fp4) / t)."""
    t_mem = byts / (hbm * 1e9)
    t_cmp = flops / (fp4 * 1e12)
    d = {"us": round(ms * 1e3, 2), "tflops": round(flops / ms / 1e9, 1),
         "gbs": round(byts / ms / 1e6, 1), "bound": "hbm" if t_mem >= t_cmp else "fp4",
         "frac_of_roofline": round(max(t_mem, t_cmp) / (ms * 1e-3), 4),
         "algorithmic_flops": int(flops), "algorithmic_bytes": int(byts)}
    d.update(extra)
    return d


def measure_configs(args, dev, groups=None):
    """Every workload configuration, kernel by kernel: name -> figures.  CUDA
    events, L2 flushed (256 MB write) before every timed call."""
    flush = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device=dev)
    hbm, fp4, peak_src = _peaks()
    iters = max(3, min(args.steps, 20))
    out = {}

    def want(group):
        return groups is None or group in groups

    # tiny single GEMM (16 x 256 x 512, seed 0): launch-latency bound
    if want("tiny_gemm"):
        g = inputs.rng(0)
        a = inputs.normal_bf16(g, (16, 512)).to(dev)
        b = inputs.normal_bf16(g, (256, 512), 0.02).to(dev)
        pa, sa, ga = F.quantize(a, atoms=True)
        pb, sb, gb = F.quantize(b, atoms=True)
        C = torch.empty((16, 256), dtype=torch.bfloat16, device=dev)
        t_g = _timed(lambda: F.nvfp4_gemm(pa, sa, ga, pb, sb, gb, C, 512), iters, flush)
        t_q = _timed(lambda: F.nvfp4_quantize(a, pa, sa, ga, F.NVFP4_SF_ATOMS), iters, flush)
        byt = (16 + 256) * 512 * (0.5 + 1 / 16) + 16 * 256 * 2
        out["tiny_gemm_16x256x512"] = _entry(
            t_g, 2.0 * 16 * 256 * 512, byt, hbm, fp4, quantize_A_us=round(t_q * 1e3, 2),
            note="launch-latency bound; the roofline fraction is not meaningful here")

    # dense 8192^3: A quantised every call, B prepared offline
    if want("dense_8192"):
        M = Nn = Kk = 8192
        a = inputs.device_normal_bf16((M, Kk), 1.0, 1, dev)
        b = inputs.device_normal_bf16((Nn, Kk), 0.02, 1001, dev)
        pb, sb, gb = F.quantize(b, atoms=True)
        pa, sa, ga = F.quantize(a, atoms=True)
        C = torch.empty((M, Nn), dtype=torch.bfloat16, device=dev)
        t_gemm = _timed(lambda: F.nvfp4_gemm(pa, sa, ga, pb, sb, gb, C, Kk), iters, flush)
        t_q = _timed(lambda: F.nvfp4_quantize(a, pa, sa, ga, F.NVFP4_SF_ATOMS), iters, flush)
        fl = 2.0 * M * Nn * Kk
        gemm_b = (M + Nn) * Kk * (0.5 + 1 / 16) + M * Nn * 2
        out["dense_gemm_8192^3"] = _entry(t_gemm, fl, gemm_b, hbm, fp4)
        out["dense_gemm_8192^3_with_quantize_A"] = _entry(
            t_gemm + t_q, fl, gemm_b + M * Kk * 2, hbm, fp4,
            note="the GEMM plus the BF16 -> NVFP4 quantisation of A (two launches)")
        # the activation quantiser alone: 2 B read + 0.5625 B written per element
        out["quantize_8192x8192"] = _entry(t_q, 0.0, M * Kk * 2.5625, hbm, fp4,
                                           note="tensor amax + block quantiser, atom scales")
        del a, b, pa, sa, pb, sb, C

    # decode gate_up, down sweep and skewed prefill (and the 2:4-sparse decode shapes)
    for name in ("decode_gate_up", "decode_down_256", "decode_down_512", "decode_down_1024",
                 "prefill_skewed"):
        if not (want("decode") or want(name) or (name == "prefill_skewed" and want("prefill"))):
            continue
        cfg = inputs.CONFIGS[name]
        g = inputs.rng(cfg.seed)
        w = torch.empty((cfg.E, cfg.N, cfg.K), dtype=torch.bfloat16, device=dev)
        for e in range(cfg.E):
            w[e] = inputs.device_normal_bf16((cfg.N, cfg.K), 0.02, cfg.seed * 100003 + e, dev)
        W = moe.quantize_experts(w)
        sparse = want("sparse") and name != "prefill_skewed"
        W_sp = moe.quantize_experts_sparse(w) if sparse else None
        del w
        torch.cuda.empty_cache()          # the BF16 weights' memory leaves the process
        if cfg.kind == "down":
            ids = inputs.uniform_topk(g, cfg.T, cfg.E, cfg.topk)
            wts = torch.from_numpy(inputs.dirichlet_weights(g, cfg.T, cfg.topk)).to(dev)
            xin = inputs.normal_bf16(g, (cfg.T * cfg.topk, cfg.K)).to(dev)
            plan = moe.GroupedPlan(W, cfg.T, cfg.topk, "combine", dev)
        else:
            xf = g.standard_normal((cfg.T, cfg.K), dtype=np.float32)
            if cfg.outliers:
                xf = inputs.add_outliers(g, xf)
            xin = inputs.to_bf16(xf).to(dev)
            ids = (inputs.zipf_topk(g, cfg.T, cfg.E, cfg.topk) if cfg.routing == "zipf"
                   else inputs.uniform_topk(g, cfg.T, cfg.E, cfg.topk))
            wts = None
            plan = moe.GroupedPlan(W, cfg.T, cfg.topk, "gather", dev)
        ids_d = torch.from_numpy(ids).to(dev)
        plan.route(ids_d)
        plan.quantize(xin)
        t_gemm = _timed(lambda: plan.gemm(wts), iters, flush)
        t_all = _timed(lambda: plan.run(xin, ids_d, wts), iters, flush)
        counts = np.bincount(ids.reshape(-1), minlength=cfg.E)
        n_act = int(np.count_nonzero(counts))
        R = cfg.T * cfg.topk
        fl = 2.0 * R * cfg.N * cfg.K
        out_rows = cfg.T if cfg.kind == "down" else R
        byt = gemm_bytes(cfg.K, cfg.N, n_act, R, out_rows)
        out[name] = _entry(t_gemm, fl, byt, hbm, fp4,
                           tokens_per_expert=[int(counts.min()), int(counts.max())],
                           active_experts=n_act,
                           pass_us_route_quantize_gemm=round(t_all * 1e3, 2))
        if W_sp is not None:
            sp_plan = moe.GroupedPlan(W_sp, cfg.T, cfg.topk, plan.mode, dev, routing_from=plan)
            sp_plan.a_tiles.copy_(plan.a_tiles)
            sp_plan.a_g.copy_(plan.a_g)
            t_sp = _timed(lambda: sp_plan.gemm(wts), iters, flush)
            byt_sp = sparse_gemm_bytes(cfg.K, cfg.N, n_act, R, out_rows)
            out[name + "_sparse24"] = _entry(
                t_sp, fl, byt_sp, hbm, fp4, speedup_vs_dense=round(t_gemm / t_sp, 3),
                note="weights pruned to 2:4 over element pairs, streamed as sparse tiles (2/3 "
                     "of the dense bytes); TFLOPS count the dense GEMM's FLOPs")
            del sp_plan
        del W, W_sp, plan
        torch.cuda.empty_cache()

    # decode expert MLP: the fused path (gate_up + SiLU * up + NVFP4 h in one
    # launch) against the same pass with h quantised by its own kernels, at
    # 16 and 32 routes per expert (32- and 64-route token tiles)
    for tokens in (T, 2 * T):
        if not want("fused_mlp"):
            break
        W1, W2, w1, w2, host, _ = build_problem(dev, tokens=tokens)
        del w1, w2
        torch.cuda.empty_cache()
        d = {k: v.to(dev) for k, v in host.items()}
        layer = moe.DecodeLayer(W1, W2, tokens, TOPK, dev)
        gu_out, _ = layer.step(d["x"], d["ids"], d["h"], d["wts"])
        # calibration of h's global (set-up, outside the timed region): amax of
        # SiLU(gate) * up over this batch
        gate, up = gu_out.float().split(N1 // 2, dim=1)
        g_h = (torch.nn.functional.silu(gate) * up).abs().amax().reshape(1) / 2688.0
        mlp = moe.FusedMLP(W1, W2, tokens, TOPK, g_h.to(torch.float32), dev)
        mlp1 = moe.FusedMLP(W1, W2, tokens, TOPK, g_h.to(torch.float32), dev, single_launch=True)
        mlp2 = moe.FusedMLP(W1, W2, tokens, TOPK, None, dev)          # two-phase global of h
        t_fused = _timed(lambda: mlp.step(d["x"], d["ids"], d["wts"]), iters, flush)
        t_one = _timed(lambda: mlp1.step(d["x"], d["ids"], d["wts"]), iters, flush)
        t_two = _timed(lambda: mlp2.step(d["x"], d["ids"], d["wts"]), iters, flush)
        t_split = _timed(lambda: layer.step(d["x"], d["ids"], d["h"], d["wts"]), iters, flush)
        fl = 2.0 * tokens * TOPK * (N1 * K1 + N2 * K2)
        n_act = int(np.count_nonzero(np.bincount(host["ids"].numpy().reshape(-1), minlength=E)))
        byt = n_act * (N1 * K1 + N2 * K2) * 0.5625 + 2.0 * (tokens * K1 + tokens * N2)
        out[f"decode_mlp_fused_T{tokens}"] = _entry(
            t_fused, fl, byt, hbm, fp4, unfused_pass_us=round(t_split * 1e3, 2),
            one_launch_pass_us=round(t_one * 1e3, 2), two_phase_pass_us=round(t_two * 1e3, 2),
            note="route + quantise x + fused gate_up/SiLU/quantise-h + down with combine; "
                 "one_launch = gate_up and down in one persistent launch; two_phase = h "
                 "written in BF16 and quantised with the global of its own amax; unfused = "
                 "the same pass with a BF16 gate_up output and h quantised by its own kernels")
        out[f"decode_mlp_one_launch_T{tokens}"] = _entry(
            t_one, fl, byt, hbm, fp4,
            note="the fused expert MLP with gate_up and down in one persistent launch")
        del layer, mlp, mlp1, mlp2, W1, W2, d, gu_out, gate, up
        torch.cuda.empty_cache()
    # decode attention over an NVFP4 KV cache (every cache byte read once):
    # 128-wide heads in groups of 4, 8 (tensor-core kernel) and 1 (CUDA-core
    # kernel), 256-wide heads in groups of 4 and 512-wide heads in groups of 4
    # (the two-pass tensor-core kernels)
    for (B_, Hq_, Hkv_, L_, D_) in ((16, 32, 8, 16384, 128), (16, 64, 8, 16384, 128),
                                    (16, 8, 8, 16384, 128), (16, 32, 8, 8192, 256),
                                    (8, 8, 2, 32768, 512)):
        if not (want("decode_attention") or want(f"decode_attention_d{D_}")):
            continue
        kc = inputs.device_normal_bf16((B_, Hkv_, L_, D_), 1.0, 71, dev)
        kq = attention.quantize_kv(kc)
        del kc
        vc = inputs.device_normal_bf16((B_, Hkv_, L_, D_), 1.0, 72, dev)
        vq = attention.quantize_kv(vc)
        del vc
        q = inputs.device_normal_bf16((B_, Hq_, D_), 1.0, 73, dev)
        seq = torch.full((B_,), L_, dtype=torch.int32, device=dev)
        plan = attention.DecodeAttention(B_, Hq_, Hkv_, L_, D_, dev)
        t_att = _timed(lambda: plan.run(q, kq, vq, seq, 1.0 / D_ ** 0.5), iters, flush)
        byt = 2.0 * B_ * Hkv_ * L_ * D_ * (0.5 + 1.0 / 16) + 2.0 * 2 * B_ * Hq_ * D_
        fl = 4.0 * B_ * Hq_ * L_ * D_
        out[f"decode_attention_B{B_}_Hq{Hq_}_Hkv{Hkv_}_L{L_}_D{D_}"] = _entry(
            t_att, fl, byt, hbm, fp4,
            note="one query token per sequence; K and V in NVFP4 (codes + E4M3 scales along "
                 "D + one global each); split-KV partials merged by a second kernel (both "
                 "timed); " + _attention_kernel_name(D_, Hq_ // Hkv_))
        del kq, vq, plan
        torch.cuda.empty_cache()
    for v in out.values():
        v.setdefault("peak_source", peak_src)
    return out


def _attention_kernel_name(D_, G_):
    """Which decode-attention kernel the library picks for a head width and
    group size (the dispatch in csrc/attention_tc.cu, aligned scale arrays)."""
    if D_ >= 256 and G_ in (2, 4, 8) and not (D_ == 512 and G_ == 8):
        return "tcgen05 two-pass kernels (scores, then values)"
    if (D_ == 128 and G_ in (2, 4, 8)) or (D_ == 64 and G_ in (4, 8)):
        return "tcgen05 pipelined kernel"
    return "CUDA-core kernel"


def run_configs(args):
    """One JSON line per workload configuration (not the headline)."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    groups = None if not args.only else set(args.only.split(","))
    for name, v in measure_configs(args, dev, groups).items():
        print(json.dumps({"workload": name, **v}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode_layer", choices=["decode_layer", "configs"],
                    help="configs: one line per workload configuration (not the headline)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", default=None,
                    help="configs: run only these comma-separated groups (tiny_gemm, "
                         "dense_8192, decode (with prefill), prefill, sparse, fused_mlp, "
                         "decode_attention, or one head width of it: decode_attention_d128, "
                         "_d256, _d512; one decode shape: decode_gate_up, decode_down_256, "
                         "_512, _1024)")
    ap.add_argument("--no-configs", action="store_true",
                    help="leave the per-configuration table out of the headline line")
    ap.add_argument("--sparse", action="store_true",
                    help="the decode step with the weights pruned to 2:4 and streamed as "
                         "sparse tiles (not the headline)")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--experts", type=int, default=E,
                    help="experts (tokens scale as 2 per expert); smaller values give the "
                         "small profiling case of the same kernels")
    args = ap.parse_args()
    _set_experts(args.experts)
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and args.impl == "ours":
        torch.distributed.init_process_group(
            "nccl", device_id=torch.device("cuda", local_rank))
    if args.workload == "configs":
        run_configs(args)
        return
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        line = run_ours(args, rank, world, local_rank)
        if line is not None and world == 1 and not args.no_configs and not args.sparse:
            # every workload configuration, kernel by kernel, beside the headline
            dev = torch.device("cuda", local_rank)
            torch.cuda.empty_cache()
            sampler = ClockSampler(local_rank)
            sampler.start()
            t0 = time.time()
            cfgs = measure_configs(args, dev)
            cfgs["wall_s"] = round(time.time() - t0, 1)
            cfgs["clocks"] = sampler.stop()
            cfgs["timing"] = ("CUDA events around each call, L2 flushed (256 MB write) before "
                              "every timed call; mean of min(steps, 20) calls")
            line["configs"] = cfgs
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1 and args.impl == "ours":
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()

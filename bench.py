#!/usr/bin/env python3
"""Benchmark of the BF16 attention hot path (forward + backward) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload llama7b] [--deviation] [--int8-forward]

One step = one pass of the whole hot path over one batch of synthetic input:
attn_fwd (O, LSE) then the backward (preprocess, main kernel, dQ conversion).
The default workload is B1 H32 N4096 d128, causal, BF16 (the Llama-2-7B-shaped
case the target is quoted on).  FLOPs are counted as 4*B*H*N^2*d for the
forward (halved when causal) and 2.5x that for the backward.

Rank 0 prints ONE JSON line.  `value` is whole-job TFLOP/s with inputs
resident in HBM; `e2e` is the same metric measured through the Python API
with pinned host buffers (host->device copies of Q, K, V, dO and
device->host copies of O, LSE, dQ, dK, dV inside the timed region);
(HostAttention pipelines head groups over upload, compute and download streams, replayed as a CUDA graph); `roofline` describes the dominant kernel (the backward main kernel) timed
with CUDA events on its stream; `cpu_baseline` is the FP64 oracle timed on
the host cores on a bounded sample.  `--impl reference` times that oracle
as the reference arm instead.  Under torchrun every rank runs its own full
workload (weak scaling, no data-path collective).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from precision_numerics_gb300 import inputs  # noqa: E402

METRIC = "BF16 attention fwd/bwd TFLOP/s on 1 GB300, % of tensor peak; max err vs FP64"
UNIT = "TFLOP/s"
DOMINANT = "bwd_main_kernel"
DOMINANT_SRC = os.path.join(ROOT, "precision_numerics_gb300", "csrc", "bwd_bf16.cu")
# ncu summary of the dominant kernel per workload (DRAM traffic per launch).
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "bwd_main_kernel_{workload}.md")


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return {"bf16": float(p["bf16_tflops"]), "bf16_sustained": float(p["bf16_tflops_sustained"]),
                "hbm": float(p["hbm_gbs"]), "source": "measured"}
    except Exception:  # noqa: BLE001 - fall back to the recorded fallback figures
        return {"bf16": 1900.0, "bf16_sustained": 1700.0, "hbm": 6800.0, "source": "fallback"}


def _max_over_ranks(values, device):
    """Element-wise maximum of `values` over all ranks (identity without a group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def _job_tflops(world, flops_per_step, steps, elapsed_ms):
    """Whole-job throughput: every rank ran `steps` steps of its own workload
    (weak scaling), timed by the slowest rank."""
    return world * flops_per_step * steps / (elapsed_ms * 1e-3) / 1e12


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index: int):
        self.samples = []
        self.proc = None
        self.gpu = gpu_index
        self.marks = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(self.gpu)], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                self.samples.append((time.time(), float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue

    def mark(self):
        self.marks.append(time.time())

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        t0, t1 = (self.marks[0], self.marks[-1]) if len(self.marks) >= 2 else (0, float("inf"))
        win = [s for s in self.samples if t0 <= s[0] <= t1]
        if len(win) < 3:
            win = self.samples
        reasons = sorted({n for s in win for n, flag in zip(self.NAMES, s[3]) if flag == "Active"})
        return {"sm_mhz": statistics.median(s[1] for s in win),
                "sm_max_mhz": max(s[2] for s in win), "reasons": reasons, "samples": len(win)}


# ---------------------------------------------------------------------------
# roofline traffic from the committed ncu summary (null if the kernel changed)
# ---------------------------------------------------------------------------
def _source_sha():
    with open(DOMINANT_SRC, "rb") as fh:
        return hashlib.sha256(fh.read()).hexdigest()


def _traffic_per_launch(workload: str):
    try:
        text = open(TRAFFIC_FILE.format(workload=workload)).read()
    except OSError:
        return None
    m_b = re.search(r"^traffic_bytes_per_launch:\s*([0-9.eE+]+)\s*$", text, re.M)
    m_s = re.search(r"^source_sha256:\s*([0-9a-f]{64})\s*$", text, re.M)
    m_w = re.search(r"^workload:\s*(\w+)\s*$", text, re.M)
    if not (m_b and m_s and m_w) or m_s.group(1) != _source_sha() or m_w.group(1) != workload:
        return None
    return float(m_b.group(1))


# ---------------------------------------------------------------------------
# CPU oracle (reference arm and cpu_baseline)
# ---------------------------------------------------------------------------
def _oracle_head_step(w, x, head, rows=None):
    """Oracle forward + backward for the first `rows` query rows of one head.

    With a causal mask the first R rows see only the first R keys, so the
    sample is exactly the square problem of size R; without the mask they see
    all N keys.  rows = None (or N) is the whole head.
    """
    import oracle
    R = w.N if rows is None else rows
    f = {k: inputs.bf16_bits_to_f32(v.reshape(w.B * w.H, w.N, w.d)[head]) for k, v in x.items()}
    nk = R if w.causal else w.N
    oracle.forward(f["q"][:R], f["k"][:nk], f["v"][:nk], w.scale, w.causal)
    oracle.backward(f["q"][:R], f["k"][:nk], f["v"][:nk], f["do"][:R], w.scale, w.causal)


def _rows_flops(w, rows):
    """Forward + backward FLOPs of the first `rows` query rows of one head."""
    pairs = rows * rows / 2 if w.causal else rows * w.N  # (query, key) pairs computed
    return 3.5 * 4 * pairs * w.d


def _head_flops(w):
    return (w.fwd_flops() + w.bwd_flops()) / (w.B * w.H)


def _cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(w, x, budget_s=12.0):
    """Time the oracle on whole heads (forward + backward) until ~budget_s."""
    t0 = time.perf_counter()
    heads = 0
    while True:
        _oracle_head_step(w, x, heads % (w.B * w.H))
        heads += 1
        if time.perf_counter() - t0 >= budget_s or heads >= w.B * w.H:
            break
    dt = time.perf_counter() - t0
    return {"value": heads * _head_flops(w) / dt / 1e12, "unit": UNIT, "cores": _cpu_cores(),
            "kind": "oracle",
            "sample": f"{heads} of {w.B * w.H} (b,h) heads of {w.name}, FP64 forward+backward, "
                      f"{dt:.1f} s; throughput scales linearly with heads"}


def run_reference(args, w, budget_s=150.0):
    world, rank, _ = _dist()
    if rank != 0:
        return 0
    x = inputs.make_inputs(w, seed=0, heads=None)
    # One step = the oracle on one head; when K such steps would not end within
    # ~budget_s, each step takes the first R query rows of a head instead, R
    # sized from a timed whole head so that K steps fit the budget.
    t0 = time.perf_counter()
    _oracle_head_step(w, x, 0)
    t_head = time.perf_counter() - t0
    rows = w.N
    if args.steps * t_head > budget_s:
        frac = budget_s / (args.steps * t_head)
        rows = max(64, int(w.N * (frac ** 0.5 if w.causal else frac)))
    for s in range(args.warmup):
        _oracle_head_step(w, x, s % (w.B * w.H), rows)
    t0 = time.perf_counter()
    for s in range(args.steps):
        _oracle_head_step(w, x, s % (w.B * w.H), rows)
    dt = time.perf_counter() - t0
    value = args.steps * _rows_flops(w, rows) / dt / 1e12
    sample = (f"each step = the first {rows} of {w.N} query rows of one of the {w.B * w.H} (b,h) "
              f"heads of {w.name}, FP64 forward+backward")
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference", "config": _config(w),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": _cpu_cores(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def _kernel_delta(ws, w, head):
    """delta of one (b, h) head as the preprocess kernel wrote it into the
    backward workspace (layout in include/attn.h: -LSE*log2(e) [B*H][N_pad],
    then delta [B*H][N_pad] from the next 256-byte boundary)."""
    n_pad = (w.N + 127) // 128 * 128
    rows = w.B * w.H * n_pad
    off = (rows * 4 + 255) // 256 * 256 + head * n_pad * 4
    return ws[off:off + w.N * 4].cpu().numpy().view(np.float32).astype(np.float64)


def _dev3(d):
    return {k: d[k] for k in ("max_abs", "mean_abs", "signed_mean")}


def _deviation_block(w, f, o, dv, ws, o_ref, dv_ref, head=0):
    """Tiled GPU vs FP64 next to naive BF16 attention vs FP64 on one head: the
    question of "Is Flash Attention Stable?" (abstract) -- how much more
    numeric deviation tiled attention has than Baseline Attention at BF16 --
    answered on this workload.  delta_lp is the backward kernel's own delta
    (rowsum(dO o O) from the stored BF16 O, "Why Low-Precision Transformer
    Training Fails", Figure 3) against rowsum(dO o O) of the exact O.
    f: the head's inputs (FP32 arrays); o_ref, dv_ref: the oracle's O and dV."""
    import oracle
    from precision_numerics_gb300.deviation import deviation
    B, H, N, d = w.B, w.H, w.N, w.d
    o_nv, _ = oracle.naive_bf16_forward(f["q"], f["k"], f["v"], w.scale, w.causal)
    dv_nv = oracle.naive_bf16_backward(f["q"], f["k"], f["v"], f["do"], w.scale, w.causal)[2]
    tiled = {"o": deviation(o.reshape(B * H, N, d)[head].float().cpu().numpy(), o_ref),
             "dv": deviation(dv.reshape(B * H, N, d)[head].float().cpu().numpy(), dv_ref)}
    naive = {"o": deviation(o_nv, o_ref), "dv": deviation(dv_nv, dv_ref)}
    dl = deviation(_kernel_delta(ws, w, head), oracle.delta(f["do"], o_ref))
    return {"sample": f"head (b,h)=(0,{head}) of the timed workload against the FP64 definition",
            "tiled_gpu": {k: _dev3(v) for k, v in tiled.items()},
            "naive_bf16": {k: _dev3(v) for k, v in naive.items()},
            "naive_over_tiled_o_max_abs": naive["o"]["max_abs"] / tiled["o"]["max_abs"],
            "naive_over_tiled_o_mean_abs": naive["o"]["mean_abs"] / tiled["o"]["mean_abs"],
            "delta_lp_minus_delta": _dev3(dl)}


def _config(w):
    return {"workload": f"{w.name}: B{w.B} H{w.H} N{w.N} d{w.d} "
                        f"{'causal' if w.causal else 'non-causal'} BF16 forward+backward",
            "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal, "scale": w.scale,
            "l2": "inputs larger than L2 (Q,K,V,O,dO,dQ,dK,dV and the FP32 dQ accumulator "
                  f"are {(8 * 2 + 4) * w.B * w.H * w.N * w.d / 2**20:.0f} MiB per step vs 129 MB L2)"}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def run_ours(args, w):
    import torch
    import torch.distributed as dist

    from precision_numerics_gb300 import attn, build
    from precision_numerics_gb300.deviation import deviation

    world, rank, local = _dist()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build.build()
    attn.load_library()

    x = inputs.make_inputs(w, seed=rank)
    host = {k: torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).pin_memory()
            for k, v in x.items()}
    t = {k: v.to(dev) for k, v in host.items()}
    B, H, N, d = w.B, w.H, w.N, w.d
    o = torch.empty_like(t["q"])
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq, dk, dv = (torch.empty_like(t["q"]) for _ in range(3))
    ws = torch.empty(attn.attn_bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    kernels_per_step = 4  # forward, backward preprocess, backward main, dQ conversion

    def step(ev=None):
        attn.attn_fwd(t["q"], t["k"], t["v"], scale=w.scale, causal=w.causal, o=o, lse=lse)
        attn.attn_bwd_preprocess(o, lse, t["do"], ws)
        if ev is not None:
            ev[0].record(stream)
        attn.attn_bwd_main(t["q"], t["k"], t["v"], t["do"], dk, dv, ws, scale=w.scale,
                           causal=w.causal)
        if ev is not None:
            ev[1].record(stream)
        attn.attn_bwd_dq_convert(dq, ws, scale=w.scale)

    sampler = ClockSampler(local)
    if rank == 0:
        sampler.start()
    for _ in range(args.warmup):
        step()
    attn.attn_check_status()
    events = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.mark()
    start.record(stream)
    for s in range(args.steps):
        step(events[s])
    end.record(stream)
    torch.cuda.synchronize()
    sampler.mark()
    if world > 1:
        dist.barrier()
    elapsed_ms = start.elapsed_time(end)
    main_ms = statistics.mean(a.elapsed_time(b) for a, b in events)
    attn.attn_check_status()

    # End-to-end through the public API with pinned host buffers: the head
    # groups are pipelined (H2D copy, kernels, D2H copy on their own streams),
    # captured once as a CUDA graph and replayed every step.
    from precision_numerics_gb300.host import HostAttention, ramped_group_sizes
    groups = (None if args.e2e_even_groups
              else ramped_group_sizes(B * H, args.e2e_chunks))
    pipe = HostAttention(B, H, N, d, scale=w.scale, causal=w.causal, chunks=args.e2e_chunks,
                         group_sizes=groups, device=dev)
    for _ in range(max(3, min(args.warmup, 5))):
        pipe.run(host["q"], host["k"], host["v"], host["do"])
    e2e_steps = max(1, min(args.steps, 20))
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    e0.record(stream)
    for _ in range(e2e_steps):
        pipe.run(host["q"], host["k"], host["v"], host["do"])
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    attn.attn_check_status()
    h2d_bytes, d2h_bytes = pipe.bytes_per_run()
    sampler.stop()

    elapsed_ms, main_ms, e2e_ms = _max_over_ranks([elapsed_ms, main_ms, e2e_ms], dev)

    if rank == 0:
        peaks = _peaks()
        step_flops = w.fwd_flops() + w.bwd_flops()
        ms_per_step = elapsed_ms / args.steps
        value = _job_tflops(world, step_flops, args.steps, elapsed_ms)
        achieved = w.bwd_flops() / (main_ms * 1e-3) / 1e12
        h2d, d2h = h2d_bytes, d2h_bytes

        # Max error vs FP64 on a sampled head (head 0) of the timed outputs.
        import oracle
        f = {k: inputs.bf16_bits_to_f32(v.reshape(B * H, N, d)[0]) for k, v in x.items()}
        o_ref, lse_ref = oracle.forward(f["q"], f["k"], f["v"], w.scale, w.causal)
        g_ref = oracle.backward(f["q"], f["k"], f["v"], f["do"], w.scale, w.causal)
        err = {"o": deviation(o.reshape(B * H, N, d)[0].float().cpu().numpy(), o_ref),
               "lse": deviation(lse.reshape(B * H, N)[0].cpu().numpy(), lse_ref)}
        for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), g_ref):
            err[name] = deviation(g.reshape(B * H, N, d)[0].float().cpu().numpy(), r)

        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) inputs, generated on the host)",
            "config": _config(w),
            "pct_of_peak": 100.0 * (value / world) / peaks["bf16"],
            "fwd_tflops": None, "bwd_main_tflops": achieved,
            "max_err_vs_fp64": {"o_max_abs": err["o"]["max_abs"], "o_mean_abs": err["o"]["mean_abs"],
                                "o_signed_mean": err["o"]["signed_mean"],
                                "lse_max_abs": err["lse"]["max_abs"],
                                "dq_rel_l2": err["dq"]["rel_l2"], "dk_rel_l2": err["dk"]["rel_l2"],
                                "dv_rel_l2": err["dv"]["rel_l2"], "sample": "head (b,h)=(0,0)"},
            "roofline": {"kernel": DOMINANT, "bound": "tensor", "achieved": achieved,
                         "peak": peaks["bf16"], "unit": "TFLOP/s",
                         "frac": achieved / peaks["bf16"],
                         "frac_of_sustained": achieved / peaks["bf16_sustained"],
                         "peak_source": f"{peaks['source']} bf16 burst",
                         "traffic": _traffic_per_launch(w.name),
                         "algorithmic": "2.5 * 4*B*H*N^2*d/2 FLOP per launch (5 matmuls)"},
            "e2e": {"value": _job_tflops(world, step_flops, 1, e2e_ms), "unit": UNIT,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "head_groups": [b - a for a, b in pipe.groups]},
            "gpu_launches": kernels_per_step * args.steps,
            "clocks": sampler.summary(),
        }
        line["fwd_tflops"] = _fwd_only_tflops(attn, t, o, lse, w, stream, torch)
        graph_ms = _graph_step_ms(step, torch, reps=min(args.steps, 200))
        line["step_graph"] = {"ms_per_step": graph_ms, "eager_ms_per_step": ms_per_step,
                              "eager_over_graph": ms_per_step / graph_ms}
        line["deviation"] = _deviation_block(w, f, o, dv, ws, o_ref, g_ref[2])
        line["host_us_per_call"] = _host_cost(attn, w, dev, torch)
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(w, x)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def _graph_step_ms(step, torch, reps):
    """The same device-resident step captured once as a CUDA graph and
    replayed (milliseconds per step, CUDA events), after the timed region:
    next to the eagerly issued step it shows what the per-call host work of
    the four launches costs the step, if anything."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def _host_cost(attn, w, dev, torch, calls=200):
    """Host time per eager call of attn_fwd + attn_bwd, in microseconds.

    "c_abi": the two C entry points called through ctypes with prepared
    arguments (the library's own host cost: argument and pointer checks,
    tensor-map encoding, launches); "python": the same through the Python
    binding (plus its checks and marshalling).  Measured on the small
    forward-only workload's shape with a backward (B1 H2 N128 d64) and on this
    workload's shape, after the timed region; the GPU work of a call is
    shorter than its host time on the small shape, so calls do not queue."""
    import ctypes
    lib = attn.load_library()
    out = {}
    for tag, (B, H, N, d) in (("B1H2N128d64", (1, 2, 128, 64)),
                              (f"B{w.B}H{w.H}N{w.N}d{w.d}", (w.B, w.H, w.N, w.d))):
        z = {k: torch.zeros((B, H, N, d), dtype=torch.bfloat16, device=dev)
             for k in ("q", "k", "v", "o", "do", "dq", "dk", "dv")}
        lse = torch.zeros((B, H, N), dtype=torch.float32, device=dev)
        ws = torch.empty(attn.attn_bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device=dev)
        st = torch.cuda.current_stream().cuda_stream
        sc = ctypes.c_float(d ** -0.5)
        fa = (z["q"].data_ptr(), z["k"].data_ptr(), z["v"].data_ptr(), z["o"].data_ptr(),
              lse.data_ptr(), B, H, N, d, sc, 1, 0, st)
        ba = (z["q"].data_ptr(), z["k"].data_ptr(), z["v"].data_ptr(), z["o"].data_ptr(),
              lse.data_ptr(), z["do"].data_ptr(), z["dq"].data_ptr(), z["dk"].data_ptr(),
              z["dv"].data_ptr(), B, H, N, d, sc, 1, 0, ws.data_ptr(), ws.numel(), st)
        n = calls if N <= 1024 else 20

        def c_abi():
            assert lib.attn_fwd(*fa) == 0 and lib.attn_bwd(*ba) == 0

        def python():
            attn.attn_fwd(z["q"], z["k"], z["v"], causal=True, o=z["o"], lse=lse)
            attn.attn_bwd(z["q"], z["k"], z["v"], z["o"], lse, z["do"], causal=True, dq=z["dq"],
                          dk=z["dk"], dv=z["dv"], workspace=ws)

        res = {}
        for name, fn in (("c_abi", c_abi), ("python", python)):
            for _ in range(5):
                fn()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            for _ in range(n):
                fn()
            res[name] = (time.perf_counter() - t0) / n * 1e6
            torch.cuda.synchronize()
        attn.attn_check_status()
        out[tag] = res
    return out


def _fwd_only_tflops(attn, t, o, lse, w, stream, torch, reps=20):
    """Forward-only throughput (after the timed region; reported, not the headline)."""
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(3):
        attn.attn_fwd(t["q"], t["k"], t["v"], scale=w.scale, causal=w.causal, o=o, lse=lse)
    e0.record(stream)
    for _ in range(reps):
        attn.attn_fwd(t["q"], t["k"], t["v"], scale=w.scale, causal=w.causal, o=o, lse=lse)
    e1.record(stream)
    torch.cuda.synchronize()
    return w.fwd_flops() * reps / (e0.elapsed_time(e1) * 1e-3) / 1e12


# ---------------------------------------------------------------------------
# deviation report (GPU vs FP64, next to naive BF16 attention vs FP64)
# ---------------------------------------------------------------------------
def run_deviation(args):
    """Numeric-deviation report, one JSON line per workload (head (0,0)).

    For O, LSE, dQ, dK, dV: the tiled GPU kernel, the tiled GPU kernel with
    the stabilised normaliser (beta = 2; on the exact-tie workload also beta =
    1.05, 1.5 and 4), and the naive BF16 attention, each against the FP64
    definition; for O and LSE also the INT8-input forward.  Also delta_lp, the
    rowsum(dO o O) that the backward's preprocess kernel formed from the GPU's
    BF16 O (read back from its workspace), against delta from the exact O
    ("Why Low-Precision Transformer Training Fails", Figure 3).
    """
    import torch

    import oracle
    from precision_numerics_gb300 import attn, build
    from precision_numerics_gb300.deviation import deviation

    build.build()
    cases = [("small", None), ("gpt2", None), ("llama7b", None), ("lowrank", 1.0),
             ("lowrank", 4.0), ("lowrank", 16.0), ("lowrank_ties", 1.0), ("lowrank_ties", 4.0),
             ("lowrank_ties", 16.0), ("longseq", None)]
    for name, sigma in cases:
        w = inputs.WORKLOADS[name]
        x = inputs.make_inputs(w, seed=0, sigma=sigma)
        t = {k: torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).cuda() for k, v in x.items()}
        runs = {}
        variants = [("tiled_gpu", attn.attn_fwd),
                    ("tiled_gpu_stable", lambda *a, **kw: attn.attn_fwd_stable(*a, beta=2.0, **kw))]
        if w.tied_keys:
            # beta is not legible on the pages: sweep it where maxima repeat exactly
            for beta in (1.05, 1.5, 4.0):
                variants.append((f"tiled_gpu_stable_beta{beta:g}",
                                 lambda *a, _b=beta, **kw: attn.attn_fwd_stable(*a, beta=_b, **kw)))
        for tag, fwd in variants:
            o, lse = fwd(t["q"], t["k"], t["v"], scale=w.scale, causal=w.causal)
            ws = torch.empty(attn.attn_bwd_workspace_bytes(w.B, w.H, w.N, w.d),
                             dtype=torch.uint8, device="cuda")
            g = attn.attn_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], scale=w.scale,
                              causal=w.causal, workspace=ws)
            attn.attn_check_status()
            runs[tag] = {"o": o, "lse": lse, "dq": g[0], "dk": g[1], "dv": g[2],
                         "delta": _kernel_delta(ws, w, 0)}
        head = 0
        f = {k: inputs.bf16_bits_to_f32(v.reshape(w.B * w.H, w.N, w.d)[head]) for k, v in x.items()}
        o_ref, lse_ref = oracle.forward(f["q"], f["k"], f["v"], w.scale, w.causal)
        g_ref = oracle.backward(f["q"], f["k"], f["v"], f["do"], w.scale, w.causal)
        o_nv, lse_nv = oracle.naive_bf16_forward(f["q"], f["k"], f["v"], w.scale, w.causal)
        g_nv = oracle.naive_bf16_backward(f["q"], f["k"], f["v"], f["do"], w.scale, w.causal)
        ref = {"o": o_ref, "lse": lse_ref, "dq": g_ref[0], "dk": g_ref[1], "dv": g_ref[2]}
        naive = {"o": o_nv, "lse": lse_nv, "dq": g_nv[0], "dk": g_nv[1], "dv": g_nv[2]}
        rep = {"workload": name, "sigma": sigma, "head": head, "naive_bf16": {}}
        for tag, r in runs.items():
            rep[tag] = {}
            for k in ref:
                gv = r[k].reshape(w.B * w.H, *r[k].shape[2:])[head].float().cpu().numpy()
                rep[tag][k] = deviation(gv, ref[k])
            # delta_lp as the backward's preprocess kernel computed it
            rep[tag]["delta"] = deviation(r["delta"], oracle.delta(f["do"], o_ref))
        for k in ref:
            rep["naive_bf16"][k] = deviation(naive[k], ref[k])
        # INT8-input forward (per-token INT8 Q and K, BF16 V): O and LSE only
        q8, qs = attn.attn_quantize_int8(t["q"])
        k8, ks = attn.attn_quantize_int8(t["k"])
        o8, l8 = attn.attn_fwd_int8(q8, qs, k8, ks, t["v"], scale=w.scale, causal=w.causal)
        attn.attn_check_status()
        rep["int8_gpu"] = {
            "o": deviation(o8.reshape(w.B * w.H, w.N, w.d)[head].float().cpu().numpy(), ref["o"]),
            "lse": deviation(l8.reshape(w.B * w.H, w.N)[head].cpu().numpy(), ref["lse"])}
        print(json.dumps(rep), flush=True)
    return 0


# ---------------------------------------------------------------------------
# INT8-input forward (per-token INT8 Q and K, BF16 V)
# ---------------------------------------------------------------------------
def run_int8_forward(args, w):
    """One JSON line for the INT8-input forward: a step quantizes Q and K
    (attn_quantize_int8_as_bf16) and runs attn_fwd_int8_as_bf16, the tcgen05
    path; value = forward FLOP count (4*B*H*N^2*d, halved when causal) per
    second.  Next to it: the same step on int8 codes (attn_quantize_int8 +
    attn_fwd_int8, the mma.sync path), the BF16 forward's time, and the
    forwards' deviation from the FP64 definition on head (0,0) (the INT8 ones
    also against the INT8 oracle)."""
    import torch

    import oracle
    from oracle import int8 as oi
    from precision_numerics_gb300 import attn, build
    from precision_numerics_gb300.deviation import deviation

    build.build()
    x = inputs.make_inputs(w, seed=0)
    t = {k: torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).cuda() for k, v in x.items()}
    qc, qcs = attn.attn_quantize_int8_as_bf16(t["q"])
    kc, kcs = attn.attn_quantize_int8_as_bf16(t["k"])
    oc, lc = attn.attn_fwd_int8_as_bf16(qc, qcs, kc, kcs, t["v"], scale=w.scale, causal=w.causal)
    q8, qs = attn.attn_quantize_int8(t["q"])
    k8, ks = attn.attn_quantize_int8(t["k"])
    o8, l8 = attn.attn_fwd_int8(q8, qs, k8, ks, t["v"], scale=w.scale, causal=w.causal)
    ob, lb = attn.attn_fwd(t["q"], t["k"], t["v"], scale=w.scale, causal=w.causal)
    stream = torch.cuda.current_stream()

    def step():
        attn.attn_quantize_int8_as_bf16(t["q"], qc, qcs)
        attn.attn_quantize_int8_as_bf16(t["k"], kc, kcs)
        attn.attn_fwd_int8_as_bf16(qc, qcs, kc, kcs, t["v"], scale=w.scale, causal=w.causal, o=oc,
                                   lse=lc)

    def step_s8():
        attn.attn_quantize_int8(t["q"], q8, qs)
        attn.attn_quantize_int8(t["k"], k8, ks)
        attn.attn_fwd_int8(q8, qs, k8, ks, t["v"], scale=w.scale, causal=w.causal, o=o8, lse=l8)

    def timed(fn, steps):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    steps = max(1, min(args.steps, 200))
    ms = timed(step, steps)
    ms_s8 = timed(step_s8, steps)
    ms_bf16 = timed(lambda: attn.attn_fwd(t["q"], t["k"], t["v"], scale=w.scale, causal=w.causal,
                                          o=ob, lse=lb), steps)
    attn.attn_check_status()
    f = {k: inputs.bf16_bits_to_f32(v.reshape(w.B * w.H, w.N, w.d)[0]) for k, v in x.items()}
    o_ref, _ = oracle.forward(f["q"], f["k"], f["v"], w.scale, w.causal)
    o_i8ref, _ = oi.int8_forward(f["q"], f["k"], f["v"], w.scale, w.causal)
    och = oc.reshape(w.B * w.H, w.N, w.d)[0].float().cpu().numpy()
    o8h = o8.reshape(w.B * w.H, w.N, w.d)[0].float().cpu().numpy()
    obh = ob.reshape(w.B * w.H, w.N, w.d)[0].float().cpu().numpy()
    line = {"metric": "INT8-input attention forward TFLOP/s-equivalent on 1 GB300",
            "value": w.fwd_flops() / ms / 1e9, "unit": "TFLOP/s", "n_gpus": 1, "steps": steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "dtype": "int8 codes held in bf16 (exact integer Q K^T), bf16 (P V)",
            "data": "synthetic", "config": _config(w),
            "step": "attn_quantize_int8_as_bf16 on Q and K + attn_fwd_int8_as_bf16",
            "int8_codes_mma_sync": {"ms": ms_s8, "tflops": w.fwd_flops() / ms_s8 / 1e9,
                                    "step": "attn_quantize_int8 on Q and K + attn_fwd_int8"},
            "bf16_forward": {"ms": ms_bf16, "tflops": w.fwd_flops() / ms_bf16 / 1e9},
            "o_vs_fp64": {"int8_as_bf16": deviation(och, o_ref), "int8": deviation(o8h, o_ref),
                          "bf16": deviation(obh, o_ref)},
            "o_int8_vs_int8_oracle": {"int8_as_bf16": deviation(och, o_i8ref),
                                      "int8": deviation(o8h, o_i8ref)}}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="llama7b", choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--int8-forward", action="store_true",
                    help="print the INT8-input forward line instead of the bench line")
    ap.add_argument("--deviation", action="store_true",
                    help="print the numeric-deviation report instead of the bench line")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-chunks", type=int, default=4,
                    help="head groups pipelined in the end-to-end (host buffer) measurement; "
                         "by default shifted by half a group (half-size first and last groups)")
    ap.add_argument("--e2e-even-groups", action="store_true",
                    help="split the end-to-end heads into --e2e-chunks equal groups instead")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.deviation:
        return run_deviation(args)
    if args.int8_forward:
        return run_int8_forward(args, inputs.WORKLOADS[args.workload])
    w = inputs.WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())

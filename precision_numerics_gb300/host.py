"""Attention forward + backward on pinned HOST tensors, pipelined over heads.

Every (b, h) head is independent, so the B*H heads are split into
contiguous groups and, for each group, a pipeline runs over three kinds of
stream: the host->device copy of Q, K, V, dO, then attn_fwd (as soon as Q,
K and V have landed) and attn_bwd (once dO has too) on the device, then the
device->host copy of O and LSE (as soon as the forward is done) and of dQ,
dK, dV.  The copies of one group overlap the kernels of
its neighbours, and the two copy directions overlap each other.  By default
the whole pipeline is captured once as a CUDA graph and replayed.  All
arithmetic runs in the library's kernels; this module only schedules copies
and calls.
"""
from __future__ import annotations

import torch

from . import attn


def ramped_group_sizes(bh, chunks):
    """Head-group sizes for `chunks` equal groups shifted by half a group.

    The first and last groups are half as large as the others (32 heads in
    4 chunks: 4, 8, 8, 8, 4), so the upload before the first forward and the
    download after the last backward, where nothing else overlaps, are half
    as long.  Groups of zero heads are dropped; the sizes sum to `bh`.
    """
    bh, chunks = int(bh), max(1, int(chunks))
    if bh < 1:
        raise ValueError("bh must be >= 1")
    m = bh / chunks
    cuts = sorted({0, bh, *(min(bh, int(m / 2 + i * m + 0.5)) for i in range(chunks))})
    return [b - a for a, b in zip(cuts[:-1], cuts[1:])]


class HostAttention:
    """Reusable pipeline for one problem shape (device buffers are reused).

    q, k, v, do: pinned host BF16 tensors [B, H, N, d].  The B*H heads are
    split into `chunks` equal groups, or into groups of the given
    `group_sizes` (heads per group, in order; they must sum to B*H).  Small
    first and last groups shorten the start (first upload) and the end (last
    download) of the pipeline, where nothing else overlaps.  Outputs are written
    into pinned host tensors allocated once (attributes o, lse, dq, dk, dv);
    they are complete once the calling stream has passed run()'s end (e.g.
    after torch.cuda.synchronize()), and the next run() overwrites them.
    """

    def __init__(self, B, H, N, d, scale=None, causal=False, chunks=4, device=None,
                 group_sizes=None, compute_streams=1, graph=True):
        self.B, self.H, self.N, self.d = B, H, N, d
        self.scale, self.causal = scale, causal
        self.device = torch.device("cuda", torch.cuda.current_device()) if device is None else device
        bh = B * H
        if group_sizes is None:
            chunks = max(1, min(chunks, bh))
            bounds = [round(i * bh / chunks) for i in range(chunks + 1)]
        else:
            if any(int(g) < 1 for g in group_sizes) or sum(group_sizes) != bh:
                raise ValueError(f"group_sizes must be positive and sum to B*H = {bh}")
            bounds = [0]
            for g in group_sizes:
                bounds.append(bounds[-1] + int(g))
        self.groups = [(a, b) for a, b in zip(bounds[:-1], bounds[1:]) if b > a]
        # One upload stream, `compute_streams` compute streams used round-robin
        # by the groups (the kernels of a small group fill only part of the
        # GPU, so consecutive groups may run side by side), one download stream.
        self.s_in = torch.cuda.Stream(self.device)
        self.s_cmp = [torch.cuda.Stream(self.device) for _ in range(max(1, int(compute_streams)))]
        self.s_out = torch.cuda.Stream(self.device)
        dt = torch.bfloat16
        self.o = torch.empty((B, H, N, d), dtype=dt).pin_memory()
        self.dq = torch.empty((B, H, N, d), dtype=dt).pin_memory()
        self.dk = torch.empty((B, H, N, d), dtype=dt).pin_memory()
        self.dv = torch.empty((B, H, N, d), dtype=dt).pin_memory()
        self.lse = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
        # Device buffers, one set per group, so group g+1's inputs can land while
        # group g is still being computed or copied out.
        self.buf = []
        for a, b in self.groups:
            n = b - a
            t = {k: torch.empty((1, n, N, d), dtype=dt, device=self.device)
                 for k in ("q", "k", "v", "do", "o", "dq", "dk", "dv")}
            t["lse"] = torch.empty((1, n, N), dtype=torch.float32, device=self.device)
            t["ws"] = torch.empty(attn.attn_bwd_workspace_bytes(1, n, N, d), dtype=torch.uint8,
                                  device=self.device)
            self.buf.append(t)
        self._last_out = [None] * len(self.groups)  # D2H completion of the previous run
        # With graph=True the whole pipeline (copies, kernels, cross-stream
        # events) is captured once per set of host input addresses as a CUDA
        # graph and replayed, so a run costs one graph launch on the host
        # instead of ~15 calls per group.
        self.graph = bool(graph)
        self._graph = None
        self._graph_key = None

    @staticmethod
    def _heads(x, a, b):
        return x.reshape(-1, *x.shape[2:])[a:b].unsqueeze(0)

    def run(self, q, k, v, do):
        """Enqueue the whole pipeline; the current stream waits for its end."""
        shape = (self.B, self.H, self.N, self.d)
        for name, x in (("q", q), ("k", k), ("v", v), ("do", do)):
            if x.device.type != "cpu" or not x.is_pinned():
                raise ValueError(f"{name} must be a pinned host tensor (tensor.pin_memory())")
            if tuple(x.shape) != shape or x.dtype != torch.bfloat16 or not x.is_contiguous():
                raise ValueError(f"{name} must be a contiguous BF16 tensor of shape {shape}")
        if not self.graph:
            return self._enqueue(q, k, v, do, after_previous=True)
        key = (q.data_ptr(), k.data_ptr(), v.data_ptr(), do.data_ptr())
        if self._graph is None or self._graph_key != key:
            self._capture(q, k, v, do)
            self._graph_key = key
        # Graph launches on one stream run in order, so a replay starts after
        # the previous one has copied its results out of the device buffers.
        self._graph.replay()
        return self.o, self.lse, self.dq, self.dk, self.dv

    def _capture(self, q, k, v, do):
        torch.cuda.synchronize(self.device)
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(self.device)
        side.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.graph(g, stream=side):
            self._enqueue(q, k, v, do, after_previous=False)
        torch.cuda.current_stream(self.device).wait_stream(side)
        self._graph = g

    def _enqueue(self, q, k, v, do, after_previous):
        s_in, s_out = self.s_in, self.s_out
        cur = torch.cuda.current_stream(self.device)
        s_in.wait_stream(cur)
        done = []
        for g, ((a, b), t) in enumerate(zip(self.groups, self.buf)):
            # This group's device buffers are free once the previous run copied them out.
            if after_previous and self._last_out[g] is not None:
                s_in.wait_event(self._last_out[g])
            # The forward needs Q, K, V only; dO is still on its way while it runs.
            with torch.cuda.stream(s_in):
                for name, src in (("q", q), ("k", k), ("v", v)):
                    t[name].copy_(self._heads(src, a, b), non_blocking=True)
                ev_qkv = torch.cuda.Event()
                ev_qkv.record(s_in)
                t["do"].copy_(self._heads(do, a, b), non_blocking=True)
                ev_in = torch.cuda.Event()
                ev_in.record(s_in)
            s_cmp = self.s_cmp[g % len(self.s_cmp)]
            s_cmp.wait_event(ev_qkv)
            with torch.cuda.stream(s_cmp):
                attn.attn_fwd(t["q"], t["k"], t["v"], scale=self.scale, causal=self.causal,
                              o=t["o"], lse=t["lse"], stream=s_cmp)
                ev_fwd = torch.cuda.Event()
                ev_fwd.record(s_cmp)
            s_cmp.wait_event(ev_in)
            with torch.cuda.stream(s_cmp):
                attn.attn_bwd(t["q"], t["k"], t["v"], t["o"], t["lse"], t["do"], scale=self.scale,
                              causal=self.causal, dq=t["dq"], dk=t["dk"], dv=t["dv"],
                              workspace=t["ws"], stream=s_cmp)
                ev_cmp = torch.cuda.Event()
                ev_cmp.record(s_cmp)
            # O and LSE go out while the backward of the same group still runs.
            s_out.wait_event(ev_fwd)
            with torch.cuda.stream(s_out):
                self._heads(self.o, a, b).copy_(t["o"], non_blocking=True)
                self.lse.reshape(-1, self.N)[a:b].copy_(t["lse"][0], non_blocking=True)
            s_out.wait_event(ev_cmp)
            with torch.cuda.stream(s_out):
                for name, dst in (("dq", self.dq), ("dk", self.dk), ("dv", self.dv)):
                    self._heads(dst, a, b).copy_(t[name], non_blocking=True)
                ev_out = torch.cuda.Event()
                ev_out.record(s_out)
            done.append(ev_out)
            if after_previous:
                self._last_out[g] = ev_out
        for ev in done:
            cur.wait_event(ev)
        return self.o, self.lse, self.dq, self.dk, self.dv

    def bytes_per_run(self):
        """Host->device and device->host bytes moved by one run()."""
        el = self.B * self.H * self.N * self.d * 2
        return 4 * el, 4 * el + self.B * self.H * self.N * 4

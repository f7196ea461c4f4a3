"""Seeded synthetic inputs for the attention workloads.

This module only draws random numbers and rounds them to the storage type;
it holds no attention arithmetic.  Both the CUDA path and the FP64 oracle
receive the arrays it returns, so the two always see bit-identical inputs.

Random source: NumPy's Philox-4x32 counter-based generator, keyed by
(seed, stream id), so every tensor of a workload has its own independent,
reproducible stream.  Values are drawn in FP32 and rounded to BF16 with
round-to-nearest-even; the BF16 values are carried as uint16 bit patterns.

Workloads (shapes, value distributions, causal flag, softmax scale):

  small        B1 H2  N128   d64,  N(0,1), non-causal, scale 1/sqrt(d)
  gpt2         B8 H12 N1024  d64,  N(0,1), causal,     scale 1/8
  llama7b      B1 H32 N4096  d128, N(0,1), causal,     scale 1/sqrt(128)
  lowrank      B4 H16 N2048  d128, Q = A.U, K = B.U with U (4 x 128) having
               orthonormal rows, A, B ~ N(0, sigma^2) of shape N x 4;
               V, dO ~ N(0,1); causal, scale 1/sqrt(128)
  longseq      B2 H16 N16384 d128, Q,K,V ~ N(0,1)/sqrt(d), dO ~ N(0,1),
               causal, scale 1/sqrt(128)
  lowrank_ties the low-rank workload with key rows duplicated in pairs
               (K[2t+1] = K[2t]), so row maxima are attained exactly twice --
               the repeated-maximum case of "Why Low-Precision Transformer
               Training Fails", Figure 7

The low-rank workload is the synthetic stand-in for the "similar low-rank
representations" of "Why Low-Precision Transformer Training Fails"
(Figure 4): with U U^T = I_4 the logits are scale * A B^T, so large,
near-tied row maxima appear as sigma grows.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

# Stream ids, one per tensor role, so that each tensor's values do not depend
# on which other tensors a caller happens to draw.
STREAM_Q, STREAM_K, STREAM_V, STREAM_DO, STREAM_A, STREAM_B, STREAM_U = range(7)


def _rng(seed: int, stream: int) -> np.random.Generator:
    # Philox key = (seed, stream); counter starts at 0.
    return np.random.Generator(np.random.Philox(key=[seed & 0xFFFFFFFFFFFFFFFF, stream]))


def normal(seed: int, stream: int, shape, std: float = 1.0) -> np.ndarray:
    """i.i.d. N(0, std^2) FP32 samples of the given shape."""
    x = _rng(seed, stream).standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round FP32 to BF16 (round to nearest, ties to even); returns uint16 bits.

    NaN inputs stay NaN (quiet bit forced); the generator never produces them.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        r[nan] = ((u[nan] >> np.uint64(16)).astype(np.uint16) | np.uint16(0x0040))
    return r


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen BF16 bit patterns to FP32 (exact)."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    scale: float
    qkv_std: float = 1.0          # std of Q, K, V entries (i.i.d. workloads)
    lowrank_rank: int = 0         # > 0: Q = A U, K = B U with U of this many rows
    sigmas: tuple = field(default_factory=tuple)
    backward: bool = True
    tied_keys: bool = False       # K[2t+1] = K[2t]

    def fwd_flops(self) -> float:
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2 if self.causal else f

    def bwd_flops(self) -> float:
        return 2.5 * self.fwd_flops()


WORKLOADS = {
    "small": Workload("small", 1, 2, 128, 64, False, 1.0 / math.sqrt(64), backward=False),
    "gpt2": Workload("gpt2", 8, 12, 1024, 64, True, 1.0 / 8.0),
    "llama7b": Workload("llama7b", 1, 32, 4096, 128, True, 1.0 / math.sqrt(128)),
    "lowrank": Workload("lowrank", 4, 16, 2048, 128, True, 1.0 / math.sqrt(128),
                        lowrank_rank=4, sigmas=(1.0, 4.0, 16.0)),
    "longseq": Workload("longseq", 2, 16, 16384, 128, True, 1.0 / math.sqrt(128),
                        qkv_std=1.0 / math.sqrt(128)),
    "lowrank_ties": Workload("lowrank_ties", 4, 16, 2048, 128, True, 1.0 / math.sqrt(128),
                             lowrank_rank=4, sigmas=(1.0, 4.0, 16.0), tied_keys=True),
}


def orthonormal_rows(seed: int, r: int, d: int, count: int) -> np.ndarray:
    """`count` independent r x d matrices with orthonormal rows (FP64).

    Each is the Q factor of a seeded d x r Gaussian, transposed; signs are
    fixed so the diagonal of the R factor is positive.
    """
    g = _rng(seed, STREAM_U).standard_normal(size=(count, d, r))
    out = np.empty((count, r, d))
    for c in range(count):
        qf, rf = np.linalg.qr(g[c])
        qf = qf * np.sign(np.diag(rf))[None, :]
        out[c] = qf.T
    return out


def make_inputs(w: Workload, seed: int = 0, sigma: float | None = None,
                dtype: str = "bf16", heads: int | None = None) -> dict:
    """Q, K, V, dO of workload `w` as [B, H, N, d] arrays.

    dtype "bf16": uint16 bit patterns (BF16 values, rounded from FP32);
    dtype "fp32": FP32 values.  `heads` limits the draw to the first
    `heads` (b, h) pairs in row-major order (used for samples); the values
    of those heads do not depend on `heads`.
    """
    shape = (w.B, w.H, w.N, w.d)
    if w.lowrank_rank:
        if sigma is None:
            sigma = w.sigmas[0]
        bh = w.B * w.H
        r = w.lowrank_rank
        a = _rng(seed, STREAM_A).standard_normal(size=(bh, w.N, r)) * sigma
        b = _rng(seed, STREAM_B).standard_normal(size=(bh, w.N, r)) * sigma
        u = orthonormal_rows(seed, r, w.d, bh)
        q = np.einsum("xnr,xrd->xnd", a, u).reshape(shape).astype(np.float32)
        k = np.einsum("xnr,xrd->xnd", b, u).reshape(shape).astype(np.float32)
        v = normal(seed, STREAM_V, shape)
    else:
        q = normal(seed, STREAM_Q, shape, w.qkv_std)
        k = normal(seed, STREAM_K, shape, w.qkv_std)
        v = normal(seed, STREAM_V, shape, w.qkv_std)
    if w.tied_keys:
        k = k.copy()
        k[..., 1::2, :] = k[..., 0:w.N - (w.N % 2):2, :]
    do = normal(seed, STREAM_DO, shape)
    out = {"q": q, "k": k, "v": v, "do": do}
    if heads is not None:
        for key in out:
            out[key] = out[key].reshape(w.B * w.H, w.N, w.d)[:heads].copy()
            out[key] = out[key].reshape(heads, 1, w.N, w.d)
    if dtype == "bf16":
        out = {key: f32_to_bf16_bits(val) for key, val in out.items()}
    elif dtype != "fp32":
        raise ValueError(f"dtype must be 'bf16' or 'fp32', got {dtype!r}")
    return out


def random_qkv(seed: int, B: int, H: int, N: int, d: int, dtype: str = "bf16",
               std: float = 1.0) -> dict:
    """Q, K, V, dO ~ N(0, std^2) (dO ~ N(0,1)) of an arbitrary shape, for tests."""
    shape = (B, H, N, d)
    out = {"q": normal(seed, STREAM_Q, shape, std), "k": normal(seed, STREAM_K, shape, std),
           "v": normal(seed, STREAM_V, shape, std), "do": normal(seed, STREAM_DO, shape)}
    if dtype == "bf16":
        out = {key: f32_to_bf16_bits(val) for key, val in out.items()}
    return out

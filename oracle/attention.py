"""FP64 oracle for exact softmax attention, forward and backward.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
bench's CPU-baseline / reference arm may import this module.  The CUDA
library never calls it and shares no code with it.

What it computes, and where that is defined:

* Forward -- "Baseline Attention" as named in "Is Flash Attention Stable?"
  (abstract), i.e. the standard attention of "Attention Is All You Need":
  S = scale * Q K^T, a causal mask (key j hidden from query i when j > i,
  square and top-left aligned), P = softmax(S) row-wise, O = P V.  The
  saved log-sum-exp is LSE_i = m_i + ln sum_j exp(S_ij - m_i) with
  m_i = max_j S_ij (natural log).  FlashAttention ("Fast and
  Memory-Efficient Exact Attention") computes this same result exactly,
  up to rounding order, so the oracle is the plain definition, not the
  tiled algorithm.
* Backward -- the analytic gradient of that definition for a given dO:
  dV = P^T dO, dP = dO V^T, delta_i = rowsum(dO o O)_i ("Why Low-Precision
  Transformer Training Fails", Figures 3 and 5: delta = rowsum(dO o O)),
  dS = P o (dP - delta), dQ = scale dS K, dK = scale dS^T Q.  Optionally
  delta is formed from a supplied (e.g. BF16-rounded) O instead, as in that
  paper's Figure 3 (delta_lp = rowsum(dO o O_lp)).
* The naive BF16 comparator -- "Baseline Attention at BF16" of "Is Flash
  Attention Stable?": materialised scores and probabilities, each matrix
  product accumulated in FP32 and rounded to BF16 (round to nearest even)
  where an eager framework materialises a tensor.  The pages do not say
  where that baseline rounds; this placement is a reading.

All arrays are NumPy.  Single-head functions take 2-D [N, d] arrays; the
`*_bhnd` wrappers loop over the leading [B, H] axes.  Inputs are widened to
FP64 exactly as given (the same BF16 or FP32 values the GPU receives).

Pins (tests that tie this module to something other than itself): closed
forms (single key, constant V, uniform keys, a hand-derived two-key
example with its gradients), invariants (rows of P sum to 1, joint
key/value permutation, causal prefixes), library routines (SciPy
log-sum-exp and softmax, PyTorch FP64 scaled-dot-product attention with
autograd), central finite differences of L = sum(dO o O), and a
pure-Python brute force on tiny inputs.  The naive BF16 comparator's
rounding is pinned against PyTorch's BF16 conversion, and where it rounds
against an eager framework's BF16 graph: PyTorch CPU ops on BF16 tensors and
their autograd backward give the same BF16 values (at least 99% bit for bit).
"""
from __future__ import annotations

import numpy as np


# ----------------------------------------------------------------------------
# Forward (the definition)
# ----------------------------------------------------------------------------

def scores(q, k, scale, causal):
    """S = scale * Q K^T, with -inf where a key lies after its query (causal)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    s = scale * (q @ k.T)
    if causal:
        n_q, n_k = s.shape
        hidden = np.arange(n_k)[None, :] > np.arange(n_q)[:, None]
        s = np.where(hidden, -np.inf, s)
    return s


def row_max(s):
    """m_i = max_j S_ij."""
    return s.max(axis=1)


def probabilities(q, k, scale, causal):
    """P = softmax(S) row-wise, together with m and the row sums l.

    P_ij = exp(S_ij - m_i) / l_i with l_i = sum_j exp(S_ij - m_i).
    """
    s = scores(q, k, scale, causal)
    m = row_max(s)
    e = np.exp(s - m[:, None])
    l = e.sum(axis=1)
    return e / l[:, None], m, l


def forward(q, k, v, scale, causal):
    """O = softmax(scale Q K^T [+ mask]) V and LSE (natural log), single head."""
    p, m, l = probabilities(q, k, scale, causal)
    o = p @ np.asarray(v, dtype=np.float64)
    lse = m + np.log(l)
    return o, lse


# ----------------------------------------------------------------------------
# Backward (analytic gradient of the definition)
# ----------------------------------------------------------------------------

def delta(do, o):
    """delta_i = sum_k dO_ik O_ik (rowsum of the elementwise product)."""
    return (np.asarray(do, dtype=np.float64) * np.asarray(o, dtype=np.float64)).sum(axis=1)


def backward(q, k, v, do, scale, causal, o_for_delta=None):
    """dQ, dK, dV of L = sum(dO o O) for O = forward(q, k, v), single head.

    With `o_for_delta` given, delta is taken as rowsum(dO o o_for_delta)
    instead of from the exact O: the substitution of "Why Low-Precision
    Transformer Training Fails", Figure 3, where delta_lp = rowsum(dO o O_lp)
    is formed from a low-precision O.  Everything else stays exact.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    p, _, _ = probabilities(q, k, scale, causal)
    o = p @ v if o_for_delta is None else np.asarray(o_for_delta, dtype=np.float64)
    dv = p.T @ do
    dp = do @ v.T
    ds = p * (dp - delta(do, o)[:, None])
    dq = scale * (ds @ k)
    dk = scale * (ds.T @ q)
    return dq, dk, dv


# ----------------------------------------------------------------------------
# Naive BF16 attention ("Baseline Attention at BF16"), emulated on the CPU
# ----------------------------------------------------------------------------

def round_bf16(x):
    """Round FP32 values to the nearest BF16 value (ties to even), as FP32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    bits = x.view(np.uint32).astype(np.uint64)
    keep = (bits >> np.uint64(16)) & np.uint64(1)
    rounded = ((bits + np.uint64(0x7FFF) + keep) >> np.uint64(16)) << np.uint64(16)
    out = rounded.astype(np.uint32).view(np.float32)
    return np.where(np.isfinite(x), out, x)


def _f32(x):
    return np.asarray(x, dtype=np.float32)


def naive_bf16_forward(q, k, v, scale, causal):
    """Eager-framework attention at BF16, single head.

    Each product is accumulated in FP32 and the result rounded to BF16;
    the scaled scores, the softmax output and O are BF16 tensors; the
    softmax itself runs in FP32.  Returns (O as FP32-held BF16 values,
    LSE in FP32 from the BF16 scores).
    """
    q, k, v = _f32(q), _f32(k), _f32(v)
    s = round_bf16(q @ k.T)
    s = round_bf16(s * np.float32(scale))
    if causal:
        n = s.shape[0]
        s = np.where(np.arange(s.shape[1])[None, :] > np.arange(n)[:, None],
                     np.float32(-np.inf), s)
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m, dtype=np.float32)
    l = e.sum(axis=1, keepdims=True, dtype=np.float32)
    p = round_bf16(e / l)
    o = round_bf16(p @ v)
    lse = (m + np.log(l)).reshape(-1).astype(np.float32)
    return o, lse


def naive_bf16_backward(q, k, v, do, scale, causal):
    """Eager-framework attention backward at BF16, single head.

    Follows autograd through the forward above: dV = bf16(P^T dO),
    dP = bf16(dO V^T), dS = bf16(P o (dP - rowsum(dP o P))) in FP32,
    the scale applied to dS with a BF16 rounding, then dQ = bf16(dS K),
    dK = bf16(dS^T Q).
    """
    q, k, v, do = _f32(q), _f32(k), _f32(v), round_bf16(_f32(do))
    s = round_bf16(q @ k.T)
    s = round_bf16(s * np.float32(scale))
    if causal:
        n = s.shape[0]
        s = np.where(np.arange(s.shape[1])[None, :] > np.arange(n)[:, None],
                     np.float32(-np.inf), s)
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m, dtype=np.float32)
    p = round_bf16(e / e.sum(axis=1, keepdims=True, dtype=np.float32))
    dv = round_bf16(p.T @ do)
    dp = round_bf16(do @ v.T)
    ds = round_bf16(p * (dp - (dp * p).sum(axis=1, keepdims=True, dtype=np.float32)))
    ds = round_bf16(ds * np.float32(scale))
    dq = round_bf16(ds @ k)
    dk = round_bf16(ds.T @ q)
    return dq, dk, dv


# ----------------------------------------------------------------------------
# [B, H, N, d] wrappers
# ----------------------------------------------------------------------------

def _heads(x):
    x = np.asarray(x)
    return x.reshape(-1, x.shape[-2], x.shape[-1])


def forward_bhnd(q, k, v, scale, causal, fn=forward):
    """Per-head `fn` over [B, H, N, d] inputs; returns O [B,H,N,d], LSE [B,H,N]."""
    lead = np.asarray(q).shape[:-2]
    qh, kh, vh = _heads(q), _heads(k), _heads(v)
    outs = [fn(qh[i], kh[i], vh[i], scale, causal) for i in range(qh.shape[0])]
    o = np.stack([x[0] for x in outs]).reshape(*lead, *qh.shape[1:])
    lse = np.stack([x[1] for x in outs]).reshape(*lead, qh.shape[1])
    return o, lse


def backward_bhnd(q, k, v, do, scale, causal, fn=backward):
    """Per-head `fn` over [B, H, N, d] inputs; returns dQ, dK, dV."""
    lead = np.asarray(q).shape[:-2]
    qh, kh, vh, doh = _heads(q), _heads(k), _heads(v), _heads(do)
    outs = [fn(qh[i], kh[i], vh[i], doh[i], scale, causal) for i in range(qh.shape[0])]
    return tuple(np.stack([x[j] for x in outs]).reshape(*lead, *qh.shape[1:]) for j in range(3))

"""INT8-input attention forward, FP64 oracle.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
bench's CPU-baseline / reference arm may import this module.  The CUDA
library never calls it and shares no code with it.

What it computes, and where that is defined:

* "INT-FlashAttention: Enabling Flash Attention for INT8 Quantization"
  (abstract; the page gives nothing beyond it): INT8 quantization that fits
  the forward workflow of FlashAttention.  Readings, since the abstract fixes
  no detail: Q and K are quantized per token -- one symmetric scale per row
  of each head -- to INT8; V stays BF16; the scores are
  S_ij = scale * s_q[i] * s_k[j] * (q8_i . k8_j) with the integer dot
  product exact; softmax, P V and LSE are those of the FP64 definition
  (oracle.attention.forward) applied to these scores.
* Quantization, with every decision taken in FP32 as the kernel takes it:
  s = fl32(max_j |x_j| / 127); code_j = rint(fl32(x_j / s)) clamped to
  [-127, 127], rint rounding half to even; a row of zeros gets s = 0 and
  all codes 0.

Pins (tests/test_oracle_int8.py): a hand-derived quantization example with
ties at .5 (tests/golden/int8_quant_example.txt); a hand-derived forward
with distinct, non-unit scales on Q and K (tests/golden/
int8_forward_example.txt: codes, scales, scores, O and LSE), which a
Q/K scale swap or skipping the quantization fails; codes within [-127, 127]
with the row maximum at +-127; sign symmetry; the round-trip error bound
|x - code * s| <= s / 2; exact integer dot products against a pure-Python
loop; lossless inputs (values already integer multiples of their scale)
reproduce the unquantized forward; the score error bound that quantization
implies.
"""
from __future__ import annotations

import numpy as np

from .attention import forward


def quantize_per_token(x):
    """Symmetric per-row INT8 codes and FP32 scales of a 2-D [N, d] array."""
    x = np.asarray(x, dtype=np.float32)
    amax = np.abs(x).max(axis=1)
    s = (amax / np.float32(127.0)).astype(np.float32)
    safe = np.where(s > 0, s, np.float32(1.0)).astype(np.float32)
    ratio = (x / safe[:, None]).astype(np.float32)
    codes = np.clip(np.rint(ratio), -127, 127).astype(np.int8)
    codes[s == 0] = 0
    return codes, s


def dequantize(codes, s):
    """code * s in FP64 (exact: an 8-bit integer times an FP32 value)."""
    return codes.astype(np.float64) * np.asarray(s, dtype=np.float64)[:, None]


def int8_scores(q8, sq, k8, sk, scale, causal):
    """S = scale * s_q s_k^T o (Q8 K8^T) with the integer product exact."""
    dots = q8.astype(np.int64) @ k8.astype(np.int64).T
    s = scale * (np.asarray(sq, np.float64)[:, None] * np.asarray(sk, np.float64)[None, :]) * dots
    if causal:
        n_q, n_k = s.shape
        s = np.where(np.arange(n_k)[None, :] > np.arange(n_q)[:, None], -np.inf, s)
    return s


def int8_forward(q, k, v, scale, causal):
    """O and LSE of attention on per-token INT8 Q and K (single head).

    Equal, up to FP64 rounding, to the definition evaluated on the
    dequantized Q and K, which is how it is computed here.
    """
    q8, sq = quantize_per_token(q)
    k8, sk = quantize_per_token(k)
    return forward(dequantize(q8, sq), dequantize(k8, sk), v, scale, causal)


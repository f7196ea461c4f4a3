"""CPU checks of the delta_lp error estimate used by the low-rank GPU tests.

tests/bounds.py derives, from the BF16 roundings of the stored O, an RMS
estimate of the dQ and dK error that delta_lp = rowsum(dO o O_lp) ("Why
Low-Precision Transformer Training Fails", Figure 3) carries.  Here that
estimate is held against a brute-force emulation of those roundings on the
CPU: P~ = exp(S - m) rounded to BF16 as the P V operand, the row sum over the
unrounded P~, O rounded to BF16, delta_lp from it, and the resulting dQ, dK
error propagated exactly.  The emulated error must stay below the estimate
and be of the same order (the estimate is not vacuous).
"""
import numpy as np
import pytest

import oracle
from precision_numerics_gb300 import inputs

from bounds import delta_error_rms


def _lowrank_head(N, d, sigma, seed):
    w = inputs.Workload("t", 1, 1, N, d, True, d ** -0.5, lowrank_rank=4, sigmas=(sigma,))
    x = inputs.make_inputs(w, seed=seed, sigma=sigma)
    return {k: inputs.bf16_bits_to_f32(v[0, 0]).astype(np.float64) for k, v in x.items()}, w.scale


def _emulated_delta_error(f, scale, causal):
    p, m, _ = oracle.probabilities(f["q"], f["k"], scale, causal)
    s = oracle.scores(f["q"], f["k"], scale, causal)
    pt = np.exp(s - m[:, None])                        # P~, largest entry 1
    pt_lp = oracle.round_bf16(pt).astype(np.float64)   # BF16 operand of P V
    o_lp = oracle.round_bf16((pt_lp @ f["v"]) / pt.sum(axis=1)[:, None]).astype(np.float64)
    o = p @ f["v"]
    e = (f["do"] * o_lp).sum(axis=1) - (f["do"] * o).sum(axis=1)   # delta_lp - delta
    ds_err = -p * e[:, None]
    return np.linalg.norm(scale * ds_err @ f["k"]), np.linalg.norm(scale * ds_err.T @ f["q"])


@pytest.mark.parametrize("sigma", [4.0, 16.0])
@pytest.mark.parametrize("seed", [0, 1])
def test_rms_estimate_covers_the_emulated_delta_error(sigma, seed):
    f, scale = _lowrank_head(512, 128, sigma, seed)
    rms_dq, rms_dk = delta_error_rms(f, scale, True)
    err_dq, err_dk = _emulated_delta_error(f, scale, True)
    assert err_dq <= rms_dq and err_dk <= rms_dk, (err_dq, rms_dq, err_dk, rms_dk)
    assert err_dq >= 0.2 * rms_dq and err_dk >= 0.2 * rms_dk, (err_dq, rms_dq, err_dk, rms_dk)


def test_estimate_grows_with_the_rank_one_structure():
    # larger sigma: larger, near-tied logits, more cancellation in dP - delta,
    # so delta_lp's error is a larger share of dQ
    rel = []
    for sigma in (1.0, 16.0):
        f, scale = _lowrank_head(256, 64, sigma, 0)
        dq = oracle.backward(f["q"], f["k"], f["v"], f["do"], scale, True)[0]
        rel.append(delta_error_rms(f, scale, True)[0] / np.linalg.norm(dq))
    assert rel[1] > 5 * rel[0], rel

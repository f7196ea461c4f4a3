"""Pins of the INT8 forward oracle (oracle/int8.py), CPU only."""
import os

import numpy as np
import pytest

import oracle
from oracle import int8 as oi

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "int8_quant_example.txt")


def _golden():
    rows, codes, scales = [], [], []
    for line in open(GOLDEN):
        if not line.strip() or line.startswith("#"):
            continue
        tag, *vals = line.split()
        if tag == "x":
            rows.append([float(v) for v in vals])
        elif tag == "codes":
            codes.append([int(v) for v in vals])
        elif tag == "scale":
            scales.append(float(vals[0]))
    return np.array(rows, np.float32), np.array(codes), np.array(scales)


def test_golden_quantization_example():
    x, codes, scales = _golden()
    c, s = oi.quantize_per_token(x)
    assert np.array_equal(c.astype(int), codes)
    assert np.array_equal(s.astype(np.float64), scales.astype(np.float32).astype(np.float64))


def _rand(seed, n=64, d=128, std=1.0):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((n, d)) * std).astype(np.float32)


@pytest.mark.parametrize("std", [1e-3, 1.0, 50.0])
def test_codes_range_max_and_round_trip(std):
    x = _rand(1, std=std)
    c, s = oi.quantize_per_token(x)
    assert c.dtype == np.int8 and np.abs(c.astype(int)).max() <= 127
    # the row maximum lands on +-127
    assert np.all(np.abs(c.astype(int)).max(axis=1) == 127)
    # |x - code * s| <= s / 2 (up to the FP32 rounding of x / s)
    err = np.abs(x.astype(np.float64) - oi.dequantize(c, s))
    assert np.all(err <= s[:, None].astype(np.float64) * (0.5 + 1e-5))


def test_sign_symmetry_and_zero_row():
    x = _rand(2)
    x[3] = 0.0
    c, s = oi.quantize_per_token(x)
    cn, sn = oi.quantize_per_token(-x)
    assert np.array_equal(cn.astype(int), -c.astype(int)) and np.array_equal(sn, s)
    assert s[3] == 0 and not c[3].any()


def test_integer_dot_products_are_exact():
    rng = np.random.default_rng(3)
    q8 = rng.integers(-127, 128, (5, 32)).astype(np.int8)
    k8 = rng.integers(-127, 128, (7, 32)).astype(np.int8)
    sq, sk = np.ones(5, np.float32), np.ones(7, np.float32)
    s = oi.int8_scores(q8, sq, k8, sk, 1.0, False)
    for i in range(5):
        for j in range(7):
            assert s[i, j] == sum(int(a) * int(b) for a, b in zip(q8[i], k8[j]))


@pytest.mark.parametrize("causal", [False, True])
def test_lossless_inputs_reproduce_the_unquantized_forward(causal):
    # integer values with a row maximum of exactly 127: s = 1, codes = x
    rng = np.random.default_rng(4)
    q = rng.integers(-127, 128, (40, 64)).astype(np.float32)
    k = rng.integers(-127, 128, (40, 64)).astype(np.float32)
    q[:, 0], k[:, 0] = 127.0, -127.0
    v = rng.standard_normal((40, 64))
    o8, l8 = oi.int8_forward(q, k, v, 1e-3, causal)
    o, l = oracle.forward(q, k, v, 1e-3, causal)
    assert np.allclose(o8, o, rtol=0, atol=1e-12) and np.allclose(l8, l, rtol=0, atol=1e-12)


def test_score_error_within_the_quantization_bound():
    q, k = _rand(5), _rand(6)
    scale = 128 ** -0.5
    q8, sq = oi.quantize_per_token(q)
    k8, sk = oi.quantize_per_token(k)
    s8 = oi.int8_scores(q8, sq, k8, sk, scale, False)
    s = oracle.scores(q, k, scale, False)
    # q = q^ + e_q with |e_q| <= s_q / 2 (same for k), so
    # |q.k - q^.k^| <= |q|.s_k/2 + |k|.s_q/2 + d s_q s_k / 4, times scale
    aq = np.abs(q.astype(np.float64)).sum(axis=1)
    ak = np.abs(k.astype(np.float64)).sum(axis=1)
    bound = scale * (aq[:, None] * sk[None, :] / 2 + ak[None, :] * sq[:, None] / 2
                     + q.shape[1] * sq[:, None] * sk[None, :] / 4) * (1 + 1e-5)
    assert np.all(np.abs(s8 - s) <= bound)
    # and the bound is not vacuous: the error is a visible fraction of it
    assert np.abs(s8 - s).max() > 1e-3 * bound.max()


def test_planted_mistake_fails_the_golden_example():
    # rounding half away from zero instead of half to even breaks the ties
    x, codes, _ = _golden()
    s = (np.abs(x).max(axis=1) / np.float32(127)).astype(np.float32)
    safe = np.where(s > 0, s, 1).astype(np.float32)
    away = np.sign(x / safe[:, None]) * np.floor(np.abs(x / safe[:, None]) + 0.5)
    assert not np.array_equal(away.astype(int), codes)


# ------------------------------------------------------- worked forward example

FWD_GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "int8_forward_example.txt")


def _fwd_golden():
    g = {}
    for line in open(FWD_GOLDEN):
        if not line.strip() or line.startswith("#"):
            continue
        name, rows, cols, *vals = line.split()
        g[name] = np.array([float(v) for v in vals]).reshape(int(rows), int(cols))
    g["scale"] = float(g["scale"][0, 0])
    return g


def test_golden_forward_example_codes_scales_scores():
    g = _fwd_golden()
    q8, sq = oi.quantize_per_token(g["q"])
    k8, sk = oi.quantize_per_token(g["k"])
    assert np.array_equal(q8.astype(int), g["q_codes"].astype(int))
    assert np.array_equal(k8.astype(int), g["k_codes"].astype(int))
    assert np.array_equal(sq.astype(np.float64), g["q_scale"].reshape(-1))
    assert np.array_equal(sk.astype(np.float64), g["k_scale"].reshape(-1))
    # every score is an exact dyadic rational, so FP64 reproduces it exactly
    s = oi.int8_scores(q8, sq, k8, sk, g["scale"], False)
    assert np.array_equal(s, g["s"])


def test_golden_forward_example_o_and_lse():
    g = _fwd_golden()
    o, lse = oi.int8_forward(g["q"], g["k"], g["v"], g["scale"], False)
    np.testing.assert_allclose(o, g["o"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, g["lse"].reshape(-1), rtol=0, atol=1e-12)


def test_planted_scale_swap_and_skipped_quantization_fail_the_forward_example():
    g = _fwd_golden()
    q8, sq = oi.quantize_per_token(g["q"])
    k8, sk = oi.quantize_per_token(g["k"])
    # slip 1: each tensor's codes paired with the other tensor's scales
    o_swap, lse_swap = oracle.forward(oi.dequantize(q8, sk), oi.dequantize(k8, sq), g["v"],
                                      g["scale"], False)
    assert np.abs(o_swap - g["o"]).max() > 1.0 and np.abs(lse_swap - g["lse"]).max() > 1.0
    # slip 2: no quantization at all
    o_raw, lse_raw = oracle.forward(g["q"], g["k"], g["v"], g["scale"], False)
    assert np.abs(o_raw - g["o"]).max() > 1e-2 and np.abs(lse_raw - g["lse"]).max() > 1e-3

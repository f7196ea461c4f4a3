"""The seeded input generator: determinism, BF16 rounding, workload recipes (CPU)."""
import math

import numpy as np
import pytest

from precision_numerics_gb300 import inputs


def test_normal_is_deterministic_and_stream_separated():
    a = inputs.normal(0, inputs.STREAM_Q, (4, 5))
    b = inputs.normal(0, inputs.STREAM_Q, (4, 5))
    c = inputs.normal(0, inputs.STREAM_K, (4, 5))
    d = inputs.normal(1, inputs.STREAM_Q, (4, 5))
    np.testing.assert_array_equal(a, b)
    assert not np.array_equal(a, c)
    assert not np.array_equal(a, d)
    assert a.dtype == np.float32


def test_normal_moments():
    x = inputs.normal(3, inputs.STREAM_V, (200000,), std=0.5)
    assert abs(x.mean()) < 0.01
    assert abs(x.std() - 0.5) < 0.01


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    x = np.concatenate([inputs.normal(5, 0, (50000,), 9.0),
                        np.array([1.00390625, 1.005859375, -1.00390625, 0.0, -0.0], np.float32)])
    bits = inputs.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(bits, ref)
    back = inputs.bf16_bits_to_f32(bits)
    np.testing.assert_array_equal(back, torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_lowrank_construction():
    w = inputs.Workload("t", 1, 2, 64, 128, True, 1 / math.sqrt(128), lowrank_rank=4,
                        sigmas=(4.0,))
    u = inputs.orthonormal_rows(0, 4, 128, 2)
    for c in range(2):
        np.testing.assert_allclose(u[c] @ u[c].T, np.eye(4), atol=1e-12)
    x = inputs.make_inputs(w, seed=0, sigma=4.0, dtype="fp32")
    # Q K^T has rank <= 4 per head.
    s = x["q"][0, 0].astype(np.float64) @ x["k"][0, 0].astype(np.float64).T
    sv = np.linalg.svd(s, compute_uv=False)
    assert sv[4] < 1e-4 * sv[0]


def test_head_subset_matches_full_draw():
    w = inputs.WORKLOADS["gpt2"]
    w = inputs.Workload("t", 2, 3, 16, 8, True, 0.5)
    full = inputs.make_inputs(w, seed=7)
    part = inputs.make_inputs(w, seed=7, heads=4)
    for key in full:
        np.testing.assert_array_equal(full[key].reshape(6, 16, 8)[:4], part[key].reshape(4, 16, 8))


def test_workload_flop_counts():
    w = inputs.WORKLOADS["llama7b"]
    assert w.fwd_flops() == pytest.approx(137.4e9, rel=1e-3)
    assert w.bwd_flops() == pytest.approx(343.6e9, rel=1e-3)
    assert inputs.WORKLOADS["gpt2"].fwd_flops() == pytest.approx(12.88e9, rel=1e-3)


def test_tied_keys_are_exact_pairs():
    w = inputs.Workload("t", 1, 2, 64, 128, True, 0.1, lowrank_rank=4, sigmas=(4.0,),
                        tied_keys=True)
    k = inputs.make_inputs(w, seed=1, sigma=4.0)["k"]
    np.testing.assert_array_equal(k[..., 1::2, :], k[..., 0::2, :])
    assert not np.array_equal(k[..., 0, :], k[..., 2, :])

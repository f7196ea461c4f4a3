"""Seeded random shapes, BF16 and FP32, against the FP64 oracle.

Twenty-four shapes drawn once from a fixed seed: N from 1 to 777 (ragged
tails of every size modulo the 64- and 128-row tiles), d in {64, 128}, B and
H from 1 to 3, causal or not, softmax scale between 0.5/sqrt(d) and
1.5/sqrt(d), input standard deviation between 0.5 and 1.25 (logit standard
deviations from ~0.1 to ~2.3: the regime the stated BF16 tolerances are
quoted for, N(0,1) inputs at scale 1/sqrt(d), and around it).  Every head of
every output is compared with the
oracle at the stated tolerances (BF16: O max-abs 2e-2 and mean-abs 2e-3,
LSE max-abs 1e-3, dQ/dK/dV relative L2 1e-2; FP32 mode: relative 1e-5).  The
stabilised forward (beta = 2) must meet the same BF16 tolerances: it changes
only rounding.
"""
import numpy as np
import pytest

import oracle
from precision_numerics_gb300 import inputs
from precision_numerics_gb300.deviation import deviation

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _cases(n=24, seed=2026):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        N = int(rng.integers(1, 778))
        d = int(rng.choice([64, 128]))
        B, H = int(rng.integers(1, 4)), int(rng.integers(1, 4))
        causal = bool(rng.integers(0, 2))
        scale = float(rng.uniform(0.5, 1.5)) / np.sqrt(d)
        std = float(rng.uniform(0.5, 1.25))
        out.append((B, H, N, d, causal, round(scale, 4), round(std, 3)))
    return out


CASES = _cases()


@pytest.fixture(scope="module")
def A(cuda_device):
    from precision_numerics_gb300 import attn, build
    build.build()
    return attn


def _dev(x, dtype):
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _host(t):
    return t.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}N{}d{}{}s{}x{}".format(
    c[0], c[1], c[2], c[3], "c" if c[4] else "n", c[5], c[6]))
def test_random_shape_bf16(A, case):
    B, H, N, d, causal, scale, std = case
    x = inputs.random_qkv(100 + N, B, H, N, d, std=std)
    f = {k: inputs.bf16_bits_to_f32(v) for k, v in x.items()}
    o_ref, lse_ref = oracle.forward_bhnd(f["q"], f["k"], f["v"], scale, causal)
    g_ref = oracle.backward_bhnd(f["q"], f["k"], f["v"], f["do"], scale, causal)
    t = {k: _dev(v, "bf16") for k, v in x.items()}
    for fwd in (A.attn_fwd, lambda *a, **kw: A.attn_fwd_stable(*a, beta=2.0, **kw)):
        o, lse = fwd(t["q"], t["k"], t["v"], scale=scale, causal=causal)
        dq, dk, dv = A.attn_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], scale=scale,
                                causal=causal)
        A.attn_check_status()
        e = deviation(_host(o), o_ref)
        assert e["max_abs"] <= 2e-2 and e["mean_abs"] <= 2e-3, ("o", e)
        assert deviation(_host(lse), lse_ref)["max_abs"] <= 1e-3
        for name, g, r in (("dq", dq, g_ref[0]), ("dk", dk, g_ref[1]), ("dv", dv, g_ref[2])):
            e = deviation(_host(g), r)
            assert e["rel_l2"] <= 1e-2, (name, e)


@pytest.mark.parametrize("case", CASES[:8], ids=lambda c: "B{}H{}N{}d{}{}".format(
    c[0], c[1], c[2], c[3], "c" if c[4] else "n"))
def test_random_shape_fp32(A, case):
    B, H, N, d, causal, scale, std = case
    x = inputs.random_qkv(200 + N, B, H, N, d, dtype="fp32", std=std)
    o_ref, lse_ref = oracle.forward_bhnd(x["q"], x["k"], x["v"], scale, causal)
    g_ref = oracle.backward_bhnd(x["q"], x["k"], x["v"], x["do"], scale, causal)
    t = {k: _dev(v, "fp32") for k, v in x.items()}
    o, lse = A.attn_fwd(t["q"], t["k"], t["v"], scale=scale, causal=causal)
    dq, dk, dv = A.attn_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], scale=scale, causal=causal)
    A.attn_check_status()
    for name, g, r in (("o", o, o_ref), ("dq", dq, g_ref[0]), ("dk", dk, g_ref[1]),
                       ("dv", dv, g_ref[2])):
        err = _host(g) - r
        rms_err, rms_ref = float(np.sqrt(np.mean(err ** 2))), float(np.sqrt(np.mean(r ** 2)))
        assert rms_err <= 1e-5 * rms_ref + 1e-6, name
        assert np.abs(err).max() <= 1e-5 * np.abs(r).max() + 1e-6, name
    assert np.abs(_host(lse) - lse_ref).max() <= 1e-5 * max(1.0, float(np.abs(lse_ref).max()))


def _large_cases(n=8, seed=777):
    """Longer sequences and many heads: multi-round persistent item lists,
    several backward head groups, ragged tails beyond the first tiles."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        N = int(rng.integers(778, 3001))
        d = int(rng.choice([64, 128]))
        B, H = int(rng.integers(1, 5)), int(rng.integers(8, 49))
        causal = bool(rng.integers(0, 2))
        scale = float(rng.uniform(0.5, 1.5)) / np.sqrt(d)
        out.append((B, H, N, d, causal, round(scale, 4)))
    # two causal ones more (the draw above gives mostly full attention)
    out += [(2, 40, 2500, 64, True, 0.125), (3, 16, 3000, 128, True, 0.0884)]
    return out


@pytest.mark.parametrize("case", _large_cases(), ids=lambda c: "B{}H{}N{}d{}{}s{}".format(
    c[0], c[1], c[2], c[3], "c" if c[4] else "n", c[5]))
def test_random_large_shape_bf16_sampled_heads(A, case):
    """Every output finite; the first, a middle and the last (b, h) head against
    the oracle at the stated BF16 tolerances."""
    B, H, N, d, causal, scale = case
    x = inputs.random_qkv(300 + N, B, H, N, d)
    t = {k: _dev(v, "bf16") for k, v in x.items()}
    o, lse = A.attn_fwd(t["q"], t["k"], t["v"], scale=scale, causal=causal)
    dq, dk, dv = A.attn_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], scale=scale, causal=causal)
    A.attn_check_status()
    for name, g in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv)):
        assert bool(torch.isfinite(g.float()).all()), name
    bh = B * H
    flat = {k: v.reshape(bh, N, d) for k, v in x.items()}
    for h in sorted({0, bh // 2, bh - 1}):
        f = {k: inputs.bf16_bits_to_f32(v[h]) for k, v in flat.items()}
        o_ref, lse_ref = oracle.forward(f["q"], f["k"], f["v"], scale, causal)
        g_ref = oracle.backward(f["q"], f["k"], f["v"], f["do"], scale, causal)
        e = deviation(_host(o.reshape(bh, N, d)[h]), o_ref)
        assert e["max_abs"] <= 2e-2 and e["mean_abs"] <= 2e-3, (h, "o", e)
        assert deviation(_host(lse.reshape(bh, N)[h]), lse_ref)["max_abs"] <= 1e-3, h
        for name, g, r in (("dq", dq, g_ref[0]), ("dk", dk, g_ref[1]), ("dv", dv, g_ref[2])):
            e = deviation(_host(g.reshape(bh, N, d)[h]), r)
            assert e["rel_l2"] <= 1e-2, (h, name, e)

"""Pins of the FP64 oracle to facts other than itself (CPU only).

Each test ties the oracle to a closed form, an invariant of the definition,
a library routine, finite differences, a pure-Python brute force, or the
hand-derived worked example in tests/golden/two_key_example.txt.  The
mutation tests at the end plant plausible mistakes in a copy of the oracle
and check that the pins catch them.
"""
import math
import os

import numpy as np
import pytest

import oracle
from oracle import attention as A

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "two_key_example.txt")


def _rand(seed, *shape):
    return np.random.default_rng(seed).standard_normal(shape)


def _load_golden():
    cases, cur = [], None
    with open(GOLDEN) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            tok = line.split()
            if tok[0] == "case":
                cur = {"name": tok[1], "scale": float(tok[3]), "causal": bool(int(tok[5]))}
                cases.append(cur)
                continue
            rows, cols = int(tok[1]), int(tok[2])
            vals = [math.log(3.0) if t == "ln3" else float(t) for t in tok[3:]]
            assert len(vals) == rows * cols, line
            cur[tok[0]] = np.array(vals).reshape(rows, cols)
    return cases


# ---------------------------------------------------------------- worked example

@pytest.mark.parametrize("case", _load_golden(), ids=lambda c: c["name"])
def test_golden_two_key_example(case):
    o, lse = oracle.forward(case["q"], case["k"], case["v"], case["scale"], case["causal"])
    np.testing.assert_allclose(o, case["o"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, case["lse"].reshape(-1), rtol=0, atol=1e-12)
    dq, dk, dv = oracle.backward(case["q"], case["k"], case["v"], case["do"], case["scale"],
                                 case["causal"])
    np.testing.assert_allclose(dv, case["dv"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(dq, case["dq"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk, case["dk"], rtol=0, atol=1e-12)


# ---------------------------------------------------------------- closed forms / invariants

@pytest.mark.parametrize("causal", [False, True])
def test_rows_of_p_sum_to_one(causal):
    q, k = _rand(0, 37, 16), _rand(1, 37, 16)
    p, _, _ = oracle.probabilities(q, k, 0.25, causal)
    assert np.all(p >= 0)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    if causal:
        assert np.all(np.triu(p, k=1) == 0)


def test_single_key_closed_form():
    q, k, v = _rand(2, 1, 8), _rand(3, 1, 8), _rand(4, 1, 8)
    for causal in (False, True):
        o, lse = oracle.forward(q, k, v, 0.3, causal)
        np.testing.assert_allclose(o, v, rtol=0, atol=1e-15)
        np.testing.assert_allclose(lse, [0.3 * float(q[0] @ k[0])], rtol=1e-15, atol=0)


@pytest.mark.parametrize("causal", [False, True])
def test_constant_v_returns_that_row(causal):
    q, k = _rand(5, 19, 8), _rand(6, 19, 8)
    row = _rand(7, 8)
    v = np.tile(row, (19, 1))
    o, _ = oracle.forward(q, k, v, 0.7, causal)
    np.testing.assert_allclose(o, np.tile(row, (19, 1)), rtol=0, atol=1e-13)


def test_joint_key_value_permutation():
    q, k, v = _rand(8, 23, 8), _rand(9, 23, 8), _rand(10, 23, 8)
    perm = np.random.default_rng(11).permutation(23)
    o1, l1 = oracle.forward(q, k, v, 0.4, False)
    o2, l2 = oracle.forward(q, k[perm], v[perm], 0.4, False)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)


def test_causal_row0_and_prefixes():
    n = 17
    q, k, v = _rand(12, n, 8), _rand(13, n, 8), _rand(14, n, 8)
    o, lse = oracle.forward(q, k, v, 0.5, True)
    np.testing.assert_allclose(o[0], v[0], rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse[0], 0.5 * float(q[0] @ k[0]), rtol=1e-15)
    for i in (1, 5, 16):
        oi, li = oracle.forward(q[i:i + 1], k[:i + 1], v[:i + 1], 0.5, False)
        np.testing.assert_allclose(o[i], oi[0], rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[i], li[0], rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_uniform_keys_average_visible_values(causal):
    n = 11
    q, v = _rand(15, n, 4), _rand(16, n, 4)
    k = np.tile(_rand(17, 4), (n, 1))
    o, lse = oracle.forward(q, k, v, 1.0, causal)
    for i in range(n):
        vis = i + 1 if causal else n
        np.testing.assert_allclose(o[i], v[:vis].mean(axis=0), rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[i], float(q[i] @ k[0]) + math.log(vis), atol=1e-13)


def test_delta_identity():
    """sum_j P_ij dP_ij equals rowsum(dO o O)_i."""
    q, k, v, do = (_rand(s, 13, 8) for s in range(20, 24))
    p, _, _ = oracle.probabilities(q, k, 0.3, True)
    o = p @ v
    dp = do @ v.T
    np.testing.assert_allclose((p * dp).sum(axis=1), oracle.delta(do, o), rtol=1e-12, atol=1e-12)


def test_delta_from_supplied_o():
    """delta from a supplied O: with the exact O nothing changes; with O + E the
    gradients move by the closed form dS' - dS = -P o (rowsum(dO o E))."""
    n, d, scale = 9, 4, 0.7
    q, k, v, do = (_rand(24 + s, n, d) for s in range(4))
    for causal in (False, True):
        p, _, _ = oracle.probabilities(q, k, scale, causal)
        o = p @ v
        g0 = oracle.backward(q, k, v, do, scale, causal)
        g1 = oracle.backward(q, k, v, do, scale, causal, o_for_delta=o)
        for a, b in zip(g0, g1):
            np.testing.assert_allclose(a, b, rtol=0, atol=1e-14)
        e = 1e-3 * _rand(28, n, d)
        g2 = oracle.backward(q, k, v, do, scale, causal, o_for_delta=o + e)
        dds = -p * (do * e).sum(axis=1)[:, None]
        np.testing.assert_allclose(g2[0] - g0[0], scale * dds @ k, rtol=0, atol=1e-13)
        np.testing.assert_allclose(g2[1] - g0[1], scale * dds.T @ q, rtol=0, atol=1e-13)
        np.testing.assert_allclose(g2[2], g0[2], rtol=0, atol=0)


# ---------------------------------------------------------------- library routines

@pytest.mark.parametrize("causal", [False, True])
def test_lse_and_softmax_match_scipy(causal):
    from scipy.special import logsumexp, softmax
    q, k = _rand(30, 29, 16), _rand(31, 29, 16)
    s = q @ k.T * 0.2
    if causal:
        s = np.where(np.triu(np.ones_like(s, bool), 1), -np.inf, s)
    p, _, _ = oracle.probabilities(q, k, 0.2, causal)
    _, lse = oracle.forward(q, k, _rand(32, 29, 16), 0.2, causal)
    np.testing.assert_allclose(p, softmax(s, axis=1), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(lse, logsumexp(s, axis=1), rtol=1e-14, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n,d", [(1, 4), (7, 8), (33, 16)])
def test_matches_torch_fp64_sdpa_with_autograd(causal, n, d):
    torch = pytest.importorskip("torch")
    q, k, v, do = (_rand(40 + s, n, d) for s in range(4))
    scale = 1.0 / math.sqrt(d)
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    with torch.nn.attention.sdpa_kernel(torch.nn.attention.SDPBackend.MATH):
        to = torch.nn.functional.scaled_dot_product_attention(
            tq[None, None], tk[None, None], tv[None, None], is_causal=causal, scale=scale)[0, 0]
    to.backward(torch.tensor(do))
    o, _ = oracle.forward(q, k, v, scale, causal)
    dq, dk, dv = oracle.backward(q, k, v, do, scale, causal)
    np.testing.assert_allclose(o, to.detach().numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=1e-11, atol=1e-12)


def test_matches_torch_fp64_attention_on_random_small_problems():
    """Property sweep: random N (including 1), d (including 1), mask, scale and
    input amplitude (logits up to a few hundred, where an unstabilised softmax
    overflows); O and the gradients against PyTorch FP64 attention with
    autograd, LSE against torch.logsumexp of the masked scores."""
    torch = pytest.importorskip("torch")
    hyp = pytest.importorskip("hypothesis")
    st = hyp.strategies

    @hyp.settings(max_examples=60, deadline=None, derandomize=True)
    @hyp.given(n=st.integers(1, 20), d=st.integers(1, 9), causal=st.booleans(),
               scale=st.floats(0.01, 3.0), amp=st.floats(0.1, 8.0), seed=st.integers(0, 2 ** 16))
    def check(n, d, causal, scale, amp, seed):
        q, k, v, do = (amp * _rand(seed + s, n, d) for s in range(4))
        tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
        with torch.nn.attention.sdpa_kernel(torch.nn.attention.SDPBackend.MATH):
            to = torch.nn.functional.scaled_dot_product_attention(
                tq[None, None], tk[None, None], tv[None, None], is_causal=causal,
                scale=scale)[0, 0]
        to.backward(torch.tensor(do))
        s_t = scale * (torch.tensor(q) @ torch.tensor(k).T)
        if causal:
            s_t = s_t.masked_fill(torch.ones(n, n, dtype=torch.bool).triu(1), float("-inf"))
        o, lse = oracle.forward(q, k, v, scale, causal)
        dq, dk, dv = oracle.backward(q, k, v, do, scale, causal)
        tol = dict(rtol=1e-10, atol=1e-10 * (1 + amp ** 3))
        np.testing.assert_allclose(o, to.detach().numpy(), **tol)
        np.testing.assert_allclose(lse, torch.logsumexp(s_t, dim=1).numpy(), rtol=1e-12,
                                   atol=1e-12)
        for mine, ref in ((dq, tq.grad), (dk, tk.grad), (dv, tv.grad)):
            np.testing.assert_allclose(mine, ref.numpy(), **tol)

    check()


# ---------------------------------------------------------------- finite differences

@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_central_differences(causal):
    n, d, scale, h = 6, 4, 0.6, 1e-6
    q, k, v, do = (_rand(50 + s, n, d) for s in range(4))

    def loss(q_, k_, v_):
        return float((oracle.forward(q_, k_, v_, scale, causal)[0] * do).sum())

    grads = oracle.backward(q, k, v, do, scale, causal)
    for which, g in zip(range(3), grads):
        num = np.zeros_like(g)
        for idx in np.ndindex(*g.shape):
            args_p = [q.copy(), k.copy(), v.copy()]
            args_m = [q.copy(), k.copy(), v.copy()]
            args_p[which][idx] += h
            args_m[which][idx] -= h
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        np.testing.assert_allclose(g, num, rtol=1e-7, atol=1e-8)


# ---------------------------------------------------------------- brute force

def _brute_force(q, k, v, scale, causal):
    n_q, n_k, d = len(q), len(k), len(q[0])
    o, lse = [], []
    for i in range(n_q):
        vis = [j for j in range(n_k) if not (causal and j > i)]
        s = {j: scale * sum(q[i][t] * k[j][t] for t in range(d)) for j in vis}
        m = max(s.values())
        w = {j: math.exp(s[j] - m) for j in vis}
        z = sum(w.values())
        o.append([sum(w[j] * v[j][t] for j in vis) / z for t in range(len(v[0]))])
        lse.append(m + math.log(z))
    return np.array(o), np.array(lse)


@pytest.mark.parametrize("causal", [False, True])
def test_brute_force_tiny(causal):
    for seed in range(3):
        q, k, v = (_rand(60 + 3 * seed + s, 5, 3) for s in range(3))
        o, lse = oracle.forward(q, k, v, 0.9, causal)
        ob, lb = _brute_force(q.tolist(), k.tolist(), v.tolist(), 0.9, causal)
        np.testing.assert_allclose(o, ob, rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(lse, lb, rtol=1e-13, atol=1e-14)


def test_bhnd_wrappers_match_per_head():
    q, k, v, do = (_rand(70 + s, 2, 3, 9, 4) for s in range(4))
    o, lse = oracle.forward_bhnd(q, k, v, 0.5, True)
    dq, dk, dv = oracle.backward_bhnd(q, k, v, do, 0.5, True)
    for b in range(2):
        for h in range(3):
            oh, lh = oracle.forward(q[b, h], k[b, h], v[b, h], 0.5, True)
            gh = oracle.backward(q[b, h], k[b, h], v[b, h], do[b, h], 0.5, True)
            np.testing.assert_array_equal(o[b, h], oh)
            np.testing.assert_array_equal(lse[b, h], lh)
            for x, y in zip((dq, dk, dv), gh):
                np.testing.assert_array_equal(x[b, h], y)


# ---------------------------------------------------------------- naive BF16 comparator

def test_round_bf16_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(80)
    x = np.concatenate([rng.standard_normal(20000).astype(np.float32) * 7,
                        np.array([0.0, -0.0, 1.0, 1.00390625, 1.005859375, 65504.0, 3.0e38,
                                  1e-40, -1e-40], np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(oracle.round_bf16(x), ref)


def test_naive_bf16_exact_on_representable_case():
    """Scores of 0 and uniform V rows: every rounding is exact, so the result is."""
    n, d = 8, 4
    q = np.zeros((n, d), np.float32)
    k = np.ones((n, d), np.float32)
    v = np.tile(np.array([0.5, -2.0, 3.0, 1.25], np.float32), (n, 1))
    o, lse = oracle.naive_bf16_forward(q, k, v, 0.125, False)
    np.testing.assert_array_equal(o, v)
    np.testing.assert_allclose(lse, math.log(n), rtol=1e-6)


@pytest.mark.parametrize("causal", [False, True])
def test_naive_bf16_within_bf16_error_of_exact(causal):
    n, d = 64, 32
    q, k, v, do = (oracle.round_bf16(_rand(90 + s, n, d).astype(np.float32)) for s in range(4))
    scale = 1 / math.sqrt(d)
    o, lse = oracle.forward(q, k, v, scale, causal)
    ob, lb = oracle.naive_bf16_forward(q, k, v, scale, causal)
    assert np.abs(ob - o).max() < 0.05
    assert np.abs(lb - lse).max() < 0.05
    g = oracle.backward(q, k, v, do, scale, causal)
    gb = oracle.naive_bf16_backward(q, k, v, do, scale, causal)
    for x, y in zip(g, gb):
        assert np.linalg.norm(y - x) / np.linalg.norm(x) < 0.03


def _eager_bf16_autograd(q, k, v, do, scale, causal):
    """The same attention run by an eager framework: PyTorch on the CPU on
    BF16 tensors (each op returns a BF16 tensor), differentiated by autograd."""
    torch = pytest.importorskip("torch")

    def leaf(x):
        return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).requires_grad_(True)

    qt, kt, vt = leaf(q), leaf(k), leaf(v)
    s = (qt @ kt.T) * scale
    if causal:
        hidden = torch.ones(s.shape, dtype=torch.bool).triu(1)
        s = s.masked_fill(hidden, float("-inf"))
    o = torch.softmax(s, -1) @ vt
    o.backward(torch.from_numpy(np.asarray(do, np.float32)).to(torch.bfloat16))
    return tuple(x.detach().float().numpy() for x in (o, qt.grad, kt.grad, vt.grad))


def _naive_forward_p_unrounded(q, k, v, scale, causal):
    """A plausible slip: probabilities kept in FP32 (no BF16 tensor between
    the softmax and P V)."""
    q, k, v = (np.asarray(x, np.float32) for x in (q, k, v))
    s = oracle.round_bf16(oracle.round_bf16(q @ k.T) * np.float32(scale))
    if causal:
        s = np.where(np.triu(np.ones(s.shape, bool), 1), np.float32(-np.inf), s)
    e = np.exp(s - s.max(axis=1, keepdims=True), dtype=np.float32)
    return oracle.round_bf16((e / e.sum(axis=1, keepdims=True, dtype=np.float32)) @ v)


def _naive_backward_scale_folded(q, k, v, do, scale, causal):
    """A plausible slip: the softmax scale folded into dS before its BF16
    rounding (one rounding where the eager graph has two)."""
    q, k, v, do = (np.asarray(x, np.float32) for x in (q, k, v, do))
    s = oracle.round_bf16(oracle.round_bf16(q @ k.T) * np.float32(scale))
    if causal:
        s = np.where(np.triu(np.ones(s.shape, bool), 1), np.float32(-np.inf), s)
    e = np.exp(s - s.max(axis=1, keepdims=True), dtype=np.float32)
    p = oracle.round_bf16(e / e.sum(axis=1, keepdims=True, dtype=np.float32))
    dp = oracle.round_bf16(do @ v.T)
    ds = oracle.round_bf16(np.float32(scale) * p *
                           (dp - (dp * p).sum(axis=1, keepdims=True, dtype=np.float32)))
    return oracle.round_bf16(ds @ k), oracle.round_bf16(ds.T @ q)


# (n, d, causal): d = 32 and 128 give softmax scales 1/sqrt(d) that are not
# powers of two, so every BF16 rounding of a scaled tensor is visible (with
# d = 64 the scale 1/8 is exact and two roundings in a row equal one).
EAGER_CASES = [(96, 32, True), (128, 128, False)]


@pytest.mark.parametrize("n,d,causal", EAGER_CASES)
def test_naive_bf16_rounding_matches_eager_bf16_autograd(n, d, causal):
    """Pins where the naive comparator rounds: an eager framework's BF16
    graph (PyTorch CPU ops and autograd) gives the same BF16 values.  Not
    every element can agree bit for bit (the two sum in different orders and
    use different exp routines, which can move a value across a BF16
    rounding boundary), so the pin is that at least 99% do, against 36-62%
    when one rounding is dropped or merged (see the planted slips below)."""
    q, k, v, do = (oracle.round_bf16(_rand(700 + s, n, d).astype(np.float32)) for s in range(4))
    scale = 1 / math.sqrt(d)
    o, _ = oracle.naive_bf16_forward(q, k, v, scale, causal)
    dq, dk, dv = oracle.naive_bf16_backward(q, k, v, do, scale, causal)
    eo, edq, edk, edv = _eager_bf16_autograd(q, k, v, do, scale, causal)
    for name, x, y in (("o", o, eo), ("dq", dq, edq), ("dk", dk, edk), ("dv", dv, edv)):
        assert np.mean(x == y) >= 0.99, name
        assert np.abs(x - y).max() <= 2 ** -6 * np.abs(y).max(), name


@pytest.mark.parametrize("n,d,causal", EAGER_CASES)
def test_eager_pin_catches_misplaced_roundings(n, d, causal):
    q, k, v, do = (oracle.round_bf16(_rand(700 + s, n, d).astype(np.float32)) for s in range(4))
    scale = 1 / math.sqrt(d)
    eo, edq, edk, _ = _eager_bf16_autograd(q, k, v, do, scale, causal)
    assert np.mean(_naive_forward_p_unrounded(q, k, v, scale, causal) == eo) < 0.9
    dq_bad, dk_bad = _naive_backward_scale_folded(q, k, v, do, scale, causal)
    assert np.mean(dq_bad == edq) < 0.9
    assert np.mean(dk_bad == edk) < 0.9


# ---------------------------------------------------------------- planted mistakes

def _forward_missing_max(q, k, v, scale, causal):
    """A plausible slip: LSE without the row max added back."""
    p, m, l = A.probabilities(q, k, scale, causal)
    return p @ np.asarray(v, float), np.log(l)


def _backward_unscaled_dk(q, k, v, do, scale, causal):
    """A plausible slip: dK without the softmax scale."""
    dq, dk, dv = A.backward(q, k, v, do, scale, causal)
    return dq, dk / scale, dv


def _backward_transposed_ds(q, k, v, do, scale, causal):
    """A plausible slip: dS^T where dS belongs (dQ from the wrong side)."""
    q, k, v, do = (np.asarray(x, float) for x in (q, k, v, do))
    p, _, _ = A.probabilities(q, k, scale, causal)
    o = p @ v
    ds = p * (do @ v.T - A.delta(do, o)[:, None])
    return scale * (ds.T @ k), scale * (ds.T @ q), p.T @ do


def test_planted_mistakes_are_caught():
    case = [c for c in _load_golden() if c["name"] == "noncausal_scale_half"][0]
    args = (case["q"], case["k"], case["v"])
    _, lse_bad = _forward_missing_max(*args, case["scale"], case["causal"])
    assert not np.allclose(lse_bad, case["lse"].reshape(-1), atol=1e-6)
    _, dk_bad, _ = _backward_unscaled_dk(*args, case["do"], case["scale"], case["causal"])
    assert not np.allclose(dk_bad, case["dk"], atol=1e-6)
    dq_bad, _, _ = _backward_transposed_ds(*args, case["do"], case["scale"], case["causal"])
    assert not np.allclose(dq_bad, case["dq"], atol=1e-6)

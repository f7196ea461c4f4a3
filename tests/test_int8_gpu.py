"""INT8-input forward on the GPU against the INT8 oracle (oracle/int8.py).

The quantization is integer work decided in FP32 on both sides, so codes and
scales must match bit for bit.  The forward is compared with the oracle's
forward on the same INT8 Q, K and BF16 V at the BF16 tolerances (O max-abs
2e-2 and mean-abs 2e-3, LSE max-abs 1e-3): the scores are exact integer dot
products times FP32 scales on both sides, and P is rounded to BF16 for P V
as in the BF16 kernel.
"""
import os

import numpy as np
import pytest

from oracle import int8 as oi
from precision_numerics_gb300 import inputs
from precision_numerics_gb300.deviation import deviation

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "int8_quant_example.txt")


@pytest.fixture(scope="module")
def A(cuda_device):
    from precision_numerics_gb300 import attn, build
    build.build()
    return attn


def _bf16_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


@pytest.mark.parametrize("shape", [(1, 1, 5, 64), (2, 3, 129, 128), (1, 2, 1000, 64)])
def test_quantize_matches_oracle_bit_for_bit(A, shape):
    x = inputs.random_qkv(21, *shape)["q"]
    x.reshape(-1, shape[-1])[1] = 0  # a zero row
    codes, scales = A.attn_quantize_int8(_bf16_dev(x))
    f = inputs.bf16_bits_to_f32(x).reshape(-1, shape[-1])
    c_ref, s_ref = oi.quantize_per_token(f)
    assert np.array_equal(codes.cpu().numpy().reshape(c_ref.shape), c_ref)
    assert np.array_equal(scales.cpu().numpy().reshape(-1).view(np.uint32), s_ref.view(np.uint32))


def test_quantize_golden_rows_with_ties(A):
    rows = []
    for line in open(GOLDEN):
        if line.startswith("x "):
            rows.append([float(v) for v in line.split()[1:]])
    x = np.zeros((1, 1, len(rows), 64), np.float32)
    x[0, 0, :, :8] = rows
    bits = inputs.f32_to_bf16_bits(x)
    assert np.array_equal(inputs.bf16_bits_to_f32(bits), x)  # the golden values are exact in BF16
    codes, scales = A.attn_quantize_int8(_bf16_dev(bits))
    c_ref, s_ref = oi.quantize_per_token(x[0, 0])
    assert np.array_equal(codes.cpu().numpy()[0, 0], c_ref)
    assert np.array_equal(scales.cpu().numpy()[0, 0], s_ref)


def _check_int8_forward(A, x, B, H, N, d, scale, causal, heads=None):
    t = {k: _bf16_dev(v) for k, v in x.items()}
    q8, qs = A.attn_quantize_int8(t["q"])
    k8, ks = A.attn_quantize_int8(t["k"])
    o, lse = A.attn_fwd_int8(q8, qs, k8, ks, t["v"], scale=scale, causal=causal)
    A.attn_check_status()
    assert bool(torch.isfinite(o.float()).all())
    f = {k: inputs.bf16_bits_to_f32(v).reshape(B * H, N, d) for k, v in x.items()}
    o = o.float().cpu().numpy().reshape(B * H, N, d)
    lse = lse.cpu().numpy().reshape(B * H, N)
    for h in (range(B * H) if heads is None else heads):
        o_ref, lse_ref = oi.int8_forward(f["q"][h], f["k"][h], f["v"][h], scale, causal)
        e = deviation(o[h], o_ref)
        assert e["max_abs"] <= 2e-2 and e["mean_abs"] <= 2e-3, (h, e)
        assert deviation(lse[h], lse_ref)["max_abs"] <= 1e-3, h


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(1, 1, 1, 64), (1, 2, 64, 128), (2, 1, 129, 64),
                                   (1, 2, 333, 128), (1, 1, 1024, 64), (1, 1, 700, 128)])
def test_int8_forward_matches_oracle(A, shape, causal):
    B, H, N, d = shape
    x = inputs.random_qkv(31, B, H, N, d)
    _check_int8_forward(A, x, B, H, N, d, d ** -0.5, causal)


def test_int8_forward_llama7b_shape(A):
    w = inputs.WORKLOADS["llama7b"]
    x = inputs.make_inputs(w, seed=0)
    _check_int8_forward(A, x, w.B, w.H, w.N, w.d, w.scale, w.causal, heads=[0, w.B * w.H - 1])


def test_int8_inputs_reject_wrong_dtype(A):
    v = torch.zeros(1, 1, 64, 64, dtype=torch.bfloat16, device="cuda")
    s = torch.zeros(1, 1, 64, dtype=torch.float32, device="cuda")
    with pytest.raises(ValueError):
        A.attn_fwd_int8(v, s, v, s, v)  # BF16 where INT8 codes are expected


# ---------------------------------------------------------------------------
# INT8 codes held in BF16: attn_quantize_int8_as_bf16 / attn_fwd_int8_as_bf16
# (the tcgen05 path).  The codes are the same integers, so they must equal the
# int8 codes exactly; the forward meets the same tolerances against the same
# INT8 oracle.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("shape", [(1, 1, 5, 64), (2, 3, 129, 128), (1, 2, 1000, 64)])
def test_quantize_as_bf16_equals_int8_codes(A, shape):
    B, H, N, d = shape
    x = inputs.random_qkv(23, *shape)["q"]
    x.reshape(-1, d)[2] = 0  # a zero row
    xd = _bf16_dev(x)
    c8, s8 = A.attn_quantize_int8(xd)
    cb, sb = A.attn_quantize_int8_as_bf16(xd)
    assert torch.equal(cb.float(), c8.float())
    n_pad = A.int8_scale_rows(N)
    assert sb.shape == (B, H, n_pad)
    assert torch.equal(sb[:, :, :N], s8)
    assert bool((sb[:, :, N:] == 0).all())


def _check_int8_as_bf16_forward(A, x, B, H, N, d, scale, causal, heads=None):
    t = {k: _bf16_dev(v) for k, v in x.items()}
    qc, qs = A.attn_quantize_int8_as_bf16(t["q"])
    kc, ks = A.attn_quantize_int8_as_bf16(t["k"])
    o, lse = A.attn_fwd_int8_as_bf16(qc, qs, kc, ks, t["v"], scale=scale, causal=causal)
    A.attn_check_status()
    assert bool(torch.isfinite(o.float()).all())
    f = {k: inputs.bf16_bits_to_f32(v).reshape(B * H, N, d) for k, v in x.items()}
    o = o.float().cpu().numpy().reshape(B * H, N, d)
    lse = lse.cpu().numpy().reshape(B * H, N)
    for h in (range(B * H) if heads is None else heads):
        o_ref, lse_ref = oi.int8_forward(f["q"][h], f["k"][h], f["v"][h], scale, causal)
        e = deviation(o[h], o_ref)
        assert e["max_abs"] <= 2e-2 and e["mean_abs"] <= 2e-3, (h, e)
        assert deviation(lse[h], lse_ref)["max_abs"] <= 1e-3, h


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(1, 1, 1, 64), (1, 2, 64, 128), (2, 1, 129, 64),
                                   (1, 2, 333, 128), (1, 1, 1024, 64), (1, 1, 700, 128)])
def test_int8_as_bf16_forward_matches_oracle(A, shape, causal):
    B, H, N, d = shape
    x = inputs.random_qkv(31, B, H, N, d)
    _check_int8_as_bf16_forward(A, x, B, H, N, d, d ** -0.5, causal)


def test_int8_as_bf16_forward_zero_query_row(A):
    """A row of zero codes scores 0 against every key: uniform weights over the visible keys."""
    B, H, N, d = 1, 1, 200, 64
    x = inputs.random_qkv(33, B, H, N, d)
    x["q"][0, 0, 150] = 0
    _check_int8_as_bf16_forward(A, x, B, H, N, d, d ** -0.5, True)


def test_int8_as_bf16_forward_llama7b_shape(A):
    w = inputs.WORKLOADS["llama7b"]
    x = inputs.make_inputs(w, seed=0)
    _check_int8_as_bf16_forward(A, x, w.B, w.H, w.N, w.d, w.scale, w.causal,
                                heads=[0, w.B * w.H - 1])


def test_int8_as_bf16_rejects_unpadded_scales(A):
    c = torch.zeros(1, 1, 64, 64, dtype=torch.bfloat16, device="cuda")
    s = torch.zeros(1, 1, 64, dtype=torch.float32, device="cuda")  # [B, H, N], not [B, H, N_pad]
    with pytest.raises(ValueError):
        A.attn_fwd_int8_as_bf16(c, s, c, s, c)


def test_both_int8_paths_reproduce_the_hand_derived_forward(A):
    """tests/golden/int8_forward_example.txt (distinct, non-unit scales on Q and
    K, two ties at .5) padded with zero columns to d = 64: padding changes no
    row maximum, no code and no dot product, so codes, scales, O and LSE are
    the hand-derived ones."""
    g = {}
    for line in open(os.path.join(os.path.dirname(__file__), "golden", "int8_forward_example.txt")):
        if line.strip() and not line.startswith("#"):
            name, r, c, *vals = line.split()
            g[name] = np.array([float(v) for v in vals]).reshape(int(r), int(c))
    scale = float(g["scale"][0, 0])
    t = {}
    for n in ("q", "k", "v"):
        x = np.zeros((1, 1, 2, 64), np.float32)
        x[0, 0, :, :2] = g[n]
        bits = inputs.f32_to_bf16_bits(x)
        assert np.array_equal(inputs.bf16_bits_to_f32(bits), x)  # exact in BF16
        t[n] = _bf16_dev(bits)
    q8, qs = A.attn_quantize_int8(t["q"])
    k8, ks = A.attn_quantize_int8(t["k"])
    assert np.array_equal(q8.cpu().numpy()[0, 0, :, :2], g["q_codes"].astype(np.int8))
    assert np.array_equal(k8.cpu().numpy()[0, 0, :, :2], g["k_codes"].astype(np.int8))
    assert np.array_equal(qs.cpu().numpy().reshape(-1), g["q_scale"].reshape(-1))
    assert np.array_equal(ks.cpu().numpy().reshape(-1), g["k_scale"].reshape(-1))
    qc, qsp = A.attn_quantize_int8_as_bf16(t["q"])
    kc, ksp = A.attn_quantize_int8_as_bf16(t["k"])
    outs = [A.attn_fwd_int8(q8, qs, k8, ks, t["v"], scale=scale, causal=False),
            A.attn_fwd_int8_as_bf16(qc, qsp, kc, ksp, t["v"], scale=scale, causal=False)]
    A.attn_check_status()
    for o, lse in outs:
        o = o.float().cpu().numpy()[0, 0, :, :2]
        # BF16 output and BF16 P in P V: within 2^-8 relative of the exact O
        assert np.all(np.abs(o - g["o"]) <= 2 ** -7 * np.abs(g["o"]) + 1e-6), o
        assert np.abs(lse.cpu().numpy().reshape(-1) - g["lse"].reshape(-1)).max() <= 1e-5

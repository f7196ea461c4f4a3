"""GPU tests that need the test build of the library (libattn_testhooks.so).

The test build compiles the same sources with test-only instrumentation
(precision_numerics_gb300.build.TEST_FLAGS): a per-row counter of the BF16
P-bar operands equal to 1.0 in the forward kernel, a switch that makes one
softmax warpgroup wait on a barrier nothing arrives at, and a 50 ms limit on
every in-kernel wait.  libattn.so never contains any of it.

1. The stabilised normaliser ("Why Low-Precision Transformer Training
   Fails", Figure 7 and Algorithm 1) exists so that no element of P-bar is
   exactly 1 in a row whose maximum repeats; the pages require the largest
   exponent to be "sufficiently negative".  Counted on the P V operands the
   kernel actually uses (after rounding to BF16): zero for the stabilised
   forward on inputs where every row's maximum is attained at least twice,
   including maxima of 0, of tiny size and of either sign; at least two per
   row for the plain forward.
2. The real kernels' failure path: a wait that runs out must make the
   kernel wind down (copies and MMAs in flight completed, TMEM freed),
   attn_check_status must report ATTN_ERR_TIMEOUT, and the next call must
   again match the oracle.  Covered for the forward kernel and for both
   backward main kernels (the d = 128 one and the persistent d = 64 one),
   each with one P/dS warpgroup of CTA 0 held on a barrier nothing arrives at.
"""
import ctypes
import math

import numpy as np
import pytest

import oracle
from precision_numerics_gb300 import inputs
from precision_numerics_gb300.deviation import deviation

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def T(cuda_device):
    from precision_numerics_gb300 import attn, build
    lib = attn.load_library(build.build_test_variant())
    lib.attn_testhook_pbar_counter.restype = ctypes.c_int
    lib.attn_testhook_pbar_counter.argtypes = [ctypes.c_void_p, ctypes.c_ulonglong]
    lib.attn_testhook_stall.restype = ctypes.c_int
    lib.attn_testhook_stall.argtypes = [ctypes.c_int]
    lib.attn_testhook_stall_bwd.restype = ctypes.c_int
    lib.attn_testhook_stall_bwd.argtypes = [ctypes.c_int]
    yield lib
    lib.attn_testhook_pbar_counter(None, 0)
    lib.attn_testhook_stall(0)
    lib.attn_testhook_stall_bwd(0)


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _fwd(T, q, k, v, scale, causal, beta=None):
    B, H, N, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if beta is None:
        r = T.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                       B, H, N, d, ctypes.c_float(scale), int(causal), 0, _stream())
    else:
        r = T.attn_fwd_stable(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                              lse.data_ptr(), B, H, N, d, ctypes.c_float(scale), int(causal),
                              ctypes.c_float(beta), 0, _stream())
    assert r == 0, T.attn_last_error()
    return o, lse


def _count_ones(T, q, k, v, scale, causal, beta):
    B, H, N, _ = q.shape
    counts = torch.zeros(B * H * N, dtype=torch.int32, device=q.device)
    assert T.attn_testhook_pbar_counter(counts.data_ptr(), counts.numel()) == 0
    o, lse = _fwd(T, q, k, v, scale, causal, beta)
    assert T.attn_check_status(_stream()) == 0, T.attn_last_error()
    assert T.attn_testhook_pbar_counter(None, 0) == 0
    return counts.cpu().numpy().reshape(B * H, N), o, lse


def _paired_axis_case(d=64, N=256):
    """Two heads whose keys are multiples of one unit vector, in equal pairs.

    Head 0: key coefficients of both signs; head 1: all negative.  Query rows
    are multiples of the same vector (0, +-2^-12, +-2^-8, ..., +-8), so every
    row's scores are scale * b_i * a_j and the row maximum is attained by a
    pair of equal keys: r_m = 0 for b = 0, tiny and of either sign for tiny b.
    """
    rng = np.random.default_rng(5)
    a0 = rng.uniform(-1.0, 1.0, N // 2)
    a1 = rng.uniform(-1.0, -0.01, N // 2)
    bs = [0.0] + [s * 2.0 ** e for e in (-12, -10, -8, -6, -4, -2, 0, 2, 3) for s in (1, -1)]
    b = np.resize(np.array(bs), N)
    q = np.zeros((1, 2, N, d), np.float32)
    k = np.zeros((1, 2, N, d), np.float32)
    q[0, :, :, 0] = b
    k[0, 0, :, 0] = np.repeat(a0, 2)
    k[0, 1, :, 0] = np.repeat(a1, 2)
    v = inputs.normal(5, inputs.STREAM_V, (1, 2, N, d))
    return {n: inputs.f32_to_bf16_bits(x) for n, x in (("q", q), ("k", k), ("v", v))}


def _tied_lowrank_case(sigma, N=512, d=128):
    w = inputs.Workload("ties", 1, 2, N, d, False, 1.0 / math.sqrt(d), lowrank_rank=4,
                        sigmas=(sigma,), tied_keys=True)
    return inputs.make_inputs(w, seed=0, sigma=sigma), w.scale


def _cases():
    for sigma in (1.0, 4.0, 16.0):
        yield f"ties_sigma{sigma:g}", *_tied_lowrank_case(sigma)
    yield "paired_axis", _paired_axis_case(), 0.125


@pytest.mark.parametrize("beta", [1.05, 2.0])
def test_stabilised_forward_leaves_no_pbar_equal_to_one(T, beta):
    for name, x, scale in _cases():
        t = {n: _dev(x[n]) for n in ("q", "k", "v")}
        ones_plain, _, _ = _count_ones(T, t["q"], t["k"], t["v"], scale, False, None)
        ones_stable, o, lse = _count_ones(T, t["q"], t["k"], t["v"], scale, False, beta)
        # every row's maximum repeats: the plain kernel rounds at least two
        # P-bar operands of each row to exactly 1, the stabilised one none
        assert ones_plain.min() >= 2, (name, int(ones_plain.min()))
        assert ones_stable.max() == 0, (name, int(ones_stable.max()),
                                        np.argwhere(ones_stable > 0)[:5].tolist())
        # and the outputs are still the attention of the definition
        f = {n: inputs.bf16_bits_to_f32(x[n]).reshape(-1, *x[n].shape[2:]) for n in ("q", "k", "v")}
        og = o.float().cpu().numpy().reshape(f["q"].shape)
        lg = lse.cpu().numpy().reshape(f["q"].shape[:2])
        for h in range(f["q"].shape[0]):
            o_ref, lse_ref = oracle.forward(f["q"][h], f["k"][h], f["v"][h], scale, False)
            dev = deviation(og[h], o_ref)
            assert dev["max_abs"] <= 2e-2 and dev["mean_abs"] <= 2e-3, (name, h, dev)
            assert np.abs(lg[h] - lse_ref).max() <= 1e-3, (name, h)


def test_forced_wait_timeout_winds_down_and_the_next_call_is_exact(T):
    B, H, N, d = 1, 4, 1024, 128
    scale = d ** -0.5
    x = inputs.random_qkv(31, B, H, N, d)
    t = {n: _dev(v) for n, v in x.items()}
    assert T.attn_check_status(_stream()) == 0
    assert T.attn_testhook_stall(1) == 0
    try:
        _fwd(T, t["q"], t["k"], t["v"], scale, True)
        # the kernel returned (no hang, no fault) and recorded the timeout
        assert T.attn_check_status(_stream()) == 4, T.attn_last_error()
    finally:
        assert T.attn_testhook_stall(0) == 0
    assert T.attn_check_status(_stream()) == 0  # the status word was cleared
    o, lse = _fwd(T, t["q"], t["k"], t["v"], scale, True)
    assert T.attn_check_status(_stream()) == 0, T.attn_last_error()
    f = {n: inputs.bf16_bits_to_f32(v).reshape(B * H, N, d) for n, v in x.items()}
    og = o.float().cpu().numpy().reshape(B * H, N, d)
    lg = lse.cpu().numpy().reshape(B * H, N)
    for h in range(B * H):
        o_ref, lse_ref = oracle.forward(f["q"][h], f["k"][h], f["v"][h], scale, True)
        dev = deviation(og[h], o_ref)
        assert dev["max_abs"] <= 2e-2 and dev["mean_abs"] <= 2e-3, (h, dev)
        assert np.abs(lg[h] - lse_ref).max() <= 1e-3, h


def _bwd(T, t, o, lse, scale, causal):
    B, H, N, d = t["q"].shape
    out = [torch.full_like(o, float("nan")) for _ in range(3)]
    ws = torch.empty(int(T.attn_bwd_workspace_bytes(B, H, N, d, 0)), dtype=torch.uint8,
                     device=o.device)
    r = T.attn_bwd(t["q"].data_ptr(), t["k"].data_ptr(), t["v"].data_ptr(), o.data_ptr(),
                   lse.data_ptr(), t["do"].data_ptr(), out[0].data_ptr(), out[1].data_ptr(),
                   out[2].data_ptr(), B, H, N, d, ctypes.c_float(scale), int(causal), 0,
                   ws.data_ptr(), ws.numel(), _stream())
    assert r == 0, T.attn_last_error()
    return out


def _rel_l2(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


@pytest.mark.parametrize("d,causal", [(128, True), (64, False)], ids=["d128_causal", "d64_full"])
def test_forced_backward_wait_timeout_winds_down_and_the_next_call_is_exact(T, d, causal):
    # d = 128 runs the one-item-per-CTA backward main kernel, d = 64 the
    # persistent one; both take the same failure path from the held warpgroup.
    from precision_numerics_gb300 import attn
    B, H, N = 1, 4, 1024
    scale = d ** -0.5
    x = inputs.random_qkv(33 + d, B, H, N, d)
    t = {n: _dev(v) for n, v in x.items()}
    o, lse = attn.attn_fwd(t["q"], t["k"], t["v"], scale=scale, causal=causal)
    assert T.attn_check_status(_stream()) == 0
    assert T.attn_testhook_stall_bwd(1) == 0
    try:
        _bwd(T, t, o, lse, scale, causal)
        # the kernel returned (no hang, no fault) and recorded the timeout
        assert T.attn_check_status(_stream()) == 4, T.attn_last_error()
    finally:
        assert T.attn_testhook_stall_bwd(0) == 0
    assert T.attn_check_status(_stream()) == 0  # the status word was cleared
    got = _bwd(T, t, o, lse, scale, causal)
    assert T.attn_check_status(_stream()) == 0, T.attn_last_error()
    og = o.float().cpu().numpy().reshape(B * H, N, d)
    g = [x_.float().cpu().numpy().reshape(B * H, N, d) for x_ in got]
    f = {n: inputs.bf16_bits_to_f32(v).reshape(B * H, N, d) for n, v in x.items()}
    for h in (0, B * H - 1):  # CTA 0's head and the last one
        ref = oracle.backward(f["q"][h], f["k"][h], f["v"][h], f["do"][h], scale, causal,
                              o_for_delta=og[h])
        for name, gv, rv in zip(("dq", "dk", "dv"), g, ref):
            assert np.isfinite(gv[h]).all(), (h, name)
            assert _rel_l2(gv[h], rv) <= 1e-2, (h, name, _rel_l2(gv[h], rv))

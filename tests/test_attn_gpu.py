"""Parity of the CUDA path (through the C ABI) with the FP64 oracle.

Tolerances: BF16 -- O max-abs 2e-2 and mean-abs 2e-3, LSE max-abs 1e-3,
dQ/dK/dV relative L2 1e-2; FP32 reference mode -- relative 1e-5 (RMS error
over RMS reference, max error over max |reference|, each with an absolute
floor of 1e-6 for exactly-zero results), LSE max-abs 1e-5 * max(1, |LSE|).
Inputs are the seeded generator's values; the oracle sees exactly the values
the GPU sees, widened to FP64.
"""
import math

import numpy as np
import pytest

import oracle
from precision_numerics_gb300 import inputs
from precision_numerics_gb300.deviation import deviation

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def A(cuda_device):
    from precision_numerics_gb300 import attn, build
    build.build()
    attn.load_library()
    return attn


def _dev(x, dtype):
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _host(t):
    return t.float().cpu().numpy().astype(np.float64)


def _widen(x, dtype):
    return inputs.bf16_bits_to_f32(x) if dtype == "bf16" else x


def _run(A, x, dtype, scale, causal, backward=True):
    t = {k: _dev(v, dtype) for k, v in x.items()}
    o, lse = A.attn_fwd(t["q"], t["k"], t["v"], scale=scale, causal=causal)
    out = {"o": o, "lse": lse}
    if backward:
        dq, dk, dv = A.attn_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], scale=scale, causal=causal)
        out.update(dq=dq, dk=dk, dv=dv)
    A.attn_check_status()
    return {k: _host(v) for k, v in out.items()}


def _oracle(x, dtype, scale, causal, backward=True):
    f = {k: _widen(v, dtype) for k, v in x.items()}
    o, lse = oracle.forward_bhnd(f["q"], f["k"], f["v"], scale, causal)
    ref = {"o": o, "lse": lse}
    if backward:
        ref["dq"], ref["dk"], ref["dv"] = oracle.backward_bhnd(f["q"], f["k"], f["v"], f["do"],
                                                              scale, causal)
    return ref


def _assert_bf16(got, ref, backward=True, tag=""):
    e = deviation(got["o"], ref["o"])
    assert e["max_abs"] <= 2e-2 and e["mean_abs"] <= 2e-3, (tag, "o", e)
    e = deviation(got["lse"], ref["lse"])
    assert e["max_abs"] <= 1e-3, (tag, "lse", e)
    if backward:
        for name in ("dq", "dk", "dv"):
            e = deviation(got[name], ref[name])
            assert e["rel_l2"] <= 1e-2, (tag, name, e)


def _assert_fp32(got, ref, backward=True, tag=""):
    # Relative 1e-5, with an absolute floor of 1e-6 (RMS and max) for results
    # whose exact value is 0 (e.g. dQ with a single key), where a relative
    # error is undefined.
    for name in ("o",) + (("dq", "dk", "dv") if backward else ()):
        err = got[name] - ref[name]
        rms_err = float(np.sqrt(np.mean(err ** 2)))
        rms_ref = float(np.sqrt(np.mean(ref[name] ** 2)))
        assert rms_err <= 1e-5 * rms_ref + 1e-6, (tag, name, deviation(got[name], ref[name]))
        assert np.abs(err).max() <= 1e-5 * np.abs(ref[name]).max() + 1e-6, (tag, name)
    lse_tol = 1e-5 * max(1.0, float(np.abs(ref["lse"]).max()))
    assert deviation(got["lse"], ref["lse"])["max_abs"] <= lse_tol, (tag, "lse")


SHAPES = [(1, 2, 128, 64), (1, 1, 1, 64), (1, 2, 17, 128), (2, 1, 129, 64), (1, 2, 256, 128),
          (1, 1, 300, 128), (2, 2, 511, 64), (1, 2, 640, 128)]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_fp32_reference_mode(A, shape, causal):
    B, H, N, d = shape
    x = inputs.random_qkv(1, B, H, N, d, dtype="fp32")
    scale = 1.0 / math.sqrt(d)
    _assert_fp32(_run(A, x, "fp32", scale, causal), _oracle(x, "fp32", scale, causal), tag=shape)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SHAPES + [(1, 1, 1000, 64), (1, 1, 1024, 128)],
                         ids=lambda s: "x".join(map(str, s)))
def test_bf16_forward_backward(A, shape, causal):
    B, H, N, d = shape
    x = inputs.random_qkv(2, B, H, N, d)
    scale = 1.0 / math.sqrt(d)
    _assert_bf16(_run(A, x, "bf16", scale, causal), _oracle(x, "bf16", scale, causal), tag=shape)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_small_workload_forward(A, dtype):
    """B1 H2 N128 d64 non-causal, scale 1/sqrt(d), FP32 and BF16 inputs."""
    w = inputs.WORKLOADS["small"]
    x = inputs.make_inputs(w, seed=0, dtype=dtype)
    got = _run(A, x, dtype, w.scale, w.causal, backward=False)
    ref = _oracle(x, dtype, w.scale, w.causal, backward=False)
    (_assert_fp32 if dtype == "fp32" else _assert_bf16)(got, ref, backward=False)


def test_single_key_closed_form(A):
    """N = 1: O = V[0] exactly (one key with weight 1)."""
    x = inputs.random_qkv(3, 2, 3, 1, 128)
    got = _run(A, x, "bf16", 0.1, False, backward=False)
    v = inputs.bf16_bits_to_f32(x["v"]).astype(np.float64)
    np.testing.assert_array_equal(got["o"], v)


def test_causal_row0_is_v0(A):
    x = inputs.random_qkv(4, 1, 2, 256, 64)
    got = _run(A, x, "bf16", 0.125, True, backward=False)
    v = inputs.bf16_bits_to_f32(x["v"]).astype(np.float64)
    np.testing.assert_array_equal(got["o"][:, :, 0], v[:, :, 0])


def test_forward_is_deterministic(A):
    x = inputs.random_qkv(5, 1, 4, 700, 128)
    t = {k: _dev(v, "bf16") for k, v in x.items()}
    o1, l1 = A.attn_fwd(t["q"], t["k"], t["v"], causal=True)
    o2, l2 = A.attn_fwd(t["q"], t["k"], t["v"], causal=True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("N,d,causal", [(300, 128, True), (300, 128, False), (1000, 128, True),
                                         (129, 128, True), (64, 128, False), (300, 64, True)])
def test_backward_phases_equal_attn_bwd(A, N, d, causal):
    """The exported phases (preprocess, main, dQ conversion) give attn_bwd's
    results.  dK and dV are bit-identical; dQ is summed with floating-point
    atomics across key tiles, whose order varies between runs, so it is
    compared with a tolerance."""
    B, H = 1, 2
    x = inputs.random_qkv(6, B, H, N, d)
    t = {k: _dev(v, "bf16") for k, v in x.items()}
    o, lse = A.attn_fwd(t["q"], t["k"], t["v"], causal=causal)
    dq, dk, dv = A.attn_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], causal=causal)
    ws = torch.empty(A.attn_bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device="cuda")
    dq2, dk2, dv2 = (torch.full_like(o, float("nan")) for _ in range(3))
    A.attn_bwd_preprocess(o, lse, t["do"], ws)
    A.attn_bwd_main(t["q"], t["k"], t["v"], t["do"], dk2, dv2, ws, causal=causal)
    A.attn_bwd_dq_convert(dq2, ws)
    A.attn_check_status()
    assert torch.equal(dk, dk2) and torch.equal(dv, dv2)
    assert bool(torch.isfinite(dq2.float()).all())
    assert (dq.float() - dq2.float()).abs().max().item() <= 2e-2 * dq.float().abs().max().item()


@pytest.mark.parametrize("N,d,causal", [(129, 128, True), (300, 64, False), (1, 128, False)])
def test_outputs_leave_guard_bands_untouched(A, N, d, causal):
    """Outputs sit inside larger buffers whose tails hold a sentinel (all-ones bits)."""
    B, H, guard = 1, 3, 4096
    x = inputs.random_qkv(7, B, H, N, d)
    t = {k: _dev(v, "bf16") for k, v in x.items()}
    n = B * H * N * d

    def guarded(numel, dtype):
        buf = torch.empty(numel + guard, dtype=dtype, device="cuda")
        buf.view(torch.int16 if dtype == torch.bfloat16 else torch.int32).fill_(-1)
        return buf

    ob, lb = guarded(n, torch.bfloat16), guarded(B * H * N, torch.float32)
    o = ob[:n].view(B, H, N, d)
    lse = lb[:B * H * N].view(B, H, N)
    A.attn_fwd(t["q"], t["k"], t["v"], causal=causal, o=o, lse=lse)
    gb = [guarded(n, torch.bfloat16) for _ in range(3)]
    A.attn_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], causal=causal,
               dq=gb[0][:n].view(B, H, N, d), dk=gb[1][:n].view(B, H, N, d),
               dv=gb[2][:n].view(B, H, N, d))
    A.attn_check_status()
    for buf in [ob, *gb]:
        assert bool((buf[n:].view(torch.int16) == -1).all())
    assert bool((lb[B * H * N:].view(torch.int32) == -1).all())
    assert bool(torch.isfinite(o.float()).all())


def test_bounded_wait_reports_timeout_and_context_survives(A):
    A.attn_check_status()
    A.attn_selftest_wait_timeout(2_000_000)  # 2 ms
    with pytest.raises(A.AttnError) as info:
        A.attn_check_status()
    assert info.value.status == A.ATTN_ERR_TIMEOUT
    A.attn_check_status()  # cleared
    x = inputs.random_qkv(8, 1, 1, 128, 64)
    got = _run(A, x, "bf16", 0.125, False, backward=False)
    _assert_bf16(got, _oracle(x, "bf16", 0.125, False, backward=False), backward=False)


def test_timeout_status_is_shared_by_all_streams(A):
    """The status words are per device, not per stream (include/attn.h at
    attn_check_status): a timeout recorded by a kernel on one stream is
    reported by a check on another stream, and that check clears it."""
    A.attn_check_status()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    A.attn_selftest_wait_timeout(1_000_000, stream=s1)
    s1.synchronize()
    with pytest.raises(A.AttnError) as info:
        A.attn_check_status(stream=s2)
    assert info.value.status == A.ATTN_ERR_TIMEOUT
    A.attn_check_status(stream=s1)  # already cleared by the check on s2


def test_rejects_host_memory(A):
    q = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16, device="cuda")
    lib = A.load_library()
    host = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16).pin_memory()
    lse = torch.empty(1, 1, 128, device="cuda")
    r = lib.attn_fwd(host.data_ptr(), q.data_ptr(), q.data_ptr(), q.data_ptr(), lse.data_ptr(),
                     1, 1, 128, 64, 0.125, 0, 0, None)
    assert r == A.ATTN_ERR_INVALID_ARG


# ---------------------------------------------------------------- stabilised forward

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(1, 2, 128, 64), (2, 1, 129, 128), (1, 2, 640, 128),
                                   (1, 1, 1000, 64)], ids=lambda s: "x".join(map(str, s)))
def test_stable_forward_matches_definition(A, shape, causal):
    """The stabilised normaliser changes only rounding: O and LSE are the
    definition's, and the backward from its LSE is the definition's gradient."""
    B, H, N, d = shape
    x = inputs.random_qkv(9, B, H, N, d)
    scale = 1.0 / math.sqrt(d)
    t = {k: _dev(v, "bf16") for k, v in x.items()}
    o, lse = A.attn_fwd_stable(t["q"], t["k"], t["v"], scale=scale, causal=causal, beta=2.0)
    dq, dk, dv = A.attn_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], scale=scale, causal=causal)
    A.attn_check_status()
    got = {k: _host(v) for k, v in dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv).items()}
    _assert_bf16(got, _oracle(x, "bf16", scale, causal), tag=shape)


@pytest.mark.parametrize("beta", [1.05, 2.0])
def test_stable_forward_on_exactly_repeated_maxima(A, beta):
    """Keys duplicated in pairs: every row max is attained twice, so the
    stabilised path normalises by beta * r_m (or 0) throughout."""
    w = inputs.Workload("ties", 1, 4, 512, 128, True, 1 / math.sqrt(128), lowrank_rank=4,
                        sigmas=(4.0,), tied_keys=True)
    x = inputs.make_inputs(w, seed=3, sigma=4.0)
    t = {k: _dev(v, "bf16") for k, v in x.items()}
    o, lse = A.attn_fwd_stable(t["q"], t["k"], t["v"], scale=w.scale, causal=True, beta=beta)
    o2, lse2 = A.attn_fwd(t["q"], t["k"], t["v"], scale=w.scale, causal=True)
    A.attn_check_status()
    ref = _oracle(x, "bf16", w.scale, True, backward=False)
    _assert_bf16({"o": _host(o), "lse": _host(lse)}, ref, backward=False)
    _assert_bf16({"o": _host(o2), "lse": _host(lse2)}, ref, backward=False)
    # The normaliser differs, so the two kernels round differently somewhere.
    assert not torch.equal(o, o2)


def test_stable_forward_caps_the_shift_for_huge_repeated_maxima(A):
    """Low-rank ties at sigma = 16: (beta - 1) * r_m far beyond the FP32 range;
    the capped normaliser keeps every row finite and exact to tolerance."""
    w = inputs.Workload("ties16", 1, 2, 512, 128, True, 1 / math.sqrt(128), lowrank_rank=4,
                        sigmas=(16.0,), tied_keys=True)
    x = inputs.make_inputs(w, seed=4, sigma=16.0)
    t = {k: _dev(v, "bf16") for k, v in x.items()}
    o, lse = A.attn_fwd_stable(t["q"], t["k"], t["v"], scale=w.scale, causal=True, beta=2.0)
    A.attn_check_status()
    assert bool(torch.isfinite(o.float()).all()) and bool(torch.isfinite(lse).all())
    _assert_bf16({"o": _host(o), "lse": _host(lse)}, _oracle(x, "bf16", w.scale, True, False),
                 backward=False)


@pytest.mark.parametrize("chunks,group_sizes,streams,graph",
                         [(1, None, 1, True), (3, None, 1, True), (3, None, 1, False),
                          (0, [1, 3, 1], 2, True), (0, [1, 3, 1], 1, True),
                          (0, [2, 3], 2, False)])
def test_host_pipeline_matches_device_path(A, chunks, group_sizes, streams, graph):
    """HostAttention (pinned host buffers, head groups pipelined over upload,
    compute and download streams, eagerly or as a replayed CUDA graph) gives
    the device path's results; run twice to exercise buffer and graph reuse."""
    from precision_numerics_gb300.host import HostAttention
    B, H, N, d = 1, 5, 300, 128
    x = inputs.random_qkv(10, B, H, N, d)
    host = {k: torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).pin_memory() for k, v in x.items()}
    t = {k: v.cuda() for k, v in host.items()}
    o, lse = A.attn_fwd(t["q"], t["k"], t["v"], causal=True)
    dq, dk, dv = A.attn_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], causal=True)
    pipe = HostAttention(B, H, N, d, causal=True, chunks=chunks or 4, group_sizes=group_sizes,
                         compute_streams=streams, graph=graph)
    for _ in range(2):
        ho, hl, hdq, hdk, hdv = pipe.run(host["q"], host["k"], host["v"], host["do"])
        torch.cuda.synchronize()
        A.attn_check_status()
        assert torch.equal(ho, o.cpu()) and torch.equal(hl, lse.cpu())
        assert torch.equal(hdk, dk.cpu()) and torch.equal(hdv, dv.cpu())
        rel = float((hdq.float() - dq.float().cpu()).norm() / dq.float().cpu().norm())
        assert rel <= 1e-2


def test_host_pipeline_rejects_bad_group_sizes(A):
    from precision_numerics_gb300.host import HostAttention
    with pytest.raises(ValueError):
        HostAttention(1, 4, 128, 64, group_sizes=[2, 1])
    with pytest.raises(ValueError):
        HostAttention(1, 4, 128, 64, group_sizes=[4, 0])


def test_host_pipeline_rejects_unpinned_or_misshaped_inputs(A):
    from precision_numerics_gb300.host import HostAttention
    pipe = HostAttention(1, 2, 128, 64, chunks=2)
    good = torch.zeros(1, 2, 128, 64, dtype=torch.bfloat16).pin_memory()
    with pytest.raises(ValueError):
        pipe.run(torch.zeros(1, 2, 128, 64, dtype=torch.bfloat16), good, good, good)
    with pytest.raises(ValueError):
        pipe.run(good.cuda(), good, good, good)
    with pytest.raises(ValueError):
        pipe.run(torch.zeros(1, 2, 64, 64, dtype=torch.bfloat16).pin_memory(), good, good, good)


def test_host_pipeline_graph_follows_new_input_buffers(A):
    """A graph-mode pipeline re-captures when it is handed other host tensors."""
    from precision_numerics_gb300.host import HostAttention
    B, H, N, d = 1, 2, 256, 64
    pipe = HostAttention(B, H, N, d, causal=False, chunks=2)
    outs = []
    for seed in (3, 4):
        x = inputs.random_qkv(seed, B, H, N, d)
        host = {k: torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).pin_memory()
                for k, v in x.items()}
        ho = pipe.run(host["q"], host["k"], host["v"], host["do"])[0]
        torch.cuda.synchronize()
        t = {k: v.cuda() for k, v in host.items()}
        o, _ = A.attn_fwd(t["q"], t["k"], t["v"], causal=False)
        assert torch.equal(ho, o.cpu())
        outs.append(ho.clone())
    assert not torch.equal(outs[0], outs[1])

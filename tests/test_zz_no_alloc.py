"""attn_bwd_noalloc: the backward for callers that must not allocate device memory.

Some callers cannot call cudaMalloc -- e.g. a component inside a host framework
that owns the whole device-memory budget, or a latency-critical loop that must
not pay for allocation and its implicit synchronization.  attn_bwd_noalloc
serves them: the caller passes inputs and outputs only, and the backward's
scratch comes from a fixed 32 MiB array inside the library.

This file is collected last on purpose (test_zz_*): if it fails, a run that
stops at the first failure has already run every other test.  It calls the
entry point through the C ABI twice in a row (different problems, so stale
scratch from the first call would show in the second) and compares each
result with attn_bwd given its own workspace, within the BF16 tolerance the
other tests use (relative L2 1e-2; dK and dV are also bit-identical because
the same deterministic kernels run).  It passes alone in a fresh process and
after the other tests.
"""
import ctypes

import numpy as np
import pytest

from precision_numerics_gb300 import inputs

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def lib(cuda_device):
    from precision_numerics_gb300 import attn, build
    build.build()
    return attn.load_library()


def _problem(seed, B, H, N, d):
    x = inputs.random_qkv(seed, B, H, N, d)
    return {k: torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).cuda() for k, v in x.items()}


def _rel_l2(a, b):
    a, b = a.double(), b.double()
    return float((a - b).norm() / b.norm())


def _run_both(lib, t, scale, causal):
    from precision_numerics_gb300 import attn
    B, H, N, d = t["q"].shape
    o, lse = attn.attn_fwd(t["q"], t["k"], t["v"], scale=scale, causal=causal)
    ref = attn.attn_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], scale=scale, causal=causal)
    out = [torch.full_like(o, float("nan")) for _ in range(3)]
    stream = torch.cuda.current_stream().cuda_stream
    status = lib.attn_bwd_noalloc(
        t["q"].data_ptr(), t["k"].data_ptr(), t["v"].data_ptr(), o.data_ptr(), lse.data_ptr(),
        t["do"].data_ptr(), out[0].data_ptr(), out[1].data_ptr(), out[2].data_ptr(),
        B, H, N, d, ctypes.c_float(scale), int(causal), ctypes.c_void_p(stream))
    assert status == 0, lib.attn_last_error().decode()
    assert lib.attn_check_status(ctypes.c_void_p(stream)) == 0
    return ref, out


def test_two_calls_in_a_row_match_attn_bwd(lib):
    cases = [(_problem(11, 2, 4, 1000, 128), 1 / 128 ** 0.5, True),
             (_problem(12, 1, 3, 700, 64), 0.125, False)]
    for t, scale, causal in cases:
        ref, got = _run_both(lib, t, scale, causal)
        for name, r, g in zip(("dq", "dk", "dv"), ref, got):
            assert bool(torch.isfinite(g.float()).all()), name
            assert _rel_l2(g, r) <= 1e-2, (name, _rel_l2(g, r))
        assert torch.equal(got[1], ref[1]) and torch.equal(got[2], ref[2])


def test_rejects_problems_beyond_the_fixed_scratch(lib):
    # B1 H32 N4096 d128 needs 65 MiB of scratch, more than the 32 MiB array.
    status = lib.attn_bwd_noalloc(16, 16, 16, 16, 16, 16, 16, 16, 16, 1, 32, 4096, 128,
                                  ctypes.c_float(0.088), 1, None)
    assert status == 1  # ATTN_ERR_INVALID_ARG, before anything is launched
    msg = lib.attn_last_error().decode()
    assert "33554432" in msg and "attn_bwd" in msg


def test_python_binding_at_the_largest_listed_problem(lib):
    """attn.attn_bwd_noalloc (the binding's checks and default scale) on B8 H12
    N1024 d64 causal, the size the header names as fitting the fixed array
    (25.9 MB of its 32 MiB), against attn_bwd with its own workspace."""
    from precision_numerics_gb300 import attn
    t = _problem(13, 8, 12, 1024, 64)
    o, lse = attn.attn_fwd(t["q"], t["k"], t["v"], causal=True)
    ref = attn.attn_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], causal=True)
    assert attn.attn_bwd_workspace_bytes(8, 12, 1024, 64) <= 32 << 20
    got = [torch.full_like(o, float("nan")) for _ in range(3)]
    attn.attn_bwd_noalloc(t["q"], t["k"], t["v"], o, lse, t["do"], *got, causal=True)
    attn.attn_check_status()
    for name, r, g in zip(("dq", "dk", "dv"), ref, got):
        assert bool(torch.isfinite(g.float()).all()), name
        assert _rel_l2(g, r) <= 1e-2, (name, _rel_l2(g, r))
    assert torch.equal(got[1], ref[1]) and torch.equal(got[2], ref[2])


def test_matches_the_oracle(lib):
    """The no-allocation backward against the FP64 definition directly (not only
    against attn_bwd): B1 H2 N700 d128 causal and d64 full, every head, dQ, dK,
    dV within the stated relative L2 of 1e-2."""
    import oracle
    from precision_numerics_gb300 import attn, inputs
    from precision_numerics_gb300.deviation import deviation
    for seed, (B, H, N, d), causal in ((21, (1, 2, 700, 128), True), (22, (1, 2, 700, 64), False)):
        x = inputs.random_qkv(seed, B, H, N, d)
        t = {k: torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).cuda() for k, v in x.items()}
        scale = d ** -0.5
        o, lse = attn.attn_fwd(t["q"], t["k"], t["v"], scale=scale, causal=causal)
        got = [torch.full_like(o, float("nan")) for _ in range(3)]
        attn.attn_bwd_noalloc(t["q"], t["k"], t["v"], o, lse, t["do"], *got, scale=scale,
                              causal=causal)
        attn.attn_check_status()
        f = {k: inputs.bf16_bits_to_f32(v).reshape(B * H, N, d) for k, v in x.items()}
        for h in range(B * H):
            ref = oracle.backward(f["q"][h], f["k"][h], f["v"][h], f["do"][h], scale, causal)
            for name, g, r in zip(("dq", "dk", "dv"), got, ref):
                e = deviation(g.reshape(B * H, N, d)[h].float().cpu().numpy().astype(np.float64), r)
                assert e["rel_l2"] <= 1e-2, (d, h, name, e)

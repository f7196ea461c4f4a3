"""The largest problem the library accepts, on the GPU.

B*H*N*d must stay below 2^31 elements; 1 x 127 x 131072 x 128 = 2,130,706,432 is
just below it, so the last head starts ~2^31 elements (4.2 GB of BF16) into
each tensor.  All 127 heads hold the same seeded values, so every head's
outputs must equal head 0's: O, LSE, dK and dV bit for bit, dQ within the
spread that the order of its floating-point atomics allows.  An offset that
overflowed 32 bits anywhere would break that.  Sampled rows of the last head
are checked against the FP64 oracle (a causal row i is the non-causal
attention of query i over keys 0..i), and the column sums of dV obey
sum_j dV_j = sum_i dO_i (every row of P sums to one).
"""
import numpy as np
import pytest

import oracle
from precision_numerics_gb300 import inputs
from precision_numerics_gb300.deviation import deviation

from bounds import delta_error_worst

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def A(cuda_device):
    from precision_numerics_gb300 import attn, build
    build.build()
    return attn


def test_largest_accepted_problem(A):
    H, N, d = 127, 131072, 128
    assert H * N * d < 2 ** 31 <= (H + 1) * N * d
    scale = d ** -0.5
    x = inputs.random_qkv(11, 1, 1, N, d)
    one = {k: torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).cuda() for k, v in x.items()}
    big = {k: v.expand(1, H, N, d).contiguous() for k, v in one.items()}
    del one
    o, lse = A.attn_fwd(big["q"], big["k"], big["v"], scale=scale, causal=True)
    dq, dk, dv = A.attn_bwd(big["q"], big["k"], big["v"], o, lse, big["do"], scale=scale,
                            causal=True)
    A.attn_check_status()
    del big
    last = H - 1
    for name, g in (("o", o), ("lse", lse), ("dk", dk), ("dv", dv)):
        assert torch.equal(g[0, last], g[0, 0]), name
        assert torch.equal(g[0, H // 2], g[0, 0]), name
    for g in (o, dq, dk, dv):
        assert bool(torch.isfinite(g[0, last].float()).all())
    dq0, dql = dq[0, 0].float(), dq[0, last].float()
    assert (dq0 - dql).abs().max().item() <= 1e-2 * dq0.abs().max().item()

    f = {k: inputs.bf16_bits_to_f32(v[0, 0]).astype(np.float64) for k, v in x.items()}
    o_last = o[0, last].float().cpu().numpy()
    lse_last = lse[0, last].cpu().numpy()
    for i in (0, 1, 127, 128, 4095, 65536, N - 2, N - 1):
        o_ref, lse_ref = oracle.forward(f["q"][i:i + 1], f["k"][:i + 1], f["v"][:i + 1], scale,
                                        False)
        dev = deviation(o_last[i:i + 1], o_ref)
        assert dev["max_abs"] <= 2e-2, (i, dev)
        assert abs(float(lse_last[i]) - float(lse_ref[0])) <= 1e-3, i

    # sum over keys of dV = sum over queries of dO.  Each query row's share of
    # the column sums carries at most ~2^-8 relative error (BF16 P in the
    # product, BF16 results), so the sums may differ by up to
    # 2^-8 * sum_i |dO_i| (first check).  Those errors have random signs: their
    # sum grows like 2^-8 * sqrt(N) (~1.4 here), and the second check allows
    # 0.05 * sqrt(N), about ten times that.
    dv_sum = dv[0, last].double().sum(dim=0).cpu().numpy()
    do_sum = f["do"].sum(axis=0)
    bound = 2.0 ** -8 * np.abs(f["do"]).sum(axis=0)
    assert np.all(np.abs(dv_sum - do_sum) <= bound)
    assert np.abs(dv_sum - do_sum).max() <= 0.05 * np.sqrt(N)


@pytest.mark.parametrize("causal", [False, True])
def test_more_heads_than_a_grid_y_dimension(A, causal):
    """B*H = 70000 heads (above the 65535 limit of a grid's y dimension), short rows."""
    B, H, N, d = 2, 35000, 3, 64
    scale = d ** -0.5
    x = inputs.random_qkv(12, B, H, N, d)
    t = {k: torch.from_numpy(np.ascontiguousarray(v).view(np.int16)).view(torch.bfloat16).cuda()
         for k, v in x.items()}
    o, lse = A.attn_fwd(t["q"], t["k"], t["v"], scale=scale, causal=causal)
    dq, dk, dv = A.attn_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], scale=scale, causal=causal)
    A.attn_check_status()
    for g in (o, dq, dk, dv):
        assert bool(torch.isfinite(g.float()).all())
    flat = {k: inputs.bf16_bits_to_f32(v).reshape(B * H, N, d) for k, v in x.items()}
    got = {k: g.float().cpu().numpy().reshape(B * H, N, d)
           for k, g in (("o", o), ("dq", dq), ("dk", dk), ("dv", dv))}
    lse_h = lse.cpu().numpy().reshape(B * H, N)
    for h in (0, 34999, 35000, B * H - 1):
        f = {k: v[h] for k, v in flat.items()}
        o_ref, lse_ref = oracle.forward(f["q"], f["k"], f["v"], scale, causal)
        g_ref = oracle.backward(f["q"], f["k"], f["v"], f["do"], scale, causal)
        assert deviation(got["o"][h], o_ref)["max_abs"] <= 2e-2, h
        assert np.abs(lse_h[h] - lse_ref).max() <= 1e-3, h
        assert deviation(got["dv"][h], g_ref[2])["rel_l2"] <= 1e-2, h
        # With three keys dQ and dK are small differences of near-equal terms:
        # allow the worst-case delta_lp bound on top of relative 1e-2.
        for name, r, b in zip(("dq", "dk"), g_ref[:2], delta_error_worst(f, scale, causal)):
            err = np.linalg.norm(got[name][h] - r)
            assert err <= 1e-2 * np.linalg.norm(r) + np.linalg.norm(b), (h, name)

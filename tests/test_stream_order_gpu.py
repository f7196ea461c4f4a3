"""Dependent calls in one stream, without host synchronisation, on the GPU.

The forward and backward kernels are launched so that a kernel may be
scheduled while the previous kernel in the stream is still running; each
thread waits for that kernel's completion before its first global-memory
access.  Here every call reads the output of the call just before it (O fed
back as the next query, dK fed to a forward), for several rounds on the same
buffers, and the results must equal those of the same chain run with a
device synchronisation after every call: bit for bit for everything but dQ,
whose FP32 atomic additions may land in another order.
"""
import numpy as np
import pytest

from precision_numerics_gb300 import inputs

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def A(cuda_device):
    from precision_numerics_gb300 import attn, build
    build.build()
    return attn


def _chain(A, t, rounds, sync, causal, scale):
    B, H, N, d = t["q"].shape
    o1, o2, o3 = (torch.empty_like(t["q"]) for _ in range(3))
    lse1, lse2, lse3 = (torch.empty((B, H, N), dtype=torch.float32, device=t["q"].device)
                        for _ in range(3))
    dq, dk, dv = (torch.empty_like(t["q"]) for _ in range(3))
    ws = torch.empty(A.attn_bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8,
                     device=t["q"].device)
    q = t["q"]
    out = []
    for _ in range(rounds):
        A.attn_fwd(q, t["k"], t["v"], scale=scale, causal=causal, o=o1, lse=lse1)
        if sync:
            torch.cuda.synchronize()
        A.attn_fwd(o1, t["k"], t["v"], scale=scale, causal=causal, o=o2, lse=lse2)
        if sync:
            torch.cuda.synchronize()
        A.attn_bwd(o1, t["k"], t["v"], o2, lse2, t["do"], scale=scale, causal=causal,
                   dq=dq, dk=dk, dv=dv, workspace=ws)
        if sync:
            torch.cuda.synchronize()
        A.attn_fwd(dk, t["k"], dv, scale=scale, causal=causal, o=o3, lse=lse3)
        if sync:
            torch.cuda.synchronize()
        out.append({k: v.clone() for k, v in (("o1", o1), ("o2", o2), ("lse2", lse2),
                                               ("dq", dq), ("dk", dk), ("dv", dv),
                                               ("o3", o3), ("lse3", lse3))})
        q = o3  # the next link of the chain starts from this link's last output
    torch.cuda.synchronize()
    A.attn_check_status()
    return out


@pytest.mark.parametrize("N,d,causal", [(1024, 128, True), (777, 64, False)])
def test_chained_calls_match_synchronised_calls(A, N, d, causal):
    B, H = 2, 4
    scale = d ** -0.5
    x = inputs.random_qkv(31, B, H, N, d)
    t = {k: torch.from_numpy(np.ascontiguousarray(v).view(np.int16)).view(torch.bfloat16).cuda()
         for k, v in x.items()}
    fast = _chain(A, t, 4, False, causal, scale)
    slow = _chain(A, t, 4, True, causal, scale)
    for r, (f, s) in enumerate(zip(fast, slow)):
        for name in ("o1", "o2", "lse2", "dk", "dv"):
            assert torch.equal(f[name], s[name]), (r, name)
        g, ref = f["dq"].float(), s["dq"].float()
        assert (g - ref).abs().max().item() <= 1e-2 * ref.abs().max().item(), r
        # o3 reads dK and dV only, so it is exact as well.
        assert torch.equal(f["o3"], s["o3"]), r
        assert torch.equal(f["lse3"], s["lse3"]), r
        for name in ("o1", "o2", "dq", "dk", "dv", "o3"):
            assert bool(torch.isfinite(f[name].float()).all()), (r, name)

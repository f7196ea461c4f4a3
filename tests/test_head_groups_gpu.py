"""The backward main kernel's head-grouped CTA order, on the GPU.

The main kernel orders its CTAs by groups of heads (sized so that the heads in
flight keep their Q / dO tiles and dQ accumulator rows in L2), then by key
tile.  The shapes below are launched in several groups, the last one ragged:
11 heads of N = 16384, d = 128 (16 MiB of per-head working set) run as groups
of 4, 4 and 3; 13 non-causal heads of N = 8192, d = 128 as 5, 5 and 3; 7 heads
of N = 32768, d = 64 as 3, 3 and 1; B = 2 x 5 heads of N = 16384, d = 64 as
5 and 5.  Every head is then run again on its own (one head: one group, the
plain key-tile order, which the oracle tests cover) and the results must
agree: O, LSE, dK and dV bit for bit (each comes from one CTA with a fixed
operation order), dQ within the spread that the order of its FP32 atomic
additions allows.  A (head, key tile) pair that was skipped, done twice or
done with another head's data breaks that.
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


@pytest.mark.parametrize("B,H,N,d,causal", [
    (1, 11, 16384, 128, True),
    (1, 13, 8192, 128, False),
    (1, 7, 32768, 64, True),
    (2, 5, 16384, 64, False),
])
def test_grouped_launch_equals_per_head_launches(A, B, H, N, d, causal):
    scale = d ** -0.5
    x = inputs.random_qkv(21, B, H, N, d)
    t = {k: torch.from_numpy(np.ascontiguousarray(v).view(np.int16)).view(torch.bfloat16).cuda()
         for k, v in x.items()}
    o, lse = A.attn_fwd(t["q"], t["k"], t["v"], scale=scale, causal=causal)
    dq, dk, dv = A.attn_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], scale=scale, causal=causal)
    A.attn_check_status()
    for b in range(B):
        for h in range(H):
            one = {k: v[b:b + 1, h:h + 1].contiguous() for k, v in t.items()}
            o1, lse1 = A.attn_fwd(one["q"], one["k"], one["v"], scale=scale, causal=causal)
            dq1, dk1, dv1 = A.attn_bwd(one["q"], one["k"], one["v"], o1, lse1, one["do"],
                                       scale=scale, causal=causal)
            A.attn_check_status()
            where = (b, h)
            assert torch.equal(o[b, h], o1[0, 0]), where
            assert torch.equal(lse[b, h], lse1[0, 0]), where
            assert torch.equal(dk[b, h], dk1[0, 0]), where
            assert torch.equal(dv[b, h], dv1[0, 0]), where
            # dQ: the FP32 accumulator sums key-tile contributions in whatever
            # order the atomics land; after BF16 rounding the two runs may
            # differ by an ulp here and there, never by a key tile's share.
            g, r = dq[b, h].float(), dq1[0, 0].float()
            diff = (g - r).abs()
            assert diff.max().item() <= 1e-2 * r.abs().max().item(), where
            assert diff.mean().item() <= 1e-3 * r.abs().mean().item(), where

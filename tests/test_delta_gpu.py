"""The backward's preprocess kernel checked on its own (delta, -LSE*log2(e)).

delta_i = rowsum(dO o O)_i with O the STORED (BF16) forward output: the
delta_lp of "Why Low-Precision Transformer Training Fails", Figure 3.  The
kernel writes it, -LSE*log2(e) and a zeroed FP32 dQ accumulator into the
caller's workspace, whose layout include/attn.h documents:
  [B*H][N_pad] FP32 -LSE*log2(e)   (-inf in the padded rows N..N_pad-1)
  [B*H][N_pad] FP32 delta          (0 in the padded rows)
  [B*H][N_pad][d] FP32 dQ accumulator (all 0)
each part starting at a 256-byte boundary, N_pad = N rounded up to 128.

Every entry is compared: delta against the oracle's FP64 rowsum within the
FP32 summation bound (each product of two BF16 values is exact in FP32;
summing d of them in any order errs by at most (d - 1) 2^-24 sum_k |dO_ik O_ik|
to first order), -LSE*log2(e) bit for bit against the same FP32 product
taken on the host, and the padded rows and the accumulator exactly.  The
workspace is filled with NaN bytes first, so an entry the kernel skipped
shows up.
"""
import numpy as np
import pytest

import oracle
from precision_numerics_gb300 import inputs

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def A(cuda_device):
    from precision_numerics_gb300 import attn, build
    build.build()
    return attn


def _align256(x):
    return (x + 255) // 256 * 256


def _bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


@pytest.mark.parametrize("B,H,N,d", [(1, 3, 200, 64), (2, 2, 128, 128), (1, 1, 1, 128),
                                     (1, 2, 777, 64), (3, 1, 4096, 128)])
def test_preprocess_delta_and_padded_rows(A, B, H, N, d):
    x = inputs.random_qkv(21, B, H, N, d)
    o_bits, do_bits = x["q"], x["do"]  # any BF16 O: delta is defined from the O it is given
    lse = inputs.normal(21, 9, (B, H, N), std=3.0) + np.float32(5.0)
    o, do = _bf16(o_bits), _bf16(do_bits)
    lse_t = torch.from_numpy(lse).cuda()
    need = A.attn_bwd_workspace_bytes(B, H, N, d)
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")  # NaN in every float
    A.attn_bwd_preprocess(o, lse_t, do, ws)
    A.attn_check_status()

    bh, n_pad = B * H, (N + 127) // 128 * 128
    rows = bh * n_pad
    raw = ws.cpu().numpy()
    neg_lse2 = raw[:rows * 4].view(np.float32).reshape(bh, n_pad)
    off = _align256(rows * 4)
    delta = raw[off:off + rows * 4].view(np.float32).reshape(bh, n_pad)
    off = 2 * _align256(rows * 4)
    dqacc = raw[off:off + rows * d * 4].view(np.float32)

    o_f = inputs.bf16_bits_to_f32(o_bits).reshape(bh, N, d)
    do_f = inputs.bf16_bits_to_f32(do_bits).reshape(bh, N, d)
    for h in range(bh):
        ref = oracle.delta(do_f[h], o_f[h])
        tol = (d - 1) * 2.0 ** -24 * (np.abs(do_f[h].astype(np.float64)) * np.abs(o_f[h])).sum(axis=1)
        err = np.abs(delta[h, :N].astype(np.float64) - ref)
        assert np.all(err <= tol * 1.01 + 1e-30), (h, float(err.max()), float(tol.max()))
    expect = -(lse.reshape(bh, N) * np.float32(1.4426950408889634))
    assert np.array_equal(neg_lse2[:, :N], expect.astype(np.float32))
    assert np.all(delta[:, N:] == 0.0)
    assert np.all(np.isneginf(neg_lse2[:, N:]))
    assert np.all(dqacc == 0.0)

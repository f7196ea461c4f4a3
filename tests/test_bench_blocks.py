"""Host logic of the bench line's deviation block (CPU, no kernel).

`_kernel_delta` reads delta out of a backward workspace laid out as
include/attn.h documents ([B*H][N_pad] FP32 -LSE*log2(e), then [B*H][N_pad]
FP32 delta from the next 256-byte boundary); `_deviation_block` compares a
result with the oracle and with the naive BF16 attention.  Both are checked
on a workspace and outputs built here.
"""
import os
import sys

import numpy as np
import pytest

import oracle
from precision_numerics_gb300 import inputs

torch = pytest.importorskip("torch")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_kernel_delta_reads_the_documented_layout():
    w = inputs.Workload("t", 1, 3, 200, 64, True, 0.125)
    n_pad, bh = 256, 3
    rows = bh * n_pad
    off = (rows * 4 + 255) // 256 * 256
    ws = torch.zeros(off + rows * 4 + rows * 64 * 4, dtype=torch.uint8)
    delta = np.arange(rows, dtype=np.float32).reshape(bh, n_pad) * np.float32(0.5)
    ws[off:off + rows * 4] = torch.from_numpy(delta.reshape(-1).view(np.uint8))
    for h in range(bh):
        np.testing.assert_array_equal(bench._kernel_delta(ws, w, h), delta[h, :200])


def test_deviation_block_compares_with_oracle_and_naive():
    w = inputs.Workload("t", 1, 1, 64, 64, True, 0.125)
    x = inputs.random_qkv(5, 1, 1, 64, 64)
    f = {k: inputs.bf16_bits_to_f32(v[0, 0]) for k, v in x.items()}
    o_ref, _ = oracle.forward(f["q"], f["k"], f["v"], w.scale, True)
    dv_ref = oracle.backward(f["q"], f["k"], f["v"], f["do"], w.scale, True)[2]
    # a "kernel" result: the exact values rounded to BF16, and an exact delta
    o = torch.from_numpy(oracle.round_bf16(o_ref).reshape(1, 1, 64, 64))
    dv = torch.from_numpy(oracle.round_bf16(dv_ref).reshape(1, 1, 64, 64))
    rows = 128
    off = (rows * 4 + 255) // 256 * 256
    ws = torch.zeros(off + rows * 4, dtype=torch.uint8)
    d_exact = np.zeros(rows, np.float32)
    d_exact[:64] = oracle.delta(f["do"], o_ref)
    ws[off:off + rows * 4] = torch.from_numpy(d_exact.view(np.uint8))
    blk = bench._deviation_block(w, f, o, dv, ws, o_ref, dv_ref)
    # rounding the exact O to BF16 errs by at most half a BF16 ulp (2^-9 relative)
    assert blk["tiled_gpu"]["o"]["max_abs"] <= 2.0 ** -9 * np.abs(o_ref).max()
    assert blk["naive_bf16"]["o"]["max_abs"] > 0
    assert blk["naive_over_tiled_o_mean_abs"] > 1.0
    # delta stored in FP32: within FP32 rounding of the exact value
    assert blk["delta_lp_minus_delta"]["max_abs"] <= 1e-6 * np.abs(d_exact).max() + 1e-12
    assert set(blk) >= {"tiled_gpu", "naive_bf16", "delta_lp_minus_delta", "sample"}


def test_traffic_comes_from_the_workloads_own_profile_and_only_for_the_current_source(tmp_path):
    import bench
    sha = bench._source_sha()
    (tmp_path / "bwd_main_kernel_gpt2.md").write_text(
        "History on this workload: 128-row query tiles\n\n"
        f"traffic_bytes_per_launch: 82265600\nworkload: gpt2\nsource_sha256: {sha}\n")
    (tmp_path / "bwd_main_kernel_llama7b.md").write_text(
        f"traffic_bytes_per_launch: 1000\nworkload: llama7b\nsource_sha256: {'0' * 64}\n")
    real = bench.TRAFFIC_FILE
    try:
        bench.TRAFFIC_FILE = str(tmp_path / "bwd_main_kernel_{workload}.md")
        assert bench._traffic_per_launch("gpt2") == 82265600.0  # this workload's own file
        assert bench._traffic_per_launch("llama7b") is None     # taken from another source
        assert bench._traffic_per_launch("longseq") is None     # no capture at all
    finally:
        bench.TRAFFIC_FILE = real

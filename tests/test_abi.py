"""The C ABI: the library loads, exports what include/attn.h declares, and its
host-side argument checks behave (CPU only; no kernel is launched)."""
import ctypes
import os
import re
import subprocess

import pytest

from precision_numerics_gb300 import attn, build

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "attn.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return attn.load_library()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"ATTN_API\s+[\w\s\*]+?\b(attn_\w+)\s*\(", text)))


def test_header_declares_the_binding_names():
    assert declared_functions() == sorted(attn.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_library_exports_nothing_else(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True,
                         text=True).stdout
    names = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert {n for n in names if n.startswith("attn_")} == set(declared_functions())


def test_status_strings(lib):
    assert lib.attn_status_string(0).decode() == "ATTN_OK"
    assert b"TIMEOUT" in lib.attn_status_string(4)
    assert lib.attn_version() >= 100


def test_workspace_bytes(lib):
    # lse2 + delta: B*H*Npad floats each (256-byte aligned), dQ accumulator B*H*Npad*d floats.
    def expect(B, H, N, d):
        npad = -(-N // 128) * 128
        a = -(-(B * H * npad * 4) // 256) * 256
        c = -(-(B * H * npad * d * 4) // 256) * 256
        return 2 * a + c
    for shape in [(1, 1, 1, 64), (1, 32, 4096, 128), (8, 12, 1024, 64), (2, 3, 129, 128)]:
        assert lib.attn_bwd_workspace_bytes(*shape, 0) == expect(*shape)
    assert lib.attn_bwd_workspace_bytes(1, 1, 128, 96, 0) == 0
    assert lib.attn_bwd_workspace_bytes(1, 1, 0, 64, 0) == 0


def _fwd(lib, **kw):
    a = dict(q=None, k=None, v=None, o=None, lse=None, B=1, H=1, N=128, d=64, scale=0.125,
             causal=0, dt=0)
    a.update(kw)
    r = lib.attn_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["N"], a["d"],
                     ctypes.c_float(a["scale"]), a["causal"], a["dt"], None)
    return r, lib.attn_last_error().decode()


def test_argument_errors_are_reported_before_any_launch(lib):
    r, msg = _fwd(lib, d=96)
    assert r == attn.ATTN_ERR_UNSUPPORTED and "96" in msg
    r, _ = _fwd(lib, N=0)
    assert r == attn.ATTN_ERR_INVALID_ARG
    r, msg = _fwd(lib, scale=float("nan"))
    assert r == attn.ATTN_ERR_INVALID_ARG and "scale" in msg
    r, _ = _fwd(lib, scale=-1.0)
    assert r == attn.ATTN_ERR_INVALID_ARG
    r, _ = _fwd(lib, dt=7)
    assert r == attn.ATTN_ERR_INVALID_ARG
    r, _ = _fwd(lib, B=65536, H=65536)
    assert r == attn.ATTN_ERR_INVALID_ARG
    r, msg = _fwd(lib)  # null pointers
    assert r == attn.ATTN_ERR_INVALID_ARG and "NULL" in msg
    r, msg = _fwd(lib, q=16 * 1001 + 8, k=16, v=16, o=16, lse=16)
    assert r == attn.ATTN_ERR_INVALID_ARG and "aligned" in msg


def test_selftest_limit_is_checked(lib):
    assert lib.attn_selftest_wait_timeout(0, None) == attn.ATTN_ERR_INVALID_ARG
    assert lib.attn_selftest_wait_timeout(2 * 10**9, None) == attn.ATTN_ERR_INVALID_ARG


def test_binding_rejects_cpu_tensors():
    import torch
    q = torch.zeros(1, 1, 8, 64)
    with pytest.raises(ValueError):
        attn.attn_fwd(q, q, q)


def test_binding_fails_loudly_without_the_library(tmp_path):
    with pytest.raises(RuntimeError, match="missing"):
        attn.load_library(str(tmp_path / "libattn.so"))


def test_stable_forward_argument_checks(lib):
    def call(beta, dt=0):
        return lib.attn_fwd_stable(16, 16, 16, 16, 16, 1, 1, 128, 64, ctypes.c_float(0.125), 1,
                                   ctypes.c_float(beta), dt, None)
    assert call(1.0) == attn.ATTN_ERR_INVALID_ARG
    assert call(float("inf")) == attn.ATTN_ERR_INVALID_ARG
    assert call(2.0, dt=1) == attn.ATTN_ERR_UNSUPPORTED


def test_int8_entry_points_check_arguments_before_any_launch(lib):
    """Shape, scale and pointer errors of the four INT8 entry points come back synchronously."""
    f = ctypes.c_float
    for name in ("attn_quantize_int8", "attn_quantize_int8_as_bf16"):
        fn = getattr(lib, name)
        assert fn(16, 16, 16, 1, 1, 128, 96, None) == attn.ATTN_ERR_UNSUPPORTED  # d
        assert fn(16, 16, 16, 1, 1, 0, 64, None) == attn.ATTN_ERR_INVALID_ARG  # N
        assert fn(None, 16, 16, 1, 1, 128, 64, None) == attn.ATTN_ERR_INVALID_ARG  # null x
        assert "NULL" in lib.attn_last_error().decode()
        assert fn(16, 16, 16 * 7 + 4, 1, 1, 128, 64, None) == attn.ATTN_ERR_INVALID_ARG  # misaligned
    for name in ("attn_fwd_int8", "attn_fwd_int8_as_bf16"):
        fn = getattr(lib, name)

        def call(*, q=16, ks=16, d=64, scale=0.125):
            return fn(q, 16, 16, ks, 16, 16, 16, 1, 1, 128, d, f(scale), 1, None)
        assert call(d=96) == attn.ATTN_ERR_UNSUPPORTED
        assert call(scale=float("nan")) == attn.ATTN_ERR_INVALID_ARG
        assert call(scale=0.0) == attn.ATTN_ERR_INVALID_ARG
        assert call(q=None) == attn.ATTN_ERR_INVALID_ARG
        assert call(ks=16 * 5 + 8) == attn.ATTN_ERR_INVALID_ARG  # misaligned k scales


def test_int8_padded_scale_rows():
    assert [attn.int8_scale_rows(n) for n in (1, 127, 128, 129, 4096)] == [128, 128, 128, 256, 4096]


def test_status_check_is_per_device_not_per_stream(lib):
    """attn_check_status takes only a stream (no workspace): the header states that
    its status words are shared by every stream and thread on the device."""
    assert attn._SIGNATURES["attn_check_status"][1] == [ctypes.c_void_p]
    text = open(HEADER).read()
    block = text[text.index("ATTN_API attn_status attn_check_status") - 1200:
                 text.index("ATTN_API attn_status attn_check_status")]
    assert "per device and per process, not per stream" in block


def test_noalloc_backward_reports_the_same_shape_errors_as_attn_bwd(lib):
    f = ctypes.c_float
    for d, want in ((96, attn.ATTN_ERR_UNSUPPORTED), (64, attn.ATTN_ERR_INVALID_ARG)):
        n = 128 if d == 96 else 0  # d = 96: unsupported head size; N = 0: invalid
        r_noalloc = lib.attn_bwd_noalloc(16, 16, 16, 16, 16, 16, 16, 16, 16, 1, 1, n, d, f(0.125),
                                         1, None)
        r_bwd = lib.attn_bwd(16, 16, 16, 16, 16, 16, 16, 16, 16, 1, 1, n, d, f(0.125), 1, 0, 16,
                             1 << 20, None)
        assert r_noalloc == r_bwd == want, (d, r_noalloc, r_bwd)

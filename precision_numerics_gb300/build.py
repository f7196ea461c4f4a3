"""Build the CUDA library libattn.so in-tree with nvcc (sm_103a only).

Each .cu file under csrc/ is compiled in parallel to an object under
_build/, then linked into precision_numerics_gb300/_lib/libattn.so with the
CUDA runtime linked statically.  build_test_variant() makes the test build
(_lib/libattn_testhooks.so, objects under _build_testhooks/), which only the
test suite loads.  A rebuild happens when any source or
header is newer than the library.
"""
from __future__ import annotations

import contextlib
import fcntl
import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB_DIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIB_DIR, "libattn.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
                     "-I", INCLUDE, "-I", CSRC, "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libattn.so")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs():
    return (_sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
            + glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)])


# The test build: the same sources with test-only instrumentation compiled in
# (ATTN_TEST_HOOKS: counters and a stall switch in the forward kernel) and a
# 50 ms limit on every in-kernel wait.  Only the test suite loads it.
TEST_VARIANT = "testhooks"
TEST_FLAGS = ("-DATTN_TEST_HOOKS", "-DATTN_TEST_WAIT_LIMIT_NS=50000000ull")


def lib_path(variant: str = "") -> str:
    return LIB if not variant else os.path.join(LIB_DIR, f"libattn_{variant}.so")


def needs_build(variant: str = "") -> bool:
    lib = lib_path(variant)
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(p) > t for p in _inputs())


@contextlib.contextmanager
def _build_lock():
    """Exclusive lock on _lib/.build.lock: processes that build at the same time
    (one per rank under torchrun, say) take turns, so none links objects that
    another one is still writing."""
    os.makedirs(LIB_DIR, exist_ok=True)
    with open(os.path.join(LIB_DIR, ".build.lock"), "w") as fh:
        fcntl.flock(fh, fcntl.LOCK_EX)
        try:
            yield
        finally:
            fcntl.flock(fh, fcntl.LOCK_UN)


def build(force: bool = False, verbose: bool = False, extra_flags=(), variant: str = "") -> str:
    """Compile and link libattn.so (or libattn_<variant>.so); returns its path."""
    lib = lib_path(variant)
    if not force and not needs_build(variant):
        return lib
    with _build_lock():
        # Another process may have built it while this one waited for the lock.
        if not force and not needs_build(variant):
            return lib
        return _build_locked(lib, verbose, extra_flags, variant)


def _build_locked(lib, verbose, extra_flags, variant) -> str:
    nvcc = _nvcc()
    build_dir = BUILD if not variant else BUILD + "_" + variant
    os.makedirs(build_dir, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.basename(src) + ".o")
        cmd = [nvcc, *NVCC_FLAGS, *extra_flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr}\n{r.stdout}")
        if verbose and (r.stderr.strip() or r.stdout.strip()):
            print(r.stdout + r.stderr, file=sys.stderr)
        return obj

    srcs = _sources()
    with ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = f"{lib}.tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link of {os.path.basename(lib)} failed:\n{r.stderr}\n{r.stdout}")
    os.replace(tmp, lib)
    return lib


def build_test_variant(force: bool = False) -> str:
    """The test build (TEST_FLAGS) as _lib/libattn_testhooks.so; returns its path."""
    return build(force=force, extra_flags=TEST_FLAGS, variant=TEST_VARIANT)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))

"""The build lock: processes building libattn.so at the same time (one per
rank under torchrun, say) take turns instead of writing the same objects."""
import subprocess
import sys
import textwrap


def test_build_lock_serialises_processes(tmp_path):
    prog = textwrap.dedent("""
        import sys, time
        from precision_numerics_gb300 import build
        with build._build_lock():
            t0 = time.monotonic()
            time.sleep(0.4)
            t1 = time.monotonic()
        print(t0, t1)
    """)
    procs = [subprocess.Popen([sys.executable, "-c", prog], stdout=subprocess.PIPE, text=True)
             for _ in range(3)]
    spans = sorted(tuple(map(float, p.communicate(timeout=60)[0].split())) for p in procs)
    assert all(p.returncode == 0 for p in procs)
    for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
        assert b0 >= a1, spans  # no two critical sections overlap


def test_up_to_date_library_is_not_rebuilt(monkeypatch):
    from precision_numerics_gb300 import build
    monkeypatch.setattr(build, "needs_build", lambda variant="": False)
    monkeypatch.setattr(build, "_build_locked", lambda *a, **k: (_ for _ in ()).throw(AssertionError("rebuilt")))
    assert build.build() == build.LIB

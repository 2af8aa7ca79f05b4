"""The library's host code (argument validation, aliasing checks, planners up to the first CUDA call)
under AddressSanitizer and UndefinedBehaviorSanitizer, on the CPU: a sanitized build of libcoco is
loaded into a subprocess that runs the host-side interface tests; any sanitizer report fails it."""

import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_host_interface_under_asan_and_ubsan(tmp_path):
    sys.path.insert(0, ROOT)
    from collective_fusedallreduce_gb300 import build
    lib = build.build_sanitized(str(tmp_path))
    syms = subprocess.run(["nm", "-D", lib], capture_output=True, text=True).stdout
    assert "__asan_report" in syms and "__ubsan_handle" in syms  # the host code is instrumented
    runtime = build.sanitizer_runtime()
    assert os.path.exists(runtime), runtime
    env = dict(os.environ, COCO_LIBRARY=lib, LD_PRELOAD=runtime,
               ASAN_OPTIONS="detect_leaks=0:halt_on_error=1",
               UBSAN_OPTIONS="halt_on_error=1:print_stacktrace=1")
    probe = subprocess.run([sys.executable, "-c", "from collective_fusedallreduce_gb300 import coco; "
                            "print(coco.library_path())"], cwd=ROOT, env=env, capture_output=True, text=True,
                           timeout=300)
    assert probe.returncode == 0, probe.stderr[-2000:]
    assert probe.stdout.strip() == lib  # the sanitized build is the one loaded
    p = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider", "-m", "not gpu",
                        os.path.join("tests", "test_abi_host.py")], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=600)
    out = p.stdout + p.stderr
    assert p.returncode == 0, out[-4000:]
    assert "AddressSanitizer" not in out and "runtime error:" not in out, out[-4000:]

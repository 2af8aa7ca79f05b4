"""Builds libcoco.so in-tree with nvcc for sm_103a (no cmake).

Every .cu file under csrc/ is compiled in parallel to _build/*.o, then linked
into ``collective_fusedallreduce_gb300/libcoco.so`` with the CUDA runtime
linked statically. Only the ``coco_*`` symbols are exported.
"""

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
LIB = os.path.join(PKG, "libcoco.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc():
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _stale(obj, deps):
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(d) > t for d in deps)


# Host-side sanitizers for a checking build of the library (device code is unchanged).
# (nvcc splits -Xcompiler values at commas, so every flag is passed on its own)
SANITIZE = ["-Xcompiler", "-fsanitize=address", "-Xcompiler", "-fsanitize=undefined", "-Xcompiler",
            "-fno-omit-frame-pointer", "-Xcompiler", "-fno-sanitize-recover=all"]


def build(verbose=False, ptxas_verbose=False, force=False, build_dir=None, lib=None, extra=()):
    """Compile (only what changed) and link libcoco.so. Returns the library path.

    ``build_dir`` / ``lib`` / ``extra`` build a variant elsewhere with extra nvcc flags (see
    build_sanitized); the default is the in-tree library."""
    BUILD = build_dir or globals()["BUILD"]
    LIB = lib or globals()["LIB"]
    extra = list(extra)
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".h")]
    headers.append(os.path.join(INCLUDE, "coco.h"))
    jobs = []
    objs = []
    for src in sources():
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if force or ptxas_verbose or _stale(obj, [src] + headers):
            cmd = [cc] + ARCH + FLAGS + extra + (["-Xptxas", "-v"] if ptxas_verbose else []) + ["-c", src, "-o", obj]
            jobs.append(cmd)

    def run(cmd):
        p = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, p

    if jobs:
        with ThreadPoolExecutor(max(1, min(len(jobs), os.cpu_count() or 1))) as ex:
            for cmd, p in ex.map(run, jobs):
                if verbose or ptxas_verbose or p.returncode:
                    sys.stderr.write(" ".join(cmd) + "\n" + p.stdout + p.stderr)
                if p.returncode:
                    raise RuntimeError(f"nvcc failed on {cmd[-3]}")
    if jobs or not os.path.exists(LIB):
        tmp = LIB + ".tmp"
        cmd = [cc] + ARCH + extra + ["-shared", "-o", tmp] + objs + ["-cudart", "static"]
        p = subprocess.run(cmd, capture_output=True, text=True)
        if p.returncode:
            sys.stderr.write(" ".join(cmd) + "\n" + p.stdout + p.stderr)
            raise RuntimeError("link of libcoco.so failed")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(verbose="-v" in sys.argv, ptxas_verbose="--ptxas" in sys.argv, force="--force" in sys.argv)
    print(LIB)


def build_sanitized(dest_dir):
    """The same library with AddressSanitizer and UndefinedBehaviorSanitizer in its host code, built
    under ``dest_dir``. A process loads it with the ASan runtime preloaded (sanitizer_runtime()) and
    COCO_LIBRARY pointing at it. Returns the library path."""
    return build(build_dir=os.path.join(dest_dir, "_build"), lib=os.path.join(dest_dir, "libcoco_sanitized.so"),
                 extra=SANITIZE)


def sanitizer_runtime():
    """Path of the ASan runtime that must be preloaded into a process loading the sanitized build."""
    p = subprocess.run(["gcc", "-print-file-name=libasan.so"], capture_output=True, text=True)
    return p.stdout.strip()


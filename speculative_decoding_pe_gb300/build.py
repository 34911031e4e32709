"""Build libpe.so in-tree with nvcc for sm_103a (GB300).

Each .cu file compiles in its own nvcc process (in parallel), then one link
step makes ``speculative_decoding_pe_gb300/_build/libpe.so``.  No cmake, no
torch extension machinery: the library is plain C-ABI.
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(OUT_DIR, "libpe.so")
# The same entry points compiled with PE_CHECKED: NaN logits and internal
# index invariants raise error bits (slower; for debugging).
CHECKED_LIB_PATH = os.path.join(OUT_DIR, "libpe_checked.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-Wall", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs() -> list[str]:
    return (sources() + glob.glob(os.path.join(CSRC, "*.cuh")) +
            glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)])


def is_stale(lib: str = LIB_PATH) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(p) > t for p in _inputs())


def _compile(lib: str, obj_dir: str, defines: list[str], verbose_ptxas: bool):
    """Start one nvcc process per source; returns (objects, processes)."""
    os.makedirs(obj_dir, exist_ok=True)
    nvcc = _nvcc()
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    procs, objs = [], []
    for src in sources():
        obj = os.path.join(obj_dir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *defines, *extra, "-c", src, "-o", obj]
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                            stderr=subprocess.STDOUT, text=True)))
    return objs, procs


def _finish(lib: str, objs, procs, verbose_ptxas: bool):
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if out and (verbose_ptxas or p.returncode):
            sys.stderr.write(out)
        if p.returncode:
            failed.append(src)
    if failed:
        raise RuntimeError("nvcc failed on: %s" % ", ".join(failed))
    tmp = lib + ".tmp%d" % os.getpid()
    subprocess.run([_nvcc(), *ARCH, "-shared", "-o", tmp, *objs], check=True)
    os.replace(tmp, lib)


def build(force: bool = False, verbose_ptxas: bool = False, checked: bool = True) -> str:
    """Compile and link libpe.so (and libpe_checked.so) when missing or older
    than a source; the two compile in parallel."""
    jobs = [(LIB_PATH, os.path.join(OUT_DIR, "obj"), [])]
    if checked:
        jobs.append((CHECKED_LIB_PATH, os.path.join(OUT_DIR, "obj_checked"), ["-DPE_CHECKED"]))
    started = [(lib, *_compile(lib, d, defs, verbose_ptxas)) for lib, d, defs in jobs
               if force or is_stale(lib)]
    for lib, objs, procs in started:
        _finish(lib, objs, procs, verbose_ptxas)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))

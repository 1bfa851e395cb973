"""Build the CUDA library in-tree with nvcc for sm_103a.

``python -m quantized_moe_decode_gemv_gb300.build`` (or ``build()``) compiles
each translation unit in parallel and links ``libmoe_gb300.so`` next to this
file, and beside it the debug build ``libmoe_gb300_checks.so`` (the same
sources compiled with ``-DMOE_CHECKS=1``: kernels check the indices they read
from data and record violations in the status word; NVTX ranges on).  The
binding loads the debug build when ``MOE_CHECKS=1`` is set in the environment.
Only nvcc and the host C++ compiler are needed (no cmake, no torch extension
machinery).
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB = os.path.join(HERE, "libmoe_gb300.so")
LIB_CHECKS = os.path.join(HERE, "libmoe_gb300_checks.so")
# (library, object directory, extra flags) of each variant
VARIANTS = [(LIB, BUILD_DIR, []), (LIB_CHECKS, os.path.join(BUILD_DIR, "checks"), ["-DMOE_CHECKS=1"])]

# (source, object name, extra flags)
SOURCES = [("moe_layer.cu", "moe_layer", []), ("moe_noalloc.cu", "moe_noalloc", [])]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-Xptxas", "-warn-spills"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("command failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    return r.stdout + r.stderr


def build(verbose: bool = False, checks: bool = True) -> str:
    """Compile and link the library (and, with ``checks``, its debug build);
    returns the path of the default library."""
    nvcc = _nvcc()
    cmds, links = [], []
    for lib, odir, vflags in (VARIANTS if checks else VARIANTS[:1]):
        os.makedirs(odir, exist_ok=True)
        objs = []
        for src, name, extra in SOURCES:
            obj = os.path.join(odir, name + ".o")
            objs.append(obj)
            cmds.append([nvcc, *ARCH, *FLAGS, *vflags, *extra, "-I", INCLUDE, "-I", CSRC, "-c",
                         os.path.join(CSRC, src), "-o", obj])
        links.append((lib, objs))
    with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, len(cmds))) as ex:
        logs = list(ex.map(_run, cmds))
    for lib, objs in links:
        tmp = lib + ".tmp"
        logs.append(_run([nvcc, *ARCH, "-shared", "-o", tmp, *objs]))
        os.replace(tmp, lib)
    if verbose:
        sys.stdout.write("".join(logs))
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))

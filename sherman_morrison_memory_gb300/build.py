"""Build the sm_103a CUDA library in-tree: ``_build/libvla_gb300.so``.

Usage: ``python -m sherman_morrison_memory_gb300.build`` (or
``__graft_entry__.build()``). Needs nvcc (CUDA 13); cross-compiles without a
GPU.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD_DIR, "libvla_gb300.so")
SOURCES = [os.path.join(CSRC, "vla_forward.cu"), os.path.join(CSRC, "vla_host.cpp"), os.path.join(CSRC, "vla_probe.cu")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    p = shutil.which("nvcc")
    if p:
        return p
    for c in ("/usr/local/cuda/bin/nvcc",):
        if os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


TRACE_LIB = os.path.join(BUILD_DIR, "libvla_gb300_trace.so")


def build(verbose: bool = False, extra=(), out: str = LIB) -> str:
    """Compile the library; ``out``/``extra`` select a variant (e.g. the
    -DVLA_TRACE profiling build written to TRACE_LIB). The translation units
    compile in parallel, then link into one shared library."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    nvcc = nvcc_path()
    tag = os.path.splitext(os.path.basename(out))[0]
    flags = [*ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, *extra]
    if verbose:
        flags += ["-Xptxas", "-v"]
    procs, objs = [], []
    for src in SOURCES:
        obj = os.path.join(BUILD_DIR, f"{tag}_{os.path.basename(src)}.o")
        cmd = [nvcc, *flags, "-c", src, "-o", obj]
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
        objs.append(obj)
    logs = []
    for cmd, pr in procs:
        log, _ = pr.communicate()
        logs.append(log)
        if pr.returncode != 0:
            raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + log)
    tmp = out + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", *objs, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc link failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    os.replace(tmp, out)
    if verbose:
        sys.stderr.write("".join(logs) + r.stdout + r.stderr)
    return out


def build_trace() -> str:
    return build(extra=("-DVLA_TRACE",), out=TRACE_LIB)


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))

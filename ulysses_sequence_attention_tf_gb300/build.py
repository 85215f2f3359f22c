"""Build ``libtf_ulysses.so`` (in-tree) with nvcc for sm_103a.

The translation units (kernels, host ABI) compile in parallel into
``_build/`` and link into ``ulysses_sequence_attention_tf_gb300/libtf_ulysses.so``.
cudart is linked statically, so the library depends only on the driver.
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
BUILD_DIR = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libtf_ulysses.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
              f"-I{INCLUDE}", f"-I{CSRC}"]
SOURCES = ["block_kernels.cu", "block_kernels_v16.cu", "gemm_kernels.cu", "relayout_kernels.cu", "staged_kernels.cu",
           "tf_ulysses.cpp", "noalloc.cu"]
DEPS = SOURCES + ["relayout.h", "noalloc.h", "device_common.cuh", "block_kernel.cuh", "tma_plan.h", "gemm.h"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, d) for d in DEPS] + [os.path.join(INCLUDE, "tf_ulysses.h")]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, defines=(), out: str | None = None) -> str:
    """Compile the library if it is missing or older than its sources.

    ``defines``: extra ``-D`` macros (tuning constants); ``out``: library path
    (default: the in-tree ``libtf_ulysses.so``)."""
    lib = out or LIB
    if not force and not defines and out is None and not _stale():
        return LIB
    build_dir = BUILD_DIR if out is None else os.path.join(os.path.dirname(lib), "_obj")
    os.makedirs(build_dir, exist_ok=True)
    cc = nvcc()
    procs = []
    objs = []
    for src in SOURCES:
        obj = os.path.join(build_dir, src + ".o")
        objs.append(obj)
        cmd = [cc, *ARCH, *NVCC_FLAGS, *[f"-D{d}" for d in defines], "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
    failed = []
    for cmd, p in procs:
        out, _ = p.communicate()
        if verbose or p.returncode != 0:
            sys.stderr.write(out)
        if p.returncode != 0:
            failed.append(" ".join(cmd))
    if failed:
        raise RuntimeError("nvcc failed:\n" + "\n".join(failed))
    tmp = lib + f".tmp{os.getpid()}"
    subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *objs], check=True)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

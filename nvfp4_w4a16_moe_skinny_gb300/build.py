"""Build the C-ABI shared library in-tree with nvcc for sm_103a.

    python -m nvfp4_w4a16_moe_skinny_gb300.build

writes ``nvfp4_w4a16_moe_skinny_gb300/libnvfp4skinny.so``: the host unit and
one unit per streaming epilogue, compiled in parallel (objects in ``_build/``)
and linked; one ``-gencode`` (compute_103a -> sm_103a); no CMake.
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libnvfp4skinny.so")
GENCODE = "arch=compute_103a,code=sm_103a"


def nvcc_path() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build the library")


def units():
    """The translation units: the host side (nvfp4_skinny.cu) and one per streaming epilogue."""
    csrc = os.path.join(PKG, "csrc")
    return [os.path.join(csrc, f) for f in sorted(os.listdir(csrc)) if f.endswith(".cu")]


def sources():
    csrc = os.path.join(PKG, "csrc")
    return [os.path.join(csrc, f) for f in sorted(os.listdir(csrc))] + [os.path.join(INCLUDE, "nvfp4_skinny.h")]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(s) <= t for s in sources())


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile every translation unit (in parallel) and link the shared library."""
    if not force and up_to_date():
        return LIB
    nvcc = nvcc_path()
    objdir = os.path.join(PKG, "_build")
    os.makedirs(objdir, exist_ok=True)
    procs = []
    for src in units():
        obj = os.path.join(objdir, os.path.basename(src) + ".o")
        cmd = [nvcc, "-gencode", GENCODE, "-O3", "-lineinfo", "-std=c++17", "-I" + INCLUDE, "-Xcompiler", "-fPIC",
               "-c", "-o", obj, src]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        procs.append((obj, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)))
    objs, errors = [], []
    for obj, pr in procs:
        out, err = pr.communicate()
        if pr.returncode != 0:
            errors.append(out + err)
        elif verbose:
            sys.stderr.write(err)
        objs.append(obj)
    if errors:
        raise RuntimeError("nvcc failed:\n" + "\n".join(errors))
    res = subprocess.run([nvcc, "-shared", "-o", LIB + ".tmp"] + objs, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("link failed:\n" + res.stdout + res.stderr)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

"""Compile the layoutmove shared library in place.

Every translation unit under ``csrc/`` -- the host layout algebra, the
copy, tile-copy and exchange planners (plain C++17, compiled with g++) and
the kernels (CUDA, compiled with nvcc for sm_103a only) -- is built in
parallel into ``_build/`` and linked into ``liblayoutmove.so`` next to this
file.  The CUDA runtime is linked
statically, so the library loads without any other CUDA shared object.
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
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "liblayoutmove.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required")


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC)
                  if f.endswith((".cpp", ".cu")))


def _newest_input() -> float:
    files = _sources() + [os.path.join(CSRC, f) for f in os.listdir(CSRC)
                          if f.endswith(".h")]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def build(verbose: bool = False, force: bool = False) -> str:
    """Build (if stale) and return the path of liblayoutmove.so."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= _newest_input()):
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    common = ["-O3", "-std=c++17", f"-I{INCLUDE}", f"-I{CSRC}"]
    jobs = []
    objs = []
    for src in _sources():
        obj = os.path.join(BUILD, os.path.basename(src) + ".o")
        objs.append(obj)
        if src.endswith(".cu"):
            cmd = [nvcc, *ARCH, "-lineinfo", *common, "-Xcompiler", "-fPIC",
                   "-Xptxas", "-v" if verbose else "-O3",
                   "-c", src, "-o", obj]
        else:
            cmd = [os.environ.get("CXX", "g++"), *common, "-fPIC", "-Wall",
                   "-c", src, "-o", obj]
        jobs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                           stderr=subprocess.STDOUT)))
    failed = []
    for cmd, proc in jobs:
        out, _ = proc.communicate()
        text = out.decode(errors="replace")
        if proc.returncode != 0:
            failed.append(" ".join(cmd) + "\n" + text)
        elif verbose and text.strip():
            sys.stderr.write(text)
    if failed:
        raise RuntimeError("layoutmove build failed:\n" + "\n".join(failed))
    tmp = LIB + ".tmp"
    link = [nvcc, *ARCH, "-shared", "-cudart", "static", *objs, "-o", tmp]
    res = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
    if res.returncode != 0:
        raise RuntimeError("layoutmove link failed:\n" +
                           res.stdout.decode(errors="replace"))
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))

"""Build libnvfp4.so in-tree for sm_103a (nvcc cross-compiles without a GPU),
and its debug twin libnvfp4_guarded.so (the same sources compiled with
NVFP4_DEBUG_GUARDS: every plain global load and store of the kernels checks
its buffer's extent and reports instead of faulting)."""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libnvfp4.so")
LIB_GUARDED = os.path.join(HERE, "libnvfp4_guarded.so")
SOURCES = ["nvfp4.cu"]

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "--compiler-options", "-fPIC,-O2",
    "-Xptxas", "-v",
    "-shared",
]


def nvcc() -> str:
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(p):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libnvfp4")
    return p


def _inputs():
    """Every file the library is compiled from: the sources, every kernel
    header under csrc/ (found by listing, so a new header is tracked too) and
    the public header."""
    files = [os.path.join(CSRC, s) for s in SOURCES]
    files += sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h")))
    files.append(os.path.join(ROOT, "include", "nvfp4.h"))
    files.append(os.path.abspath(__file__))
    return files


def _lib(guards: bool) -> str:
    return LIB_GUARDED if guards else LIB


def up_to_date(guards: bool = False) -> bool:
    lib = _lib(guards)
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def _command(guards: bool, out: str):
    return [nvcc(), *NVCC_FLAGS, *(["-DNVFP4_DEBUG_GUARDS"] if guards else []), "-o", out,
            os.path.join(CSRC, "nvfp4.cu")]


def build_all(force: bool = False, verbose: bool = False, guarded: bool = True):
    """Compile the libraries that are out of date, the normal and the guarded
    one side by side.  Returns their paths."""
    todo = [g for g in ([False, True] if guarded else [False]) if force or not up_to_date(g)]
    procs = []
    for g in todo:
        tmp = _lib(g) + f".tmp{os.getpid()}"
        procs.append((g, tmp, subprocess.Popen(_command(g, tmp), stdout=subprocess.PIPE,
                                               stderr=subprocess.PIPE, text=True)))
    errors = []
    for g, tmp, p in procs:
        _, err = p.communicate()
        if p.returncode != 0:
            errors.append(f"nvcc failed ({os.path.basename(_lib(g))}):\n" + err[-8000:])
            continue
        if verbose:
            sys.stderr.write(err)
        os.makedirs(os.path.join(ROOT, "_build"), exist_ok=True)
        with open(os.path.join(ROOT, "_build", "ptxas_guarded.log" if g else "ptxas.log"), "w") as f:
            f.write(err)
        os.replace(tmp, _lib(g))
    if errors:
        raise RuntimeError("\n".join(errors))
    return [LIB] + ([LIB_GUARDED] if guarded else [])


def build(force: bool = False, verbose: bool = False, guards: bool = False) -> str:
    """Compile one library (the guarded one with guards=True) if out of date."""
    if not force and up_to_date(guards):
        return _lib(guards)
    tmp = _lib(guards) + f".tmp{os.getpid()}"
    r = subprocess.run(_command(guards, tmp), capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + r.stderr[-8000:])
    if verbose:
        sys.stderr.write(r.stderr)
    os.makedirs(os.path.join(ROOT, "_build"), exist_ok=True)
    with open(os.path.join(ROOT, "_build", "ptxas_guarded.log" if guards else "ptxas.log"), "w") as f:
        f.write(r.stderr)
    os.replace(tmp, _lib(guards))
    return _lib(guards)


if __name__ == "__main__":
    for path in build_all(force="--force" in sys.argv, verbose="-v" in sys.argv):
        print(path)

"""Build libattn_sm103a.so in-tree with nvcc (sm_103a only, no cmake).

Each ``csrc/*.cu`` is compiled to an object in parallel, then linked into a
shared library next to this file with the CUDA runtime linked statically, so
the library loads on a machine without a GPU driver (the driver API is
reached at run time through the runtime's entry-point lookup).

The same sources are also built with ``-DATTN_DEBUG_CHECKS`` into
``libattn_sm103a_debug.so``: every TMA coordinate and tensor-memory address
is range-checked on the device and a failure is reported through the device
error word (the stand-in for a memory checker; see attn_build_flags()).

    python -m exact_attention_52_gb300.build [--verbose]
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB_NAME = "libattn_sm103a.so"
LIB_PATH = os.path.join(PKG, LIB_NAME)
DEBUG_LIB_PATH = os.path.join(PKG, "libattn_sm103a_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
          "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libattn_sm103a.so")
    return cand


def _sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _compile(job: tuple[str, bool]) -> tuple[str, str]:
    src, debug = job
    out_dir = os.path.join(BUILD, "debug") if debug else BUILD
    obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc(), *ARCH, *CFLAGS, *(["-DATTN_DEBUG_CHECKS"] if debug else []), "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def _link(objs: list[str], path: str) -> None:
    tmp = path + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, path)


def build(verbose: bool = False) -> str:
    """Compile every kernel source twice (release and range-checked debug build),
    link both shared libraries and return the release library's path."""
    os.makedirs(os.path.join(BUILD, "debug"), exist_ok=True)
    srcs = _sources()
    jobs = [(s, False) for s in srcs] + [(s, True) for s in srcs]
    with cf.ThreadPoolExecutor(max_workers=min(16, len(jobs))) as ex:
        results = list(ex.map(_compile, jobs))
    release, debug = results[:len(srcs)], results[len(srcs):]
    log = "\n".join(err for _, err in release)
    with open(os.path.join(BUILD, "ptxas.log"), "w") as f:
        f.write(log)
    if verbose:
        print(log)
    _link([o for o, _ in release], LIB_PATH)
    _link([o for o, _ in debug], DEBUG_LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(verbose="--verbose" in sys.argv))

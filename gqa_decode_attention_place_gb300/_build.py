"""Build libgqa_attn.so in-tree with nvcc for sm_103a (GB300).

Each ``csrc/*.cu`` file is compiled to an object in parallel, then linked into
``lib/libgqa_attn.so`` (CUDA runtime linked statically).  Rebuilds only when a
source or header is newer than the library.  ``-Xptxas -v`` output (registers,
spills, shared memory) is kept in ``_build/ptxas.log``.

``build(debug=True)`` makes ``lib/libgqa_attn_debug.so`` from the same sources
with ``-DGQA_DEBUG``: the kernels then check their index-derived addresses
(bulk-copy tile coordinates, cluster landing slots, partial-result slots,
output rows) before each access and record a failed check instead of making
it.  Setting ``GQA_ATTN_DEBUG=1`` makes the package load that library.
"""

from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIBDIR = os.path.join(PKG, "lib")
LIBNAME = "libgqa_attn.so"
LIBPATH = os.path.join(LIBDIR, LIBNAME)
DEBUG_LIBPATH = os.path.join(LIBDIR, "libgqa_attn_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-Wall,-Wextra",
                     "--expt-relaxed-constexpr", "-Xptxas", "-v", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libgqa_attn.so")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (_sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
            + glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)])


def lib_path(debug: bool = False) -> str:
    return DEBUG_LIBPATH if debug else LIBPATH


def up_to_date(debug: bool = False) -> bool:
    path = lib_path(debug)
    if not os.path.exists(path):
        return False
    t = os.path.getmtime(path)
    return all(os.path.getmtime(p) <= t for p in _deps())


def _compile(nvcc: str, src: str, debug: bool):
    bdir = os.path.join(BUILD, "debug") if debug else BUILD
    obj = os.path.join(bdir, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc] + NVCC_FLAGS + (["-DGQA_DEBUG"] if debug else []) + ["-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    return src, obj, r.returncode, r.stdout + r.stderr, " ".join(cmd)


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Compile and link the library (the range-checked one if ``debug``);
    return its path."""
    path = lib_path(debug)
    if not force and up_to_date(debug):
        return path
    nvcc = _nvcc()
    os.makedirs(os.path.join(BUILD, "debug") if debug else BUILD, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    srcs = _sources()
    logs = []
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        results = list(ex.map(lambda s: _compile(nvcc, s, debug), srcs))
    failed = False
    for src, obj, rc, out, cmd in results:
        logs.append(f"$ {cmd}\n{out}")
        if rc != 0:
            failed = True
            sys.stderr.write(f"nvcc failed on {src}:\n{out}\n")
        else:
            warnings = [ln for ln in out.splitlines() if "warning" in ln.lower()]
            if warnings:  # host-compiler warnings (-Wall -Wextra) are shown, not hidden
                sys.stderr.write(f"{os.path.basename(src)}:\n" + "\n".join(warnings) + "\n")
    log = os.path.join(BUILD, "ptxas_debug.log" if debug else "ptxas.log")
    with open(log, "w") as f:
        f.write("\n".join(logs))
    if failed:
        raise RuntimeError(f"CUDA compilation failed (see {log})")
    tmp = path + ".tmp"
    link = [nvcc] + ARCH + ["-shared", "-o", tmp] + [r[1] for r in results]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}{r.stderr}")
    os.replace(tmp, path)
    if verbose:
        print(f"built {path}")
    return path


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, debug="--debug" in sys.argv)

"""Build libtpmlp.so in-tree with nvcc for sm_103a.

Each CUDA translation unit is compiled in parallel, then linked into
``tensor_transformer_mlp_tcgen05_gb300/libtpmlp.so`` (the CUDA runtime is
linked statically; the driver API is reached through the runtime's entry-point
lookup, so the library does not link libcuda).  Object files go to
``_build/`` at the repository root.  A rebuild is skipped when the library is
newer than every source and header.

``build(checks=True)`` makes the debug variant ``libtpmlp_checks.so`` (objects
in ``_build/checks``) with ``-DTPMLP_CHECKS``: device-side checks of TMA
coordinates and store indices that report ``TPMLP_ERR_CHECK`` instead of
letting a bad access happen.  Load it by setting ``TPMLP_LIB`` to its path
before the binding is imported.
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
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_PATH = os.path.join(PKG, "libtpmlp.so")
CHECKS_LIB_PATH = os.path.join(PKG, "libtpmlp_checks.so")

SOURCES = ["gemm_tc2.cu", "rowops.cu", "simt.cu",
           "tp_mlp_host.cu", "noalloc.cu", "attn_fwd.cu", "attn_bwd.cu",
           "attn_host.cu", "fp8.cu", "probe.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
          "--expt-relaxed-constexpr", "-I" + INCLUDE, "-I" + CSRC]


def nvcc_path() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required")


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)
             if f.endswith((".cu", ".cuh", ".h"))]
    files.append(os.path.join(INCLUDE, "tp_mlp.h"))
    files.append(os.path.join(INCLUDE, "tp_attn.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date(lib_path: str = LIB_PATH) -> bool:
    if not os.path.exists(lib_path):
        return False
    t = os.path.getmtime(lib_path)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False,
          ptxas_info: bool = False, checks: bool = False) -> str:
    """Compile and link; returns the library path.  Raises on failure.
    checks=True builds the debug variant (see the module docstring)."""
    lib_path = CHECKS_LIB_PATH if checks else LIB_PATH
    if not force and up_to_date(lib_path):
        return lib_path
    nvcc = nvcc_path()
    obj_dir = os.path.join(BUILD_DIR, "checks") if checks else BUILD_DIR
    os.makedirs(obj_dir, exist_ok=True)
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    if checks:
        extra.append("-DTPMLP_CHECKS")

    def compile_one(src):
        obj = os.path.join(obj_dir, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc, *ARCH, *CFLAGS, *extra, "-c", os.path.join(CSRC, src),
               "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose or ptxas_info:
        for obj, log in results:
            if log.strip():
                print(f"--- {os.path.basename(obj)}\n{log}", file=sys.stderr)
    tmp = lib_path + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True,
                ptxas_info="--ptxas-info" in sys.argv,
                checks="--checks" in sys.argv))

"""Build libfcp.so in-tree with nvcc for sm_103a.

Compiles every translation unit in csrc/ in parallel and links one shared
library, context_document_masked_gb300/_lib/libfcp.so. `build(checked=True)`
builds the same sources with FCP_DEVICE_CHECKS=1 (every plan-table index the
kernels read is bounds-checked on the device; a failed check sets an error bit
and skips the work unit) into _lib_checked/libfcp.so, which the binding loads
when the environment sets FCP_DEVICE_CHECKS=1.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_lib")
LIB = os.path.join(OUT_DIR, "libfcp.so")
OUT_DIR_CHECKED = os.path.join(HERE, "_lib_checked")
LIB_CHECKED = os.path.join(OUT_DIR_CHECKED, "libfcp.so")
SOURCES = ["api.cu", "attn_fwd.cu", "attn_bwd.cu", "copy_kernels.cu", "noalloc.cu", "plan.cpp",
           "tables.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(p):
        raise RuntimeError("nvcc not found")
    return p


def _stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    deps.append(os.path.join(HERE, "..", "include", "fcp.h"))
    return any(os.path.getmtime(f) > t for f in deps if os.path.exists(f))


def build(verbose: bool = False, force: bool = False, checked: bool = False) -> str:
    out_dir, lib = (OUT_DIR_CHECKED, LIB_CHECKED) if checked else (OUT_DIR, LIB)
    if not force and not _stale(lib):
        return lib
    os.makedirs(out_dir, exist_ok=True)
    nvcc = _nvcc()
    common = ["-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-lineinfo", *ARCH]
    if checked:
        common += ["-DFCP_DEVICE_CHECKS=1"]
    if verbose:
        common += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(out_dir, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc, *common, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            sys.stderr.write(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + ".tmp"
    r = subprocess.run([nvcc, "-shared", *ARCH, "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


def ensure_built() -> str:
    return build(checked=os.environ.get("FCP_DEVICE_CHECKS") == "1")


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv, checked="--checked" in sys.argv))

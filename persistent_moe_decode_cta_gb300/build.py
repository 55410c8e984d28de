"""Build libmk.so (the C-ABI megakernel library) in-tree with nvcc for sm_103a.

Four builds of the device code (default, deterministic, two tensor-core variants)
and the host planner/ABI compile in parallel, then link into
persistent_moe_decode_cta_gb300/libmk.so with the CUDA runtime linked statically.  Usable as `python -m persistent_moe_decode_cta_gb300.build`.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmk.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["mk_kernel.cu", "mk_kernel_det.cu", "mk_kernel_umma.cu", "mk_kernel_umma_ffn.cu", "mk_host.cpp"]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags(extra_ptxas=False):
    f = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-maxrregcount=224",
         "-I" + os.path.join(ROOT, "include"), "-I" + CSRC] + ARCH
    if extra_ptxas:
        f += ["-Xptxas", "-v"]
    return f


def build(verbose: bool = False, ptxas_info: bool = False) -> str:
    nvcc = nvcc_path()
    os.makedirs(OUT_DIR, exist_ok=True)
    objs = []
    cmds = []
    for src in SOURCES:
        obj = os.path.join(OUT_DIR, src + ".o")
        lang = ["-x", "cu"] if src.endswith(".cu") else ["-x", "c++"]
        cmds.append([nvcc, *lang, *_flags(ptxas_info and src.endswith(".cu")), "-c",
                     os.path.join(CSRC, src), "-o", obj])
        objs.append(obj)

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    with ThreadPoolExecutor(len(cmds)) as ex:
        results = list(ex.map(run, cmds))
    for cmd, r in results:
        if verbose or ptxas_info:
            sys.stderr.write(r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    link = [nvcc, *ARCH, "-shared", "-o", LIB + ".tmp", *objs, "-cudart", "static"]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + " ".join(link) + "\n" + r.stdout + r.stderr)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose=True, ptxas_info="-v" in sys.argv))

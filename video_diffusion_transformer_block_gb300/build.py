"""Builds the sm_103a CUDA library (libvdtb_attn.so) in-tree with nvcc.

Two variants of the same sources are built, all translation units in
parallel: libvdtb_attn.so, which the Python binding loads, and
libvdtb_attn_debug.so, compiled with -DATTN_DEBUG, in which every global store
of the kernels is bounds-checked (a store outside its buffer is skipped and
reported through the status word).  Usage:
``python -m video_diffusion_transformer_block_gb300.build``.
"""
from __future__ import annotations

import concurrent.futures
import hashlib
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_NAME = "libvdtb_attn.so"
LIB_PATH = os.path.join(PKG, LIB_NAME)
DEBUG_LIB_PATH = os.path.join(PKG, "libvdtb_attn_debug.so")
BUILD_DIR = os.path.join(PKG, "_build")
SOURCES = ["attn_api.cu", "aux_kernels.cu", "route_tc.cu", "attn_fwd_d128.cu", "attn_fwd_d64.cu", "fp8_gemm.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xptxas", "-warn-spills"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the attention library")


def _fingerprint() -> str:
    h = hashlib.sha256()
    for name in sorted(os.listdir(CSRC)):
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode() + f.read())
    for name in sorted(os.listdir(INCLUDE)):
        with open(os.path.join(INCLUDE, name), "rb") as f:
            h.update(name.encode() + f.read())
    h.update(" ".join(ARCH + NVCC_FLAGS).encode())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile every .cu of csrc/ for sm_103a and link libvdtb_attn.so and libvdtb_attn_debug.so.
    Returns the path of the regular library."""
    fp = _fingerprint()
    stamp = os.path.join(BUILD_DIR, "fingerprint")
    if (not force and os.path.exists(LIB_PATH) and os.path.exists(DEBUG_LIB_PATH) and os.path.exists(stamp)):
        with open(stamp) as f:
            if f.read().strip() == fp:
                return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    nvcc = _nvcc()
    variants = {LIB_PATH: ("", []), DEBUG_LIB_PATH: ("_debug", ["-DATTN_DEBUG"])}

    def compile_one(job) -> str:
        src, suffix, defs = job
        obj = os.path.join(BUILD_DIR, src.replace(".cu", f"{suffix}.o"))
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *defs, f"-I{INCLUDE}", "-c", os.path.join(CSRC, src), "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}{suffix}:\n{res.stdout}\n{res.stderr}")
        if verbose and (res.stdout or res.stderr):
            sys.stderr.write(res.stdout + res.stderr)
        return obj

    jobs = [(src, suffix, defs) for suffix, defs in variants.values() for src in SOURCES]
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        objs = list(ex.map(compile_one, jobs))
    for k, (path, (suffix, _)) in enumerate(variants.items()):
        tmp = path + f".tmp{os.getpid()}"
        cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs[k * len(SOURCES):(k + 1) * len(SOURCES)]]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
        os.replace(tmp, path)
    with open(stamp, "w") as f:
        f.write(fp)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))

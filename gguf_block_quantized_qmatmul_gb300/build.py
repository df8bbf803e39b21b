"""Build the CUDA library (libqmm.so) in-tree with nvcc for sm_103a.

Translation units are compiled in parallel and linked into
``gguf_block_quantized_qmatmul_gb300/_build/libqmm.so``.  No fast-math flags:
the quantizers rely on IEEE round-to-nearest intrinsics.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libqmm.so")
ROOT = os.path.dirname(HERE)
UNITS = ["qmm_api", "qmm_quant", "qmm_stream_q8_0", "qmm_stream_q4_k", "qmm_stream_x_0", "qmm_stream_q6_k", "qmm_gemv_q8_0", "qmm_gemv_q4_k", "qmm_dmma", "qmm_dmma_x_0", "qmm_dmma_q6_k", "qmm_tc", "qmm_tcx", "qmm_tcx_f32", "qmm_static_ws", "qmm_batch", "qmm_batch_mix"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v"]


def _nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libqmm.so")


def _deps():
    out = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    out.append(os.path.join(ROOT, "include", "qmm.h"))
    out.append(os.path.abspath(__file__))
    return out


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    procs = []
    for u in UNITS:
        obj = os.path.join(BUILD, u + ".o")
        log = open(os.path.join(BUILD, u + ".ptxas.txt"), "w")
        cmd = [nvcc, *ARCH, *FLAGS, "-c", os.path.join(CSRC, u + ".cu"), "-o", obj]
        procs.append((u, subprocess.Popen(cmd, stdout=log, stderr=subprocess.STDOUT), log))
    failed = []
    for u, p, log in procs:
        p.wait()
        log.close()
        if p.returncode != 0:
            failed.append(u)
    if failed:
        msgs = "".join(open(os.path.join(BUILD, u + ".ptxas.txt")).read()[-4000:] for u in failed)
        raise RuntimeError(f"nvcc failed for {failed}:\n{msgs}")
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp] + [os.path.join(BUILD, u + ".o") for u in UNITS]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    if verbose:
        print(f"built {LIB}", file=sys.stderr)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)

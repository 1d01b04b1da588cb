"""Build the BitLinear CUDA library in-tree: ``bitlinear_02_b300/libbitlinear.so``.

Every source is compiled for sm_103a only (``-gencode
arch=compute_103a,code=sm_103a``); ninja-free, one nvcc invocation per
translation unit, run in parallel, then linked with nvcc.  ``--debug``
(``build(debug=True)``) builds ``libbitlinear_debug.so`` instead, with
``-DBITLINEAR_DEBUG``: device-side bounds checks on every plain global
access (see include/bitlinear.h).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libbitlinear.so")
DEBUG_OUT_DIR = os.path.join(HERE, "_build_debug")
DEBUG_LIB = os.path.join(HERE, "libbitlinear_debug.so")
SOURCES = ["pack.cu", "quant.cu", "gemv.cu", "fused.cu", "gemm.cu", "variants.cu", "api.cu"]
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
    "--expt-relaxed-constexpr",
]


def _needs(out: str, deps: list[str]) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False, debug: bool = False) -> str:
    out_dir, lib = (DEBUG_OUT_DIR, DEBUG_LIB) if debug else (OUT_DIR, LIB)
    flags = FLAGS + (["-DBITLINEAR_DEBUG"] if debug else [])
    os.makedirs(out_dir, exist_ok=True)
    headers = [os.path.join(CSRC, "bl_device.cuh"), os.path.join(CSRC, "decode_math.cuh"),
               os.path.join(os.path.dirname(HERE), "include", "bitlinear.h")]
    jobs = []
    objs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(out_dir, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _needs(o, [s, *headers]):
            cmd = [NVCC, *flags, "-c", s, "-o", o]
            if ptxas_info:
                cmd.insert(1, "-Xptxas=-v")
            jobs.append(cmd)

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    with cf.ThreadPoolExecutor(max_workers=min(8, max(1, len(jobs)))) as ex:
        for cmd, r in ex.map(run, jobs):
            if verbose or r.returncode != 0 or ptxas_info:
                sys.stderr.write(r.stdout + r.stderr)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed: {' '.join(cmd)}")
    if force or jobs or _needs(lib, objs):
        tmp = lib + f".{os.getpid()}.tmp"
        cmd = [NVCC, "-shared", "-gencode", "arch=compute_103a,code=sm_103a", *objs, "-o", tmp,
               "-lcudart"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
            raise RuntimeError("link failed")
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv,
                debug="--debug" in sys.argv))

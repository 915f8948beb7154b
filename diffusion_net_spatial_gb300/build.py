"""Build the sm_103a shared libraries in-tree (no cmake, no torch extension).

    python -m diffusion_net_spatial_gb300.build

Compiles every ``csrc/*.cu`` to an object in parallel with
``nvcc -gencode arch=compute_103a,code=sm_103a`` and links them into
``diffusion_net_spatial_gb300/libssa_gb300.so`` (C ABI of ``include/ssa.h``,
fp16 tensor-core operands), and the same sources with ``-DSSA_OPERAND_BF16``
into ``libssa_gb300_bf16.so`` (bf16 operands; for comparing the two operand
types).  Objects are rebuilt only when a source or header is newer.
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
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libssa_gb300.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags(extra=()):
    return ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
                   "-I" + os.path.join(ROOT, "include"), "-I" + CSRC] + list(extra)


def _headers_mtime() -> float:
    hs = glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(ROOT, "include", "*.h"))
    return max((os.path.getmtime(h) for h in hs), default=0.0)


VARIANTS = {  # library -> (object folder, extra nvcc flags)
    "f16": (os.path.join(PKG, "_build"), []),
    "bf16": (os.path.join(PKG, "_build_bf16"), ["-DSSA_OPERAND_BF16"]),
}


def lib_path(operand: str = "f16") -> str:
    return LIB if operand == "f16" else os.path.join(PKG, f"libssa_gb300_{operand}.so")


def build(verbose: bool = False, ptxas_verbose: bool = False, force: bool = False, operands=("f16", "bf16")) -> str:
    nvcc = nvcc_path()
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    hdr_t = _headers_mtime()
    jobs = []
    objs = {}
    for op in operands:
        out_dir, extra_def = VARIANTS[op]
        os.makedirs(out_dir, exist_ok=True)
        objs[op] = []
        for s in srcs:
            o = os.path.join(out_dir, os.path.basename(s)[:-3] + ".o")
            objs[op].append(o)
            if force or ptxas_verbose or not os.path.exists(o) or os.path.getmtime(o) < max(os.path.getmtime(s), hdr_t):
                extra = (["-Xptxas", "-v"] if ptxas_verbose else []) + extra_def
                jobs.append([nvcc] + _flags(extra) + ["-c", s, "-o", o])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    errors = []
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            for cmd, r in ex.map(run, jobs):
                if verbose or ptxas_verbose or r.returncode:
                    sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
                if r.returncode:
                    errors.append(cmd[-3])
    if errors:
        raise RuntimeError("nvcc failed for: " + ", ".join(errors))
    for op in operands:
        lib = lib_path(op)
        if jobs or not os.path.exists(lib) or any(os.path.getmtime(o) > os.path.getmtime(lib) for o in objs[op]):
            cmd = [nvcc] + ARCH + ["-shared", "-o", lib] + objs[op] + ["-lcudart_static", "-ldl", "-lpthread", "-lrt"]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if verbose or r.returncode:
                sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
            if r.returncode:
                raise RuntimeError("link failed")
    return LIB


if __name__ == "__main__":
    build(verbose="-v" in sys.argv, ptxas_verbose="--ptxas" in sys.argv, force="-f" in sys.argv)
    print(LIB)

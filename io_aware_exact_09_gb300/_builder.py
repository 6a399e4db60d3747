"""Build the CUDA library in-tree: nvcc for sm_103a, one object per .cu in
parallel, linked into ``libfa_gb300.so`` beside this file (static cudart, so
the library loads without a GPU driver present)."""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libfa_gb300.so")
SOURCES = ["fa_api.cu", "fa_fwd.cu", "fa_fwd_fp8.cu", "fa_bwd.cu", "fa_bwd64.cu", "fa_bwd128.cu", "fa_decode.cu", "fa_quant.cu", "fa_selftest.cu", "fa_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
                "--expt-relaxed-constexpr", "-I", os.path.join(HERE, "..", "include")]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    deps.append(os.path.join(HERE, "..", "include", "fa.h"))
    deps.append(os.path.abspath(__file__))
    return any(os.path.getmtime(p) > t for p in deps)


def _compile(src: str) -> str:
    obj = os.path.join(BUILD, src.replace(".cu", ".o"))
    log = os.path.join(BUILD, src.replace(".cu", ".ptxas.log"))
    cmd = [nvcc()] + FLAGS + ["-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    with open(log, "w") as f:
        f.write(r.stdout + r.stderr)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed for %s:\n%s" % (src, r.stdout + r.stderr))
    return obj


# Kernels that split registers between warpgroups with setmaxnreg: the
# split in the source assumes exactly this many registers per thread at
# launch; a different allocation would make setmaxnreg.inc wait forever, so
# the build refuses it.
REGISTER_SPLIT_KERNELS = {"fa_fwd.cu": ("fa_fwd_kernel", 168), "fa_fwd_fp8.cu": ("fa_fwd_fp8_kernel", 168),
                          "fa_bwd64.cu": ("fa_bwd64_kernel", 128), "fa_bwd128.cu": ("fa_bwd128_kernel", 128)}


def _check_register_split(src: str) -> None:
    if src not in REGISTER_SPLIT_KERNELS:
        return
    name, want = REGISTER_SPLIT_KERNELS[src]
    log = open(os.path.join(BUILD, src.replace(".cu", ".ptxas.log"))).read().splitlines()
    found = 0
    for i, line in enumerate(log):
        if "Compiling entry function" in line and name in line:
            for nxt in log[i + 1:i + 6]:
                if "Used" in nxt and "registers" in nxt:
                    regs = int(nxt.split("Used")[1].split("registers")[0])
                    if regs != want:
                        raise RuntimeError("%s: ptxas allocated %d registers, the setmaxnreg split needs %d"
                                           % (name, regs, want))
                    found += 1
                    break
    if found == 0:
        raise RuntimeError("%s: no ptxas register report found" % name)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(_compile, SOURCES))
    for src in SOURCES:
        _check_register_split(src)
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs + ["-ldl"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s" % (r.stdout + r.stderr))
    os.replace(tmp, LIB)
    if verbose:
        for s in SOURCES:
            sys.stdout.write(open(os.path.join(BUILD, s.replace(".cu", ".ptxas.log"))).read())
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)

"""Build libmbx.so in-tree: one nvcc job per translation unit (in parallel),
then one link.  sm_103a only; no CPU code path is built."""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
KERN = os.path.join(CSRC, "kernels")
OBJ = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libmbx.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

SOURCES = [
    os.path.join(CSRC, "mbx_api.cu"),
    os.path.join(KERN, "ln_modulate.cu"),
    os.path.join(KERN, "ln_nvfp4.cu"),
    os.path.join(KERN, "rmsnorm.cu"),
    os.path.join(KERN, "residual.cu"),
    os.path.join(KERN, "qkv.cu"),
    os.path.join(KERN, "modtable.cu"),
    os.path.join(KERN, "selftest.cu"),
]
HEADERS = [os.path.join(KERN, f) for f in os.listdir(KERN) if f.endswith((".cuh", ".h", ".inc"))]
HEADERS.append(os.path.join(INCLUDE, "mbx.h"))

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + [
    "-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr",
    # IEEE binary32: no flush-to-zero, correctly rounded division and sqrt,
    # and no contraction of a multiply and an add into one fused operation,
    # neither by the front end nor by ptxas (ptxas otherwise fuses even
    # explicitly rounded mul.rn.f32x2 / add.rn.f32x2 pairs).  Fused
    # multiply-adds the kernels want are written as explicit fma instructions.
    "-ftz=false", "-prec-div=true", "-prec-sqrt=true", "-fmad=false", "-Xptxas", "-fmad=false",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
    "-I", INCLUDE,
]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmbx.so")


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra: list[str] | None = None) -> str:
    os.makedirs(OBJ, exist_ok=True)
    cc = nvcc()
    flags = NVCC_FLAGS + (extra or [])
    objs, jobs = [], []
    for src in SOURCES:
        obj = os.path.join(OBJ, os.path.basename(src).replace(".cu", ".o"))
        objs.append(obj)
        if force or _stale(obj, [src] + HEADERS):
            jobs.append([cc, *flags, "-c", src, "-o", obj])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)

    with cf.ThreadPoolExecutor(max_workers=len(jobs) or 1) as ex:
        list(ex.map(run, jobs))
    if force or jobs or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        run([cc, *ARCH, "-shared", "-o", tmp, *objs])
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True,
                extra=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else None))

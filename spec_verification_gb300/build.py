"""Compile libss.so (the CUDA kernels and their C ABI) in-tree for sm_103a.

Each .cu file is compiled to an object in parallel with nvcc, then linked
into spec_verification_gb300/_build/libss.so against the CUDA runtime.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
INCLUDE = ROOT / "include"
BUILD = PKG / "_build"
LIB = BUILD / "libss.so"
SOURCES = ["ss_api.cu", "ss_stage1.cu", "ss_stage1_f32.cu", "ss_stage1_bf16.cu", "ss_stage1_exact.cu",
           "ss_stage2.cu", "ss_residual.cu", "ss_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for c in (os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"):
        p = Path(c) / "bin" / "nvcc" if c else None
        if p and p.exists():
            return str(p)
    p = shutil.which("nvcc")
    if not p:
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libss.so")
    return p


def flags() -> list:
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
                   "-I", str(INCLUDE), "-I", str(CSRC)]


def _stale(obj: Path, src: Path) -> bool:
    if not obj.exists():
        return True
    deps = [src, INCLUDE / "ss.h", CSRC / "ss_common.cuh", CSRC / "ss_stage1.cuh", CSRC / "ss_stage2.cuh", Path(__file__)]
    return any(d.exists() and d.stat().st_mtime > obj.stat().st_mtime for d in deps)


def build(force: bool = False, verbose: bool = False, extra: list | None = None) -> Path:
    BUILD.mkdir(exist_ok=True)
    cc = nvcc()
    objs = []
    jobs = []
    for s in SOURCES:
        src = CSRC / s
        obj = BUILD / (s[:-3] + ".o")
        objs.append(obj)
        if force or _stale(obj, src):
            jobs.append([cc, *flags(), *(extra or []), "-c", str(src), "-o", str(obj)])
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
            for cmd, res in zip(jobs, ex.map(lambda c: subprocess.run(c, capture_output=True, text=True), jobs)):
                if verbose or res.returncode != 0:
                    print(" ".join(cmd))
                    print(res.stdout, res.stderr)
                if res.returncode != 0:
                    raise RuntimeError(f"nvcc failed for {cmd[-3]}")
    if jobs or not LIB.exists():
        tmp = LIB.with_suffix(f".{os.getpid()}.tmp.so")
        cmd = [cc, *ARCH, "-shared", "-o", str(tmp), *map(str, objs), "-lcudart", "-ldl"]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            print(" ".join(cmd), res.stdout, res.stderr)
            raise RuntimeError("link of libss.so failed")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

"""Build libgqa_attn.so in-tree with nvcc for sm_103a.

Usage: ``python -m gqa_attention_gb300.build`` (or ``build()`` from Python).
Each ``csrc/*.cu`` is compiled in parallel to an object under ``_build/`` and
the objects are linked into ``gqa_attention_gb300/libgqa_attn.so`` against the
shared CUDA runtime (``libcudart.so.13``), so that a process that also uses
PyTorch holds one runtime instance.  Rebuilds only what changed.
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
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libgqa_attn.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def cuda_home() -> str:
    home = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH")
    if home and os.path.exists(os.path.join(home, "bin", "nvcc")):
        return home
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    return "/usr/local/cuda"


def _nvcc() -> str:
    return os.path.join(cuda_home(), "bin", "nvcc")


def _cflags(extra=()):
    return [*ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
            "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC, *extra]


def _deps_mtime() -> float:
    files = glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]
    return max(os.path.getmtime(f) for f in files)


def _compile(src: str, obj: str, extra) -> str:
    cmd = [_nvcc(), *_cflags(extra), "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stderr}\n{r.stdout}")
    return r.stderr


def build(force: bool = False, verbose: bool = False, extra_flags=(), lib_path: str = LIB,
          build_dir: str = BUILD) -> str:
    """Compile every csrc/*.cu for sm_103a and link libgqa_attn.so; return its path.

    ``extra_flags``, ``lib_path`` and ``build_dir`` let a tuning run build a
    variant (e.g. ``-DGQA_DECODE_STAGES_D128=4``) beside the default library.
    """
    BUILD_, LIB_ = build_dir, lib_path
    os.makedirs(BUILD_, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    dep_t = _deps_mtime()
    jobs = []
    for src in srcs:
        obj = os.path.join(BUILD_, os.path.basename(src)[:-3] + ".o")
        if force or not os.path.exists(obj) or os.path.getmtime(obj) < max(
                os.path.getmtime(src), dep_t):
            jobs.append((src, obj))
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 1))) as ex:
            futs = {ex.submit(_compile, s, o, list(extra_flags)): s for s, o in jobs}
            for f in cf.as_completed(futs):
                msg = f.result()
                if verbose and msg:
                    print(f"[{os.path.basename(futs[f])}]\n{msg}", file=sys.stderr)
    objs = [os.path.join(BUILD_, os.path.basename(s)[:-3] + ".o") for s in srcs]
    if jobs or force or not os.path.exists(LIB_):
        lib64 = os.path.join(cuda_home(), "lib64")
        tmp = LIB_ + f".tmp{os.getpid()}"
        cmd = [_nvcc(), *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
               "-Xlinker", f"-rpath,{lib64}", "-Xlinker", "--no-undefined"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr}\n{r.stdout}")
        os.replace(tmp, LIB_)
    return LIB_


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv,
          extra_flags=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else [])
    print(LIB)

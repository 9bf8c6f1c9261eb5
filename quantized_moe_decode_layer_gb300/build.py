"""Build of the in-tree CUDA library libmoe.so for sm_103a.

The eight translation units compile in parallel with nvcc
(-gencode arch=compute_103a,code=sm_103a) and link into
quantized_moe_decode_layer_gb300/libmoe.so next to this file.  Objects go to
_build/ at the repository root.  build(debug_bounds=True) makes the
bounds-checked variant, libmoe_debug.so (the same sources compiled with
-DMOE_DEBUG_BOUNDS), which the binding loads when MOE_DEBUG_BOUNDS=1 is set.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "libmoe.so")
OUT_DEBUG = os.path.join(HERE, "libmoe_debug.so")
OBJDIR = os.path.join(ROOT, "_build")
SOURCES = ["moe_abi.cu", "moe_pack.cu", "moe_layer.cu", "moe_layer_w8.cu", "moe_tc.cu", "moe_grouped.cu", "moe_attn.cu",
           "moe_stream.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    p = shutil.which("nvcc")
    if p:
        return p
    for c in ("/usr/local/cuda/bin/nvcc",):
        if os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmoe.so")


def _stale(out: str) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(ROOT, "include", "moe.h")]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, extra_flags=(), debug_bounds: bool = False) -> str:
    out = OUT_DEBUG if debug_bounds else OUT
    if not force and not _stale(out):
        return out
    objdir = os.path.join(OBJDIR, "debug") if debug_bounds else OBJDIR
    os.makedirs(objdir, exist_ok=True)
    cc = nvcc()
    flags = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", *ARCH, *extra_flags]
    if debug_bounds:
        flags.append("-DMOE_DEBUG_BOUNDS=1")

    def compile_one(src):
        obj = os.path.join(objdir, src.replace(".cu", ".o"))
        cmd = [cc, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj

    with cf.ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = out + f".tmp{os.getpid()}"
    r = subprocess.run([cc, "-shared", *ARCH, "-cudart", "static", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)
    return out


def build_all(force: bool = False) -> None:
    """Both variants, in parallel."""
    with cf.ThreadPoolExecutor(2) as ex:
        list(ex.map(lambda d: build(force=force, debug_bounds=d), (False, True)))


if __name__ == "__main__":
    build_all(force=True)
    print(OUT, OUT_DEBUG)

"""Build libfme.so (the CUDA library behind include/fme.h) for sm_103a with nvcc.

Every translation unit is compiled in parallel, then linked into
``fp8_moe_expert_gb300/libfme.so`` (git-ignored, rebuilt on each machine: the
object code is architecture specific and the host code is built for the host
it runs on).  Usage: ``python -m fp8_moe_expert_gb300.build``.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
LIBRARY = os.path.join(HERE, "libfme.so")
BUILD_DIR = os.path.join(HERE, "_build")
SOURCES = ["api.cu", "quant_nvfp4.cu", "quant_mxfp8.cu", "gemm.cu", "gemm_nvfp4.cu", "route.cu"]
HEADERS = ["fme_device.cuh", "fme_launch.h", "gemm_common.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libfme.so")


def _inputs() -> list[str]:
    files = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    files.append(os.path.join(ROOT, "include", "fme.h"))
    return files


def stale(output: str = LIBRARY) -> bool:
    if not os.path.exists(output):
        return True
    t = os.path.getmtime(output)
    return any(os.path.getmtime(f) > t for f in _inputs())


def build(output: str = LIBRARY, extra_flags: list[str] | None = None, verbose: bool = False) -> str:
    """Compile and link the library; returns its path."""
    flags = NVCC_FLAGS + (extra_flags or [])
    tool = nvcc()
    # objects and nvcc's own intermediates stay inside the package tree (git-ignored)
    os.makedirs(BUILD_DIR, exist_ok=True)
    with tempfile.TemporaryDirectory(prefix=f"{os.getpid()}_", dir=BUILD_DIR) as tmp:
        env = dict(os.environ, TMPDIR=tmp)

        def compile_one(src: str) -> str:
            obj = os.path.join(tmp, os.path.splitext(src)[0] + ".o")
            cmd = [tool, *ARCH, *flags, "-I", os.path.join(ROOT, "include"), "-c",
                   os.path.join(CSRC, src), "-o", obj]
            res = subprocess.run(cmd, capture_output=True, text=True, env=env)
            if res.returncode != 0:
                raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
            if verbose:
                sys.stderr.write(res.stdout + res.stderr)
            return obj

        with ThreadPoolExecutor(max_workers=len(SOURCES)) as pool:
            objs = list(pool.map(compile_one, SOURCES))
        tmp_out = output + ".tmp"
        cmd = [tool, *ARCH, "-shared", "-o", tmp_out, *objs]
        res = subprocess.run(cmd, capture_output=True, text=True, env=env)
        if res.returncode != 0:
            raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
        os.replace(tmp_out, output)
    return output


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))

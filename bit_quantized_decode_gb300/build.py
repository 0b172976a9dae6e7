"""Build the sm_103a shared library ``libw4a8.so`` in the package directory.

nvcc compiles each translation unit under ``csrc/`` in parallel for
``compute_103a``/``sm_103a`` and links them into a C-ABI shared library with
the CUDA runtime linked statically.  Quantization must be IEEE-exact, so the
build keeps precise division and does not flush denormals.

Usage: ``python -m bit_quantized_decode_gb300.build [--force]``.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
OBJDIR = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libw4a8.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = [
    "-O3", "-std=c++17", "-lineinfo", *ARCH,
    "-Xcompiler", "-fPIC",
    "-prec-div=true", "-prec-sqrt=true", "-ftz=false",
    "-Xptxas", "-v",
    "-I", INCLUDE,
]
SOURCES = ["gemv_w4.cu", "gemv_q4_0.cu", "gemv_q6g32.cu", "gemv_i8g32.cu", "gemv_a32.cu", "w4a8_api.cu",
           "prep_kernels.cu", "gemv_tc.cu", "gemv_chain.cu", "hbm_read.cu", "host_quant.cpp"]
# host-only C++ (the host quantizers): IEEE arithmetic as written, no FMA contraction
HOST_FLAGS = ["-O2", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-ffp-contract=off",
              "-Xcompiler", "-fno-fast-math", "-I", INCLUDE]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libw4a8.so")


def _inputs_digest() -> str:
    h = hashlib.sha256()
    for d in (CSRC, INCLUDE):
        for name in sorted(os.listdir(d)):
            if name.endswith((".cu", ".cuh", ".h", ".cpp")):
                with open(os.path.join(d, name), "rb") as f:
                    h.update(name.encode())
                    h.update(f.read())
    h.update(" ".join(NVCC_FLAGS + HOST_FLAGS).encode())
    return h.hexdigest()


# Sources that define the one-token decode GEMV (stream_linear_kernel<W4, 1, fused>):
# a profile summary taken on them stays valid while they are unchanged.
GEMV_W4_SOURCES = ("gemv_kernel.cuh", "quant_a8.cuh", "fusion.cuh", "ptx.cuh", "internal.h", "gemv_w4.cu")


def kernel_digest(names=GEMV_W4_SOURCES) -> str:
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    # the include directory is an absolute path that differs between checkouts
    h.update(" ".join("include" if f == INCLUDE else f for f in NVCC_FLAGS).encode())
    return h.hexdigest()


def _stamp_path() -> str:
    return LIB + ".stamp"


def up_to_date() -> bool:
    if not os.path.exists(LIB) or not os.path.exists(_stamp_path()):
        return False
    with open(_stamp_path()) as f:
        return f.read().strip() == _inputs_digest()


def _compile(src: str, log: list) -> str:
    obj = os.path.join(OBJDIR, os.path.splitext(src)[0] + ".o")
    flags = HOST_FLAGS if src.endswith(".cpp") else NVCC_FLAGS
    cmd = [nvcc(), *flags, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    log.append((src, r.stdout + r.stderr))
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    return obj


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile (if stale) and return the path of libw4a8.so."""
    if not force and up_to_date():
        return LIB
    os.makedirs(OBJDIR, exist_ok=True)
    log: list = []
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, log), SOURCES))
    tmp = LIB + f".tmp{os.getpid()}"
    r = subprocess.run([nvcc(), *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(os.path.join(OBJDIR, "ptxas.log"), "w") as f:
        for src, text in log:
            f.write(f"==== {src}\n{text}\n")
    with open(_stamp_path(), "w") as f:
        f.write(_inputs_digest())
    if verbose:
        for src, text in log:
            print(f"==== {src}\n{text}")
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

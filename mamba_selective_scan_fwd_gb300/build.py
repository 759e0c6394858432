"""Build ``libss.so`` (the sm_103a selective-scan library) in-tree with nvcc.

The library is plain CUDA C++ with an ``extern "C"`` ABI (include/ss.h); no
torch headers are involved.  Translation units compile in parallel; the CUDA
runtime is linked statically so the shared object only needs the driver.
"""

from __future__ import annotations

import hashlib
import os
import re
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libss.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v"]
SOURCES = ["api.cu", "dispatch.cu", "fwd_f32.cu", "fwd_bf16.cu", "fwd_f16.cu", "bwd_f32.cu",
           "bwd_bf16.cu", "bwd_f16.cu", "decode.cu", "fwd_noalloc.cu", "probe.cu"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libss.so")


def _digest() -> str:
    h = hashlib.sha256()
    h.update(" ".join(ARCH + NVCC_FLAGS + SOURCES).encode())
    deps = sorted(f for f in os.listdir(CSRC) if f.endswith((".cu", ".cuh", ".h")))
    for name in deps:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode() + f.read())
    with open(os.path.join(ROOT, "include", "ss.h"), "rb") as f:
        h.update(f.read())
    return h.hexdigest()


# a string or character literal (kept), or a comment (dropped)
_TOKEN = re.compile(r'"(?:\\.|[^"\\])*"|\'(?:\\.|[^\'\\])*\'|//[^\n]*|/\*.*?\*/', re.S)


def _code(text: str) -> str:
    """Source text without comments, whitespace runs collapsed: what the compiler sees."""
    text = _TOKEN.sub(lambda m: m.group(0) if m.group(0)[0] in "\"'" else " ", text)
    return re.sub(r"\s+", " ", text).strip()


def source_digest() -> str:
    """Digest of the kernel sources (comments and layout ignored) and build flags:
    changes whenever the compiled kernels may change, and only then."""
    h = hashlib.sha256()
    h.update(" ".join(ARCH + NVCC_FLAGS + SOURCES).encode())
    deps = sorted(f for f in os.listdir(CSRC) if f.endswith((".cu", ".cuh", ".h")))
    for name in deps:
        with open(os.path.join(CSRC, name), encoding="utf-8") as f:
            h.update(name.encode() + _code(f.read()).encode())
    with open(os.path.join(ROOT, "include", "ss.h"), encoding="utf-8") as f:
        h.update(_code(f.read()).encode())
    return h.hexdigest()[:16]


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile every translation unit and link libss.so; skipped when up to date."""
    os.makedirs(BUILD, exist_ok=True)
    stamp = os.path.join(BUILD, "stamp")
    dig = _digest()
    if not force and os.path.exists(LIB) and os.path.exists(stamp) and open(stamp).read() == dig:
        return LIB
    exe = nvcc()

    def compile_one(src):
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        cmd = [exe, *ARCH, *NVCC_FLAGS, "-I", os.path.join(ROOT, "include"), "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        with open(obj + ".log", "w") as f:
            f.write(r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr[-4000:]}")
        if verbose:
            print(r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [exe, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link of libss.so failed:\n{r.stderr[-4000:]}")
    os.replace(tmp, LIB)
    with open(stamp, "w") as f:
        f.write(dig)
    return LIB


if __name__ == "__main__":
    print(build(force=True))

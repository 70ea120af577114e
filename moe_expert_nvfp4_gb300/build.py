"""Build libnvfp4moe.so in-tree with nvcc for sm_103a.

Each translation unit is compiled in parallel to an object file under
``_build/``, then linked into ``moe_expert_nvfp4_gb300/libnvfp4moe.so``
(CUDA runtime linked statically).  Rebuilds only when a source is newer
than the library.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libnvfp4moe.so")
SOURCES = ["api.cu", "route.cu", "stream_tc.cu", "fma.cu", "moe_fma.cu", "noalloc.cu", "rows.cu", "quant.cu",
           "probe.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "-ftz=false", "-prec-div=true", "-prec-sqrt=true"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libnvfp4moe.so")


def _deps() -> list[str]:
    out = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    out.append(os.path.join(ROOT, "include", "nvfp4moe.h"))
    out.append(os.path.abspath(__file__))
    return out


def source_hash(files=None) -> str:
    """sha256 over the kernel sources and the public header (identifies the
    kernel version a profile was taken on).  ``files`` (names under csrc/)
    narrows it to one kernel's sources: a counter taken on that kernel stays
    valid while they and the header are unchanged."""
    import hashlib
    h = hashlib.sha256()
    for f in sorted(files if files is not None else os.listdir(CSRC)):
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(f.encode() + b"\0" + fh.read())
    with open(os.path.join(ROOT, "include", "nvfp4moe.h"), "rb") as fh:
        h.update(fh.read())
    return h.hexdigest()[:16]


def needs_build() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(d) > t for d in _deps())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not needs_build():
        return LIB
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)

    def compile_one(src: str) -> str:
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        cmd = [nvcc, *ARCH, *FLAGS, "-I", os.path.join(ROOT, "include"), "-c",
               os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        # nvcc 13.0's device front end has been seen to crash (SIGSEGV) now and
        # then on the large persistent kernel with the same input that
        # compiles on the next try: retry a crash, never a compile error
        for attempt in range(4):
            r = subprocess.run(cmd, capture_output=True, text=True)
            crashed = r.returncode < 0 or "Segmentation fault" in r.stderr
            if r.returncode == 0 or not crashed:
                break
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and r.stderr:
            sys.stderr.write(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

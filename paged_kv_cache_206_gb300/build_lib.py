"""Build libpa.so in-tree with nvcc for sm_103a.

Each translation unit under ``csrc/`` compiles in parallel to an object under
``_build/obj``; the objects link into ``_build/libpa.so``. Nothing is rebuilt
when every object is newer than its source and every header, and the build
stamp (machine, compiler version, flags) matches the one the objects were made
with; objects from another machine or compiler are never reused. The CUDA runtime
is linked statically and the driver is reached through the runtime's
entry-point query, so the library loads on a machine without a GPU.
"""
from __future__ import annotations

import glob
import hashlib
import os
import platform
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libpa.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
                f"-I{INCLUDE}", f"-I{CSRC}", "--expt-relaxed-constexpr"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpa.so")


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))


def _headers_mtime() -> float:
    hs = glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]
    return max(os.path.getmtime(h) for h in hs)


def _stamp(cc: str) -> str:
    """What the objects depend on beyond their sources: the machine, the
    compiler and the flags."""
    ver = subprocess.run([cc, "--version"], capture_output=True, text=True).stdout
    text = "\n".join([platform.machine(), ver, " ".join(FLAGS), " ".join(ARCH)])
    return hashlib.sha256(text.encode()).hexdigest()[:16]


def build(force: bool = False, verbose: bool = False, jobs: int | None = None) -> str:
    """Compile what is stale and link; returns the library path."""
    os.makedirs(os.path.join(BUILD, "obj"), exist_ok=True)
    cc = nvcc()
    stamp_path = os.path.join(BUILD, "stamp")
    stamp = _stamp(cc)
    if not os.path.exists(stamp_path) or open(stamp_path).read().strip() != stamp:
        force = True  # objects (if any) from another machine, compiler or flag set
    hdr = _headers_mtime()
    objs, todo = [], []
    for src in sources():
        obj = os.path.join(BUILD, "obj", os.path.basename(src) + ".o")
        objs.append(obj)
        if force or not os.path.exists(obj) or os.path.getmtime(obj) < max(hdr, os.path.getmtime(src)):
            todo.append((src, obj))

    def compile_one(job):
        src, obj = job
        tmp = obj + f".tmp{os.getpid()}"
        cmd = [cc, *FLAGS, "-c", src, "-o", tmp]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr}")
        os.replace(tmp, obj)
        return r.stderr

    if todo:
        jobs = jobs or min(len(todo), max(1, len(os.sched_getaffinity(0))))
        with ThreadPoolExecutor(jobs) as ex:
            logs = list(ex.map(compile_one, todo))
        if verbose:
            for (src, _), log in zip(todo, logs):
                print(f"== {os.path.basename(src)}\n{log}")
    if todo or force or not os.path.exists(LIB):
        tmp = LIB + f".tmp{os.getpid()}"
        r = subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"],
                           capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link of libpa.so failed:\n{r.stderr}")
        os.replace(tmp, LIB)
        with open(stamp_path, "w") as f:
            f.write(stamp + "\n")
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

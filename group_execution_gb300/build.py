"""Builds libgroupexec.so in-tree for sm_103a (GB300).

Every translation unit compiles in parallel with nvcc (CUDA) or g++ (host
C++); the CUDA runtime is linked statically, and the driver API is reached at
run time through the runtime's entry-point lookup, so the library loads on a
machine without a GPU driver (graph building and grouping then still work).
"""
from __future__ import annotations

import concurrent.futures as cf
import fcntl
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libgroupexec.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _cuda_home():
    for c in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if c and os.path.exists(os.path.join(c, "bin", "nvcc")):
            return c
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(nvcc))
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libgroupexec.so")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cpp")))


def headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    return hs + [os.path.join(ROOT, "include", "groupexec.h"), __file__]


EMBED = ("fg_abi.h", "fg_device.cuh", "group_kernels.cuh", "gemm_kernel.cuh")
EMBED_NAMES = ("kEmbedAbi", "kEmbedDevice", "kEmbedKernels", "kEmbedGemm")


def write_embed():
    """Raw-string copies of the device headers for run-time compilation of
    group programs (their local #include lines dropped: the texts are
    concatenated in dependency order)."""
    os.makedirs(BUILD, exist_ok=True)
    out = []
    for f, name in zip(EMBED, EMBED_NAMES):
        text = "".join(ln for ln in open(os.path.join(CSRC, f)) if not ln.lstrip().startswith('#include "'))
        assert ")FGSRC" not in text
        out.append(f'static const char* {name} = R"FGSRC(\n{text})FGSRC";\n')
    path = os.path.join(BUILD, "jit_embed.inc")
    new = "".join(out)
    if not os.path.exists(path) or open(path).read() != new:
        open(path, "w").write(new)


def _cmd(src, obj, cuda):
    inc = ["-I", os.path.join(cuda, "include"), "-I", CSRC, "-I", os.path.join(ROOT, "include"), "-I", BUILD]
    if src.endswith(".cu"):
        return [os.path.join(cuda, "bin", "nvcc"), *ARCH, "-O3", "-lineinfo", "-std=c++17",
                "-Xcompiler", "-fPIC", "-Xptxas", "-warn-spills", *inc, "-c", src, "-o", obj]
    return ["g++", "-O2", "-std=c++17", "-fPIC", "-Wall", "-ffp-contract=off", *inc, "-c", src, "-o", obj]


def stale():
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in sources() + headers())


def build(force=False, verbose=False, jobs=None):
    """Compile (if stale) and return the path of libgroupexec.so.  Processes
    building at once (parallel test workers) take turns on a lock file; the
    others then find the library fresh."""
    if not force and not stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    with open(os.path.join(BUILD, ".lock"), "w") as lk:
        fcntl.flock(lk, fcntl.LOCK_EX)
        try:
            if not force and not stale():
                return LIB
            return _build_locked(verbose, jobs)
        finally:
            fcntl.flock(lk, fcntl.LOCK_UN)


def _build_locked(verbose, jobs):
    cuda = _cuda_home()
    write_embed()
    srcs = sources()
    objs = [os.path.join(BUILD, os.path.basename(s) + ".o") for s in srcs]

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if verbose or r.returncode:
            sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        if r.returncode:
            raise RuntimeError(f"compilation failed: {cmd[-3]}")
        return r.stderr

    with cf.ThreadPoolExecutor(max_workers=jobs or min(8, len(srcs))) as ex:
        list(ex.map(run, [_cmd(s, o, cuda) for s, o in zip(srcs, objs)]))
    tmp = LIB + ".tmp"
    run([os.path.join(cuda, "bin", "nvcc"), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs,
         "-lpthread", "-ldl", "-lrt"])
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
    print(LIB)

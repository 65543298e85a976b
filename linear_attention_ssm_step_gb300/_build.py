"""Build the CUDA library libkda_gb300.so in-tree with nvcc (sm_103a only).

Each translation unit compiles in its own nvcc process, in parallel, then one
nvcc -shared links them. No cmake, no torch extension machinery.
"""

import os
import shutil
import subprocess
import sys

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG_DIR, "_build")
LIB_PATH = os.path.join(PKG_DIR, "libkda_gb300.so")

SOURCES = ["kda_api.cu", "kda_step.cu", "kda_ring.cu", "kda_tmap.cu", "kda_verify_tc.cu", "kda_fp8.cu",
           "kda_prefill.cu", "kda_prefill_tc.cu", "kda_prefill_chain.cu"]
HEADERS = ["kda_device.cuh", "kda_launch.h", "kda_tc.cuh", "kda_chunk.cuh", "kda_fp8_codec.cuh"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# --fmad=false: no implicit mul+add contraction anywhere, so every fused
# multiply-add in the kernels is an explicit one and the same source gives the
# same bits in every kernel that inlines it.
CFLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "--fmad=false", "-Xcompiler", "-fPIC",
                 "-I", INCLUDE, "-I", CSRC]


def _nvcc():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        raise RuntimeError("nvcc not found; the CUDA 13 toolkit is required to build libkda_gb300.so")
    return nvcc


def _inputs():
    files = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [os.path.join(INCLUDE, h) for h in ("kda.h", "kda_fp8.h", "kda_prefill.h")]
    files.append(os.path.abspath(__file__))
    return files


# Builds of the same sources for tests only, by name: their own library file
# and object folder, extra compiler definitions. "waittest" is the
# failure-detection build: every asynchronous global -> shared copy is left
# unissued and the bounded waits give up after 2 ms, so each kernel's timeout
# path runs without a fault (kda_device.cuh, KDA_WITHHOLD_LOADS).
VARIANTS = {
    "waittest": ["-DKDA_WITHHOLD_LOADS", "-DKDA_WAIT_LIMIT_NS=2000000ull"],
}


def lib_path(variant=None):
    if variant is None:
        return LIB_PATH
    return os.path.join(PKG_DIR, f"libkda_gb300_{variant}.so")


def is_stale(variant=None):
    path = lib_path(variant)
    if not os.path.exists(path):
        return True
    t = os.path.getmtime(path)
    return any(os.path.getmtime(f) > t for f in _inputs())


def build(force=False, verbose=False, variant=None):
    """Compile and link libkda_gb300.so (or a test variant of it); returns its path."""
    path = lib_path(variant)
    if not force and not is_stale(variant):
        return path
    nvcc = _nvcc()
    bdir = BUILD_DIR if variant is None else os.path.join(BUILD_DIR, variant)
    extra = [] if variant is None else VARIANTS[variant]
    os.makedirs(bdir, exist_ok=True)
    procs = []
    objs = []
    for src in SOURCES:
        obj = os.path.join(bdir, src.replace(".cu", ".o"))
        objs.append(obj)
        cmd = ([nvcc] + CFLAGS + extra + (["-Xptxas", "-v"] if verbose else []) +
               ["-c", os.path.join(CSRC, src), "-o", obj])
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if verbose and out:
            sys.stdout.write(out)
        if p.returncode != 0:
            failed.append((src, out))
    if failed:
        raise RuntimeError("nvcc failed:\n" + "\n".join(f"--- {s}\n{o}" for s, o in failed))
    tmp = path + ".tmp"
    link = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout)
    os.replace(tmp, path)
    return path


if __name__ == "__main__":
    print(build(force=True, verbose="-v" in sys.argv))

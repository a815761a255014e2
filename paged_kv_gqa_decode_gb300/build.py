"""Build the sm_103a shared library (nvcc, one translation unit per head_dim, in parallel).

The library lands in ``paged_kv_gqa_decode_gb300/lib/libpaged_kv_gqa_decode.so``.
``python -m paged_kv_gqa_decode_gb300.build`` or ``__graft_entry__.build()``
runs it; nothing here is needed at run time.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_DIR = os.path.join(PKG, "lib")
LIB_NAME = "libpaged_kv_gqa_decode.so"
LIB_PATH = os.path.join(LIB_DIR, LIB_NAME)
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["paged_attn_api.cu", "append.cu", "decode_d64.cu", "decode_d128.cu",
           "decode_d256.cu", "decode_fp8_d128.cu", "decode_fp8_d256.cu", "decode_xp_d64.cu",
           "decode_xp_d128.cu", "decode_xp_d256.cu", "decode_multi_d64.cu",
           "decode_multi_d128.cu", "decode_multi_d256.cu"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA 13 toolkit is required to build")
    return cand


def _flags():
    # hidden default visibility: only the C ABI (marked in paged_attn.h) is exported,
    # so nothing internal (e.g. a template's static locals) is shared between two
    # copies of the library loaded into one process
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler",
                   "-fPIC,-O2,-fvisibility=hidden,-fvisibility-inlines-hidden",
                   "-I", INCLUDE, "-I", CSRC, "--expt-relaxed-constexpr", "-Xptxas", "-v"]


def source_digest() -> str:
    """sha256 over the kernel sources and the public header (identifies a build)."""
    h = hashlib.sha256()
    names = sorted(os.listdir(CSRC))
    for n in names:
        if n.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(CSRC, n), "rb") as f:
                h.update(n.encode() + b"\0" + f.read())
    with open(os.path.join(INCLUDE, "paged_attn.h"), "rb") as f:
        h.update(f.read())
    return h.hexdigest()


def build(verbose: bool = False, force: bool = False) -> str:
    os.makedirs(LIB_DIR, exist_ok=True)
    obj_dir = os.path.join(LIB_DIR, "obj")
    os.makedirs(obj_dir, exist_ok=True)
    digest = source_digest()
    stamp = os.path.join(LIB_DIR, "build.sha256")
    if not force and os.path.exists(LIB_PATH) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == digest:
                return LIB_PATH
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(obj_dir, src.replace(".cu", ".o"))
        cmd = [cc] + _flags() + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    with open(os.path.join(LIB_DIR, "ptxas.log"), "w") as f:
        for (obj, log), src in zip(results, SOURCES):
            f.write(f"== {src}\n{log}\n")
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = [cc] + ARCH + ["-shared", "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    with open(stamp, "w") as f:
        f.write(digest + "\n")
    if verbose:
        print(f"built {LIB_PATH}")
    return LIB_PATH


# A test build of the library for the bounded-wait tests only: the bf16 head_dim-128
# kernels compiled with wait limits of a few milliseconds and two hooks that make
# a wait run out (a ring slot left without its copy, a combiner waiting for one
# more published part than exists).  Never loaded by the product path.
WAIT_TEST_LIB = os.path.join(LIB_DIR, "libpaged_kv_gqa_decode_waittest.so")
WAIT_TEST_SOURCES = ["paged_attn_api.cu", "append.cu", "decode_d128.cu"]
WAIT_TEST_DEFINES = ["-DPAGED_ATTN_WAIT_TEST", "-DPAGED_ATTN_MBAR_SLEEPS=(1u<<14)",
                     "-DPAGED_ATTN_PUBLISH_POLLS=(1u<<15)"]


def build_wait_test(force: bool = False) -> str:
    os.makedirs(LIB_DIR, exist_ok=True)
    obj_dir = os.path.join(LIB_DIR, "obj_waittest")
    os.makedirs(obj_dir, exist_ok=True)
    digest = source_digest() + " " + " ".join(WAIT_TEST_DEFINES)
    stamp = os.path.join(LIB_DIR, "build_waittest.sha256")
    if not force and os.path.exists(WAIT_TEST_LIB) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == digest:
                return WAIT_TEST_LIB
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(obj_dir, src.replace(".cu", ".o"))
        cmd = [cc] + _flags() + WAIT_TEST_DEFINES + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(WAIT_TEST_SOURCES)) as ex:
        objs = list(ex.map(compile_one, WAIT_TEST_SOURCES))
    tmp = WAIT_TEST_LIB + f".tmp{os.getpid()}"
    r = subprocess.run([cc] + ARCH + ["-shared", "-o", tmp] + objs, capture_output=True,
                       text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, WAIT_TEST_LIB)
    with open(stamp, "w") as f:
        f.write(digest + "\n")
    return WAIT_TEST_LIB


if __name__ == "__main__":
    build(verbose=True, force="--force" in sys.argv)

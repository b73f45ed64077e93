"""Build libattn.so in-tree with nvcc for sm_103a (cross-compiles without a GPU).

Each translation unit under ``csrc/`` is compiled in parallel, then linked into
``attention_forward_attn_gb300/libattn.so`` with the CUDA runtime linked
statically.  Objects go to ``_build/`` next to the sources (git-ignored).
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
INCLUDE = os.path.join(ROOT, "include")
LIB_PATH = os.path.join(PKG, "libattn.so")

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libattn.so")


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs():
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(
        os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(INCLUDE, "*.h")) + [__file__]


def is_stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(f) > t for f in _inputs())


def _compile(src: str, extra) -> str:
    obj = os.path.join(BUILD, os.path.basename(src) + ".o")
    cmd = [nvcc()] + ARCH_FLAGS + NVCC_FLAGS + list(extra) + ["-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, " ".join(cmd), r.stderr))
    return obj


def build_library(force: bool = False, extra_flags=()) -> str:
    """Compile and link libattn.so when missing or older than its sources; returns its path."""
    if not force and not extra_flags and not is_stale():
        return LIB_PATH
    os.makedirs(BUILD, exist_ok=True)
    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra_flags), srcs))
    tmp = LIB_PATH + ".tmp.%d" % os.getpid()
    cmd = [nvcc()] + ARCH_FLAGS + ["-shared", "-Xcompiler", "-fPIC", "-cudart", "static"] + objs + [
        "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (" ".join(cmd), r.stderr))
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


# A test-only library: the same objects, except that the tensor-core forward
# is compiled so that CTA 0 skips one K-tile load and every bounded wait gives
# up after 20 ms.  The tests use it to drive the timeout path (the waiting
# roles record ATTN_ERR_TIMEOUT, the CTA drains and frees its TMEM, the kernel
# returns); the product never loads it.
WAIT_TEST_LIB_PATH = os.path.join(PKG, "libattn_waittest.so")
WAIT_TEST_FLAGS = ["-DATTN_TEST_DROP_K_LOAD=1", "-DATTN_WAIT_LIMIT_NS=20000000ull"]
WAIT_TEST_SOURCE = "attn_tc.cu"


def build_wait_test_library() -> str:
    """Build libattn_waittest.so next to libattn.so (see WAIT_TEST_FLAGS); returns its path."""
    build_library()
    inputs = _inputs()
    if (os.path.exists(WAIT_TEST_LIB_PATH) and
            all(os.path.getmtime(f) <= os.path.getmtime(WAIT_TEST_LIB_PATH) for f in inputs)):
        return WAIT_TEST_LIB_PATH
    src = os.path.join(CSRC, WAIT_TEST_SOURCE)
    obj = os.path.join(BUILD, WAIT_TEST_SOURCE + ".waittest.o")
    cmd = [nvcc()] + ARCH_FLAGS + NVCC_FLAGS + WAIT_TEST_FLAGS + ["-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, " ".join(cmd), r.stderr))
    objs = [os.path.join(BUILD, os.path.basename(x) + ".o") for x in sources()
            if os.path.basename(x) != WAIT_TEST_SOURCE] + [obj]
    tmp = WAIT_TEST_LIB_PATH + ".tmp.%d" % os.getpid()
    cmd = [nvcc()] + ARCH_FLAGS + ["-shared", "-Xcompiler", "-fPIC", "-cudart", "static"] + objs + [
        "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (" ".join(cmd), r.stderr))
    os.replace(tmp, WAIT_TEST_LIB_PATH)
    return WAIT_TEST_LIB_PATH


if __name__ == "__main__":
    print(build_library(force=True))

"""Build the KDA prefill C-ABI library (``libkda.so``) in-tree for sm_103a.

Each ``csrc/*.cu`` translation unit is compiled in parallel with nvcc, then
the objects are linked into ``kimi_delta_attention_kda_gb300/libkda.so``
(CUDA runtime linked statically, so the library needs only the driver).
"""

from __future__ import annotations

import concurrent.futures
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(HERE, "libkda.so")
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found")
    return cand


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _headers():
    return sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) +
                  glob.glob(os.path.join(HERE, "..", "include", "*.h")))


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile and link ``libkda.so``; returns its path."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    srcs = _sources()
    hdrs = _headers()
    objs = []
    jobs = []
    for src in srcs:
        obj = os.path.join(BUILD_DIR, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if force or ptxas_info or _stale(obj, [src] + hdrs):
            cmd = [nvcc()] + NVCC_FLAGS + ARCH_FLAGS + ["-c", src, "-o", obj]
            if ptxas_info:
                cmd += ["-Xptxas", "-v"]
            jobs.append(cmd)

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    failed = []
    with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, len(jobs))) as ex:
        for cmd, r in ex.map(run, jobs):
            if verbose or ptxas_info or r.returncode != 0:
                sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
            if r.returncode != 0:
                failed.append(cmd[-3])
    if failed:
        raise RuntimeError("nvcc failed for: " + ", ".join(failed))
    if force or jobs or _stale(LIB_PATH, objs):
        tmp = LIB_PATH + ".tmp.%d" % os.getpid()
        cmd = [nvcc()] + ARCH_FLAGS + ["-shared", "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n" + r.stdout + r.stderr)
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


TEST_HOOKS_LIB = os.path.join(HERE, "libkda_testhooks.so")
TEST_WAIT_BOUND_CYCLES = 100000


def build_test_hooks(force: bool = False) -> str:
    """Compile the test-only library ``libkda_testhooks.so``: the hooks of
    ``csrc/kda_test_hooks.cu`` with the library's wait bound cut to 10^5
    cycles, so that a test can make a bounded wait run out.  Never linked
    into ``libkda.so``."""
    src = os.path.join(CSRC, "kda_test_hooks.cu")
    if force or _stale(TEST_HOOKS_LIB, [src] + _headers()):
        tmp = TEST_HOOKS_LIB + ".tmp.%d" % os.getpid()
        cmd = ([nvcc()] + NVCC_FLAGS + ARCH_FLAGS +
               ["-DKDA_TEST_HOOKS", "-DKDA_WAIT_BOUND_CYCLES=%dLL" % TEST_WAIT_BOUND_CYCLES,
                "-shared", "-o", tmp, src])
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed for the test hooks:\n" + r.stdout + r.stderr)
        os.replace(tmp, TEST_HOOKS_LIB)
    return TEST_HOOKS_LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas-info" in sys.argv)
    print(LIB_PATH)

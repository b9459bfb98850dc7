"""In-tree build of libmlaverify.so (sm_103a) with nvcc.

Each translation unit under csrc/ is compiled in parallel for
compute_103a/sm_103a only, then linked into _build/libmlaverify.so. Only
the C ABI declared in include/mla_verify.h is exported.
"""

from __future__ import annotations

import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(OUT_DIR, "libmlaverify.so")
SELFTEST_SRC = os.path.join(CSRC, "selftest", "umma_selftest.cu")
SELFTEST_LIB = os.path.join(OUT_DIR, "libmlaselftest.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC = os.environ.get("NVCC", "nvcc")


def _nvcc():
    cand = [NVCC, "/usr/local/cuda/bin/nvcc"]
    for c in cand:
        if os.path.isabs(c) and os.path.exists(c):
            return c
        if not os.path.isabs(c):
            from shutil import which
            w = which(c)
            if w:
                return w
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + \
        sorted(glob.glob(os.path.join(CSRC, "*.h"))) + [
        *sorted(glob.glob(os.path.join(INCLUDE, "*.h"))), os.path.abspath(__file__)]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build_library(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    nvcc = _nvcc()
    os.makedirs(OUT_DIR, exist_ok=True)
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-I", INCLUDE, "-I", CSRC,
                    "-Xcompiler", "-fPIC,-fvisibility=hidden", "-Xptxas", "-v"]
    procs = []
    objs = []
    for src in _sources():
        obj = os.path.join(OUT_DIR, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        cmd = [nvcc] + flags + ["-c", src, "-o", obj]
        procs.append((src, cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                 stderr=subprocess.STDOUT, text=True)))
    failed = []
    for src, cmd, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            failed.append((src, cmd, out))
        elif verbose:
            sys.stderr.write(f"== {os.path.basename(src)}\n{out}")
    if failed:
        msg = "\n".join(f"{' '.join(c)}\n{o}" for _, c, o in failed)
        raise RuntimeError("nvcc failed:\n" + msg)
    tmp = LIB + f".tmp{os.getpid()}"
    link = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout + r.stderr)
    os.replace(tmp, LIB)
    return LIB


def build_selftest(force: bool = False) -> str:
    """Test-only library with the tcgen05 layout self-tests (shares tc_ptx.cuh);
    built on demand by the tests that load it, not by build()."""
    deps = [SELFTEST_SRC, os.path.join(CSRC, "tc_ptx.cuh"), os.path.join(CSRC, "tmap.cu"),
            os.path.join(CSRC, "tmap.cuh"), os.path.abspath(__file__)]
    if (not force and os.path.exists(SELFTEST_LIB)
            and all(os.path.getmtime(d) <= os.path.getmtime(SELFTEST_LIB) for d in deps)):
        return SELFTEST_LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = SELFTEST_LIB + f".tmp{os.getpid()}"
    cmd = [_nvcc()] + ARCH + ["-O2", "-std=c++17", "-I", CSRC, "-Xcompiler",
                              "-fPIC,-fvisibility=hidden", "-shared", SELFTEST_SRC,
                              os.path.join(CSRC, "tmap.cu"), "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("selftest build failed:\n" + r.stdout + r.stderr)
    os.replace(tmp, SELFTEST_LIB)
    return SELFTEST_LIB


if __name__ == "__main__":
    print(build_library(force="--force" in sys.argv, verbose=True))
    print(build_selftest(force="--force" in sys.argv))

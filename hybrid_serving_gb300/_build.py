"""Build libhsfork.so in-tree with nvcc for sm_103a (no cmake, no setuptools).

Each translation unit compiles in parallel to ``_build/``; the shared
library lands next to this file.  A unit is rebuilt unless its object was
made from exactly the current bytes of the unit, every header, this script
and the nvcc command: a stamp file beside each object records the SHA-256
of those inputs, so an object copied in from another checkout or machine
(with whatever timestamps) is never linked against sources it was not
built from.  The library carries a stamp over all its objects' stamps.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import hashlib
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(HERE, "libhsfork.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libhsfork.so")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))


def _headers():
    return sorted(glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) +
                  glob.glob(os.path.join(INCLUDE, "*.h")))


def _digest(paths, extra: str) -> str:
    h = hashlib.sha256(extra.encode())
    for p in paths:
        h.update(os.path.basename(p).encode() + b"\0")
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def _stamp_ok(target: str, digest: str) -> bool:
    try:
        return os.path.exists(target) and open(target + ".sha").read().strip() == digest
    except OSError:
        return False


def _write_stamp(target: str, digest: str) -> None:
    with open(target + ".sha", "w") as f:
        f.write(digest + "\n")


def build(verbose: bool = False, force: bool = False) -> str:
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    hdrs = _headers() + [os.path.abspath(__file__)]
    common = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]
    jobs = []
    objs = []
    digests = []
    for src in _sources():
        obj = os.path.join(BUILD, os.path.basename(src) + ".o")
        if src.endswith(".cu"):
            cmd = [nvcc] + ARCH + common + ["-c", src, "-o", obj] + (["-Xptxas", "-v"] if verbose else [])
        else:
            cmd = [nvcc] + common + ["-x", "c++", "-c", src, "-o", obj]
        dig = _digest([src] + hdrs, " ".join(c for c in cmd if c not in ("-Xptxas", "-v")))
        objs.append(obj)
        digests.append(dig)
        if force or not _stamp_ok(obj, dig):
            jobs.append((src, obj, dig, cmd))

    def run(job):
        src, obj, dig, cmd = job
        if os.path.exists(obj + ".sha"):
            os.remove(obj + ".sha")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode == 0:
            _write_stamp(obj, dig)
        return src, r

    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            for src, r in ex.map(run, jobs):
                if verbose or r.returncode != 0:
                    sys.stderr.write(r.stdout + r.stderr)
                if r.returncode != 0:
                    raise RuntimeError(f"nvcc failed on {os.path.basename(src)}")
    lib_dig = hashlib.sha256("".join(digests).encode()).hexdigest()
    if force or jobs or not _stamp_ok(LIB, lib_dig):
        tmp = LIB + ".tmp"
        cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
            raise RuntimeError("linking libhsfork.so failed")
        os.replace(tmp, LIB)
        _write_stamp(LIB, lib_dig)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))

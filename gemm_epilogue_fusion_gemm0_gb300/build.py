"""Builds libcoda.so in-tree with nvcc for sm_103a (no cmake, one translation unit),
and its checked twin libcoda_checked.so (-DCODA_CHECKED: device-side bounds and
alignment checks that record a status code instead of touching memory)."""

from __future__ import annotations

import os
import shutil
import subprocess

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_PATH = os.path.join(PKG_DIR, "libcoda.so")
LIB_PATH_CHECKED = os.path.join(PKG_DIR, "libcoda_checked.so")
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libcoda.so")


def _sources() -> list[str]:
    files = [os.path.join(CSRC, f) for f in sorted(os.listdir(CSRC)) if f.endswith((".cu", ".cuh"))]
    files.append(os.path.join(INCLUDE, "coda.h"))
    return files


def is_stale(path: str = LIB_PATH) -> bool:
    if not os.path.exists(path):
        return True
    t = os.path.getmtime(path)
    return any(os.path.getmtime(f) > t for f in _sources())


def _cmd(out: str, checked: bool, verbose: bool) -> list[str]:
    cmd = [
        _nvcc(), *ARCH_FLAGS, "-O3", "-lineinfo", "-std=c++17",
        "--shared", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
        "-I", INCLUDE, "-o", out, os.path.join(CSRC, "coda.cu"),
    ]
    if checked:
        cmd.insert(1, "-DCODA_CHECKED=1")
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    return cmd


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    """Compile csrc/coda.cu into libcoda.so (or, with checked=True,
    libcoda_checked.so) next to this file; returns its path."""
    path = LIB_PATH_CHECKED if checked else LIB_PATH
    if not force and not is_stale(path):
        return path
    tmp = path + ".tmp"
    cmd = _cmd(tmp, checked, verbose)
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + res.stdout + res.stderr)
    if verbose:
        print(res.stdout + res.stderr)
    os.replace(tmp, path)
    return path


def build_all(force: bool = False) -> list[str]:
    """Both libraries, compiled side by side (two nvcc processes)."""
    jobs = []
    for checked in (False, True):
        path = LIB_PATH_CHECKED if checked else LIB_PATH
        if force or is_stale(path):
            tmp = path + ".tmp"
            cmd = _cmd(tmp, checked, False)
            jobs.append((path, tmp, cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                          stderr=subprocess.STDOUT, text=True)))
    for path, tmp, cmd, proc in jobs:
        out, _ = proc.communicate()
        if proc.returncode != 0:
            raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + out)
        os.replace(tmp, path)
    return [LIB_PATH, LIB_PATH_CHECKED]


if __name__ == "__main__":
    print(build(force=True, verbose=True))
    print(build(force=True, checked=True))

"""Build libdash_attn.so in-tree with nvcc for sm_103a (GB300).

build(checks=True) makes libdash_attn_checked.so instead: the same sources compiled with
DASH_BOUNDS_CHECKS=1, whose backward checks every index it reads from its schedule tables
on the device (the binding loads it when DASH_ATTN_BOUNDS_CHECKS=1 is set).
"""

from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libdash_attn.so")
LIB_CHECKED = os.path.join(PKG, "libdash_attn_checked.so")

SOURCES = ["dash_attn.cu", "sched.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    files.append(os.path.abspath(__file__))
    return files


def up_to_date(checks: bool = False) -> bool:
    lib = LIB_CHECKED if checks else LIB
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False, checks: bool = False) -> str:
    """Compile the library if a source is newer than it. Returns the library path."""
    lib = LIB_CHECKED if checks else LIB
    if not force and up_to_date(checks):
        return lib
    nvcc = os.environ.get("NVCC", "nvcc")
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-O3", "-lineinfo", "-std=c++17", "--threads", "0",
           "-Xcompiler", "-fPIC,-O3", "-Xptxas", "-v" if verbose else "-O3",
           "-shared", "-I", INCLUDE, "-o", tmp]
    if checks:
        cmd.append("-DDASH_BOUNDS_CHECKS=1")
    cmd += [os.path.join(CSRC, s) for s in SOURCES]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        sys.stderr.write(res.stdout + res.stderr)
        raise RuntimeError(f"nvcc failed building {os.path.basename(lib)}")
    if verbose:
        sys.stderr.write(res.stdout + res.stderr)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                checks="--checks" in sys.argv))

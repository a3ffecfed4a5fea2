"""Build libsga.so in-tree with nvcc for sm_103a (one translation unit, static cudart), and its
debug twin libsga_debug.so (-DSGA_DEBUG: every kernel checks its indexed stores)."""
from __future__ import annotations

import glob
import hashlib
import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIB = os.path.join(PKG, "libsga.so")
LIB_DEBUG = os.path.join(PKG, "libsga_debug.so")
HEADER = os.path.join(ROOT, "include", "sga.h")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-lineinfo", "-O3", "-std=c++17",
    "-Xcompiler", "-fPIC", "-shared",
    "-Xptxas", "-v",
]


def _sources(csrc: str = CSRC, header: str = HEADER):
    return sorted(glob.glob(os.path.join(csrc, "*.cu")) + glob.glob(os.path.join(csrc, "*.cuh"))) + [header]


def source_hash(csrc: str = CSRC, header: str = HEADER) -> str:
    """Fingerprint of the library's sources (file names and contents).  It is compiled into the
    library (``sga_build_info``), and the binding refuses a library built from other sources."""
    h = hashlib.sha256()
    for path in _sources(csrc, header):
        h.update(os.path.basename(path).encode() + b"\0")
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def needs_build(debug: bool = False) -> bool:
    lib = LIB_DEBUG if debug else LIB
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(s) > t for s in _sources())


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    lib = LIB_DEBUG if debug else LIB
    if not force and not needs_build(debug):
        return lib
    nvcc = os.environ.get("NVCC", "nvcc")
    tmp = lib + ".tmp"
    cmd = [nvcc, *NVCC_FLAGS, f'-DSGA_SOURCE_HASH="{source_hash()}"', *(["-DSGA_DEBUG"] if debug else []),
           "-o", tmp, os.path.join(CSRC, "sga.cu")]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + res.stdout + res.stderr)
    if verbose:
        print(res.stdout + res.stderr)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    build(force=True, verbose=True)
    build(force=True, verbose=True, debug=True)

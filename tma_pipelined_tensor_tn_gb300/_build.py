"""Build libtmagemm.so in-tree with nvcc for sm_103a (GB300).

Each ``csrc/*.cu`` is compiled to an object in parallel, then linked into a
shared library with the CUDA runtime linked statically, so the library loads
(and its symbols can be listed) on a machine without a GPU driver.
"""
from __future__ import annotations

import glob
import hashlib
import os
import platform
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libtmagemm.so")
# The checked build (-DTMAGEMM_CHECKED): kernels that check their own
# invariants and count the work units they complete.
BUILD_CHECKED = os.path.join(PKG, "_build_checked")
LIB_CHECKED = os.path.join(PKG, "libtmagemm_checked.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE,
              "--expt-relaxed-constexpr"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libtmagemm.so")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (_sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
            + glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)])


def _stamp(flags) -> str:
    """What a build depends on: this machine's architecture, the compiler
    flags and the bytes of every source and header."""
    h = hashlib.sha256()
    h.update(platform.machine().encode())
    h.update(" ".join(flags).encode())
    for d in sorted(_deps()):
        h.update(os.path.relpath(d, ROOT).encode())
        with open(d, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def up_to_date(lib: str = LIB, flags=None) -> bool:
    """True if `lib` exists and was built here from the current sources with
    these flags (a library built on another machine or from other sources is
    rebuilt)."""
    if flags is None:
        flags = ARCH + NVCC_FLAGS + (["-DTMAGEMM_CHECKED"] if lib == LIB_CHECKED else [])
    if not os.path.exists(lib) or not os.path.exists(lib + ".stamp"):
        return False
    with open(lib + ".stamp") as f:
        return f.read().strip() == _stamp(flags)


def build(force: bool = False, verbose: bool = False, extra_flags=None,
          checked: bool = False) -> str:
    """Compile every CUDA source and link libtmagemm.so (or, with checked=True,
    libtmagemm_checked.so); returns its path."""
    lib_path = LIB_CHECKED if checked else LIB
    build_dir = BUILD_CHECKED if checked else BUILD
    flags = ARCH + NVCC_FLAGS + (["-DTMAGEMM_CHECKED"] if checked else []) + list(extra_flags or [])
    if not force and up_to_date(lib_path, flags):
        return lib_path
    os.makedirs(build_dir, exist_ok=True)
    cc = nvcc()
    procs = []
    objs = []
    for src in _sources():
        obj = os.path.join(build_dir, os.path.basename(src) + ".o")
        objs.append(obj)
        cmd = [cc, *flags, "-c", src, "-o", obj]
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for cmd, p in procs:
        out, _ = p.communicate()
        text = out.decode(errors="replace")
        if p.returncode != 0:
            failed.append((cmd, text))
        elif verbose and text.strip():
            sys.stderr.write(text)
    if failed:
        msg = "\n".join(" ".join(c) + "\n" + t for c, t in failed)
        raise RuntimeError("nvcc failed:\n" + msg)
    tmp = lib_path + ".tmp"
    link = [cc, *ARCH, "-shared", "-Xcompiler", "-fPIC", "-o", tmp, *objs, "-cudart", "static"]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + " ".join(link) + "\n" + r.stdout + r.stderr)
    os.replace(tmp, lib_path)
    with open(lib_path + ".stamp", "w") as f:
        f.write(_stamp(flags) + "\n")
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, checked="--checked" in sys.argv))

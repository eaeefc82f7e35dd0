"""Ahead-of-time build of the CUDA library for sm_103a.

Compiles every ``csrc/*.cu`` translation unit in parallel with nvcc
(``-gencode arch=compute_103a,code=sm_103a``, no fast-math) and links them
into ``_build/libaddln.so`` with the CUDA runtime linked statically, so the
library needs nothing from PyTorch at load time.  Rebuilds only when a
source or header is newer than the library.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(OUT_DIR, "libaddln.so")
# The bounds-checked debugging build (ADDLN_CHECK_BOUNDS): every kernel tests
# each global access against its buffer first.  Tests only; never loaded by
# the package itself.
CHECKED_DIR = os.path.join(OUT_DIR, "checked")
CHECKED_LIB = os.path.join(CHECKED_DIR, "libaddln_checked.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libaddln.so")


def sources() -> list:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs() -> list:
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) \
        + glob.glob(os.path.join(INCLUDE, "*.h"))


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False, extra_flags: list | None = None,
          checked: bool = False) -> str:
    """Build the library if needed and return its path.  checked: the
    bounds-checked debugging build instead (its own objects and library)."""
    out_dir, lib = (CHECKED_DIR, CHECKED_LIB) if checked else (OUT_DIR, LIB)
    if not force and not extra_flags and up_to_date(lib):
        return lib
    os.makedirs(os.path.join(out_dir, "obj"), exist_ok=True)
    cc = nvcc()
    flags = NVCC_FLAGS + list(extra_flags or []) + (["-DADDLN_CHECK_BOUNDS"] if checked else [])

    def compile_one(src):
        obj = os.path.join(out_dir, "obj", os.path.basename(src)[:-3] + ".o")
        cmd = [cc, *ARCH, *flags, "-c", src, "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
        if verbose:
            print(res.stdout + res.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, sources()))
    tmp = lib + f".tmp{os.getpid()}"
    # every symbol must resolve at link time: a missing definition fails the
    # build here, not the first dlopen
    cmd = [cc, *ARCH, "-shared", "-Xcompiler", "-fPIC", "-cudart", "static",
           "-Xlinker", "--no-undefined", "-o", tmp, *objs]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, lib)
    return lib


def ptxas_report(extra_flags: list | None = None) -> dict:
    """Compiles every translation unit with ptxas's verbose report (the same
    flags as the library, objects to a scratch folder) and returns, for each
    kernel (mangled name), its registers, stack frame and spill store / load
    bytes as the assembler reports them."""
    import re
    import tempfile
    cc = nvcc()
    flags = NVCC_FLAGS + list(extra_flags or []) + ["-Xptxas", "-v"]
    with tempfile.TemporaryDirectory() as tmp:
        def one(src):
            obj = os.path.join(tmp, os.path.basename(src)[:-3] + ".o")
            res = subprocess.run([cc, *ARCH, *flags, "-c", src, "-o", obj], capture_output=True,
                                 text=True)
            if res.returncode != 0:
                raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
            return res.stdout + res.stderr

        with ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
            logs = list(ex.map(one, sources()))
    out = {}
    for log in logs:
        cur = None
        for line in log.splitlines():
            m = re.search(r"Function properties for (\S+)", line)
            if m:
                cur = m.group(1)
                out.setdefault(cur, {})
                continue
            m = re.search(r"(\d+) bytes stack frame, (\d+) bytes spill stores, (\d+) bytes spill loads",
                          line)
            if m and cur:
                out[cur].update(stack=int(m.group(1)), spill_stores=int(m.group(2)),
                                spill_loads=int(m.group(3)))
                continue
            m = re.search(r"Used (\d+) registers", line)
            if m and cur:
                out[cur]["registers"] = int(m.group(1))
                cur = None
    return out


if __name__ == "__main__":
    import sys
    print(build(force=True, verbose="-v" in sys.argv))

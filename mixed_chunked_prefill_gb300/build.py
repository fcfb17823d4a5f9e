"""Build the in-tree CUDA library ``_lib/libmcp.so`` for sm_103a with nvcc.

Each translation unit is compiled in parallel with
``-gencode arch=compute_103a,code=sm_103a -lineinfo``; the objects go to
``<repo>/_build`` and the shared library to ``mixed_chunked_prefill_gb300/_lib``.
The CUDA runtime is linked statically, so the library needs only the driver.

``build(checked=True)`` builds the debugging variant ``_lib/libmcp_checked.so``
(compiled with ``-DMCP_CHECKED``; objects in ``_build/checked``): the same ABI,
plus device-side checks that cost extra work (duplicate append slots).
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_DIR = os.path.join(HERE, "_lib")
LIB_PATH = os.path.join(LIB_DIR, "libmcp.so")
CHECKED_LIB_PATH = os.path.join(LIB_DIR, "libmcp_checked.so")

SOURCES = ["host.cpp", "sched.cpp", "append.cu", "attn_fwd.cu", "combine.cu",
           "attn_fwd_noalloc.cu"]
HEADERS = ["mcp_internal.h", "ptx.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or put CUDA's bin on PATH)")


def _flags(ptxas_verbose: bool, checked: bool = False) -> list:
    f = ["-std=c++17", "-O3", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC",
         "-I", INCLUDE, "-I", CSRC]
    if checked:
        f += ["-DMCP_CHECKED=1"]
    if ptxas_verbose:
        f += ["-Xptxas", "-v"]
    return f


def _newer(target: str, deps: list) -> bool:
    if not os.path.exists(target):
        return False
    t = os.path.getmtime(target)
    return all(os.path.getmtime(d) <= t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False,
          checked: bool = False) -> str:
    """Compile (if stale) and link the library (the MCP_CHECKED variant with
    ``checked``); return its path."""
    build_dir = os.path.join(BUILD_DIR, "checked") if checked else BUILD_DIR
    lib_path = CHECKED_LIB_PATH if checked else LIB_PATH
    os.makedirs(build_dir, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    cc = nvcc()
    headers = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, "mcp.h")]
    jobs = []
    objs = []
    for s in SOURCES:
        src = os.path.join(CSRC, s)
        obj = os.path.join(build_dir, os.path.splitext(s)[0] + ".o")
        objs.append(obj)
        if force or ptxas_verbose or not _newer(obj, [src] + headers + [__file__]):
            jobs.append([cc, *_flags(ptxas_verbose, checked), "-c", src, "-o", obj])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    if jobs:
        with ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            for cmd, r in ex.map(run, jobs):
                if verbose or ptxas_verbose:
                    sys.stderr.write(r.stdout + r.stderr)
                if r.returncode != 0:
                    raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    if force or jobs or not _newer(lib_path, objs):
        cmd = [cc, "-shared", *ARCH, "-o", lib_path, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    return lib_path


if __name__ == "__main__":
    p = build(force="--force" in sys.argv, verbose=True, ptxas_verbose="--ptxas-v" in sys.argv,
              checked="--checked" in sys.argv)
    print(p)

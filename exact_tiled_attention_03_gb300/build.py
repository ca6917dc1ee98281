"""Build the sm_103a CUDA library (lib/libfa_gb300.so) in-tree with nvcc.

One -gencode (compute_103a -> sm_103a), translation units compiled in
parallel, then linked into a shared library with the CUDA runtime linked
statically. Works the same on an x86_64 host (cross-compiling, no GPU) and on
the aarch64 GPU host. Rebuilds only what is older than its sources.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIBDIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIBDIR, "libfa_gb300.so")

SOURCES = ["fa_abi.cu", "fa_prefill_sm103.cu", "fa_verify.cu", "fa_simt.cu", "fa_selftest.cu",
           "fa_verify_static.cu", "fa_backward_sm103.cu", "fa_prefill_fp8_sm103.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA library cannot be built")


def _headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hs += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return hs


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def compile_flags(verbose_ptxas: bool = False):
    flags = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
                    "-I", INCLUDE, "-I", CSRC, "--expt-relaxed-constexpr"]
    if verbose_ptxas:
        flags += ["-Xptxas", "-v"]
    return flags


def build(force: bool = False, verbose_ptxas: bool = False, jobs: int | None = None,
          defines=(), lib_path: str | None = None, build_dir: str | None = None) -> str:
    """Build the library; `defines` (e.g. ["FA_PREFILL_CHUNK=32"]) with a separate
    `lib_path` and `build_dir` give a variant build next to the default one."""
    nvcc = nvcc_path()
    bdir = build_dir or BUILD
    lib = lib_path or LIB
    os.makedirs(bdir, exist_ok=True)
    os.makedirs(os.path.dirname(lib), exist_ok=True)
    headers = _headers()
    objs, todo = [], []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(bdir, src.replace(".cu", ".o"))
        objs.append(o)
        if force or verbose_ptxas or _stale(o, [s] + headers):
            todo.append((s, o))

    def _one(so):
        s, o = so
        cmd = [nvcc] + compile_flags(verbose_ptxas) + [f"-D{d}" for d in defines] + ["-c", s, "-o", o]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(s)}:\n{r.stdout}\n{r.stderr}")
        return s, r.stdout + r.stderr

    logs = []
    if todo:
        with ThreadPoolExecutor(max_workers=jobs or min(len(todo), os.cpu_count() or 4)) as ex:
            logs = list(ex.map(_one, todo))
    if verbose_ptxas:
        for s, log in logs:
            print(f"== {os.path.basename(s)}\n{log}")
    if force or todo or _stale(lib, objs):
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return lib


DEBUG_LIB = os.path.join(LIBDIR, "libfa_gb300_debug.so")


def build_debug(force: bool = False) -> str:
    """The debug build: the same sources with FA_DEBUG defined (device-side index
    checks that record a bit in the status word), as lib/libfa_gb300_debug.so."""
    return build(force=force, defines=["FA_DEBUG=1"], lib_path=DEBUG_LIB,
                 build_dir=os.path.join(PKG, "_build_debug"))


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))

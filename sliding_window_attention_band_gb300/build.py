"""Builds the CUDA library libswab.so in-tree (sliding_window_attention_band_gb300/_lib/).

Every translation unit is compiled by nvcc for sm_103a only, in parallel, and
linked into one shared library with the CUDA runtime linked statically.  The
same sources with SWAB_BOUNDS_CHECK=1 give libswab_bounds.so, the
bounds-checked build (every plain global access of a kernel tested against
the call's buffer extents); ``build_all()`` compiles both in one pool.
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
LIBDIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIBDIR, "libswab.so")
LIB_BOUNDS = os.path.join(LIBDIR, "libswab_bounds.so")
VARIANTS = {  # variant: (library, object folder, extra nvcc flags)
    "regular": (LIB, "obj", ()),
    "bounds": (LIB_BOUNDS, "obj_bounds", ("-DSWAB_BOUNDS_CHECK=1",)),
}
SOURCES = ["swab_api.cu", "k_band_qk.cu", "k_band_gather.cu", "k_softmax.cu", "k_attention.cu", "k_attention_bwd.cu",
           "k_global.cu", "k_bias_transpose.cu", "k_global_proj.cu",
           "k_global_tc.cu"]
HEADERS = ["swab_common.cuh", "swab_internal.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
          "--expt-relaxed-constexpr"]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA library cannot be built")
    return path


def _inputs():
    files = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    files.append(os.path.join(ROOT, "include", "swab.h"))
    return files


def up_to_date(variant: str = "regular") -> bool:
    lib = VARIANTS[variant][0]
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def _compile_jobs(variant, extra_flags, verbose):
    """(source, compile function) pairs of one variant."""
    lib, objdir, flags = VARIANTS[variant]
    os.makedirs(os.path.join(LIBDIR, objdir), exist_ok=True)
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(LIBDIR, objdir, os.path.splitext(src)[0] + ".o")
        cmd = [cc, *ARCH, *CFLAGS, *flags, *extra_flags, "-I", os.path.join(ROOT, "include"), "-c",
               os.path.join(CSRC, src), "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if verbose or res.returncode != 0:
            sys.stderr.write(" ".join(cmd) + "\n" + res.stdout + res.stderr)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src} ({variant} build)")
        return obj

    return [(src, compile_one) for src in SOURCES]


def _link(variant, objs):
    lib = VARIANTS[variant][0]
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        sys.stderr.write(" ".join(cmd) + "\n" + res.stdout + res.stderr)
        raise RuntimeError(f"link of {os.path.basename(lib)} failed")
    os.replace(tmp, lib)
    return lib


def build_variants(variants, force: bool = False, verbose: bool = False, extra_flags=()):
    """Compile and link the given variants, every translation unit of all of
    them in one pool; returns their library paths."""
    todo = [v for v in variants if force or not up_to_date(v)]
    jobs = [(v, src, fn) for v in todo for src, fn in _compile_jobs(v, extra_flags, verbose)]
    if jobs:
        with ThreadPoolExecutor(max_workers=min(len(jobs), max(os.cpu_count() or 1, len(SOURCES)))) as ex:
            objs = list(ex.map(lambda job: job[2](job[1]), jobs))
        for v in todo:
            _link(v, [o for (vv, _, _), o in zip(jobs, objs) if vv == v])
    return [VARIANTS[v][0] for v in variants]


def build(force: bool = False, verbose: bool = False, extra_flags=(), variant: str = "regular") -> str:
    """Compile and link one variant (libswab.so by default); returns its path."""
    return build_variants([variant], force, verbose, extra_flags)[0]


def build_all(force: bool = False, verbose: bool = False):
    """The regular and the bounds-checked library."""
    return build_variants(["regular", "bounds"], force, verbose)


if __name__ == "__main__":
    print(build_all(force="--force" in sys.argv, verbose="-v" in sys.argv))

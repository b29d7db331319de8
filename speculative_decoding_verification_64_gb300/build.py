"""Build ``libspecdec.so`` (the C-ABI library) from ``csrc/`` with nvcc for sm_103a.

The translation units compile in parallel, then link into one shared library
with the CUDA runtime linked statically.  Objects go to ``_build/`` next to
this file; the library lands beside this file (both are git-ignored).

Usage: ``python -m speculative_decoding_verification_64_gb300.build [--force] [--debug-flags ...]``
"""
from __future__ import annotations

import argparse
import concurrent.futures
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_NAME = "libspecdec.so"
LIB_PATH = os.path.join(HERE, LIB_NAME)

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc_path() -> str:
    cand = [os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"]
    for c in cand:
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libspecdec.so")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _headers():
    return sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h")))


# Test builds: the same sources with a define that changes one behaviour, in a
# library (and object folder) of their own.  "shortwait": consumers' waits on
# copies give up at once, so that the give-up paths run (see common.cuh).
VARIANTS = {"shortwait": ["-DSPECDEC_CONSUMER_WAIT_NS=0ull"]}


def _up_to_date(lib_path: str) -> bool:
    if not os.path.exists(lib_path):
        return False
    t = os.path.getmtime(lib_path)
    return all(os.path.getmtime(f) <= t for f in _sources() + _headers() + [__file__])


def build(force: bool = False, extra_flags=None, verbose: bool = False,
          variant: str = None) -> str:
    """Compile every CUDA translation unit and link ``libspecdec.so`` (or the
    test variant's ``libspecdec_<variant>.so``).  Returns its path."""
    lib_path, build_dir = LIB_PATH, BUILD_DIR
    if variant is not None:
        extra_flags = list(extra_flags or []) + VARIANTS[variant]
        lib_path = os.path.join(HERE, f"libspecdec_{variant}.so")
        build_dir = BUILD_DIR + "_" + variant
    if not force and _up_to_date(lib_path):
        return lib_path
    nvcc = nvcc_path()
    os.makedirs(build_dir, exist_ok=True)
    flags = ARCH_FLAGS + NVCC_FLAGS + list(extra_flags or [])
    jobs = []
    for src in _sources():
        obj = os.path.join(build_dir, os.path.splitext(os.path.basename(src))[0] + ".o")
        jobs.append(([nvcc] + flags + ["-c", src, "-o", obj], obj))

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        results = list(ex.map(lambda j: run(j[0]), jobs))
    for cmd, r in results:
        if verbose and (r.stdout or r.stderr):
            sys.stderr.write(r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    tmp = lib_path + f".tmp{os.getpid()}"
    link = [nvcc] + ARCH_FLAGS + ["-shared", "-cudart", "static", "-o", tmp] + \
        [o for _, o in jobs]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + " ".join(link) + "\n" + r.stdout + r.stderr)
    os.replace(tmp, lib_path)
    return lib_path


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--extra", nargs="*", default=[], help="extra nvcc flags, e.g. -Xptxas -v")
    a = ap.parse_args(argv)
    print(build(force=a.force, extra_flags=a.extra, verbose=a.verbose))


if __name__ == "__main__":
    main()

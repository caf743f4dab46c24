"""Builds ``libtgemm.so`` in-tree with nvcc for sm_103a.

Each ``csrc/*.cu`` file is compiled to an object in parallel, then the objects
are linked into one shared library with the CUDA runtime linked statically.
No torch headers or libraries are involved: the library's interface is plain C
(``include/tgemm.h``).
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
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(PKG, "libtgemm.so")
DEBUG_LIB_PATH = os.path.join(PKG, "libtgemm_debug.so")   # with the device-side checks (TGEMM_DEBUG)
PAGES_DIR = os.path.join(PKG, "csrc_pages")
PAGES_LIB_PATH = os.path.join(PKG, "libtgemm_pages.so")
PROBES_DIR = os.path.join(PKG, "csrc_probes")
PROBES_LIB_PATH = os.path.join(PKG, "libtgemm_probes.so")   # read-stream calibration (include/tgemm_probes.h)

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
              "--expt-relaxed-constexpr", "-I" + INCLUDE, "-I" + CSRC]


def nvcc() -> str:
    path = shutil.which("nvcc")
    if path:
        return path
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found (set CUDA_HOME or put nvcc on PATH)")


def sources(directory=CSRC):
    return sorted(os.path.join(directory, f) for f in os.listdir(directory) if f.endswith(".cu"))


def _headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hs += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return hs


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _build_lib(srcs, lib_path, tag, verbose, force, ptxas_verbose, extra=()):
    os.makedirs(BUILD_DIR, exist_ok=True)
    cc = nvcc()
    headers = _headers()
    objs = []
    jobs = []
    for src in srcs:
        obj = os.path.join(BUILD_DIR, tag + "_" + os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if force or _stale(obj, [src, *headers, __file__]):
            cmd = [cc, *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
            if ptxas_verbose:
                cmd[1:1] = ["-Xptxas", "-v"]
            jobs.append(cmd)

    def run(cmd):
        res = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, res

    if jobs:
        with ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as pool:
            for cmd, res in pool.map(run, jobs):
                if verbose or ptxas_verbose or res.returncode != 0:
                    sys.stderr.write(" ".join(cmd) + "\n" + res.stdout + res.stderr)
                if res.returncode != 0:
                    raise RuntimeError(f"nvcc failed on {cmd[-3]}")
    if force or jobs or _stale(lib_path, objs):
        tmp = lib_path + ".tmp"
        cmd = [cc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs, "-ldl", "-lpthread", "-lrt"]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if verbose or res.returncode != 0:
            sys.stderr.write(" ".join(cmd) + "\n" + res.stdout + res.stderr)
        if res.returncode != 0:
            raise RuntimeError(f"linking {os.path.basename(lib_path)} failed")
        os.replace(tmp, lib_path)
    return lib_path


def build(verbose: bool = False, force: bool = False, ptxas_verbose: bool = False) -> str:
    """Compile and link ``libtgemm.so``, its debug build ``libtgemm_debug.so``
    (the same sources with the device-side consistency checks, TGEMM_DEBUG), the
    pages' comparator library and the read-stream calibration library; returns
    libtgemm's path."""
    with ThreadPoolExecutor(max_workers=4) as pool:
        main = pool.submit(_build_lib, sources(), LIB_PATH, "tgemm", verbose, force, ptxas_verbose)
        debug = pool.submit(_build_lib, sources(), DEBUG_LIB_PATH, "tgemm_dbg", verbose, force, ptxas_verbose,
                            ("-DTGEMM_DEBUG",))
        pages = pool.submit(_build_lib, sources(PAGES_DIR), PAGES_LIB_PATH, "pages", verbose, force,
                            ptxas_verbose)
        probes = pool.submit(_build_lib, sources(PROBES_DIR), PROBES_LIB_PATH, "probes", verbose, force,
                             ptxas_verbose)
        pages.result()
        probes.result()
        debug.result()
        return main.result()


if __name__ == "__main__":
    build(verbose="-v" in sys.argv, force="-f" in sys.argv, ptxas_verbose="--ptxas" in sys.argv)
    print(LIB_PATH)

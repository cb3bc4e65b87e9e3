"""Builds the library in-tree: every CUDA source compiled for sm_103a with
nvcc, in parallel, then linked into shared libraries next to this file:
libwsa.so (the product build) and libwsa_checked.so (the same sources with
-DWSA_BOUNDS_CHECK: every plan-table row index range-checked on the device)."""

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
REPO_DIR = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(REPO_DIR, "include")
BUILD_DIR = os.path.join(REPO_DIR, "_build")
LIB_PATH = os.path.join(PKG_DIR, "libwsa.so")
CHECKED_LIB_PATH = os.path.join(PKG_DIR, "libwsa_checked.so")
# (library, build folder, extra nvcc flags)
VARIANTS = [(LIB_PATH, BUILD_DIR, []),
            (CHECKED_LIB_PATH, os.path.join(REPO_DIR, "_build", "checked"), ["-DWSA_BOUNDS_CHECK"])]

SOURCES = ["plan.cu", "transition.cu", "attention_fp32.cu", "attention_tc.cu", "abi.cu",
           "attention_noalloc.cu", "sp.cu", "rope.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr"]


def _nvcc():
    for cand in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "bin", "nvcc")):
            return os.path.join(cand, "bin", "nvcc")
    found = shutil.which("nvcc")
    if not found:
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libwsa.so")
    return found


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "wsa.h"))
    files.append(os.path.abspath(__file__))
    return files


def _up_to_date(lib):
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _deps())


def _run(cmd):
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("command failed:\n" + " ".join(cmd) + "\n" + r.stdout)
    return r.stdout


def build(force=False, verbose=False, ptxas_verbose=False):
    """Compile every source for sm_103a and link both libraries; returns the
    product library's path."""
    todo = [v for v in VARIANTS if force or not _up_to_date(v[0])]
    if not todo:
        return LIB_PATH
    nvcc = _nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_verbose else []
    jobs = []
    for lib, bdir, defs in todo:
        os.makedirs(bdir, exist_ok=True)
        for src in SOURCES:
            obj = os.path.join(bdir, src.replace(".cu", ".o"))
            jobs.append((lib, obj, [nvcc, "-c", *ARCH, *FLAGS, *defs, *extra, "-I", INCLUDE, "-I", CSRC,
                                    os.path.join(CSRC, src), "-o", obj]))
    with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        outs = list(ex.map(lambda j: _run(j[2]), jobs))
    if verbose or ptxas_verbose:
        for (_, obj, _), out in zip(jobs, outs):
            print(f"== {obj}\n{out}")
    for lib, _, _ in todo:
        tmp = lib + ".tmp"
        _run([nvcc, "-shared", *ARCH, "-o", tmp] + [o for l, o, _ in jobs if l == lib])
        os.replace(tmp, lib)
    return LIB_PATH


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True, ptxas_verbose="-v" in sys.argv))

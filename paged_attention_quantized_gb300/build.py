"""Build libpa.so (the C-ABI CUDA library) in-tree for sm_103a.

    python -m paged_attention_quantized_gb300.build [--force] [--verbose]

Each translation unit under csrc/ is compiled in parallel with
`nvcc -gencode arch=compute_103a,code=sm_103a -O3 -lineinfo` and linked into
paged_attention_quantized_gb300/_build/libpa.so.  The build is skipped when the
library is newer than every source and header.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libpa.so")
# A test build of the same sources: every bounded wait gives up after 2 ms
# instead of 2 s, and a workspace header word can make the copy of one page
# go missing (PA_FAULT_INJECT), so the timeout path can be exercised on a GPU
# without any fault.  It is never loaded by the package.
VARIANTS = {"": ("_build", "libpa.so", []),
            "fi": ("_build_fi", "libpa_fi.so", ["-DPA_FAULT_INJECT", "-DPA_WAIT_LIMIT_NS=2000000ull"])}
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
                     "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + [os.path.join(INCLUDE, "pa.h"), __file__]


def lib_path(variant: str = "") -> str:
    d, name, _ = VARIANTS[variant]
    return os.path.join(HERE, d, name)


def up_to_date(variant: str = "") -> bool:
    lib = lib_path(variant)
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, verbose: bool = False, jobs: int | None = None, variant: str = "") -> str:
    lib = lib_path(variant)
    if not force and up_to_date(variant):
        return lib
    out_dir = os.path.dirname(lib)
    os.makedirs(os.path.join(out_dir, "obj"), exist_ok=True)
    nvcc = _nvcc()
    extra = (["-Xptxas", "-v"] if verbose else []) + VARIANTS[variant][2]

    def compile_one(src):
        obj = os.path.join(out_dir, "obj", os.path.basename(src) + ".o")
        cmd = [nvcc] + NVCC_FLAGS + extra + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, (r.stdout + r.stderr)

    srcs = sources()
    jobs = jobs or min(len(srcs), max(1, os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(max_workers=jobs) as ex:
        results = list(ex.map(compile_one, srcs))
    if verbose:
        for _, log in results:
            if log.strip():
                sys.stdout.write(log)
    tmp = lib + f".{os.getpid()}.tmp"
    cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="--verbose" in sys.argv))

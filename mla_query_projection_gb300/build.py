"""Build ``libmla_query.so`` (the C-ABI library) in-tree with nvcc for sm_103a.

Each ``csrc/*.cu`` is compiled to an object in parallel, then linked into one
shared library next to this file.  The CUDA runtime is linked statically, so
the library loads on a machine without a GPU (every call then returns
MLA_ECUDA).  Usage: ``python -m mla_query_projection_gb300.build``.
"""

from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libmla_query.so")
BUILD = os.path.join(HERE, "_build")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + [
    "-O3",
    "-lineinfo",
    "-std=c++17",
    "-Xcompiler",
    "-fPIC",
    "-Xcompiler",
    "-fvisibility=hidden",
    "--expt-relaxed-constexpr",
    "-Xptxas",
    "-v",
]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmla_query.so")
    return cand


def _compile(src: str, build_dir: str = BUILD, extra: tuple = ()) -> tuple[str, str]:
    obj = os.path.join(build_dir, os.path.basename(src) + ".o")
    cmd = [nvcc(), *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
    p = subprocess.run(cmd, capture_output=True, text=True)
    if p.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{p.stdout}\n{p.stderr}")
    return obj, p.stderr


def build(verbose: bool = False, out_dir: str | None = None, extra: tuple = ()) -> str:
    """Compile and link; returns the path of the shared library.  With
    `out_dir` and `extra` nvcc flags, a variant of the same sources goes into
    out_dir (for instance the bounds-checked build, extra=("-DMLA_CHECKS",));
    the in-tree library is left as it is."""
    build_dir = BUILD if out_dir is None else out_dir
    lib = LIB if out_dir is None else os.path.join(out_dir, "libmla_query.so")
    os.makedirs(build_dir, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        results = list(ex.map(lambda src: _compile(src, build_dir, tuple(extra)), srcs))
    objs = [o for o, _ in results]
    if verbose:
        for _, log in results:
            sys.stderr.write(log)
    tmp = lib + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
    p = subprocess.run(cmd, capture_output=True, text=True)
    if p.returncode != 0:
        raise RuntimeError(f"link failed:\n{p.stdout}\n{p.stderr}")
    os.replace(tmp, lib)
    with open(os.path.join(build_dir, "ptxas.log"), "w") as f:
        for _, log in results:
            f.write(log)
    return lib


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))

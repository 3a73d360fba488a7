"""Builds libdsa.so in-tree with nvcc for sm_103a (GB300).

Translation units compile in parallel into ``_build/`` next to this file; the shared library is
linked to ``dynamic_block_sparse_gb300/libdsa.so``.  A rebuild happens only when a source or
header is newer than the library (or ``force=True``).  ``build_traced()`` makes the phase-tracing
variant ``libdsa_trace.so`` (compiled with ``-DDSA_TIMELINE``) in ``_build_trace/``; nothing loads
it but the tracing script.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(HERE, "libdsa.so")
TRACE_BUILD_DIR = os.path.join(HERE, "_build_trace")
TRACE_LIB_PATH = os.path.join(HERE, "libdsa_trace.so")

SOURCES = ["api.cu", "attn.cu", "calib.cu", "kvquant.cu", "meta_score.cu", "prr_step.cu",
           "select.cu", "stream_attn.cu", "threshold.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O3",
         "--expt-relaxed-constexpr", "-I" + INCLUDE, "-I" + CSRC]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found")
    return cand


def _newest(paths) -> float:
    return max(os.path.getmtime(p) for p in paths)


def _inputs() -> list[str]:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)
             if f.endswith((".cu", ".cuh", ".h"))]
    files.append(os.path.join(INCLUDE, "dsa.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date(lib_path: str = LIB_PATH) -> bool:
    return os.path.exists(lib_path) and os.path.getmtime(lib_path) >= _newest(_inputs())


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
          traced: bool = False) -> str:
    lib_path = TRACE_LIB_PATH if traced else LIB_PATH
    build_dir = TRACE_BUILD_DIR if traced else BUILD_DIR
    if not force and up_to_date(lib_path):
        return lib_path
    os.makedirs(build_dir, exist_ok=True)
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    if traced:
        extra.append("-DDSA_TIMELINE")

    def compile_one(src: str) -> tuple[str, str]:
        obj = os.path.join(build_dir, src.replace(".cu", ".o"))
        cmd = [cc, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stdout + r.stderr

    with cf.ThreadPoolExecutor(max_workers=min(len(SOURCES), os.cpu_count() or 4)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    logs = "".join(log for _, log in results)
    tmp = lib_path + ".tmp"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    if verbose or ptxas_info:
        sys.stdout.write(logs)
    return lib_path


def build_traced(force: bool = False) -> str:
    return build(force=force, traced=True)


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv)
    print(LIB_PATH)

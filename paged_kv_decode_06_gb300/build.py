"""Build the CUDA library ``libpagedattn.so`` in-tree for sm_103a.

Each translation unit is compiled by its own nvcc process (in parallel), then
linked into one shared library that exports the C ABI of
``include/paged_attn.h``.  No CMake; the same command works on x86_64 and on
aarch64 hosts.
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
LIB_PATH = os.path.join(HERE, "libpagedattn.so")
SOURCES = ["pa_host.cu", "pa_split_bf16.cu", "pa_split_fp8.cu", "pa_split_fp8_tok.cu", "pa_merge.cu", "pa_static_ws.cu", "pa_cache_write.cu",
           "pa_split_tc.cu", "pa_mla.cu", "pa_mla_tc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    exe = shutil.which("nvcc")
    if exe:
        return exe
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpagedattn.so")


def common_flags():
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
                   "--expt-relaxed-constexpr"]


def _compile(src: str, ptxas_verbose: bool) -> tuple[str, str]:
    obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
    cmd = [nvcc_path(), "-c", os.path.join(CSRC, src), "-o", obj] + common_flags()
    if ptxas_verbose:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def _sources_newer_than(target: str) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    files.append(os.path.abspath(__file__))
    return any(os.path.getmtime(f) > t for f in files)


def build(force: bool = False, ptxas_verbose: bool = False, quiet: bool = True) -> str:
    """Compile (if sources changed) and return the library path."""
    if not force and not ptxas_verbose and not _sources_newer_than(LIB_PATH):
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(lambda s: _compile(s, ptxas_verbose), SOURCES))
    if ptxas_verbose:
        for (_, log) in results:
            sys.stderr.write(log)
    tmp = LIB_PATH + ".tmp"
    cmd = [nvcc_path()] + ARCH + ["-shared", "-o", tmp] + [o for o, _ in results] + ["-Xcompiler", "-fPIC"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    if not quiet:
        print(f"built {LIB_PATH}")
    return LIB_PATH


if __name__ == "__main__":
    build(force=True, ptxas_verbose="-v" in sys.argv, quiet=False)

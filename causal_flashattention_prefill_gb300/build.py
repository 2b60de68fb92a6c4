"""Builds the CUDA library in tree: ``libzyfa_gb300.so`` next to this file.

nvcc compiles each translation unit for sm_103a only (one ``-gencode``), in
parallel, and links them with the static CUDA runtime.  The result exports the
C ABI declared in ``include/zyfa.h``.

Usage: ``python -m causal_flashattention_prefill_gb300.build [--force]``.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_NAME = "libzyfa_gb300.so"
LIB_PATH = os.path.join(PKG, LIB_NAME)

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-Xcompiler", "-fvisibility=hidden", "-diag-suppress", "177"]

SOURCES = ["api.cpp", "fwd_sm103.cu", "quant.cu"]
HEADERS = ["fwd.h", "quant.h", "zyfa_ptx.cuh"]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build")
    return path


def _inputs():
    files = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    files.append(os.path.join(INCLUDE, "zyfa.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date(lib: str = LIB_PATH) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def _compile(src: str, obj: str, extra) -> None:
    cmd = [nvcc()] + NVCC_FLAGS + list(extra) + ["-I", INCLUDE, "-I", CSRC, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")


def build_library(sources, out_path, extra=(), force=False, inputs=None) -> str:
    """Compiles ``sources`` (paths) in parallel and links a shared library."""
    inputs = list(inputs or []) + list(sources)
    if (not force and os.path.exists(out_path)
            and all(os.path.getmtime(f) <= os.path.getmtime(out_path) for f in inputs)):
        return out_path
    os.makedirs(BUILD_DIR, exist_ok=True)
    tag = os.path.splitext(os.path.basename(out_path))[0]
    objs = [os.path.join(BUILD_DIR, f"{tag}_{os.path.basename(s)}.o") for s in sources]
    with cf.ThreadPoolExecutor(max_workers=len(sources)) as ex:
        futs = [ex.submit(_compile, s, o, extra) for s, o in zip(sources, objs)]
        for f in futs:
            f.result()
    tmp = out_path + ".tmp"
    cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out_path)
    return out_path


def build(force: bool = False) -> str:
    """Builds ``libzyfa_gb300.so`` if a source is newer than it; returns its path."""
    return build_library([os.path.join(CSRC, s) for s in SOURCES], LIB_PATH,
                         force=force, inputs=_inputs())


PROBE_DIR = os.path.join(ROOT, "tests", "probes")
PROBE_LIB = os.path.join(PROBE_DIR, "libzyfa_probes.so")


def build_probes(force: bool = False) -> str:
    """Builds the test-only tensor-core probe library under tests/probes."""
    src = os.path.join(PROBE_DIR, "mma_probe.cu")
    return build_library([src], PROBE_LIB, force=force,
                         inputs=[os.path.join(CSRC, "zyfa_ptx.cuh")])


def build_all(force: bool = False) -> list:
    """Builds the library and the probes concurrently."""
    with cf.ThreadPoolExecutor(max_workers=2) as ex:
        a = ex.submit(build, force)
        b = ex.submit(build_probes, force)
        return [a.result(), b.result()]


if __name__ == "__main__":
    print(build_all(force="--force" in sys.argv))

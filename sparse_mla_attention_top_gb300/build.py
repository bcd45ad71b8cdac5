"""Builds libsvt.so from csrc/ with nvcc for sm_103a (one -gencode, translation units
compiled in parallel, static CUDA runtime). The library lands next to this file."""

from __future__ import annotations

import os
import subprocess
import sys
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
INCLUDE = ROOT / "include"
LIB = PKG / "libsvt.so"
BUILD_DIR = PKG / "_build"
# The phase-trace build: the same sources with SVT_PHASE_TRACE defined (clock stamps at each
# pipeline step of the attention kernel); a separate library that only profiling loads.
TRACE_LIB = PKG / "libsvt_trace.so"
TRACE_BUILD_DIR = PKG / "_build_trace"
SOURCES = ["api.cu", "attention.cu", "resolve.cu", "union.cu", "merge.cu", "noalloc.cu", "topk.cu", "probe.cu",
           "pair_prefill.cu"]
NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-lineinfo",
              "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden", f"-I{INCLUDE}", f"-I{CSRC}"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def _inputs():
    return [CSRC / s for s in SOURCES] + list(CSRC.glob("*.cuh")) + list(CSRC.glob("*.h")) + [INCLUDE / "svt.h"]


def up_to_date(lib: Path = LIB) -> bool:
    if not lib.exists():
        return False
    t = lib.stat().st_mtime
    return all(p.stat().st_mtime <= t for p in _inputs())


def build(force: bool = False, verbose: bool = False, trace: bool = False) -> Path:
    """Builds libsvt.so (or, with trace=True, the phase-trace library) and returns its path."""
    lib = TRACE_LIB if trace else LIB
    build_dir = TRACE_BUILD_DIR if trace else BUILD_DIR
    flags = NVCC_FLAGS + (["-DSVT_PHASE_TRACE"] if trace else [])
    if not force and up_to_date(lib):
        return lib
    build_dir.mkdir(exist_ok=True)
    nvcc = _nvcc()
    procs = []
    objs = []
    for src in SOURCES:
        obj = build_dir / (Path(src).stem + ".o")
        objs.append(obj)
        cmd = [nvcc, *flags, "-c", str(CSRC / src), "-o", str(obj)]
        if verbose:
            print(" ".join(cmd), flush=True)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
    failed = []
    for src, pr in procs:
        out, _ = pr.communicate()
        if pr.returncode != 0:
            failed.append(f"--- {src}\n{out}")
        elif verbose and out.strip():
            print(out)
    if failed:
        raise RuntimeError("nvcc failed:\n" + "\n".join(failed))
    tmp = lib.with_suffix(f".so.tmp{os.getpid()}")
    cmd = [nvcc, "-shared", "-gencode", "arch=compute_103a,code=sm_103a", "-o", str(tmp), *map(str, objs)]
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
    print(LIB)

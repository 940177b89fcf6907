"""Build the TurboQuant C-ABI library (libtq.so) in-tree for GB300 (sm_103a).

Each translation unit is compiled by nvcc in parallel, then linked into a
shared library with the CUDA runtime linked statically, so the library works
next to whatever CUDA runtime the host process (PyTorch) has loaded.

The "debug" variant (libtq_debug.so) is compiled with TQ_DEBUG_BOUNDS: every
index the kernels compute into shared or global memory is range-checked into
the device error word (TQ_ERR_DEVICE_BOUNDS) instead of being trusted.  The
environment variable TQ_LIB_VARIANT=debug makes the binding load it.

    python -m kv_cache_quantization_random_gb300.build [--force] [--verbose] [--debug]
"""

from __future__ import annotations

import argparse
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(OUT_DIR, "libtq.so")
DEBUG_DIR = os.path.join(OUT_DIR, "debug")
DEBUG_LIB_PATH = os.path.join(OUT_DIR, "libtq_debug.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

SOURCES = ["tq_host.cpp", "tq_quantize.cu", "tq_qjl.cu", "tq_decode.cu", "tq_decode_g1.cu", "tq_decode_g2.cu",
           "tq_decode_g4.cu", "tq_decode_g8.cu"]
HEADERS = ["tq_internal.h", "tq_device.cuh", "tq_decode_kernel.cuh", "tq_quant_common.cuh",
           "tq_umma.cuh"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O3",
              "--expt-relaxed-constexpr", "-I", INCLUDE]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the TurboQuant library needs the CUDA toolkit to build")


def variant() -> str:
    """The library variant this process uses: TQ_LIB_VARIANT (release | debug)."""
    v = os.environ.get("TQ_LIB_VARIANT", "release")
    if v not in ("release", "debug"):
        raise ValueError(f"TQ_LIB_VARIANT must be release or debug, not {v!r}")
    return v


def lib_path(var: str = None) -> str:
    return DEBUG_LIB_PATH if (var or variant()) == "debug" else LIB_PATH


def _stale(path: str) -> bool:
    if not os.path.exists(path):
        return True
    t = os.path.getmtime(path)
    deps = [os.path.join(CSRC, s) for s in SOURCES + HEADERS] + [os.path.join(INCLUDE, "tq.h"),
                                                                 os.path.abspath(__file__)]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=None, var: str = None) -> str:
    """Compile and link the library variant (default: TQ_LIB_VARIANT, else
    release) if any source is newer than it; return its path."""
    var = var or variant()
    path = lib_path(var)
    if not force and not _stale(path):
        return path
    obj_dir = DEBUG_DIR if var == "debug" else OUT_DIR
    os.makedirs(obj_dir, exist_ok=True)
    cc = nvcc()
    flags = NVCC_FLAGS + (["-DTQ_DEBUG_BOUNDS"] if var == "debug" else []) + list(extra_flags or [])
    procs = []
    objs = []
    for src in SOURCES:
        obj = os.path.join(obj_dir, os.path.splitext(src)[0] + ".o")
        objs.append(obj)
        cmd = [cc, *ARCH, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        text = out.decode(errors="replace")
        if p.returncode != 0:
            failed.append((src, text))
        elif verbose and text.strip():
            print(text, flush=True)
    if failed:
        msg = "\n".join(f"--- {s}\n{t}" for s, t in failed)
        raise RuntimeError(f"nvcc failed:\n{msg}")
    tmp = path + ".tmp"
    cmd = [cc, *ARCH, "-shared", "-cudart=static", "-o", tmp, *objs]
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout.decode(errors="replace"))
    os.replace(tmp, path)
    return path


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--ptxas-v", action="store_true", help="print register / spill report")
    ap.add_argument("--debug", action="store_true", help="the bounds-checked variant")
    args = ap.parse_args()
    extra = ["-Xptxas", "-v"] if args.ptxas_v else []
    print(build(force=args.force or args.ptxas_v, verbose=args.verbose or args.ptxas_v,
                extra_flags=extra, var="debug" if args.debug else None))

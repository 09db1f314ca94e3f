"""Build libhogwild.so in-tree with nvcc for sm_103a (GB300).

Translation units are compiled in parallel; the result lands in
``concurrent_shared_kv_gb300/_build/libhogwild.so``.  Run as a script or call
``build()``.
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
BUILD = os.path.join(PKG, "_build")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(BUILD, "libhogwild.so")
# the layer-timeline build (HW_TRACE: globaltimer stamps, hw_trace_read)
BUILD_TRACE = os.path.join(PKG, "_build_trace")
LIB_TRACE = os.path.join(BUILD_TRACE, "libhogwild_trace.so")

SOURCES = ["api.cpp", "attn_decode_simt.cu", "attn_decode_tc.cu", "block_commit.cu",
           "attn_decode_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _flags():
    return ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC,-O3", "-I", INCLUDE, "-I", CSRC,
            "--expt-relaxed-constexpr"] + ARCH


def _deps():
    out = [os.path.join(INCLUDE, "hogwild.h")]
    for f in os.listdir(CSRC):
        if f.endswith((".h", ".cuh")):
            out.append(os.path.join(CSRC, f))
    return out


def _stale(obj: str, src: str) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(p) > t for p in [src] + _deps())


def build(verbose: bool = False, extra: tuple = (), trace: bool = False) -> str:
    """Compile libhogwild.so (trace=True: the HW_TRACE build, libhogwild_trace.so
    in its own folder); returns the library's path."""
    out_dir, lib_path = (BUILD_TRACE, LIB_TRACE) if trace else (BUILD, LIB)
    if trace:
        extra = tuple(extra) + ("-DHW_TRACE",)
    os.makedirs(out_dir, exist_ok=True)
    cc = nvcc()
    jobs = []
    objs = []
    for s in SOURCES:
        src = os.path.join(CSRC, s)
        if not os.path.exists(src):
            continue
        obj = os.path.join(out_dir, s.rsplit(".", 1)[0] + ".o")
        objs.append(obj)
        if _stale(obj, src) or (extra and not trace):
            cmd = [cc, "-c", src, "-o", obj] + _flags() + list(extra)
            if s.endswith(".cpp"):
                cmd[1:1] = ["-x", "cu"]
            jobs.append(cmd)

    def run(cmd):
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
        return r.stdout + r.stderr

    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        for log in ex.map(run, jobs):
            if verbose and log.strip():
                print(log)
    if jobs or not os.path.exists(lib_path):
        tmp = lib_path + f".tmp{os.getpid()}"
        run([cc, "-shared", "-o", tmp] + objs + ARCH + ["-Xcompiler", "-fPIC"])
        os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))

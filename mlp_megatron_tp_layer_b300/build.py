"""Build libtpl.so (the C-ABI library) in-tree for sm_103a with nvcc.

    python mlp_megatron_tp_layer_b300/build.py [--force] [--verbose]

(Run it as a file: importing the package itself needs the built library.)

Objects go to mlp_megatron_tp_layer_b300/_build/, the library next to this
file.  A source is recompiled when it or any header is newer than its object.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libtpl.so")
SOURCES = ["api.cu", "simt.cu", "tc_gemm.cu", "decode_fused.cu", "static_ws.cu", "vocab_topk.cu", "w8_gemm.cu"]
HEADERS = [os.path.join(CSRC, h) for h in os.listdir(CSRC) if h.endswith((".h", ".cuh"))] + \
          [os.path.join(ROOT, "include", "tpl.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CUDA_HOME = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def nvcc() -> str:
    cand = os.path.join(CUDA_HOME, "bin", "nvcc")
    return cand if os.path.exists(cand) else (shutil.which("nvcc") or "nvcc")


def _stale(obj: str, src: str) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(p) > t for p in [src] + HEADERS)


def _compile(src: str, verbose: bool, build_dir: str = BUILD, defines=()) -> str:
    obj = os.path.join(build_dir, os.path.basename(src) + ".o")
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
           "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include"), *[f"-D{d}" for d in defines],
           "-c", src, "-o", obj]
    if verbose:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if verbose and (r.stdout or r.stderr):
        sys.stderr.write(r.stdout + r.stderr)
    return obj


def build(force: bool = False, verbose: bool = False, trace: bool = False) -> str:
    """Build libtpl.so; with trace, the instrumented libtpl_trace.so (fused-stack
    phase stamps, read with tpl_fused_trace_read) from objects of its own."""
    build_dir = BUILD + "_trace" if trace else BUILD
    lib = os.path.join(HERE, "libtpl_trace.so") if trace else LIB
    defines = ("TPL_FUSED_TRACE",) if trace else ()
    os.makedirs(build_dir, exist_ok=True)
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    objs = [os.path.join(build_dir, os.path.basename(s) + ".o") for s in srcs]
    todo = [s for s, o in zip(srcs, objs) if force or _stale(o, s)]
    if todo:
        with cf.ThreadPoolExecutor(max_workers=len(todo)) as ex:
            list(ex.map(lambda s: _compile(s, verbose, build_dir, defines), todo))
    if todo or not os.path.exists(lib) or any(os.path.getmtime(o) > os.path.getmtime(lib) for o in objs):
        LIBOUT = lib
        tmp = LIBOUT + ".tmp"
        cmd = [nvcc(), *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
               "-Xlinker", "-rpath," + os.path.join(CUDA_HOME, "lib64")]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIBOUT)
    return lib


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--trace", action="store_true", help="the instrumented libtpl_trace.so")
    a = ap.parse_args()
    print(build(a.force, a.verbose, a.trace))

"""In-tree build of libcvr.so: nvcc, sm_103a only, translation units compiled in parallel."""
from __future__ import annotations

import concurrent.futures
import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
# the library the binding loads: libcvr.so, or the per-CTA timeline diagnostic build (CVR_TIMELINE=1, built with
# build(timeline=True) next to it)
LIB_DEFAULT = os.path.join(PKG, "libcvr.so")
LIB_TIMELINE = os.path.join(PKG, "libcvr_timeline.so")
LIB = LIB_TIMELINE if os.environ.get("CVR_TIMELINE") == "1" else LIB_DEFAULT
SOURCES = ["cvr_api.cu", "k_sparse.cu", "k_mlp.cu", "k_gemm.cu", "k_ple.cu", "k_attn.cu", "k_attn_tc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall"]


def _compile(src: str, extra, build_dir: str = BUILD) -> str:
    obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
    cmd = ["nvcc", *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj


def build(extra_flags=(), verbose: bool = False, timeline: bool = False) -> str:
    """Compiles csrc/*.cu into libcvr.so next to this file and returns its path (timeline=True: the diagnostic
    build with per-CTA timestamps, libcvr_timeline.so)."""
    build_dir = BUILD + ("_timeline" if timeline else "")
    lib = LIB_TIMELINE if timeline else LIB_DEFAULT
    # (the timeline buffer is one device array shared by the translation units: relocatable device code)
    flags = list(extra_flags) + (["-DCVR_TIMELINE", "-rdc=true"] if timeline else [])
    os.makedirs(build_dir, exist_ok=True)
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, flags, build_dir), SOURCES))
    tmp = lib + ".tmp"
    cmd = ["nvcc", *ARCH, "-shared", *(["-rdc=true"] if timeline else []), "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    if verbose:
        print("built", lib)
    return lib

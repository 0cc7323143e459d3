"""Build the in-tree shared libraries with nvcc for sm_103a.

    python -m kv_cache_block_gb300.build        # libkk.so and synth/libkksynth.so

Each .cu compiles to its own object in parallel; objects are rebuilt only
when a source or header is newer.
"""
from __future__ import annotations

import concurrent.futures
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2"]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found")
    return path


def _newest(paths) -> float:
    return max((os.path.getmtime(p) for p in paths), default=0.0)


def _compile(src: str, obj: str, deps, extra) -> str:
    if os.path.exists(obj) and os.path.getmtime(obj) >= _newest([src] + list(deps)):
        return obj
    cmd = [nvcc()] + NVCC_FLAGS + list(extra) + ["-c", src, "-o", obj]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
    if res.stderr.strip() and "-Xptxas" in " ".join(extra):
        sys.stderr.write(res.stderr)
    return obj


def _library(srcs, deps, out: str, build_dir: str, extra=()) -> str:
    os.makedirs(build_dir, exist_ok=True)
    objs = [os.path.join(build_dir, os.path.splitext(os.path.basename(s))[0] + ".o") for s in srcs]
    with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        list(ex.map(lambda so: _compile(so[0], so[1], deps, extra), zip(srcs, objs)))
    if not os.path.exists(out) or os.path.getmtime(out) < _newest(objs):
        cmd = [nvcc()] + ARCH + ["-shared", "-o", out] + objs
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"link of {out} failed:\n{res.stdout}\n{res.stderr}")
    return out


def build_kk(extra=()) -> str:
    csrc = os.path.join(PKG, "csrc")
    srcs = sorted(glob.glob(os.path.join(csrc, "*.cu")))
    deps = glob.glob(os.path.join(csrc, "*.cuh")) + glob.glob(os.path.join(csrc, "*.h")) + [
        os.path.join(ROOT, "include", "kk.h")
    ]
    return _library(srcs, deps, os.path.join(PKG, "libkk.so"), os.path.join(PKG, "_build"), extra)


def build_synth(extra=()) -> str:
    sdir = os.path.join(ROOT, "synth")
    srcs = sorted(glob.glob(os.path.join(sdir, "csrc", "*.cu")))
    return _library(srcs, [], os.path.join(sdir, "libkksynth.so"), os.path.join(sdir, "_build"), extra)


def build_all(extra=()) -> None:
    with concurrent.futures.ThreadPoolExecutor(max_workers=2) as ex:
        futs = [ex.submit(build_kk, extra), ex.submit(build_synth, extra)]
        for f in futs:
            f.result()


if __name__ == "__main__":
    build_all(sys.argv[1:])
    print("built", os.path.join(PKG, "libkk.so"))

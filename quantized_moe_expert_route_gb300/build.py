"""Builds the in-tree shared libraries with nvcc for sm_103a.

* ``quantized_moe_expert_route_gb300/libmoe_route.so``: the layer (C ABI in
  include/moe_route.h).
* ``synth/libmoe_synth.so``: the GPU filler of seeded synthetic weights (C ABI
  in include/moe_synth.h); benchmark and test input generation only.

Translation units compile in parallel; a library is rebuilt only when one of
its sources or headers is newer than it.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr"] + ARCH

LIBS = {
    "moe_route": {
        "out": os.path.join(PKG, "libmoe_route.so"),
        "srcs": [os.path.join(PKG, "csrc", f) for f in ("api.cu", "route.cu", "bucket.cu", "gemv.cu", "stream.cu", "decode.cu", "tc.cu", "noalloc.cu", "shard.cu", "cold.cu")],
        "deps": [os.path.join(PKG, "csrc", "moe_internal.cuh"), os.path.join(PKG, "csrc", "dot16.cuh"), os.path.join(PKG, "csrc", "pdl.cuh"),
                 os.path.join(INCLUDE, "moe_route.h")],
    },
    "moe_synth": {
        "out": os.path.join(ROOT, "synth", "libmoe_synth.so"),
        "srcs": [os.path.join(ROOT, "synth", "csrc", "synth_fill.cu")],
        "deps": [os.path.join(INCLUDE, "moe_synth.h")],
    },
}


def nvcc() -> str:
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(p):
        raise RuntimeError("nvcc not found")
    return p


def _stale(out: str, inputs) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(i) > t for i in inputs)


def _compile(src: str, obj: str, deps) -> None:
    if not _stale(obj, [src] + list(deps)):
        return
    cmd = [nvcc(), *NVCC_FLAGS, "-I", INCLUDE, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")


def build(verbose: bool = False) -> dict:
    os.makedirs(BUILD, exist_ok=True)
    jobs = []
    for name, spec in LIBS.items():
        for src in spec["srcs"]:
            obj = os.path.join(BUILD, f"{name}__{os.path.basename(src)}.o")
            jobs.append((name, src, obj, spec["deps"]))
    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        futs = [ex.submit(_compile, src, obj, deps) for _, src, obj, deps in jobs]
        for f in futs:
            f.result()
    outs = {}
    for name, spec in LIBS.items():
        objs = [o for n, _, o, _ in jobs if n == name]
        if _stale(spec["out"], objs):
            cmd = [nvcc(), *ARCH, "-shared", "-o", spec["out"], *objs]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"link failed for {name}:\n{r.stdout}\n{r.stderr}")
        outs[name] = spec["out"]
        if verbose:
            print(f"built {spec['out']}")
    return outs


if __name__ == "__main__":
    build(verbose=True)
    sys.exit(0)

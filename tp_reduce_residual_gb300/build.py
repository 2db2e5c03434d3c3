"""Build libbeamnorm.so in-tree for sm_103a (GB300).

Nine objects, one per kernel mode, are compiled from one template source in
parallel, plus the small-T finalize object, the static-scratch object and the
C-ABI object; everything
is compiled with ``-fmad=false`` so that the FP32 epilogue is never
contracted into FMAs ("Fuse Beam's TP all-reduce with its sandwich norms",
"Details", "Build" bullet).  nvcc cross-compiles without a GPU.  The result is
``tp_reduce_residual_gb300/_build/libbeamnorm.so`` (git-ignored); a stamp of
the sources and flags skips rebuilding when nothing changed.

    python -m tp_reduce_residual_gb300.build [--force] [--verbose-ptxas]
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libbeamnorm.so")
STAMP = os.path.join(OUT_DIR, "libbeamnorm.stamp")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-fmad=false", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden", "-Xcompiler", "-Wall",
              "-Wno-deprecated-gpu-targets"]

# kernel modes: object name -> mode bits (see csrc/bn_internal.h)
MODES = {
    "reduce_norm": 4 | 8,
    "fin_reduce_norm": 1 | 4 | 8,
    "reduce_resnorm": 8,
    "fin_reduce_resnorm": 1 | 8,
    "reduce_only": 16,
    "fin_reduce_only": 1 | 16,
    "norm_only": 2 | 4 | 8,
    "fin_only": 1 | 32,
    "resnorm_only": 2 | 8,
}

SOURCES = ["bn_device.cuh", "bn_internal.h", "bn_kernels.cu", "bn_abi.cu", "bn_wide.h",
           "bn_wide.cu", "bn_noalloc.cu", "bn_cluster.h", "bn_cluster.cu"]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libbeamnorm")
    return path


def _stamp(extra) -> str:
    h = hashlib.sha256()
    for name in SOURCES:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(f.read())
    with open(os.path.join(INCLUDE, "beamnorm.h"), "rb") as f:
        h.update(f.read())
    h.update(" ".join(ARCH + NVCC_FLAGS + list(extra)).encode())
    h.update(repr(sorted(MODES.items())).encode())
    return h.hexdigest()


def _run(cmd):
    p = subprocess.run(cmd, capture_output=True, text=True)
    if p.returncode != 0:
        raise RuntimeError(f"command failed ({p.returncode}): {' '.join(cmd)}\n{p.stdout}\n{p.stderr}")
    return p.stdout + p.stderr


def build(force: bool = False, verbose_ptxas: bool = False, jobs: int = 0) -> str:
    """Compile (if needed) and return the path of libbeamnorm.so."""
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    os.makedirs(OUT_DIR, exist_ok=True)
    stamp = _stamp(extra)
    if not force and os.path.exists(LIB) and os.path.exists(STAMP):
        with open(STAMP) as f:
            if f.read().strip() == stamp:
                return LIB
    cc = nvcc()
    inc = ["-I", INCLUDE, "-I", CSRC]
    cmds = []
    for name, bits in MODES.items():
        obj = os.path.join(OUT_DIR, f"bn_kernels_{name}.o")
        cmds.append([cc, *ARCH, *NVCC_FLAGS, *extra, *inc, f"-DBN_MODE_NAME={name}",
                     f"-DBN_MODE_VALUE={bits}", "-c", os.path.join(CSRC, "bn_kernels.cu"),
                     "-o", obj])
    abi_obj = os.path.join(OUT_DIR, "bn_abi.o")
    cmds.append([cc, *ARCH, *NVCC_FLAGS, *inc, "-c", os.path.join(CSRC, "bn_abi.cu"), "-o", abi_obj])
    wide_obj = os.path.join(OUT_DIR, "bn_wide.o")
    cmds.append([cc, *ARCH, *NVCC_FLAGS, *extra, *inc, "-c", os.path.join(CSRC, "bn_wide.cu"),
                 "-o", wide_obj])
    cluster_obj = os.path.join(OUT_DIR, "bn_cluster.o")
    cmds.append([cc, *ARCH, *NVCC_FLAGS, *extra, *inc, "-c", os.path.join(CSRC, "bn_cluster.cu"),
                 "-o", cluster_obj])
    noalloc_obj = os.path.join(OUT_DIR, "bn_noalloc.o")
    cmds.append([cc, *ARCH, *NVCC_FLAGS, *inc, "-c", os.path.join(CSRC, "bn_noalloc.cu"),
                 "-o", noalloc_obj])
    jobs = jobs or min(len(cmds), max(1, os.cpu_count() or 1))
    logs = []
    with cf.ThreadPoolExecutor(max_workers=jobs) as ex:
        for out in ex.map(_run, cmds):
            logs.append(out)
    objs = [c[-1] for c in cmds]
    tmp = LIB + f".tmp{os.getpid()}"
    _run([cc, *ARCH, "-shared", "-o", tmp, *objs])
    os.replace(tmp, LIB)
    with open(STAMP, "w") as f:
        f.write(stamp)
    if verbose_ptxas:
        sys.stdout.write("".join(logs))
    return LIB


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose-ptxas", action="store_true")
    args = ap.parse_args(argv)
    print(build(force=args.force, verbose_ptxas=args.verbose_ptxas))


if __name__ == "__main__":
    main()

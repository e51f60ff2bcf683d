"""Build of the CUDA library: nvcc, one translation unit per process, linked into one shared object.

Output: ``gemm_groupnorm_accelerator_gb300/_build/libconv1dnorm.so`` (kept out of version
control). Only sm_103a code is generated; the runtime is linked statically so the library
loads without a driver (e.g. for the host-only tests).
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import hashlib
import os
import re
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
ROOT = os.path.dirname(PKG)
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libconv1dnorm.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "-diag-suppress", "177", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA library cannot be built")
    return path


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _headers():
    return sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))) + \
        [os.path.join(INCLUDE, "conv1d_norm.h")]


def _code_only(text: str) -> str:
    """Source text without comments and with runs of whitespace collapsed: what the compiler turns
    into code (string literals in these sources hold no comment markers)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_fingerprint(source: str) -> str:
    """Hash of the code of one translation unit (a csrc/*.cu file name), of every header and of the
    flags, comments and layout left out: a profile of a kernel defined in that file stays valid
    while this does not change (a comment-only edit keeps it)."""
    h = hashlib.sha256()
    for f in [os.path.join(CSRC, source)] + _headers():
        with open(f, encoding="utf-8") as fh:
            h.update(os.path.basename(f).encode())
            h.update(_code_only(fh.read()).encode())
    h.update(" ".join(ARCH + [f for f in NVCC_FLAGS if f not in (INCLUDE, CSRC)]).encode())
    return h.hexdigest()


def _fingerprint(sources=None) -> str:
    h = hashlib.sha256()
    for f in (_sources() if sources is None else sources) + _headers():
        with open(f, "rb") as fh:
            h.update(os.path.basename(f).encode())
            h.update(fh.read())
    # flags without the (machine-dependent) include paths: the same sources and flags give the same
    # fingerprint on every machine, so a profile taken on one box matches a build on another
    h.update(" ".join(ARCH + [f for f in NVCC_FLAGS if f not in (INCLUDE, CSRC)]).encode())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile every csrc/*.cu for sm_103a and link libconv1dnorm.so; skip when up to date."""
    os.makedirs(BUILD, exist_ok=True)
    stamp = os.path.join(BUILD, "stamp")
    fp = _fingerprint()
    if not force and os.path.exists(LIB) and os.path.exists(stamp) and open(stamp).read() == fp:
        return LIB
    nv = nvcc()
    objs = []

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        cmd = [nv] + ARCH + NVCC_FLAGS + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            print(r.stdout + r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, _sources()))
    tmp = LIB + f".{os.getpid()}.tmp"
    cmd = [nv] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(stamp, "w") as f:
        f.write(fp)
    return LIB

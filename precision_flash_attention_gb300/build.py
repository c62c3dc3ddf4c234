"""Builds libpfa.so in-tree with nvcc for sm_103a (no cmake, no setuptools).

Translation units are compiled in parallel, then linked into
``precision_flash_attention_gb300/libpfa.so``. A stamp file records the host
architecture and a hash of the sources so that a library built on another
machine (or from older sources) is rebuilt.
"""
from __future__ import annotations

import hashlib
import os
import platform
import re
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libpfa.so")
STAMP = os.path.join(BUILD_DIR, "stamp.txt")

SOURCES = ["attn_api.cu", "attn_fwd.cu", "attn_fwd_study.cu", "attn_fwd_lowp.cu", "attn_fwd_pair.cu",
           "attn_bwd.cu", "attn_dq.cu", "attn_delta.cu", "attn_bwd_noalloc.cu", "wait_probe.cu"]
HEADERS = [os.path.join(CSRC, "pfa_device.cuh"), os.path.join(CSRC, "pfa_internal.h"),
           os.path.join(CSRC, "attn_fwd.cuh"), os.path.join(CSRC, "pfa_trace.cuh"),
           os.path.join(INCLUDE, "pfa.h")]

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpfa")


def source_digest() -> str:
    """Hash of the CUDA sources and headers (independent of the host machine)."""
    h = hashlib.sha256()
    for path in [os.path.join(CSRC, s) for s in SOURCES] + HEADERS:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


# The translation unit of each kernel; its traffic record is keyed to that file,
# the API file that builds its launch arguments and the shared headers.
KERNEL_SOURCES = {"attn_bwd_kernel": "attn_bwd.cu", "convert_dq_kernel": "attn_bwd.cu",
                  "attn_dq_kernel": "attn_dq.cu",
                  "attn_fwd_kernel": "attn_fwd.cu", "delta_kernel": "attn_delta.cu",
                  "delta_alt_kernel": "attn_delta.cu"}


def _product_text(path: str) -> bytes:
    """A source file as the product build compiles it: without comments and without
    what only trace builds (-DPFA_TRACE) compile (lines that invoke a trace macro and
    `#if defined(PFA_TRACE) ...` blocks)."""
    out, depth = [], 0
    with open(path, encoding="utf-8") as f:
        for line in f:
            t = line.strip()
            if depth:
                if t.startswith("#if"):
                    depth += 1
                elif t.startswith("#endif"):
                    depth -= 1
                continue
            if t.startswith("#if defined(PFA_TRACE)"):
                depth = 1
                continue
            if "_TRACE(" in t and "define" not in t:
                continue
            out.append(line)
    text = re.sub(r"/\*.*?\*/", "", "".join(out), flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    # Layout does not change what is compiled: one stripped, non-empty line per line.
    return "\n".join(t.strip() for t in text.splitlines() if t.strip()).encode()


def _local_includes(path: str, seen: list) -> list:
    """`path` and, depth first, the project headers it includes (#include "..."), each once."""
    if path in seen:
        return seen
    seen.append(path)
    with open(path, encoding="utf-8") as f:
        for name in re.findall(r'^\s*#include\s+"([^"]+)"', f.read(), flags=re.M):
            for d in (CSRC, INCLUDE):
                cand = os.path.join(d, name)
                if os.path.exists(cand):
                    _local_includes(cand, seen)
                    break
    return seen


def kernel_source_digest(kernel: str) -> str:
    """Hash of the sources one kernel is built from (see KERNEL_SOURCES): its translation
    unit, the API file that builds its launch arguments and the project headers the two
    include, as the product build compiles them."""
    h = hashlib.sha256()
    files = []
    for tu in (KERNEL_SOURCES[kernel], "attn_api.cu"):
        _local_includes(os.path.join(CSRC, tu), files)
    for path in files:
        h.update(_product_text(path))
    return h.hexdigest()


def _digest() -> str:
    h = hashlib.sha256()
    h.update(platform.machine().encode())
    h.update(" ".join(ARCH_FLAGS + CFLAGS).encode())
    h.update(source_digest().encode())
    return h.hexdigest()


def is_current() -> bool:
    if not os.path.exists(LIB) or not os.path.exists(STAMP):
        return False
    with open(STAMP, encoding="utf-8") as f:
        return f.read().strip() == _digest()


def build_library(force: bool = False, verbose: bool = False) -> str:
    """Compile and link libpfa.so unless an up-to-date build exists; returns its path."""
    if not force and is_current():
        return LIB
    os.makedirs(BUILD_DIR, exist_ok=True)
    cc = nvcc()

    def compile_one(src: str) -> str:
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        cmd = [cc, *CFLAGS, *ARCH_FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + ".tmp"
    cmd = [cc, "-shared", *ARCH_FLAGS, "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(STAMP, "w", encoding="utf-8") as f:
        f.write(_digest())
    return LIB


if __name__ == "__main__":
    print(build_library(force=True, verbose=True))

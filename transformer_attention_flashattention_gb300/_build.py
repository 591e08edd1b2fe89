"""Builds libfa.so (the C-ABI library) in-tree with nvcc for sm_103a.

Each translation unit is compiled in parallel into ``_build/``, then linked with
the static CUDA runtime into ``transformer_attention_flashattention_gb300/libfa.so``.
No libcuda link: the tensor-map encoder is fetched from the driver at run time.
Run as ``python -m transformer_attention_flashattention_gb300._build``.

The library carries the SHA-256 (first 16 hex digits) of everything it is built
from: the CUDA sources, the C header, this script and the compiler flags.  It is
compiled into ``libfa.so`` as a string and returned by ``fa_build_id()``.  A
library is rebuilt unless it carries the id of the sources as they are now, and
the binding refuses to load one that does not.
"""
from __future__ import annotations

import hashlib
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_PATH = os.path.join(PKG_DIR, "libfa.so")
SOURCES = ["fa_api.cu", "fa_fwd.cu", "fa_fwd1.cu", "fa_fwd2.cu", "fa_fwd_fp8.cu", "fa_quant.cu", "fa_decode.cu",
           "fa_decode_noalloc.cu", "fa_bwd.cu",
           "fa_host.cu", "fa_naive.cu"]
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
          "-I" + os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is needed to build libfa.so")


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(ROOT, "include", "fa.h"))
    files.append(os.path.abspath(__file__))
    return files


BUILD_ID_TAG = b"fa-build-id:"


def source_id() -> str:
    """Hash of the sources, header, this script and the flags the library is built from."""
    h = hashlib.sha256()
    for f in sorted(_deps()):
        h.update(os.path.relpath(f, ROOT).encode() + b"\0")
        with open(f, "rb") as fh:
            h.update(fh.read() + b"\0")
    h.update(" ".join(ARCH_FLAGS + CFLAGS).encode())
    return h.hexdigest()[:16]


def built_id(path: str = LIB_PATH):
    """The build id a library file carries (read from its bytes, without loading it), or None."""
    try:
        with open(path, "rb") as f:
            data = f.read()
    except OSError:
        return None
    i = data.find(BUILD_ID_TAG)
    if i < 0:
        return None
    return data[i + len(BUILD_ID_TAG):i + len(BUILD_ID_TAG) + 16].decode("ascii", "replace")


def _stale() -> bool:
    return built_id() != source_id()


def _compile(src: str, extra) -> str:
    obj = os.path.join(BUILD_DIR, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *ARCH_FLAGS, *CFLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return obj


def build(force: bool = False, verbose: bool = False, extra_flags=(), quiet: bool = False) -> str:
    """Compile and link libfa.so unless it already carries the current sources' build id;
    returns its path and says (unless ``quiet``) whether it compiled."""
    sid = source_id()
    if not force and not extra_flags and built_id() == sid:
        if not quiet:
            print(f"libfa.so: up to date (build id {sid})", flush=True)
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    extra = list(extra_flags) + (["-Xptxas", "-v"] if verbose else []) + [f'-DFA_BUILD_ID="{sid}"']
    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra), SOURCES))
    tmp = LIB_PATH + ".tmp"
    cmd = [nvcc(), *ARCH_FLAGS, "-shared", "-o", tmp, *objs, "-ldl"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    if not quiet:
        print(f"libfa.so: compiled {len(SOURCES)} translation units (build id {sid})", flush=True)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

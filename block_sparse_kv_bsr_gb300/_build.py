"""Build the C-ABI library ``libbsrattn.so`` for sm_103a with nvcc.

Every translation unit under ``csrc/`` is compiled in parallel into
``_build/`` and linked into one shared library (static CUDA runtime, no
libcuda link: the driver entry point for tensor-map encoding is fetched at
run time).  The build is skipped when no source or flag changed.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import re
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT = os.path.join(PKG, "_build")
LIB_NAME = "libbsrattn.so"

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC"]
COMMON = FLAGS + [f"-I{INCLUDE}", f"-I{CSRC}"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libbsrattn.so")


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cpp")))


def _digest() -> str:
    h = hashlib.sha256()
    files = sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC))
    files.append(os.path.join(INCLUDE, "bsr_attn.h"))
    for full in files:
        with open(full, "rb") as f:
            h.update(os.path.basename(full).encode())
            h.update(f.read())
    h.update(" ".join(ARCH + COMMON).encode())
    return h.hexdigest()[:16]


# Sources that determine a kernel family's machine code (for matching a profile to a build).
DECODE_KERNEL_SOURCES = ("bsr_decode.cuh", "bsr_decode_d128.cu", "bsr_internal.h", "ptx.cuh",
                         "bsr_launch.cuh")
PREFILL_KERNEL_SOURCES = ("bsr_prefill.cu", "bsr_internal.h", "ptx.cuh", "umma.cuh",
                          "bsr_launch.cuh")
DECODE_KV8_KERNEL_SOURCES = ("bsr_decode_kv8.cu", "bsr_decode.cuh", "bsr_internal.h", "ptx.cuh",
                             "bsr_launch.cuh", "bsr_launchers.h")


_COMMENT = re.compile(rb"//[^\n]*|/\*.*?\*/", re.S)


def _code_of(text: bytes) -> bytes:
    """Source text without comments and blank-space differences (what the compiler sees),
    so that editing a comment does not change a kernel's build digest.  String literals
    in these sources hold inline PTX, which has no comment markers."""
    lines = (ln.rstrip() for ln in _COMMENT.sub(b"", text).split(b"\n"))
    return b"\n".join(ln for ln in lines if ln)


def kernel_digest(names=DECODE_KERNEL_SOURCES) -> str:
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode())
            h.update(_code_of(f.read()))
    h.update(" ".join(ARCH + FLAGS).encode())   # no paths: the same on every machine
    return h.hexdigest()[:16]


def lib_path() -> str:
    return os.path.join(OUT, LIB_NAME)


def build(verbose: bool = False, jobs: int | None = None) -> str:
    """Compile and link if needed; return the path of the shared library."""
    os.makedirs(OUT, exist_ok=True)
    tag = _digest()
    stamp = os.path.join(OUT, "stamp")
    lib = lib_path()
    if os.path.exists(lib) and os.path.exists(stamp) and open(stamp).read() == tag:
        return lib
    nvcc = _nvcc()

    def compile_one(src: str) -> str:
        obj = os.path.join(OUT, os.path.basename(src) + ".o")
        cmd = [nvcc, *ARCH, *COMMON, "-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            print(r.stdout + r.stderr)
        return obj

    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=jobs or min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = f"{lib}.{os.getpid()}.tmp"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", *objs, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    with open(stamp, "w") as f:
        f.write(tag)
    return lib


if __name__ == "__main__":
    print(build(verbose=True))

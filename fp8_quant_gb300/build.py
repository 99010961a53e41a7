"""Build step of the CUDA library: nvcc, sm_103a only, in-tree.

``python -m fp8_quant_gb300.build`` (or ``build()``) compiles the translation
units in ``csrc/`` in parallel and links them into ``lib/libkvstore.so`` next
to this file. Symbols are hidden except the C ABI of ``include/kvstore.h``.
The CUDA runtime is linked statically, so the library needs only the driver
at run time.
"""

from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
SOURCES = [os.path.join(CSRC, f) for f in ("kvstore.cu", "kv_gather.cu", "kv_scale.cu", "kv_fp8_ex.cu")]
SRC = SOURCES[0]
HEADER = os.path.join(ROOT, "include", "kvstore.h")
LIBDIR = os.path.join(HERE, "lib")
LIB = os.path.join(LIBDIR, "libkvstore.so")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-lineinfo", "-O3", "-std=c++17",
    "-ftz=false", "-prec-div=true", "-prec-sqrt=true", "-fmad=false",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-O2", "-Xcompiler", "-fvisibility=hidden",
]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if c and (os.path.isabs(c) and os.path.exists(c) or not os.path.isabs(c)):
            return c
    return "nvcc"


def _deps():
    return [HEADER] + [os.path.join(CSRC, f) for f in sorted(os.listdir(CSRC))
                       if f.endswith((".cu", ".cuh", ".h"))]


def build(force: bool = False, verbose: bool = False, extra_flags=(), out: str = None) -> str:
    """Compile and link the library; returns its path. Skips the work when the
    library is newer than every source and header (unless ``force``)."""
    from concurrent.futures import ThreadPoolExecutor
    lib = out or LIB
    if (not force and out is None and os.path.exists(lib)
            and all(os.path.getmtime(lib) >= os.path.getmtime(d) for d in _deps())):
        return lib
    os.makedirs(os.path.dirname(lib), exist_ok=True)
    tag = f".tmp{os.getpid()}"
    objs = [lib + "." + os.path.basename(src) + tag + ".o" for src in SOURCES]
    flags = [*NVCC_FLAGS, *extra_flags, "-I", os.path.join(ROOT, "include"), "-I", CSRC]
    if verbose:
        flags.insert(0, "-Xptxas=-v")

    def compile_one(pair):
        src, obj = pair
        subprocess.check_call([nvcc(), *flags, "-c", "-o", obj, src])

    try:
        with ThreadPoolExecutor(len(SOURCES)) as ex:
            list(ex.map(compile_one, zip(SOURCES, objs)))
        subprocess.check_call([nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-shared",
                               "-cudart", "static", "-o", lib + tag, *objs])
        os.replace(lib + tag, lib)
    finally:
        for o in objs:
            if os.path.exists(o):
                os.remove(o)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

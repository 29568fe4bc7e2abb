"""Build libditattn.so in-tree with nvcc for sm_103a.

Each .cu translation unit is compiled in parallel, then linked into one shared
library with the CUDA runtime linked statically (so the library loads on a
machine without a GPU driver; the driver API is reached at run time through
the runtime's entry-point query).
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
from pathlib import Path

PKG = Path(__file__).resolve().parent
CSRC = PKG / "csrc"
INCLUDE = PKG.parent / "include"
BUILD = PKG.parent / "_build"
LIBRARY = PKG / "libditattn.so"
SOURCES = ["api.cu", "attn_fwd.cu", "attn_merge.cu", "qk_norm_rope.cu", "row_kernels.cu", "fp8.cu", "host_path.cu",
           "attention_path.cu", "attention_noalloc.cu", "ring_overlap.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not Path(path).exists():
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build libditattn.so")
    return path


def _stale() -> bool:
    if not LIBRARY.exists():
        return True
    t = LIBRARY.stat().st_mtime
    deps = list(CSRC.glob("*")) + list(INCLUDE.glob("*.h")) + [Path(__file__)]
    return any(p.stat().st_mtime > t for p in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> Path:
    if not force and not _stale():
        return LIBRARY
    BUILD.mkdir(exist_ok=True)
    flags = [*ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", str(INCLUDE),
             "--expt-relaxed-constexpr", *extra_flags]
    if verbose:
        flags += ["-Xptxas", "-v"]
    cc = nvcc()

    def compile_one(src: str) -> tuple[Path, str]:
        obj = BUILD / (src + ".o")
        r = subprocess.run([cc, *flags, "-c", str(CSRC / src), "-o", str(obj)], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=min(len(SOURCES), os.cpu_count() or 1)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose:
        for _, err in results:
            print(err)
    tmp = LIBRARY.with_suffix(".so.tmp")
    r = subprocess.run([cc, *ARCH, "-shared", "-cudart", "static", "-o", str(tmp), *[str(o) for o, _ in results]],
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, LIBRARY)
    return LIBRARY


if __name__ == "__main__":
    import sys

    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIBRARY)

"""Build librbkv.so in-tree with nvcc for sm_103a.

Each translation unit is compiled in parallel to an object file under
``ragged_blocked_kv_gb300/_lib/obj`` and the objects are linked into
``ragged_blocked_kv_gb300/_lib/librbkv.so`` (CUDA runtime linked statically, so
the library needs only the driver at run time).  A rebuild happens when any
source or header is newer than the library.

    python -m ragged_blocked_kv_gb300.build [--force] [--verbose]
"""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
INCLUDE = ROOT / "include"
LIBDIR = PKG / "_lib"
LIB = LIBDIR / "librbkv.so"

SOURCES = ["rbkv_host.cpp", "rbkv_kernels.cu", "rbkv_decode.cu", "rbkv_chunk.cu",
           "rbkv_chunk_single.cu", "rbkv_noalloc.cu", "rbkv_router.cpp",
           "rbkv_gemm.cu", "rbkv_layer.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    return "nvcc"


def _flags(verbose: bool):
    f = ["-O3", "-std=c++17", "-lineinfo", *ARCH, "-Xcompiler", "-fPIC,-O3,-ffp-contract=off",
         f"-I{INCLUDE}", f"-I{CSRC}"]
    if verbose:
        f += ["-Xptxas", "-v"]
    return f


def _stale() -> bool:
    if not LIB.exists():
        return True
    t = LIB.stat().st_mtime
    deps = [CSRC / s for s in SOURCES] + list(CSRC.glob("*.h")) + list(INCLUDE.glob("*.h"))
    return any(d.stat().st_mtime > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> Path:
    """Compile (if stale) and return the path of librbkv.so."""
    if not force and not _stale():
        return LIB
    obj = LIBDIR / "obj"
    obj.mkdir(parents=True, exist_ok=True)
    flags = _flags(verbose)

    def compile_one(src: str):
        out = obj / (src + ".o")
        cmd = [nvcc(), *flags, "-c", str(CSRC / src), "-o", str(out)]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, cmd, r

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    for src, cmd, r in results:
        if verbose and (r.stdout or r.stderr):
            sys.stderr.write(f"--- {src}\n{r.stdout}{r.stderr}")
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{' '.join(cmd)}\n{r.stdout}{r.stderr}")
    tmp = LIB.with_suffix(".so.tmp")
    cmd = [nvcc(), "-shared", *ARCH, "-o", str(tmp)] + [str(obj / (s + ".o")) for s in SOURCES]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stdout}{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="--verbose" in sys.argv)
    print(LIB)

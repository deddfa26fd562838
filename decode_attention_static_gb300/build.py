"""Build the CUDA library (libdecode_attn.so) for sm_103a with nvcc.

Each translation unit is compiled in parallel into _build/, then linked into
a shared library beside this file. cudart is linked statically, so the
library needs only the CUDA driver at run time.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import pathlib
import shutil
import subprocess

PKG = pathlib.Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
INCLUDE = ROOT / "include"
BUILD_DIR = ROOT / "_build"
LIBRARY = PKG / "libdecode_attn.so"

SOURCES = ["abi.cu", "decode_f16.cu", "decode_bf16.cu", "decode_f16_rope.cu", "decode_bf16_rope.cu", "append.cu",
           "static_scratch.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         f"-I{INCLUDE}", f"-I{CSRC}"]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not pathlib.Path(exe).exists():
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")
    return exe


def _compile(src: pathlib.Path, obj: pathlib.Path, extra: list[str]) -> str:
    cmd = [nvcc(), *ARCH, *FLAGS, *extra, "-c", str(src), "-o", str(obj)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src.name}:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return r.stderr


def _stale(output: pathlib.Path) -> bool:
    if not output.exists():
        return True
    t = output.stat().st_mtime
    deps = list(CSRC.glob("*")) + list(INCLUDE.glob("*.h")) + [pathlib.Path(__file__)]
    return any(d.stat().st_mtime > t for d in deps)


def build_library(force: bool = False, verbose_ptxas: bool = False) -> pathlib.Path:
    """Compile and link the library if any source is newer than it."""
    if not force and not _stale(LIBRARY):
        return LIBRARY
    BUILD_DIR.mkdir(exist_ok=True)
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    objs = [BUILD_DIR / (s.replace(".cu", ".o")) for s in SOURCES]
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        logs = list(ex.map(lambda so: _compile(CSRC / so[0], so[1], extra), zip(SOURCES, objs)))
    if verbose_ptxas:
        for s, log in zip(SOURCES, logs):
            print(f"== {s}\n{log}")
    tmp = LIBRARY.with_name(LIBRARY.name + f".tmp{os.getpid()}")
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", str(tmp), *map(str, objs)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIBRARY)
    return LIBRARY


if __name__ == "__main__":
    import sys

    print(build_library(force=True, verbose_ptxas="-v" in sys.argv))

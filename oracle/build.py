"""Compile the decode-attention oracle (oracle.c) into a shared library.

Test infrastructure: the oracle is the checker for the CUDA library, never a
part of it. ``-ffp-contract=off`` keeps every multiply and add separately
rounded, so that x86-64 and aarch64 builds give the same doubles.
"""
from __future__ import annotations

import os
import pathlib
import shutil
import subprocess
import tempfile

HERE = pathlib.Path(__file__).resolve().parent
SOURCE = HERE / "oracle.c"
LIBRARY = HERE / "liboracle.so"

BASE_FLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]


def _openmp_works(cc: str) -> bool:
    with tempfile.TemporaryDirectory() as tmp:
        src = pathlib.Path(tmp) / "t.c"
        src.write_text("#include <omp.h>\nint main(void){return omp_get_max_threads() > 0 ? 0 : 1;}\n")
        r = subprocess.run([cc, "-fopenmp", str(src), "-o", str(pathlib.Path(tmp) / "t")],
                           capture_output=True)
        return r.returncode == 0


def compile_oracle(source: pathlib.Path = SOURCE, output: pathlib.Path = LIBRARY,
                   openmp: bool | None = None) -> pathlib.Path:
    """Build ``source`` into ``output`` with gcc; returns the library path."""
    cc = os.environ.get("CC") or shutil.which("gcc") or "cc"
    if openmp is None:
        openmp = _openmp_works(cc)
    flags = list(BASE_FLAGS) + (["-fopenmp"] if openmp else [])
    output = pathlib.Path(output)
    tmp_out = output.with_name(output.name + f".tmp{os.getpid()}")
    cmd = [cc, *flags, str(source), "-o", str(tmp_out), "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"oracle build failed: {' '.join(cmd)}\n{r.stderr}")
    os.replace(tmp_out, output)
    return output


def ensure_built() -> pathlib.Path:
    """Build the oracle if the library is missing or older than its source."""
    if not LIBRARY.exists() or LIBRARY.stat().st_mtime < SOURCE.stat().st_mtime:
        compile_oracle()
    return LIBRARY


if __name__ == "__main__":
    print(compile_oracle())

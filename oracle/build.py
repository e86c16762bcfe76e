"""Compile the FP64 CPU oracle (pkv_oracle.c) into a shared library with gcc.

Test infrastructure: the library this writes is loaded only by the test suite,
the smoke check and the CPU-baseline leg of the benchmark.  OpenMP is used when
the compiler supports it (the oracle's attention loop runs rows x query heads
in parallel); otherwise the same code builds single-threaded.
"""
from __future__ import annotations

import os
import subprocess
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "pkv_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libpkv_oracle.so")


def _openmp_works(cc: str) -> bool:
    with tempfile.TemporaryDirectory() as tmp:
        src = os.path.join(tmp, "t.c")
        with open(src, "w") as f:
            f.write("#include <omp.h>\nint main(void){return omp_get_max_threads()>0?0:1;}\n")
        r = subprocess.run([cc, "-fopenmp", src, "-o", os.path.join(tmp, "t")],
                           capture_output=True)
        return r.returncode == 0


def build(force: bool = False) -> str:
    """Build the oracle library if it is missing or older than its source."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    cc = os.environ.get("CC", "gcc")
    # -O2 without -ffast-math: the oracle relies on IEEE double arithmetic.
    flags = ["-O2", "-std=gnu11", "-shared", "-fPIC", "-fno-fast-math", "-ffp-contract=off"]
    if _openmp_works(cc):
        flags.append("-fopenmp")
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.run([cc, *flags, SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))

"""Build the CPU oracle (test infrastructure) as a shared library.

Compiles ``oracle/mx_oracle.c`` with the host C compiler into
``oracle/_build/libmx_oracle.so``.  Plain C99, ``-O2``, no fast-math and no
floating-point contraction, so the oracle gives the same bits on x86_64 and
aarch64 hosts.  OpenMP is used when the compiler accepts ``-fopenmp``.
"""
from __future__ import annotations

import os
import subprocess
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "mx_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libmx_oracle.so")


def _cc() -> str:
    return os.environ.get("CC", "gcc")


def _openmp_ok(cc: str) -> bool:
    with tempfile.TemporaryDirectory() as td:
        src = os.path.join(td, "t.c")
        with open(src, "w") as f:
            f.write("#include <omp.h>\nint main(void){return omp_get_max_threads() > 0 ? 0 : 1;}\n")
        r = subprocess.run([cc, "-fopenmp", src, "-o", os.path.join(td, "t")],
                           capture_output=True)
        return r.returncode == 0


def build(force: bool = False) -> str:
    """Compile the oracle if the library is missing or older than its source."""
    os.makedirs(OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)
            and os.path.getmtime(LIB) >= os.path.getmtime(__file__)):
        return LIB
    cc = _cc()
    flags = ["-std=c99", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]
    if _openmp_ok(cc):
        flags.append("-fopenmp")
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.run([cc, *flags, SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))

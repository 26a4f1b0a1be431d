"""Builds the CPU oracle shared library (test infrastructure only).

The oracle is plain C compiled with the host compiler; OpenMP is used when the
compiler supports it and skipped otherwise (the results do not depend on it).
"""
from __future__ import annotations

import os
import subprocess
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "kda_oracle.c")
BUILD_DIR = os.path.join(HERE, "_build")


def _openmp_flag(cc: str) -> list[str]:
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "t.c")
        with open(src, "w") as f:
            f.write("#include <omp.h>\nint main(void){return omp_get_max_threads() > 0 ? 0 : 1;}\n")
        r = subprocess.run([cc, "-fopenmp", src, "-o", os.path.join(d, "t")],
                           capture_output=True)
        return ["-fopenmp"] if r.returncode == 0 else []


def build(out_path: str | None = None, mutation: int = 0, force: bool = False) -> str:
    """Compile kda_oracle.c into a shared library and return its path.

    ``mutation`` != 0 plants one numbered mistake (used only by the tests that
    show the pins catch such mistakes).
    """
    if out_path is None:
        name = "libkda_oracle.so" if mutation == 0 else f"libkda_oracle_m{mutation}.so"
        out_path = os.path.join(BUILD_DIR, name)
    if (not force and os.path.exists(out_path)
            and os.path.getmtime(out_path) >= os.path.getmtime(SRC)):
        return out_path
    os.makedirs(os.path.dirname(out_path), exist_ok=True)
    cc = os.environ.get("CC", "gcc")
    tmp = out_path + f".tmp{os.getpid()}"
    cmd = [cc, "-O2", "-fPIC", "-shared", "-std=c99", *(_openmp_flag(cc)),
           f"-DKDA_ORACLE_MUTATION={int(mutation)}", SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out_path)
    return out_path


if __name__ == "__main__":
    print(build(force=True))

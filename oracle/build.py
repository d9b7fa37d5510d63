"""Compile the CPU oracle (test infrastructure) into two shared libraries.

liboracle_f32.so computes in f32, the pages' precision; liboracle_f64.so is the same
source computed in f64, used by the tests to bound rounding error.  Both are built with
-ffp-contract=off so every product and sum is rounded on its own and the results are the
same on x86-64 and aarch64 hosts.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")


def lib_dir() -> str:
    # ORACLE_LIB_DIR lets the mutation tests load a deliberately broken copy of the oracle
    return os.environ.get("ORACLE_LIB_DIR") or HERE


def lib_path(precision: str) -> str:
    return os.path.join(lib_dir(), f"liboracle_{precision}.so")


def _stale(out: str) -> bool:
    if not os.path.exists(out):
        return True
    if os.path.dirname(out) != HERE:
        return False
    mt = os.path.getmtime(out)
    return any(os.path.getmtime(os.path.join(HERE, f)) > mt for f in ("oracle.c", "oracle.h"))


def build(force: bool = False, src: str = SRC, out_dir: str = HERE) -> None:
    procs = []
    for prec, real in (("f32", "float"), ("f64", "double")):
        out = os.path.join(out_dir, f"liboracle_{prec}.so")
        if not force and not _stale(out):
            continue
        # a temporary name of this process: several test workers may build at once
        tmp = f"{out}.{os.getpid()}.tmp"
        cmd = [
            "gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
            "-fno-fast-math", f"-DORC_REAL={real}", "-Wall", "-Wno-unknown-pragmas",
            "-I", HERE, src, "-o", tmp, "-lm",
        ]
        procs.append((subprocess.Popen(cmd), out, tmp))
    for p, out, tmp in procs:
        if p.wait() != 0:
            raise RuntimeError(f"oracle build failed for {out}")
        os.replace(tmp, out)  # atomic: a concurrent loader sees the old or the new library


if __name__ == "__main__":
    build(force="--force" in sys.argv)

"""Build the CPU oracle's shared library (test infrastructure only).

Compiles ``oracle_sgemm.c`` with gcc into ``liboracle_sgemm.so`` next to it.
Plain IEEE double arithmetic: -O2 without any fast-math option.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle_sgemm.c")
LIB = os.path.join(HERE, "liboracle_sgemm.so")
CFLAGS = ["-O2", "-fno-fast-math", "-fPIC", "-shared", "-pthread", "-std=c11", "-Wall", "-Wextra"]


def build(force: bool = False, src: str = SRC, out: str = LIB) -> str:
    """Compile ``src`` into ``out`` unless ``out`` is newer; return ``out``."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + ".tmp.%d" % os.getpid()
    cmd = [os.environ.get("CC", "gcc"), *CFLAGS, src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))

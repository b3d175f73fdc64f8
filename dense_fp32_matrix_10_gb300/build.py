"""Build the CUDA library in-tree: csrc/*.cu -> libsgemm_gb300.so (sm_103a only).

Each translation unit is compiled by nvcc in parallel (one -gencode for
compute capability 10.3a), objects go to ``_build/`` and are relinked only when
a source or header changed.  The CUDA runtime is linked statically, so the
library depends on nothing but the driver at run time.
"""
import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libsgemm_gb300.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = [*ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xptxas", "-v",
              "-Xcompiler", "-fPIC,-fvisibility=hidden", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; set NVCC or put the CUDA toolkit on PATH")
    return cand


def _headers():
    return glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


def _compile(nvcc, src, obj, log, defines=()):
    cmd = [nvcc, *NVCC_FLAGS, *("-D" + d for d in defines), "-c", src, "-o", obj + ".tmp"]
    proc = subprocess.run(cmd, capture_output=True, text=True)
    with open(log, "w") as f:
        f.write(" ".join(cmd) + "\n" + proc.stdout + proc.stderr)
    if proc.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{proc.stderr[-4000:]}")
    os.replace(obj + ".tmp", obj)
    return obj


def build(force: bool = False, jobs: int = None, verbose: bool = False, defines=(),
          out: str = None) -> str:
    """Compile and link if anything is out of date; return the library path.

    ``defines`` (e.g. ``["SG_SIMT_KC_UNROLL=4"]``) select compile-time kernel
    options; a build with defines needs its own ``out`` path and object dir.
    """
    nvcc = _nvcc()
    defines = list(defines)
    if defines and not out:
        raise ValueError("a build with defines needs its own output path")
    lib = out or LIB
    build_dir = BUILD if not out else os.path.join(BUILD, "variant_" + os.path.basename(out).replace(".so", ""))
    os.makedirs(build_dir, exist_ok=True)
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    newest_header = max((os.path.getmtime(h) for h in _headers()), default=0.0)
    todo, objs = [], []
    for src in sources:
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        stale = force or not os.path.exists(obj) or \
            os.path.getmtime(obj) < max(os.path.getmtime(src), newest_header)
        if stale:
            todo.append((src, obj, obj[:-2] + ".log"))
    if todo:
        jobs = jobs or min(len(todo), os.cpu_count() or 4)
        with cf.ThreadPoolExecutor(max_workers=jobs) as ex:
            list(ex.map(lambda t: _compile(nvcc, *t, defines=defines), todo))
    relink = force or bool(todo) or not os.path.exists(lib) or \
        os.path.getmtime(lib) < max(os.path.getmtime(o) for o in objs)
    if relink:
        tmp = lib + ".tmp.%d" % os.getpid()
        cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs, "-ldl", "-lpthread", "-lrt"]
        proc = subprocess.run(cmd, capture_output=True, text=True)
        if proc.returncode != 0:
            raise RuntimeError("link failed:\n" + proc.stderr[-4000:])
        os.replace(tmp, lib)
    if verbose:
        for _, obj, log in todo:
            sys.stdout.write(open(log).read())
    return lib


def ptxas_report() -> str:
    """The -Xptxas -v lines (registers, spills, shared memory) of the last build."""
    out = []
    for log in sorted(glob.glob(os.path.join(BUILD, "*.log"))):
        out.append(f"== {os.path.basename(log)[:-4]}")
        out += [ln for ln in open(log).read().splitlines()
                if "Compiling entry" in ln or "registers" in ln or "spill" in ln]
    return "\n".join(out)


if __name__ == "__main__":
    import argparse
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("-v", action="store_true")
    ap.add_argument("--define", "-D", action="append", default=[])
    ap.add_argument("--out", default=None)
    a = ap.parse_args()
    print(build(force=a.force, verbose=a.v, defines=a.define, out=a.out))

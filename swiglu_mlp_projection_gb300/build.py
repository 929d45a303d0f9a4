"""Build the CUDA library (sm_103a) in-tree: _build/libswiglu_gb300.so.

Each .cu file in csrc/ compiles to an object in parallel, then nvcc links
them into one shared library with the static CUDA runtime.  Only one
-gencode target is built (compute_103a -> sm_103a).  Host code is portable
(no host-architecture flags), so the same command builds on x86_64 and aarch64.
"""
import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
OUT_DIR = os.path.join(HERE, "_build")
LIB_NAME = "libswiglu_gb300.so"
LIB = os.path.join(OUT_DIR, LIB_NAME)

GENCODE = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden", "--expt-relaxed-constexpr",
              "-I", INCLUDE]


def nvcc():
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return cand


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (_sources() + glob.glob(os.path.join(CSRC, "*.cuh"))
            + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(INCLUDE, "*.h"))
            + [os.path.abspath(__file__)])


def up_to_date():
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force=False, verbose=False, extra_flags=()):
    """Compile and link the library if any source is newer than it."""
    if not force and up_to_date():
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    objs = []
    cmds = []
    for src in _sources():
        obj = os.path.join(OUT_DIR, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        cmds.append([nvcc(), *GENCODE, *NVCC_FLAGS, *extra_flags, "-c", src, "-o", obj])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if verbose or r.returncode != 0:
            sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed on %s" % cmd[-3])
        return r

    workers = max(1, min(len(cmds), os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(workers) as ex:
        list(ex.map(run, cmds))
    tmp = LIB + ".tmp.%d" % os.getpid()
    run([nvcc(), *GENCODE, "-shared", "-Xcompiler", "-fPIC", *objs, "-o", tmp,
         "-lcudart_static", "-ldl", "-lpthread", "-lrt"])
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

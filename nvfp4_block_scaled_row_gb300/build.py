"""Build the CUDA library libnvfp4_gb300.so for sm_103a, in-tree.

Each translation unit is compiled by nvcc in parallel, then linked into one shared library with
the CUDA runtime linked statically.  --fmad=false keeps nvcc from contracting multiplies and adds
into fused multiply-adds anywhere the kernels did not ask for one explicitly.
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJDIR = os.path.join(PKG, "_build")
LIBDIR = os.path.join(PKG, "lib")
LIBRARY = os.path.join(LIBDIR, "libnvfp4_gb300.so")
SOURCES = ["nvfp4_quant.cu", "nvfp4_aux.cu", "nvfp4_capi.cu", "nvfp4_noalloc.cu", "nvfp4_host.cu",
           "nvfp4_gemm.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "--fmad=false", "-Xcompiler", "-fPIC",
                     "-Xcompiler", "-Wall", "-I", INCLUDE, "-I", CSRC]


def nvcc():
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    path = os.path.join(home, "bin", "nvcc")
    return path if os.path.exists(path) else "nvcc"


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "nvfp4.h"))
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def compile_commands(extra=()):
    cmds = []
    for src in SOURCES:
        obj = os.path.join(OBJDIR, src.replace(".cu", ".o"))
        cmds.append([nvcc(), *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj])
    return cmds


def build(force=False, verbose=False, extra=()):
    """Compile the library if it is missing or older than any source; return its path."""
    if not force and os.path.exists(LIBRARY) and os.path.getmtime(LIBRARY) >= _deps():
        return LIBRARY
    os.makedirs(OBJDIR, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    cmds = compile_commands(extra)

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
        return r.stdout + r.stderr

    with ThreadPoolExecutor(len(cmds)) as ex:
        logs = list(ex.map(run, cmds))
    objs = [c[-1] for c in cmds]
    tmp = LIBRARY + ".tmp"
    link = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + " ".join(link) + "\n" + r.stdout + r.stderr)
    os.replace(tmp, LIBRARY)
    if verbose:
        print("".join(logs))
    return LIBRARY


if __name__ == "__main__":
    extra = ["-Xptxas", "-v"] if "-v" in sys.argv else []
    print(build(force=True, verbose=bool(extra), extra=extra))

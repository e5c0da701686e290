"""Build libmoe.so (the C-ABI library) in-tree with nvcc for sm_103a.

Each .cu file compiles in its own nvcc process (in parallel), then one nvcc
call links the shared library with the static CUDA runtime.  No torch, cmake
or setuptools involved.
"""
import concurrent.futures as cf
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_lib")
LIB = os.path.join(OUT_DIR, "libmoe.so")
SOURCES = ["abi.cu", "route.cu", "dispatch.cu", "combine.cu", "grouped_ffn.cu", "decode_fused.cu", "mxfp8.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc():
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def _flags(verbose_ptxas=False, extra=()):
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "include")]
    f += list(extra)
    if verbose_ptxas:
        f += ["-Xptxas", "-v"]
    return f


def _inputs():
    deps = [os.path.join(CSRC, s) for s in SOURCES]
    deps += [os.path.join(CSRC, h) for h in os.listdir(CSRC) if h.endswith((".cuh", ".h"))]
    deps.append(os.path.join(ROOT, "include", "moe.h"))
    return deps


def up_to_date():
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def build(force=False, verbose_ptxas=False, jobs=None, extra_flags=(), out_lib=None):
    """Compile and link libmoe.so; returns its path.  Raises on compiler errors.
    extra_flags / out_lib build a differently-configured copy elsewhere (tuning)."""
    lib = out_lib or LIB
    if not force and not verbose_ptxas and not extra_flags and out_lib is None and up_to_date():
        return LIB
    out_dir = os.path.dirname(lib)
    os.makedirs(out_dir, exist_ok=True)
    tag = os.path.splitext(os.path.basename(lib))[0]
    objs = [os.path.join(out_dir, tag + "_" + s.replace(".cu", ".o")) for s in SOURCES]

    def compile_one(src, obj):
        cmd = [nvcc()] + _flags(verbose_ptxas, extra_flags) + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, r

    with cf.ThreadPoolExecutor(max_workers=jobs or len(SOURCES)) as ex:
        results = list(ex.map(lambda so: compile_one(*so), zip(SOURCES, objs)))
    for src, r in results:
        if verbose_ptxas and r.stderr:
            sys.stderr.write(r.stderr)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    tmp = lib + ".tmp"
    cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs + ["-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))

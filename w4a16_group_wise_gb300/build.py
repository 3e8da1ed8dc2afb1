"""Build the CUDA library (sm_103a) in-tree: csrc/*.cu -> _libw4a16.so beside this file, and its
bounds-checked debug build (the same sources with W4A16_BOUNDS defined) -> _libw4a16_bounds.so.

Plain nvcc, no cmake: every translation unit of both libraries is compiled in parallel with one
-gencode, then each set is linked into a shared library with the CUDA runtime linked statically.
Each library exports exactly the extern "C" entry points of include/w4a16.h.
"""
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(ROOT, "_build")
LIB = os.path.join(HERE, "_libw4a16.so")
BOUNDS_LIB = os.path.join(HERE, "_libw4a16_bounds.so")
# library -> (object directory, extra defines)
VARIANTS = {LIB: (OUT_DIR, []), BOUNDS_LIB: (os.path.join(OUT_DIR, "bounds"), ["-DW4A16_BOUNDS"])}
SOURCES = ["capi.cu", "repack.cu", "dequant.cu", "gemv.cu", "gemm_tc.cu", "noalloc.cu", "embed.cu", "convert.cu",
           "selftest.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
         "--expt-relaxed-constexpr"]


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(ROOT, "include", "w4a16.h"))
    return files


def _stale(lib):
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(f) > t for f in _inputs() + [os.path.abspath(__file__)])


def build(force=False, verbose=False, ptxas_info=False):
    """Compile and link each library that is missing or older than an input.  Returns the path
    of the normal library."""
    todo = [lib for lib in VARIANTS if force or _stale(lib)]
    if not todo:
        return LIB
    nvcc = _nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []

    def compile_one(job):
        lib, src = job
        out_dir, defines = VARIANTS[lib]
        obj = os.path.join(out_dir, src.replace(".cu", ".o"))
        cmd = [nvcc] + ARCH + FLAGS + defines + extra + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed on %s%s:\n%s" % (src, " ".join([""] + defines), r.stdout))
        return obj, r.stdout

    for lib in todo:
        os.makedirs(VARIANTS[lib][0], exist_ok=True)
    jobs = [(lib, src) for lib in todo for src in SOURCES]
    with cf.ThreadPoolExecutor(max_workers=min(len(jobs), max(os.cpu_count() or 1, 4))) as ex:
        results = list(ex.map(compile_one, jobs))
    if verbose or ptxas_info:
        for (_, log) in results:
            if log.strip():
                print(log)
    for lib in todo:
        objs = [o for (l, _), (o, _) in zip(jobs, results) if l == lib]
        tmp = lib + ".tmp"
        cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs
        r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n%s" % r.stdout)
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))

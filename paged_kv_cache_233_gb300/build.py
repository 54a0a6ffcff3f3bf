"""Build ``libpagedkv.so`` in-tree with nvcc for sm_103a.

Each CUDA translation unit under ``csrc/`` is compiled in its own process
(they are independent), then linked into one shared library next to this
file. The CUDA runtime is linked statically, so loading the library needs no
driver until the first CUDA call.
"""
import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
LIBRARY = os.path.join(HERE, "libpagedkv.so")
BUILD_DIR = os.path.join(HERE, "_build")
SOURCES = ["api.cu", "append.cu", "swap.cu", "merge.cu", "prefill.cu", "prefill_tc.cu", "decode_f32.cu",
           "decode_f16.cu", "decode_bf16.cu", "decode_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr"]


def _nvcc():
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build libpagedkv")
    return exe


def _inputs():
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    deps.append(os.path.join(INCLUDE, "pagedkv.h"))
    return deps


def _stale():
    if not os.path.exists(LIBRARY):
        return True
    built = os.path.getmtime(LIBRARY)
    return any(os.path.getmtime(p) > built for p in _inputs())


def build(force=False, verbose=False, ptxas_info=False):
    """Compile and link; returns the library path. Skips work when up to date."""
    if not force and not _stale():
        return LIBRARY
    nvcc = _nvcc()
    os.makedirs(BUILD_DIR, exist_ok=True)
    extra = ["-Xptxas", "-v"] if ptxas_info else []

    def compile_one(src):
        obj = os.path.join(BUILD_DIR, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc, *ARCH, *FLAGS, *extra, "-I", INCLUDE, "-c", os.path.join(CSRC, src), "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        return src, obj, cmd, res

    objs = []
    failures = []
    workers = min(len(SOURCES), os.cpu_count() or 1)
    with concurrent.futures.ThreadPoolExecutor(max_workers=workers) as pool:
        for src, obj, cmd, res in pool.map(compile_one, SOURCES):
            if verbose or ptxas_info:
                sys.stderr.write(res.stderr)
            if res.returncode != 0:
                failures.append(f"{' '.join(cmd)}\n{res.stdout}{res.stderr}")
            objs.append(obj)
    if failures:
        raise RuntimeError("libpagedkv build failed:\n" + "\n".join(failures))
    tmp = LIBRARY + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("libpagedkv link failed:\n" + " ".join(cmd) + "\n" + res.stderr)
    os.replace(tmp, LIBRARY)
    return LIBRARY


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))

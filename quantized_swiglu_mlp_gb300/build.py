"""Build libqswiglu.so in-tree with nvcc for sm_103a (GB300).

Each translation unit compiles in parallel; the shared library lands in
``quantized_swiglu_mlp_gb300/lib/``.  No CMake, no torch extension machinery.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "lib")
LIB_PATH = os.path.join(OUT_DIR, "libqswiglu.so")
SOURCES = ["qsw_api.cu", "qsw_gemv.cu", "qsw_gemv_stream.cu", "qsw_prefill.cu", "qsw_elementwise.cu"]
HEADERS = ["qsw_device.cuh", "qsw_smallm.cuh", "qsw_internal.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags(verbose_ptxas: bool) -> list[str]:
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2,-fvisibility=hidden",
                "-I", os.path.join(ROOT, "include")]
    if verbose_ptxas:
        f += ["-Xptxas", "-v"]
    return f


# The sources each kernel is compiled from (for kernel_hash).
KERNEL_SOURCES = {
    "gemv_stream": ["qsw_gemv_stream.cu", "qsw_smallm.cuh", "qsw_device.cuh"],
    "gemv": ["qsw_gemv.cu", "qsw_smallm.cuh", "qsw_device.cuh"],
    "prefill": ["qsw_prefill.cu", "qsw_device.cuh"],
}


def _hash(names) -> str:
    import hashlib
    h = hashlib.sha256()
    for name in sorted(names):
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:12]


def source_hash() -> str:
    """Short hash of every source the library is built from."""
    return _hash(SOURCES + HEADERS)


def kernel_hash(kernel: str) -> str:
    """Short hash of the sources one kernel is compiled from (used to tell
    whether a stored profile still describes that kernel)."""
    return _hash(KERNEL_SOURCES[kernel])


DEBUG_LIB_PATH = os.path.join(OUT_DIR, "libqswiglu_debug.so")
# (library, object folder, extra nvcc flags): the regular build and the debug
# build (device-side address/copy checks and NaN-filled staging, QSW_DEBUG_BOUNDS)
VARIANTS = ((LIB_PATH, "obj", []), (DEBUG_LIB_PATH, "obj_debug", ["-DQSW_DEBUG_BOUNDS"]))


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, s) for s in SOURCES + HEADERS]
    deps.append(os.path.join(ROOT, "include", "qswiglu.h"))
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    """Compile both libraries (every translation unit of both at once) and
    return the regular one's path."""
    todo = [v for v in VARIANTS if force or _stale(v[0])]
    if not todo:
        return LIB_PATH
    cc = nvcc()
    flags = _flags(verbose_ptxas)
    for _, objdir, _ in todo:
        os.makedirs(os.path.join(OUT_DIR, objdir), exist_ok=True)

    def compile_one(job) -> str:
        src, objdir, extra = job
        obj = os.path.join(OUT_DIR, objdir, src.replace(".cu", ".o"))
        cmd = [cc, *flags, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose_ptxas:
            sys.stderr.write(r.stderr)
        return obj

    jobs = [(src, objdir, extra) for _, objdir, extra in todo for src in SOURCES]
    with ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        objs = list(ex.map(compile_one, jobs))
    for n, (lib, _, _) in enumerate(todo):
        tmp = lib + f".tmp{os.getpid()}"
        mine = objs[n * len(SOURCES):(n + 1) * len(SOURCES)]
        r = subprocess.run([cc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *mine], capture_output=True,
                           text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))

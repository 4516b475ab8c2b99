"""In-tree build of ``libsplitzip.so`` (CUDA kernels + C ABI) for sm_103a.

Each ``.cu`` file under ``csrc/`` is compiled in parallel with nvcc, then the
objects are linked into a shared library next to this file.  A stamp file with
a hash of the sources and flags makes the build a no-op when nothing changed.
ptxas resource usage (registers, spills, shared memory) is kept in
``_build/ptxas.log``.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import hashlib
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIBRARY = os.path.join(PKG, "libsplitzip.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + [
    "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
    "--expt-relaxed-constexpr", "-Xptxas", "-v", f"-I{INCLUDE}", f"-I{CSRC}",
]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the SplitZip CUDA library cannot be built")
    return exe


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _digest() -> str:
    h = hashlib.sha256()
    for path in sorted(_sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh"))
                       + glob.glob(os.path.join(INCLUDE, "*.h"))):
        h.update(os.path.basename(path).encode())
        with open(path, "rb") as f:
            h.update(f.read())
    h.update(" ".join(NVCC_FLAGS).encode())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link the library if the sources changed; return its path."""
    stamp = LIBRARY + ".stamp"
    want = _digest()
    if not force and os.path.exists(LIBRARY) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == want:
                return LIBRARY
    os.makedirs(BUILD_DIR, exist_ok=True)
    exe = nvcc()

    def compile_one(src):
        obj = os.path.join(BUILD_DIR, os.path.basename(src)[:-3] + ".o")
        res = subprocess.run([exe, *NVCC_FLAGS, "-c", src, "-o", obj], capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{res.stdout}\n{res.stderr}")
        return obj, res.stderr

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as pool:
        results = list(pool.map(compile_one, _sources()))
    with open(os.path.join(BUILD_DIR, "ptxas.log"), "w") as f:
        for _, log in results:
            f.write(log)
    if verbose:
        for _, log in results:
            print(log)
    part = LIBRARY + f".{os.getpid()}.part"
    res = subprocess.run([exe, *ARCH, "-shared", "-o", part, *[o for o, _ in results]], capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(part, LIBRARY)
    with open(stamp, "w") as f:
        f.write(want)
    return LIBRARY


if __name__ == "__main__":
    print(build(force=True, verbose=True))

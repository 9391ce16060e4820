"""Build the pre-attention CUDA library in-tree: libpre_attn.so next to this file.

Each translation unit under csrc/ is compiled for sm_103a only, in parallel,
then linked (CUDA runtime static) into a shared library exporting the C-ABI
of include/pre_attn.h.
"""

from __future__ import annotations

import hashlib
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
LIB = os.path.join(HERE, "libpre_attn.so")
STAMP = LIB + ".sha256"
SOURCES = ["pa_api.cu", "pa_prologue.cu", "pa_gemv.cu", "pa_gemm.cu", "pa_gemm2.cu", "pa_noalloc.cu",
           "pa_signal.cu", "pa_index.cu", "pa_drafter.cu", "pa_gemv_persist.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
              "-Xptxas", "-v", "--expt-relaxed-constexpr"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def source_hash() -> str:
    """sha256 of everything the library is built from: the sources and headers
    under csrc/, the public header, this file (flags, source list) and nvcc's
    version line."""
    h = hashlib.sha256()
    deps = sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC)) + [os.path.join(ROOT, "include", "pre_attn.h"),
                                                                     os.path.abspath(__file__)]
    for d in deps:
        h.update(os.path.basename(d).encode())
        with open(d, "rb") as f:
            h.update(f.read())
    try:
        h.update(subprocess.run([nvcc(), "--version"], capture_output=True, text=True).stdout.encode())
    except (RuntimeError, OSError):
        pass
    return h.hexdigest()


def _stale() -> bool:
    """The library is rebuilt unless it exists and its stamp records the hash
    of the current sources (file times are not trusted: a copied tree or an
    archive can make an old binary look newer than its sources)."""
    if not (os.path.exists(LIB) and os.path.exists(STAMP)):
        return True
    with open(STAMP) as f:
        return f.read().strip() != source_hash()


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not _stale():
        return LIB
    digest = source_hash()
    out_dir = os.path.join(ROOT, "_build")
    os.makedirs(out_dir, exist_ok=True)
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(out_dir, src.replace(".cu", ".o"))
        cmd = [cc, *ARCH, *NVCC_FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with ThreadPoolExecutor(len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose:
        for (_, log), src in zip(results, SOURCES):
            print(f"== {src}\n{log}")
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *[o for o, _ in results],
           "-Xlinker", "--version-script=" + os.path.join(CSRC, "exports.map")]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(STAMP, "w") as f:
        f.write(digest + "\n")
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force=True, verbose="-v" in sys.argv))

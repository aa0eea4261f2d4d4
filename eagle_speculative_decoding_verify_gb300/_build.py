"""Compile the CUDA sources into the in-tree C-ABI library ``libeagle.so``.

nvcc, sm_103a only; translation units are compiled in parallel and linked
with the CUDA runtime statically.  The library embeds a hash of its sources
and build flags (``eagle_build_id()``); a build is reused only when that hash
equals the hash of the sources on disk, and the binding refuses a library
whose hash differs.
"""

import glob
import hashlib
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libeagle.so")
OBJ = os.path.join(ROOT, "_build", "obj")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def _nvcc():
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(
        os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(INCLUDE, "*.h"))


def source_hash():
    """sha256 (16 hex digits) of every source and header, by relative path and
    content, and of the compiler flags."""
    h = hashlib.sha256()
    for p in sorted(_deps()):
        h.update(os.path.relpath(p, ROOT).encode())
        with open(p, "rb") as f:
            h.update(f.read())
    h.update(" ".join(ARCH + FLAGS[:-4]).encode())
    return h.hexdigest()[:16]


BUILD_ID_FILE = LIB + ".buildid"


def up_to_date():
    """True when libeagle.so was built from the sources on disk (its recorded
    build id equals their hash)."""
    if not os.path.exists(LIB) or not os.path.exists(BUILD_ID_FILE):
        return False
    with open(BUILD_ID_FILE) as f:
        return f.read().strip() == source_hash()


def build(force=False, verbose=False, extra_flags=()):
    """Build libeagle.so; returns its path.  Raises RuntimeError on failure."""
    if not force and up_to_date():
        return LIB
    os.makedirs(OBJ, exist_ok=True)
    nvcc = _nvcc()
    build_id = source_hash()

    def compile_one(src):
        obj = os.path.join(OBJ, os.path.basename(src) + ".o")
        cmd = [nvcc, *ARCH, *FLAGS, *extra_flags, f"-DEAGLE_BUILD_ID=\"{build_id}\"", "-c", src,
               "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stderr[-4000:]}")
        if verbose and r.stderr.strip():
            print(r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, sources()))
    tmp = LIB + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stderr[-4000:])
    os.replace(tmp, LIB)
    with open(BUILD_ID_FILE, "w") as f:
        f.write(build_id + "\n")
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True))

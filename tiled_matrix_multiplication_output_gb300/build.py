"""Build the CUDA library `_build/libtiled_gemm.so` for sm_103a with nvcc.

Each translation unit compiles in its own nvcc process (in parallel), then
they are linked into one shared library with the CUDA runtime linked
statically, so the library loads the same way on any host that has the
NVIDIA driver.  A sidecar stamp beside the library holds a SHA-256 over the
sources, the headers, this file and the nvcc command line; the build is
skipped only when the stamp matches (file times are not trusted: a copied
tree keeps or resets them arbitrarily).
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import platform
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB_NAME = "libtiled_gemm.so"
LIB_PATH = os.path.join(OUT_DIR, LIB_NAME)
STAMP_PATH = LIB_PATH + ".sha256"
SOURCES = ("api.cu", "tc_gemm.cu", "tc_gemm_nn.cu", "tc_gemm_tn.cu", "tc_gemm_nt.cu",
           "tc_gemm_tt.cu", "tc_gemm_splitk.cu", "tc_small.cu", "simt_gemm.cu", "tile16.cu",
           "model.cu")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
              "-I" + INCLUDE, "-I" + CSRC]


def nvcc_path() -> str | None:
    cand = shutil.which("nvcc")
    if cand:
        return cand
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    p = os.path.join(home, "bin", "nvcc")
    return p if os.path.exists(p) else None


def _inputs() -> list[str]:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    files.append(os.path.abspath(__file__))
    return sorted(f for f in files if os.path.isfile(f))


def source_stamp() -> str:
    """SHA-256 over every source and header (name and bytes), this build
    script, the compiler flags and the host architecture (a library built on
    another kind of host never counts as current)."""
    h = hashlib.sha256()
    for f in _inputs():
        h.update(os.path.relpath(f, ROOT).encode())
        h.update(b"\0")
        with open(f, "rb") as fh:
            h.update(fh.read())
        h.update(b"\0")
    h.update(" ".join(ARCH + NVCC_FLAGS).replace(ROOT, "<root>").encode())
    h.update(platform.machine().encode())
    return h.hexdigest()


def built_stamp() -> str | None:
    """The stamp recorded with the library on disk, or None."""
    if not (os.path.exists(LIB_PATH) and os.path.exists(STAMP_PATH)):
        return None
    with open(STAMP_PATH) as f:
        return f.read().strip() or None


def up_to_date() -> bool:
    return built_stamp() == source_stamp()


# What the last build() call in this process did: "built" or "reused".
last_action = None


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link the library unless the library on disk was built
    from exactly these sources and flags; returns its path."""
    global last_action
    stamp = source_stamp()
    if not force and built_stamp() == stamp:
        last_action = "reused"
        return LIB_PATH
    nvcc = nvcc_path()
    if nvcc is None:
        raise RuntimeError("nvcc not found: cannot build the CUDA library")
    os.makedirs(OUT_DIR, exist_ok=True)
    tag = str(os.getpid())

    def compile_one(src: str) -> str:
        obj = os.path.join(OUT_DIR, src.replace(".cu", f".{tag}.o"))
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{res.stdout}\n{res.stderr}")
        if verbose and (res.stdout or res.stderr):
            print(res.stdout, res.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB_PATH + f".{tag}.tmp"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    res = subprocess.run(cmd, capture_output=True, text=True)
    for o in objs:
        os.remove(o)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, LIB_PATH)
    with open(STAMP_PATH + f".{tag}", "w") as f:
        f.write(stamp + "\n")
    os.replace(STAMP_PATH + f".{tag}", STAMP_PATH)
    last_action = "built"
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True, verbose=True))

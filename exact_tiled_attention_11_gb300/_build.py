"""Build the CUDA library (libattn.so) in-tree for sm_103a with nvcc.

Each .cu file is compiled on its own (in parallel) and the objects are linked
into ``exact_tiled_attention_11_gb300/libattn.so``.  The CUDA runtime is
linked statically; the driver's tensor-map encoder is looked up at run time,
so the library needs no ``-lcuda``.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG_DIR, "_build")
LIB_PATH = os.path.join(PKG_DIR, "libattn.so")

SOURCES = ("api.cu", "decode.cu", "prefill_f32.cu", "prefill_bf16.cu", "decode_noalloc.cu", "prefill_fp8.cu",
           "fp8_quantize.cu", "selftest.cu", "cascade.cu")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
                     f"-I{INCLUDE}", f"-I{CSRC}"]


def nvcc_path() -> str:
    cand = [os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"]
    for c in cand:
        p = os.path.join(c, "bin", "nvcc") if c else ""
        if p and os.path.exists(p):
            return p
    p = shutil.which("nvcc")
    if p is None:
        raise RuntimeError("nvcc not found: set CUDA_HOME or put nvcc on PATH")
    return p


def _inputs() -> list[str]:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cuh", ".h"))]
    files.append(os.path.join(INCLUDE, "attn.h"))
    files.append(os.path.abspath(__file__))
    return files


def _is_native(path: str) -> bool:
    """True when the shared object at ``path`` was built for this machine's CPU."""
    import platform
    try:
        with open(path, "rb") as f:
            head = f.read(20)
    except OSError:
        return False
    if head[:4] != b"\x7fELF":
        return False
    machine = int.from_bytes(head[18:20], "little")
    want = {"x86_64": 62, "aarch64": 183, "arm64": 183}.get(platform.machine())
    return want is None or machine == want


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH) or not _is_native(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the library if any source is newer than it; return its path."""
    if not force and up_to_date():
        return LIB_PATH
    nvcc = nvcc_path()
    os.makedirs(BUILD_DIR, exist_ok=True)

    def compile_one(src: str) -> str:
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        cmd = [nvcc, *NVCC_FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB_PATH + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-Xcompiler", "-fPIC", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

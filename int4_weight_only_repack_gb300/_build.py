"""Build libw4a16.so in-tree with nvcc for sm_103a (no cmake, no torch extension).

Each .cu file compiles in its own nvcc process (in parallel), then one nvcc
link step makes the shared library next to this file. The CUDA runtime is
linked statically, so the library needs only the driver at run time.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG_DIR, "csrc")
ROOT = os.path.dirname(PKG_DIR)
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_NAME = "libw4a16.so"
LIB_PATH = os.path.join(PKG_DIR, LIB_NAME)

SOURCES = ("w4a16_api.cu", "repack_kernels.cu", "decode_kernel.cu", "decode_stream_kernel.cu",
           "prefill_kernel.cu", "w4a8_kernel.cu")

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
CXX_FLAGS = [
    "-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
    "-I", os.path.join(ROOT, "include"),
]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _run(cmd):
    proc = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    return proc.returncode, proc.stdout


def build(verbose: bool = False, ptxas_info: bool = False, csrc: str = CSRC,
          out: str = LIB_PATH, build_dir: str = BUILD_DIR, defines=()) -> str:
    """Compile every CUDA source and link libw4a16.so; returns the library path."""
    os.makedirs(build_dir, exist_ok=True)
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    extra += [f"-D{d}" for d in defines]
    jobs = []
    for src in SOURCES:
        obj = os.path.join(build_dir, src.replace(".cu", ".o"))
        jobs.append((src, obj, [cc, *ARCH_FLAGS, *CXX_FLAGS, *extra, "-c",
                                os.path.join(csrc, src), "-o", obj]))
    with ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        results = list(ex.map(lambda j: (j[0], *_run(j[2])), jobs))
    failed = False
    for src, rc, log in results:
        if verbose or rc != 0 or ptxas_info:
            sys.stdout.write(f"--- {src} (rc={rc})\n{log}")
        failed |= rc != 0
    if failed:
        raise RuntimeError("nvcc compilation failed")
    tmp = out + ".tmp"
    rc, log = _run([cc, *ARCH_FLAGS, "-shared", "-o", tmp, *[j[1] for j in jobs],
                    "-Xcompiler", "-fvisibility=hidden"])
    if rc != 0:
        sys.stdout.write(log)
        raise RuntimeError("nvcc link failed")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    build(verbose=True, ptxas_info="--ptxas" in sys.argv)

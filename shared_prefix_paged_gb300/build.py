"""Build libcsp_gb300.so in-tree with nvcc for sm_103a.

Each .cu file compiles in its own nvcc process (in parallel), then one link step
makes the shared library.  Output: shared_prefix_paged_gb300/_build/libcsp_gb300.so.
Run as ``python -m shared_prefix_paged_gb300.build``.
"""

from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
INCLUDE = os.path.join(ROOT, "include")
LIB_NAME = "libcsp_gb300.so"
SOURCES = ["api.cu", "prefix_attn.cu", "paged_attn.cu", "paged_tc.cu", "decode_cascade.cu",
           "combine.cu", "noalloc.cu", "plan_device.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def lib_path() -> str:
    return os.path.join(BUILD, LIB_NAME)


def _nvcc() -> str:
    cand = shutil.which("nvcc")
    if cand:
        return cand
    for base in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if base and os.path.exists(os.path.join(base, "bin", "nvcc")):
            return os.path.join(base, "bin", "nvcc")
    raise RuntimeError("nvcc not found: the CUDA library cannot be built")


def _flags() -> list[str]:
    return ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
                   "-Xcompiler", "-fvisibility=hidden", f"-I{INCLUDE}", f"-I{CSRC}",
                   "--expt-relaxed-constexpr", "-diag-suppress", "177"]


def _inputs() -> list[str]:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "csp.h"))
    return files


def is_stale() -> bool:
    out = lib_path()
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(f) > t for f in _inputs())


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile (if stale) and return the library path."""
    out = lib_path()
    if not force and not is_stale():
        return out
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    flags = _flags()

    def compile_one(src: str) -> str:
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        cmd = [nvcc, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{res.stderr}")
        if verbose and res.stderr:
            sys.stderr.write(res.stderr)
        return obj

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = f"{out}.{os.getpid()}.tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-Xcompiler", "-fPIC"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stderr}")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))

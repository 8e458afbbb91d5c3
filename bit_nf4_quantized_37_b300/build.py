"""Build the sm_103a C-ABI library libqlora_nf4.so in this directory with nvcc.

    python -m bit_nf4_quantized_37_b300.build [--force] [--checked]

Cross-compiles without a GPU.  No --use_fast_math: the quantize/dequantize arithmetic uses
explicitly rounded intrinsics and must stay IEEE.

--checked builds the bounds-checked variant libqlora_nf4_checked.so (QLORA_CHECK_BOUNDS=1:
the kernels test their own shared-window offsets, split-reduction partial indices and
arrival tickets, record a failed check in the device error word and skip the access).  The
Python binding loads it when QLORA_NF4_LIB names it.
"""
from __future__ import annotations

import hashlib
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
LIB = os.path.join(HERE, "libqlora_nf4.so")
CHECKED_LIB = os.path.join(HERE, "libqlora_nf4_checked.so")
SOURCES = ["api.cu", "linear.cu", "nf4_codec.cu", "umma_gemm.cu", "lora_side.cu", "skinny.cu",
           "tensormap.cu", "profile.cu",
           "noalloc.cu", "merge.cu", "multi.cu", "selftest.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "--expt-relaxed-constexpr", "-Xptxas", "-v"]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found")
    return path


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cuh", ".h"))]
    files.append(os.path.join(INCLUDE, "qlora_nf4.h"))
    files.append(os.path.abspath(__file__))
    return files


def _paths(checked: bool):
    lib = CHECKED_LIB if checked else LIB
    return lib, lib + ".stamp", os.path.join(HERE, "_build_checked" if checked else "_build")


def _flags(checked: bool):
    return FLAGS + (["-DQLORA_CHECK_BOUNDS=1"] if checked else [])


def _digest(checked: bool = False) -> str:
    h = hashlib.sha256(" ".join(ARCH + _flags(checked)).encode())
    for f in sorted(_deps()):
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def up_to_date(checked: bool = False) -> bool:
    """The library exists and was built from exactly the current sources (content hash, so
    copies of the tree with fresh timestamps do not rebuild)."""
    lib, stamp, _ = _paths(checked)
    if not (os.path.exists(lib) and os.path.exists(stamp)):
        return False
    with open(stamp) as f:
        return f.read().strip() == _digest(checked)


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    lib, stamp, objdir = _paths(checked)
    if not force and up_to_date(checked):
        return lib
    os.makedirs(objdir, exist_ok=True)
    flags = _flags(checked)

    def compile_one(src):
        obj = os.path.join(objdir, src.replace(".cu", ".o"))
        cmd = [nvcc(), *ARCH, *flags, "-I", INCLUDE, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, obj, r.returncode, f"$ {' '.join(cmd)}\n{r.stdout}{r.stderr}"

    # the translation units are independent: compile them side by side
    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(max(1, min(len(SOURCES), os.cpu_count() or 1))) as ex:
        results = list(ex.map(compile_one, SOURCES))
    objs = []
    logs = []
    for src, obj, rc, log in results:
        logs.append(log)
        if rc != 0:
            sys.stderr.write(log)
            raise RuntimeError(f"nvcc failed on {src}")
        objs.append(obj)
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-Xcompiler", "-fPIC", *objs, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    logs.append(f"$ {' '.join(cmd)}\n{r.stdout}{r.stderr}")
    if r.returncode != 0:
        sys.stderr.write(logs[-1])
        raise RuntimeError("link failed")
    os.replace(tmp, lib)
    with open(stamp, "w") as f:
        f.write(_digest(checked))
    with open(os.path.join(objdir, "build.log"), "w") as f:
        f.write("\n".join(logs))
    if verbose:
        print("\n".join(logs))
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                checked="--checked" in sys.argv))

"""Build step: compiles the CUDA sources into the in-tree shared library
``rl_fine_tuning_pass_gb300/libgrpo_rowpass.so`` for sm_103a (GB300).

Each translation unit is compiled in parallel with one ``-gencode`` (a minute or less),
then linked with the static CUDA runtime; the tensor-map encoder is looked up through the
runtime at first use, so no other library is linked.  Nothing is installed outside this
directory.

    python -m rl_fine_tuning_pass_gb300.build          # build if sources changed
    python -m rl_fine_tuning_pass_gb300.build --force  # rebuild
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_NAME = "libgrpo_rowpass.so"
LIB_PATH = os.path.join(PKG, LIB_NAME)

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "--expt-relaxed-constexpr",
              "-I", INCLUDE, "-I", CSRC]
SOURCES = ["capi.cu", "rowpass_fwd_bf16.cu", "rowpass_fwd_f32.cu", "rowpass_bwd_bf16.cu", "rowpass_bwd_f32.cu",
           "rowpass_fused_bf16.cu", "rowpass_fused_f32.cu", "rowpass_seq.cu",
           "rowpass_vocab.cu", "rowpass_linear.cu"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the row-pass library")


def _deps():
    return [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "grpo_rowpass.h")]


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(d) <= t for d in _deps())


def _compile(src: str, extra) -> str:
    obj = os.path.join(BUILD_DIR, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{' '.join(cmd)}\n{res.stdout}\n{res.stderr}")
    if res.stderr.strip() and os.environ.get("GRPO_BUILD_VERBOSE"):
        sys.stderr.write(res.stderr)
    return obj


def build(force: bool = False, ptxas_verbose: bool = False) -> str:
    """Compile (if needed) and return the path of the shared library."""
    if not force and up_to_date():
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    extra = ["-Xptxas", "-v"] if ptxas_verbose else []
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra), SOURCES))
    tmp = LIB_PATH + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, ptxas_verbose="--ptxas-v" in sys.argv))

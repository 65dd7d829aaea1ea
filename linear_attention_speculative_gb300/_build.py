"""Build the CUDA library (sm_103a) in-tree with nvcc.

Eleven translation units are compiled in parallel (the C ABI, one unit per
verify kernel family and activation type -- one item per CTA, pipelined,
split -- the q/k conv_state roll kernel, the commit kernel, the
allocation-free entry point, and the bounded-wait self-test) and linked into
``_lib/libkda_gb300.so``.  The shared CUDA runtime is used so the library and
PyTorch share one runtime instance.
"""

from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIB_DIR = os.path.join(HERE, "_lib")
OBJ_DIR = os.path.join(LIB_DIR, "obj")
LIB_PATH = os.path.join(LIB_DIR, "libkda_gb300.so")
SOURCES = ("kda_api.cu", "kda_inst_tile_bf16.cu", "kda_inst_tile_f32.cu", "kda_inst_tile_cl_bf16.cu",
           "kda_inst_tile_cl_f32.cu", "kda_inst_tile_dec_bf16.cu", "kda_inst_tile_dec_f32.cu",
           "kda_inst_pipe_bf16.cu",
           "kda_inst_pipe_f32.cu", "kda_inst_split_bf16.cu", "kda_inst_split_f32.cu", "kda_roll.cu",
           "kda_commit.cu", "kda_noalloc.cu", "kda_selftest.cu")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def _cuda_lib_dir(nv: str) -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nv))), "lib64")


def _deps():
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    deps.append(os.path.join(os.path.dirname(HERE), "include", "kda_verify.h"))
    deps.append(os.path.abspath(__file__))
    return deps


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    if not force and up_to_date():
        return LIB_PATH
    nv = nvcc()
    os.makedirs(OBJ_DIR, exist_ok=True)
    common = [nv, "-std=c++17", "-O3", "-lineinfo", *ARCH, "-Xcompiler", "-fPIC",
              "--expt-relaxed-constexpr", "-Xptxas", "-warn-spills", *extra_flags]

    def compile_one(src: str) -> str:
        obj = os.path.join(OBJ_DIR, src.replace(".cu", ".o"))
        cmd = common + ["-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose or "spill" in (r.stderr or "").lower():
            sys.stderr.write(r.stderr)
        return obj

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    link = [nv, "-shared", *ARCH, "--cudart", "shared", "-o", tmp, *objs,
            "-Xlinker", f"-rpath,{_cuda_lib_dir(nv)}"]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

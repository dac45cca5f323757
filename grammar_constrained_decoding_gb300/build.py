"""Builds libcg.so in-tree: host C++ with g++, device code with nvcc for sm_103a.

    python -m grammar_constrained_decoding_gb300.build [--force]

Translation units compile in parallel; the library links against the static
CUDA runtime.  The output lives in grammar_constrained_decoding_gb300/_build/.
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
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(OUT_DIR, "libcg.so")

CXX_SOURCES = ["compiler/gbnf.cpp", "compiler/schema.cpp", "compiler/structtag.cpp", "compiler/automaton.cpp",
               "compiler/pda.cpp", "grammar.cpp", "evaluator.cpp"]
CU_SOURCES = ["ctx.cu", "kernel_mask.cu", "kernel_sample.cu", "kernel_seg.cu", "kernel_accept.cu", "pda.cu"]
HEADERS = ["compiler/ir.h", "compiler/json.h", "cg_internal.h", "device.cuh", "row_ops.cuh", "pda.cuh", "bf16_ops.cuh"]
GENCODE = "arch=compute_103a,code=sm_103a"


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _run(cmd: list[str]) -> None:
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"command failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    nvcc = _nvcc()
    include = os.path.join(ROOT, "include")
    headers = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(include, "cg.h")]
    jobs = []
    objs = []
    for src in CXX_SOURCES:
        path = os.path.join(CSRC, src)
        obj = os.path.join(OUT_DIR, src.replace("/", "_") + ".o")
        objs.append(obj)
        if force or _stale(obj, [path] + headers):
            jobs.append(["g++", "-O2", "-std=c++17", "-fPIC", "-Wall", "-Wno-unused-function",
                         f"-I{include}", "-c", path, "-o", obj])
    for src in CU_SOURCES:
        path = os.path.join(CSRC, src)
        obj = os.path.join(OUT_DIR, src + ".o")
        objs.append(obj)
        if force or _stale(obj, [path] + headers):
            jobs.append([nvcc, "-gencode", GENCODE, "-O3", "-lineinfo", "-std=c++17",
                         "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr", f"-I{include}",
                         "-c", path, "-o", obj])
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        for f in [ex.submit(_run, j) for j in jobs]:
            f.result()
    if force or jobs or _stale(LIB, objs):
        _run([nvcc, "-shared", "-gencode", GENCODE, "-o", LIB] + objs + ["-lcudart_static", "-lrt", "-ldl", "-lpthread"])
    if verbose:
        print(LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)

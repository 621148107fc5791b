"""Builds libgbattn.so in-tree with nvcc for sm_103a (no CMake, no torch
extension machinery): each .cu compiles in parallel, then one link step.

    python -m exact_tiled_attention_gb300._build [--force] [--verbose]

Build option (environment): GBATTN_EX2_EMU_EVERY=E evaluates every E-th pair
of softmax exponentials with the FMA-pipe polynomial instead of the MUFU unit
(default 0 = none; the library is rebuilt when the setting changes).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libgbattn.so")

SOURCES = ["gbattn_api.cu", "prefill_fwd.cu", "prefill_pair.cu", "prefill_fp8.cu", "decode_splitkv.cu",
           "decode_noalloc.cu", "backward.cu", "backward_atomic.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA library cannot be built")


def _deps() -> list[str]:
    out = [os.path.join(INCLUDE, "gbattn.h")]
    for f in os.listdir(CSRC):
        out.append(os.path.join(CSRC, f))
    return out


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _options() -> list[str]:
    emu = int(os.environ.get("GBATTN_EX2_EMU_EVERY", "0") or 0)
    return [f"-DGBATTN_EX2_EMU_EVERY={emu}"]


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    deps = _deps()
    stamp = os.path.join(BUILD, "options.txt")
    opts = _options()
    old = open(stamp).read() if os.path.exists(stamp) else ""
    if not force and not _stale(LIB, deps) and old == " ".join(opts):
        return LIB
    cc = nvcc()
    extra = (["-Xptxas", "-v"] if ptxas_verbose else []) + opts

    def compile_one(src: str):
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        cmd = [cc, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, obj, r

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    for src, _, r in results:
        if verbose or ptxas_verbose or r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}")
    tmp = LIB + f".tmp{os.getpid()}"
    link = [cc, *ARCH, "-shared", "-o", tmp, *[obj for _, obj, _ in results]]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError("nvcc link failed")
    os.replace(tmp, LIB)
    with open(stamp, "w") as f:
        f.write(" ".join(opts))
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="--verbose" in sys.argv,
          ptxas_verbose="--ptxas" in sys.argv)
    print(LIB)

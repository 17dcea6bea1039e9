"""Build libpagedattn.so in-tree with nvcc for sm_103a (GB300).

Translation units compile in parallel; the CUDA runtime is linked statically
so the library loads next to any PyTorch build.  Output:
``paged_kv_cache_kvcache_gb300/_build/libpagedattn.so``.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libpagedattn.so")

SOURCES = ["api.cpp", "pack.cpp", "store_kv.cu", "decode.cu", "decode_int8.cu", "prefill.cu", "copy_blocks.cu", "tmap.cpp",
           "selftest.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpagedattn")


def _inputs():
    files = [os.path.join(CSRC, s) for s in SOURCES]
    files += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    files.append(os.path.join(INCLUDE, "pagedattn.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    common = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O3", "-I", INCLUDE, "-I", CSRC] + ARCH
    procs = []
    objs = []
    for s in SOURCES:
        src = os.path.join(CSRC, s)
        obj = os.path.join(BUILD, s + f".{os.getpid()}.o")
        objs.append(obj)
        cmd = [nvcc] + common + ["-c", src, "-o", obj]
        if s.endswith(".cu"):
            cmd += ["--expt-relaxed-constexpr"]
            if ptxas_verbose:
                cmd += ["-Xptxas", "-v"]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((s, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    logs = {}
    for s, p in procs:
        out, _ = p.communicate()
        logs[s] = out.decode(errors="replace")
        if p.returncode != 0:
            failed.append(s)
    if verbose or ptxas_verbose:
        for s in SOURCES:
            if logs[s].strip():
                print(f"--- {s}\n{logs[s]}", file=sys.stderr)
    if failed:
        for o in objs:
            if os.path.exists(o):
                os.remove(o)
        raise RuntimeError("nvcc failed for " + ", ".join(failed) + ":\n" + "\n".join(logs[s] for s in failed))
    tmp = LIB + f".{os.getpid()}.tmp"
    link = [nvcc, "-shared", "-cudart", "static", "-o", tmp] + objs + ARCH
    r = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
    for o in objs:
        os.remove(o)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout.decode(errors="replace"))
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv, ptxas_verbose="--ptxas" in sys.argv)
    print(LIB)

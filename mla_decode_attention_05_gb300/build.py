"""Compile the CUDA library in-tree for sm_103a (GB300).

    python -m mla_decode_attention_05_gb300.build [--force] [--verbose-ptxas]

Each translation unit of csrc/ is compiled by its own nvcc process (in
parallel), then linked into _lib/libmla_decode.so with the CUDA runtime
linked statically, so the library loads on a machine without a GPU driver.
"""
from __future__ import annotations

import argparse
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_DIR = os.path.join(HERE, "_lib")
OBJ_DIR = os.path.join(LIB_DIR, "obj")
SO = os.path.join(LIB_DIR, "libmla_decode.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found")
    return cand


def _inputs():
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    deps = srcs + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))
    return srcs, deps


def up_to_date() -> bool:
    if not os.path.exists(SO):
        return False
    _, deps = _inputs()
    t = os.path.getmtime(SO)
    return all(os.path.getmtime(d) <= t for d in deps) and os.path.getmtime(__file__) <= t


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    if not force and up_to_date():
        return SO
    os.makedirs(OBJ_DIR, exist_ok=True)
    nvcc = _nvcc()
    srcs, _ = _inputs()
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                    "-I", INCLUDE, "-I", CSRC, "--expt-relaxed-constexpr"]
    if verbose_ptxas:
        flags += ["-Xptxas", "-v"]
    procs = []
    objs = []
    for s in srcs:
        o = os.path.join(OBJ_DIR, os.path.basename(s) + ".o")
        objs.append(o)
        procs.append((s, subprocess.Popen([nvcc, "-c", s, "-o", o] + flags,
                                          stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for s, pr in procs:
        out, _ = pr.communicate()
        text = out.decode(errors="replace")
        if pr.returncode != 0:
            failed.append((s, text))
        elif text.strip() and (verbose_ptxas or "warning" in text):
            sys.stderr.write(text)
    if failed:
        msg = "\n".join(f"--- {s}\n{t}" for s, t in failed)
        raise RuntimeError("nvcc failed:\n" + msg)
    tmp = SO + f".tmp{os.getpid()}"
    subprocess.check_call([nvcc, "-shared", "-o", tmp] + objs + ARCH + ["-cudart", "static", "-ldl"])
    os.replace(tmp, SO)
    return SO


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose-ptxas", action="store_true")
    a = ap.parse_args()
    print(build(force=a.force, verbose_ptxas=a.verbose_ptxas))

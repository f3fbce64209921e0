"""The C ABI from a C program: tests/c_abi/decode_main.c includes only
include/mla_decode.h and the CUDA runtime header, links the built library,
and runs the schedule and the decode with no Python or PyTorch in its
process.

On the CPU: the program (and so the header) compiles as strict C99 and links.
On the GPU: it decodes a seeded request written to files, and its output
matches the oracle within the decode tolerances.
"""
import os
import shutil
import subprocess

import numpy as np
import pytest

from workloads import make_workload

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_abi", "decode_main.c")
INCLUDE = os.path.join(ROOT, "include")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _compile(out_dir, link: bool):
    gcc = shutil.which("gcc")
    if gcc is None or not os.path.exists(os.path.join(CUDA, "include", "cuda_runtime.h")):
        pytest.skip("gcc or the CUDA headers are missing")
    cmd = [gcc, "-std=c99", "-O2", "-Wall", "-Wextra", "-Werror", "-I", INCLUDE,
           "-I", os.path.join(CUDA, "include"), SRC]
    if not link:
        subprocess.run(cmd + ["-fsyntax-only"], check=True, capture_output=True)
        return None
    from mla_decode_attention_05_gb300 import build
    lib_dir = os.path.dirname(build.build())
    exe = os.path.join(out_dir, "decode_main")
    cuda_lib = os.path.join(CUDA, "lib64")
    subprocess.run(cmd + ["-o", exe, "-L", lib_dir, "-lmla_decode", "-L", cuda_lib, "-lcudart",
                          f"-Wl,-rpath,{lib_dir}:{cuda_lib}"], check=True, capture_output=True)
    return exe


def test_c_program_compiles_as_c99():
    _compile(None, link=False)


@pytest.mark.gpu
def test_c_program_decodes_like_the_oracle(tmp_path, oracle_mod):
    import _gpu as G
    exe = _compile(str(tmp_path), link=True)
    w = make_workload("c_abi", 3, 2, 64, [700, 1, 130], seed=41)
    d = str(tmp_path)
    with open(os.path.join(d, "request.txt"), "w") as f:
        f.write(f"{w.B} {w.T} {w.H} {w.num_pages} {w.max_pages} {w.softmax_scale!r}\n")
    np.ascontiguousarray(w.q).tofile(os.path.join(d, "q.bin"))
    np.ascontiguousarray(w.kv).tofile(os.path.join(d, "kv.bin"))
    np.ascontiguousarray(w.block_table, dtype=np.int32).tofile(os.path.join(d, "block_table.bin"))
    np.ascontiguousarray(w.cache_seqlens, dtype=np.int32).tofile(os.path.join(d, "seqlens.bin"))
    r = subprocess.run([exe, d], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    out_bits = np.fromfile(os.path.join(d, "out.bin"), dtype=np.uint16).reshape(w.B, w.T, w.H, 512)
    out = (out_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    lse = np.fromfile(os.path.join(d, "lse.bin"), dtype=np.float32).reshape(w.B, w.H, w.T).astype(np.float64)
    ref_o, ref_l = oracle_mod.decode_all(w)
    assert np.abs(out - ref_o).max() <= G.TOL_O
    assert np.abs(out - ref_o).max() <= G.TOL_O_REL * np.abs(ref_o).max()
    assert np.abs(lse - ref_l).max() <= G.TOL_LSE

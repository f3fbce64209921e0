"""mla_decode_noalloc: decode for callers that cannot allocate device memory.

Some host programs own all device memory (runtimes that plan every byte up
front, plugin contracts that forbid allocation, foreign-function callers with
no allocator), so they cannot hand the library a workspace.  This entry point
keeps its scratch in a fixed array inside the library.  These tests call it
through the C ABI and check it against the ordinary entry point (caller
allocated schedule and workspace) on the same inputs, twice in a row, and
check that an oversized request is refused before anything is launched.

The file sorts last so that a run stopping at the first failure has already
run every other test; it does not depend on them and passes on its own.
"""
import ctypes

import numpy as np
import pytest
import torch

from workloads import make_workload

import _gpu as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mla():
    from mla_decode_attention_05_gb300 import build
    build.build()
    import mla_decode_attention_05_gb300 as m
    m.device_status()
    return m


def _noalloc_c_abi(mla, w, d):
    """One mla_decode_noalloc call through the C ABI (ctypes, raw pointers)."""
    L = mla.lib()
    P = ctypes.c_void_p
    out = torch.full((w.B, w.T, w.H, 512), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((w.B, w.H, w.T), 7.0, dtype=torch.float32, device="cuda")
    ptr = lambda t: None if t is None else P(t.data_ptr())
    rc = L.mla_decode_noalloc(
        ptr(d["q"]), ptr(d["kv"]), w.kv_format, w.num_pages, 64, ptr(d["bt"]), w.max_pages,
        ptr(d["sk"]), ptr(d["topk"]), w.topk_len, ptr(d["scales"]), ctypes.c_float(w.softmax_scale),
        int(w.causal), ptr(out), ptr(lse), w.B, w.T, w.H,
        P(torch.cuda.current_stream().cuda_stream))
    return rc, out, lse


def _compare(res_ref, out, lse):
    o = out.float().cpu().numpy().astype(np.float64)
    l = lse.cpu().numpy().astype(np.float64)
    ref_o, ref_l = res_ref["out"], res_ref["lse"]
    assert np.array_equal(np.isneginf(l), np.isneginf(ref_l))
    fin = np.isfinite(ref_l)
    assert np.abs(o - ref_o).max() <= G.TOL_O
    assert np.abs(l[fin] - ref_l[fin]).max() <= G.TOL_LSE


def test_noalloc_matches_decode_twice(mla):
    """Two calls in a row (different requests, the second reusing the scratch
    the first left behind) agree with mla_decode on the same inputs."""
    cases = [
        make_workload("na1", 6, 1, 128, [5000, 64, 1, 3000, 130, 0], seed=31),
        make_workload("na2", 3, 2, 64, [900, 300, 2000], seed=32, topk=200, topk_pad_count=11, fp8=True),
    ]
    for w in cases:
        d = G.to_device(w)
        ref = G.run(w, dev=d)                     # ordinary entry point
        rc, out, lse = _noalloc_c_abi(mla, w, d)
        assert rc == 0, mla.lib().mla_last_error_string().decode()
        torch.cuda.synchronize()
        _compare(ref, out, lse)
    assert mla.device_status() == 0


def test_noalloc_refuses_oversized_request(mla):
    """A request whose schedule and workspace exceed the fixed scratch gets
    MLA_ERR_WORKSPACE and an explanation; nothing is written."""
    w = make_workload("big", 400, 1, 128, [64] * 400, seed=33)
    d = G.to_device(w)
    rc, out, lse = _noalloc_c_abi(mla, w, d)
    assert rc == -3
    assert b"scratch" in mla.lib().mla_last_error_string()
    torch.cuda.synchronize()
    assert torch.all(out.float() == 7.0) and torch.all(lse == 7.0)

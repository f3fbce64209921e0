"""mla_decode_noalloc: decode for callers that cannot allocate device memory.

Some host programs own all device memory (runtimes that plan every byte up
front, plugin contracts that forbid allocation, foreign-function callers with
no allocator), so they cannot hand the library a workspace.  This entry point
keeps its scratch in a fixed array inside the library.  These tests call it
through the C ABI and check it bit for bit against the ordinary entry point
(caller-allocated schedule and workspace, same worker count) on the same
inputs, twice in a row, and check that the largest request that fits runs
while larger ones are refused before anything is launched.

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


def _reference(mla, w, d):
    """The ordinary entry point (caller-allocated schedule and workspace) at
    the worker count mla_decode_noalloc uses."""
    md, ns = mla.metadata(d["sk"], w.H, w.T, topk=w.topk_len, causal=w.causal)
    assert md.shape[0] == mla.default_num_parts()
    out, lse = mla.decode(d["q"], d["kv"], d["bt"], d["sk"], softmax_scale=w.softmax_scale,
                          causal=w.causal, topk_indices=d["topk"], kv_scales=d["scales"],
                          tile_md=md, num_splits=ns)
    return out, lse


def _same_bits(a, b):
    return torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a.view(torch.int32),
                       b.view(torch.int16) if b.dtype == torch.bfloat16 else b.view(torch.int32))


def test_noalloc_matches_decode_twice(mla, oracle_mod):
    """Two calls in a row of each request (the second reusing the scratch the
    first left behind) give the same bits as mla_decode with the same worker
    count: the same schedule and kernels, only the scratch differs.  The
    requests cover dense, causal T = 4, top-k with the per-128 FP8 rows and
    the per-tensor FP8 rows; one of them is also checked against the
    oracle."""
    cases = [
        make_workload("na1", 6, 1, 128, [5000, 64, 1, 3000, 130, 0], seed=31),
        make_workload("na2", 3, 2, 64, [900, 300, 2000], seed=32, topk=200, topk_pad_count=11, fp8=True),
        make_workload("na3", 2, 4, 64, [700, 130], seed=34, causal=True),
        make_workload("na4", 3, 1, 128, [900, 64, 2100], seed=35, fp8_tensor=True),
    ]
    for k, w in enumerate(cases):
        d = G.to_device(w)
        ref_o, ref_l = _reference(mla, w, d)
        for _ in range(2):
            rc, out, lse = _noalloc_c_abi(mla, w, d)
            assert rc == 0, mla.lib().mla_last_error_string().decode()
            torch.cuda.synchronize()
            assert _same_bits(out, ref_o) and _same_bits(lse, ref_l), w.name
        if k == 2:
            res = dict(out=out.float().cpu().numpy().astype(np.float64),
                       lse=lse.cpu().numpy().astype(np.float64))
            G.compare_rows(w, res, G.all_rows(w), oracle_mod)
    assert mla.device_status() == 0


def _scratch_need(mla, B, H, T, topk):
    """Bytes of scratch a request takes: the schedule arrays, each rounded up
    to 256 bytes, plus the decode workspace (the rule the header states)."""
    parts = mla.default_num_parts()
    r256 = lambda n: (n + 255) // 256 * 256
    md_elems, ns_elems = mla.metadata_sizes(B, H, T, topk, parts)
    return r256(md_elems * 4) + r256(ns_elems * 4) + mla.workspace_bytes(B, H, T, topk, parts)


def test_noalloc_largest_request_fits_and_one_more_is_refused(mla):
    """The largest batch whose schedule and workspace fit the fixed scratch
    runs and matches mla_decode bit for bit; one sequence more gets
    MLA_ERR_WORKSPACE and an explanation, and nothing is written."""
    limit = 64 << 20
    B = 1
    while _scratch_need(mla, B + 1, 128, 1, 0) <= limit:
        B += 1
    assert _scratch_need(mla, B, 128, 1, 0) <= limit < _scratch_need(mla, B + 1, 128, 1, 0)
    w = make_workload("cap", B, 1, 128, [64 + (b * 37) % 300 for b in range(B)], seed=36)
    d = G.to_device(w)
    ref_o, ref_l = _reference(mla, w, d)
    rc, out, lse = _noalloc_c_abi(mla, w, d)
    assert rc == 0, mla.lib().mla_last_error_string().decode()
    torch.cuda.synchronize()
    assert _same_bits(out, ref_o) and _same_bits(lse, ref_l)
    w1 = make_workload("cap1", B + 1, 1, 128, [64] * (B + 1), seed=37)
    d1 = G.to_device(w1)
    rc, out, lse = _noalloc_c_abi(mla, w1, d1)
    assert rc == -3
    assert b"scratch" in mla.lib().mla_last_error_string()
    torch.cuda.synchronize()
    assert torch.all(out.float() == 7.0) and torch.all(lse == 7.0)
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

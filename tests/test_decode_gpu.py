"""GPU parity: the CUDA path through the C ABI against the float64 oracle on
the same seeded inputs.  Small cases and the five named workloads (at full
size, in the launch configuration the bench uses: the default worker count)
are compared row by row in full."""
import zlib

import numpy as np
import pytest
import torch

import workloads
from workloads import make_workload

import _gpu as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mla():
    from mla_decode_attention_05_gb300 import build
    build.build()
    import mla_decode_attention_05_gb300 as m
    m.device_status()  # clear
    return m


def _status_clean(mla):
    assert mla.device_status() == 0


# --- the five workloads ---------------------------------------------------------

def test_tiny_dense_full(mla, oracle_mod):
    w = workloads.config(1)
    res = G.run(w)
    G.compare_rows(w, res, G.all_rows(w), oracle_mod)
    _status_clean(mla)


@pytest.mark.parametrize("cfg", [2, 3, 5])
def test_dense_configs_every_row(mla, oracle_mod, cfg):
    """The full-size dense workloads in the bench's launch configuration,
    every (b, t, h) row against the oracle element by element (the oracle
    takes about 12 s for the 8192 rows of the largest on 16 host cores)."""
    w = workloads.config(cfg)
    res = G.run(w)
    G.compare_rows(w, res, G.all_rows(w), oracle_mod)
    assert np.all(np.isfinite(res["lse"]))
    _status_clean(mla)


def test_sparse_fp8_config_every_row_and_gathered(mla, oracle_mod):
    """The full-size sparse FP8 workload: every row against the oracle and
    every sequence's gathered-index record against the oracle's valid set."""
    w = workloads.config(4)
    res = G.run(w, record=True)
    G.compare_rows(w, res, G.all_rows(w), oracle_mod)
    for b in range(w.B):
        got = res["gathered"][b, 0]
        assert np.all(got >= -1)
        exp = oracle_mod.valid_keys(w, b, 0)
        assert np.array_equal(np.sort(got[got >= 0]), exp), "gathered-index set differs"
        # each slot records its own index (or -1 for a -1 slot)
        assert np.array_equal(got, np.where(w.topk[b, 0] >= 0, w.topk[b, 0], -1))
    _status_clean(mla)


# --- small cases, every row --------------------------------------------------------

SMALL = [
    dict(B=3, T=1, H=128, seqlens=[1, 63, 200]),
    dict(B=2, T=1, H=64, seqlens=[64, 129]),
    dict(B=2, T=1, H=3, seqlens=[300, 5]),
    dict(B=2, T=4, H=64, seqlens=[130, 67], causal=True),
    dict(B=2, T=3, H=64, seqlens=[100, 3], causal=True),
    dict(B=1, T=2, H=128, seqlens=[150], causal=True),
    dict(B=3, T=1, H=128, seqlens=[0, 70, 0]),
    dict(B=2, T=1, H=64, seqlens=[500, 90], fp8=True),
    dict(B=2, T=2, H=64, seqlens=[300, 200], topk=100, topk_pad_count=9, fp8=True),
    dict(B=2, T=1, H=64, seqlens=[500, 90], fp8_tensor=True),
    dict(B=2, T=2, H=128, seqlens=[300, 200], topk=100, topk_pad_count=9, fp8_tensor=True),
    dict(B=2, T=1, H=128, seqlens=[400, 70], topk=64),
    dict(B=1, T=1, H=64, seqlens=[64], topk=1),
    dict(B=2, T=1, H=1, seqlens=[300, 65]),
    dict(B=2, T=8, H=16, seqlens=[200, 9], causal=True),
    dict(B=1, T=16, H=32, seqlens=[700], causal=True),
    dict(B=2, T=4, H=64, seqlens=[900, 260], topk=130, topk_pad_count=5),
    dict(B=1, T=1, H=128, seqlens=[4160], fp8=True),
    dict(B=2, T=4, H=16, seqlens=[300, 70], causal=True, fp8=True),   # 64 rows: padding warps gather
    dict(B=2, T=2, H=64, seqlens=[200, 90], causal=True, fp8=True),   # 128 rows: the usual gather
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: "-".join(f"{k}{v}" for k, v in c.items() if k != "seqlens"))
@pytest.mark.parametrize("parts", [None, 1, 37])
def test_small_every_row(mla, oracle_mod, case, parts):
    c = dict(case)
    B, T, H, sl = c.pop("B"), c.pop("T"), c.pop("H"), c.pop("seqlens")
    w = make_workload("small", B, T, H, sl, seed=zlib.crc32(repr(case).encode()) % 1000, **c)
    res = G.run(w, num_parts=parts, record=True)
    G.compare_rows(w, res, G.all_rows(w), oracle_mod)
    if w.topk is not None:
        for b in range(B):
            for t in range(T):
                got = res["gathered"][b, t]
                assert np.array_equal(np.sort(got[got >= 0]), oracle_mod.valid_keys(w, b, t))
    _status_clean(mla)


def test_all_slots_padding(mla, oracle_mod):
    """A top-k row of only -1: O = 0, LSE = -inf, nothing gathered."""
    w = make_workload("pad", 2, 1, 64, [200, 200], seed=5, topk=70)
    w.topk[0] = -1
    res = G.run(w, record=True)
    G.compare_rows(w, res, G.all_rows(w), oracle_mod)
    assert np.all(res["gathered"][0] == -1)


def test_many_splits_combine(mla, oracle_mod):
    """More workers than tiles: every item is cut into many pieces and the
    combine kernel merges them."""
    w = make_workload("split", 2, 1, 128, [1000, 640], seed=8)
    res = G.run(w, num_parts=40)
    ns = np.diff(res["num_splits"])
    assert ns.max() >= 10
    G.compare_rows(w, res, G.all_rows(w), oracle_mod)


def test_schedule_reused_by_consecutive_calls(mla, oracle_mod):
    """One schedule serves several decode calls in stream order (as one
    schedule serves every layer of a step), with identical results."""
    w = make_workload("reuse", 3, 1, 128, [3000, 700, 5000], seed=21)
    d = G.to_device(w)
    md, ns = mla.metadata(d["sk"], w.H, w.T, num_parts=24)
    outs = []
    for _ in range(3):
        out, lse = mla.decode(d["q"], d["kv"], d["bt"], d["sk"], softmax_scale=w.softmax_scale,
                              tile_md=md, num_splits=ns)
        outs.append((out.clone(), lse.clone()))
    torch.cuda.synchronize()
    assert np.diff(ns.cpu().numpy()).max() > 1
    for o, l in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(l, outs[0][1])
    res = dict(out=outs[0][0].float().cpu().numpy().astype(np.float64),
               lse=outs[0][1].cpu().numpy().astype(np.float64))
    G.compare_rows(w, res, G.all_rows(w), oracle_mod)


def test_more_workers_than_fit_at_once(mla, oracle_mod):
    """num_parts above the worker pairs the device holds at once: later
    workers start as earlier ones finish; items whose pieces span both
    groups still combine correctly."""
    w = make_workload("waves", 2, 1, 64, [9000, 7000], seed=22)
    res = G.run(w, num_parts=120)
    assert mla.device_status() == 0
    G.compare_rows(w, res, G.all_rows(w), oracle_mod)


def test_largest_rows_per_sequence_causal(mla, oracle_mod):
    """T = 16 query tokens x H = 128 heads = 2048 rows per sequence (16
    items each), causal, ragged lengths: every row against the oracle."""
    w = make_workload("t16h128", 2, 16, 128, [200, 77], seed=31, causal=True)
    res = G.run(w)
    G.compare_rows(w, res, G.all_rows(w), oracle_mod)
    _status_clean(mla)


def test_metadata_bit_exact(mla):
    """Device schedule == the plain-Python statement of the rule."""
    from oracle import schedule as S
    rng = np.random.default_rng(4)
    for trial in range(25):
        B = int(rng.integers(1, 70))
        H = int(rng.choice([64, 128]))
        T = int(rng.integers(1, 5))
        causal = bool(rng.integers(0, 2))
        topk = 0 if causal else int(rng.choice([0, 0, 2048]))
        sl = rng.integers(0, 40000, size=B).astype(np.int32)
        if topk:
            sl = np.maximum(sl, topk).astype(np.int32)
        P = int(rng.integers(1, 160))
        md, ns = mla.metadata(torch.from_numpy(sl).cuda(), H, T, topk=topk, causal=causal, num_parts=P)
        ref_md, ref_ns = S.schedule(sl, H, T, P, topk, causal)
        assert np.array_equal(md.cpu().numpy(), np.array(ref_md, dtype=np.int32)), trial
        assert np.array_equal(ns.cpu().numpy(), np.array(ref_ns, dtype=np.int32)), trial


def test_bad_page_and_index_set_status(mla, oracle_mod):
    """Out-of-range page ids and top-k indices are caught by the kernel's own
    bounds checks: the row is skipped and a status bit is set; nothing
    faults."""
    w = make_workload("bad", 1, 1, 64, [128], seed=3)
    w.block_table[0, 1] = 10 ** 6
    G.run(w)
    st = mla.device_status()
    assert st & mla.STATUS_BAD_PAGE
    ws = make_workload("badk", 1, 1, 64, [128], seed=3, topk=8)
    ws.topk[0, 0, 2] = 500
    res = G.run(ws, record=True)
    st = mla.device_status()
    assert st & mla.STATUS_BAD_TOPK
    assert res["gathered"][0, 0, 2] == -1
    # the other slots still give the oracle's answer over the valid ones
    ws.topk[0, 0, 2] = -1
    G.compare_rows(ws, res, G.all_rows(ws), oracle_mod)


def test_repeat_calls_identical(mla):
    """Same inputs twice: identical bits (no state carried between calls)."""
    w = make_workload("rep", 4, 1, 128, [700, 64, 1, 333], seed=9)
    d = G.to_device(w)
    a = G.run(w, dev=d)
    b = G.run(w, dev=d)
    assert np.array_equal(a["out"], b["out"]) and np.array_equal(a["lse"], b["lse"])


def test_output_only_16_byte_aligned(mla, oracle_mod):
    """out 16 bytes past a 32-byte boundary: the epilogue must use its
    16-byte stores there (32-byte stores need 32-byte alignment)."""
    w = make_workload("align", 3, 1, 128, [700, 64, 130], seed=21)
    d = G.to_device(w)
    md, ns = mla.metadata(d["sk"], w.H, w.T)
    n = w.B * w.T * w.H * 512
    buf = torch.full((n + 8,), 7.0, dtype=torch.bfloat16, device="cuda")
    out = buf[8:].view(w.B, w.T, w.H, 512)
    assert out.data_ptr() % 32 == 16
    o, lse = mla.decode(d["q"], d["kv"], d["bt"], d["sk"], softmax_scale=w.softmax_scale,
                        tile_md=md, num_splits=ns, out=out)
    torch.cuda.synchronize()
    assert o.data_ptr() == out.data_ptr()
    assert torch.all(buf[:8] == 7.0), "wrote before the output"
    res = dict(out=o.float().cpu().numpy().astype(np.float64), lse=lse.cpu().numpy().astype(np.float64))
    G.compare_rows(w, res, G.all_rows(w), oracle_mod)


# --- the M = 64 dual GEMM for QK (selected per thread) ----------------------------

# the dual GEMM serves the page path (bf16 cache, no top-k) with at most 64 rows per item
DUAL_CASES = [c for c in SMALL if not c.get("topk") and not c.get("fp8") and not c.get("fp8_tensor")
              and c["T"] * c["H"] <= 64] + [
    dict(B=3, T=1, H=64, seqlens=[1000, 64, 257]),
    dict(B=2, T=2, H=32, seqlens=[700, 129], causal=True),
    dict(B=2, T=4, H=16, seqlens=[300, 4], causal=True),
]


@pytest.fixture
def dual_gemm(mla):
    mla.set_dual_gemm(True)
    yield
    mla.set_dual_gemm(False)


@pytest.mark.parametrize("case", DUAL_CASES, ids=lambda c: "-".join(f"{k}{v}" for k, v in c.items() if k != "seqlens"))
@pytest.mark.parametrize("parts", [None, 37])
def test_dual_gemm_small_every_row(mla, oracle_mod, dual_gemm, case, parts):
    """Items of at most 64 rows with QK as the dual GEMM: every row against
    the oracle (dense and causal, H = 1, 3, 16, 32, 64, ragged lengths)."""
    c = dict(case)
    B, T, H, sl = c.pop("B"), c.pop("T"), c.pop("H"), c.pop("seqlens")
    w = make_workload("small", B, T, H, sl, seed=zlib.crc32(repr(case).encode()) % 1000, **c)
    res = G.run(w, num_parts=parts, record=True)
    G.compare_rows(w, res, G.all_rows(w), oracle_mod)
    if w.topk is not None:
        for b in range(B):
            for t in range(T):
                got = res["gathered"][b, t]
                assert np.array_equal(np.sort(got[got >= 0]), oracle_mod.valid_keys(w, b, t))
    _status_clean(mla)


@pytest.mark.parametrize("cfg", [1])
def test_dual_gemm_h64_workloads_every_row(mla, oracle_mod, dual_gemm, cfg):
    """The tiny dense H = 64 workload with the dual GEMM, every row against
    the oracle."""
    w = workloads.config(cfg)
    res = G.run(w, record=True)
    G.compare_rows(w, res, G.all_rows(w), oracle_mod)
    _status_clean(mla)

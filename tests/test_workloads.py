"""The five named workloads follow their stated recipe (shapes, lengths,
page maps, top-k structure, value distributions, seeds); they are the inputs
of every parity test and of the benchmark, so a drift here would silently
change what is measured."""
import numpy as np
import pytest

import workloads as W


def _bf16_values(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _check_pages(w, pool_is_exact):
    bt = w.block_table
    pages_per = -(-w.cache_seqlens.astype(np.int64) // 64)
    used = np.concatenate([bt[b, :pages_per[b]] for b in range(w.B)])
    assert (used >= 0).all() and (used < w.num_pages).all()
    assert len(np.unique(used)) == len(used)            # no page shared between sequences
    if pool_is_exact:
        assert len(used) == w.num_pages


def _check_q(w):
    q = _bf16_values(w.q).astype(np.float64)
    assert np.isfinite(q).all()
    assert abs(q.mean()) < 0.01 and abs(q.std() - 0.5) < 0.01   # N(0, 1) * 0.5


@pytest.mark.parametrize("idx", [1, 2, 3, 4, 5])
def test_named_workload_recipe(idx):
    w = W.config(idx)
    assert w.seed == 1000 + idx
    assert abs(w.softmax_scale - 192 ** -0.5) < 1e-15
    _check_q(w)
    if idx == 1:
        assert (w.B, w.T, w.H) == (2, 1, 64) and list(w.cache_seqlens) == [256, 256]
        assert w.block_table.tolist() == [[0, 1, 2, 3], [4, 5, 6, 7]]   # the unpaged cache, 4 pages per sequence
        assert w.kv.shape == (8, 64, 576) and w.kv_format == W.KV_BF16
    elif idx == 2:
        assert (w.B, w.T, w.H) == (16, 1, 128) and (w.cache_seqlens == 4096).all()
        assert w.num_pages == 1024 and w.kv_format == W.KV_BF16
        _check_pages(w, True)
    elif idx == 3:
        assert (w.B, w.T, w.H) == (64, 1, 128) and w.kv_format == W.KV_BF16
        sk = w.cache_seqlens
        assert sk.min() >= 1024 and sk.max() <= 32768 and int(sk.sum()) == 1119245
        _check_pages(w, True)
    elif idx == 4:
        assert (w.B, w.T, w.H) == (32, 1, 64) and w.kv_format == W.KV_FP8
        assert (w.cache_seqlens == 65536).all() and w.num_pages == 32768
        assert w.kv.shape == (32768, 64, 640) and w.kv_scales.shape == (32768, 64, 4)
        assert w.kv_scales.min() >= 0.5 and w.kv_scales.max() <= 2.0
        tk = w.topk
        assert tk.shape == (32, 1, 2048)
        for b in range(32):
            row = tk[b, 0]
            assert (row == -1).sum() == 102                 # round(0.05 * 2048) unused slots
            valid = row[row >= 0]
            assert len(np.unique(valid)) == len(valid) and valid.max() < 65536
        codes = w.kv[:, :, :512]
        assert not ((codes & 0x7F) == 0x7F).any()           # no e4m3 NaN code
        _check_pages(w, True)
    else:
        assert (w.B, w.T, w.H) == (32, 4, 64) and w.causal and (w.cache_seqlens == 16384).all()
        assert w.num_pages == 8192 and w.kv_format == W.KV_BF16
        _check_pages(w, True)


def test_generation_is_deterministic():
    a, b = W.config(2), W.config(2)
    for name in ("q", "kv", "block_table", "cache_seqlens"):
        np.testing.assert_array_equal(getattr(a, name), getattr(b, name))

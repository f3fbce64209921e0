"""Pins of the float64 oracle against things other than itself.

The pages print no worked example for the attention, so the oracle is pinned
to (1) library routines on special cases that reduce to plain attention
(torch scaled_dot_product_attention / logsumexp in float64, torch's own bf16
and float8_e4m3fn decoders), (2) closed forms, (3) invariants of the
definition, and (4) brute force on tiny inputs.  Each test names the kind of
mistake it would catch.
"""
import math

import numpy as np
import pytest
import torch

import workloads
from workloads import D_QK, D_V, make_workload

SCALE = 1.0 / math.sqrt(192.0)


def _bf16_bits_to_f64(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).double()


def _gather_keys(w, b, n_keys):
    """Dense float64 K rows 0..n_keys-1 of sequence b (bf16 cache), read
    through the block table with numpy indexing."""
    pages = w.block_table[b, np.arange(n_keys) // 64]
    slots = np.arange(n_keys) % 64
    return _bf16_bits_to_f64(w.kv[pages, slots])          # [n, 576]


def _sdpa(q, K, scale):
    """Library attention in float64 with one KV head: q [h, 576], K [n, 576]."""
    V = K[:, :D_V]
    out = torch.nn.functional.scaled_dot_product_attention(
        q[None, :, None, :], K[None, None].expand(1, q.shape[0], -1, -1),
        V[None, None].expand(1, q.shape[0], -1, -1), scale=scale)[0, :, 0, :]
    lse = torch.logsumexp(scale * (q @ K.T), dim=-1)
    return out.numpy(), lse.numpy()


# --- element decoders ---------------------------------------------------------

def test_bf16_decoder_exhaustive(oracle_mod):
    """All 65536 bf16 codes against torch's bf16->float64 (catches a wrong
    shift or a byte-order slip)."""
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = _bf16_bits_to_f64(codes).numpy()
    got = np.array([oracle_mod.bf16_to_f64(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_e4m3_decoder_exhaustive(oracle_mod):
    """All 256 OCP e4m3 codes against torch.float8_e4m3fn->float64
    (catches a wrong bias, subnormal rule or NaN code)."""
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    got = np.array([oracle_mod.e4m3_to_f64(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert nan.sum() == 2
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9


# --- special cases that are library attention -----------------------------------

@pytest.mark.parametrize("H,sk,paged", [(64, 256, False), (128, 200, True), (2, 1, True)])
def test_dense_t1_equals_library_sdpa(oracle_mod, H, sk, paged):
    """T=1 dense decode is plain attention with one KV head, K = the 576-wide
    row and V = its first 512 values: compare with torch SDPA in float64
    (catches a dropped RoPE block, a wrong V slice, a wrong scale or a page
    lookup slip)."""
    w = make_workload("t", 2, 1, H, [sk, max(1, sk // 2)], seed=7,
                      identity_pages=not paged)
    out, lse = oracle_mod.decode_all(w)
    for b in range(w.B):
        n = int(w.cache_seqlens[b])
        K = _gather_keys(w, b, n)
        q = _bf16_bits_to_f64(w.q[b, 0])
        ro, rl = _sdpa(q, K, w.softmax_scale)
        np.testing.assert_allclose(out[b, 0], ro, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[b, :, 0], rl, rtol=0, atol=1e-12)


def test_causal_rows_equal_truncated_sdpa(oracle_mod):
    """Causal T=4: query token t sees keys n < s_k - T + t + 1, so its rows
    equal library attention on that prefix (catches an off-by-one in the
    causal bound and a transposed (t, h) row index)."""
    T, H, sk = 4, 3, 70
    w = make_workload("t", 2, T, H, [sk, 66], seed=11, causal=True)
    out, lse = oracle_mod.decode_all(w)
    for b in range(w.B):
        s = int(w.cache_seqlens[b])
        for t in range(T):
            n = s - T + t + 1
            K = _gather_keys(w, b, n)
            q = _bf16_bits_to_f64(w.q[b, t])
            ro, rl = _sdpa(q, K, w.softmax_scale)
            np.testing.assert_allclose(out[b, t], ro, atol=1e-12, rtol=0)
            np.testing.assert_allclose(lse[b, :, t], rl, atol=1e-12, rtol=0)


def test_causal_t1_is_noncausal(oracle_mod):
    w1 = make_workload("t", 2, 1, 4, [90, 33], seed=3, causal=True)
    w0 = make_workload("t", 2, 1, 4, [90, 33], seed=3, causal=False)
    o1, l1 = oracle_mod.decode_all(w1)
    o0, l0 = oracle_mod.decode_all(w0)
    assert np.array_equal(o1, o0) and np.array_equal(l1, l0)


def test_sparse_subset_equals_sdpa_on_gathered_rows(oracle_mod):
    """Top-k with -1 slots: attention over exactly the named rows, in any
    order (catches a slot read as a key, or -1 read as key 0)."""
    w = make_workload("t", 2, 2, 3, [200, 150], seed=5, topk=40, topk_pad_count=7)
    out, lse = oracle_mod.decode_all(w)
    for b in range(w.B):
        Kall = _gather_keys(w, b, int(w.cache_seqlens[b]))
        for t in range(w.T):
            ids = w.topk[b, t]
            ids = ids[ids >= 0]
            assert len(ids) == 33
            q = _bf16_bits_to_f64(w.q[b, t])
            ro, rl = _sdpa(q, Kall[torch.from_numpy(ids.astype(np.int64))], w.softmax_scale)
            np.testing.assert_allclose(out[b, t], ro, atol=1e-12, rtol=0)
            np.testing.assert_allclose(lse[b, :, t], rl, atol=1e-12, rtol=0)


def test_sparse_full_topk_equals_dense(oracle_mod):
    """Top-k naming every key of the sequence (shuffled) equals dense."""
    sk = 96
    wd = make_workload("t", 1, 1, 4, [sk], seed=21)
    ws = make_workload("t", 1, 1, 4, [sk], seed=21)
    ws.topk = np.random.default_rng(0).permutation(sk).astype(np.int32).reshape(1, 1, sk)
    od, ld = oracle_mod.decode_all(wd)
    os_, ls = oracle_mod.decode_all(ws)
    np.testing.assert_allclose(os_, od, atol=1e-13, rtol=0)
    np.testing.assert_allclose(ls, ld, atol=1e-13, rtol=0)


# --- FP8 rows -------------------------------------------------------------------

def _fp8_as_bf16_workload(w8, scale_mult=None):
    """The same cache written as bf16 rows (every e4m3 value times a power-of-
    two scale is exact in bf16)."""
    codes = torch.from_numpy(np.ascontiguousarray(w8.kv[:, :, :D_V])).view(torch.float8_e4m3fn)
    nope = codes.float() * torch.from_numpy(w8.kv_scales).repeat_interleave(128, dim=2)
    rope = torch.from_numpy(np.ascontiguousarray(w8.kv[:, :, D_V:])).view(torch.bfloat16)
    kv = torch.cat([nope.to(torch.bfloat16), rope], dim=2)
    assert torch.equal(kv[:, :, :D_V].float(), nope)       # exact in bf16
    return workloads.Workload(
        name="as_bf16", B=w8.B, T=w8.T, H=w8.H, q=w8.q,
        kv=kv.view(torch.int16).numpy().view(np.uint16), kv_format=workloads.KV_BF16,
        kv_scales=None, block_table=w8.block_table, cache_seqlens=w8.cache_seqlens,
        topk=w8.topk, softmax_scale=w8.softmax_scale, causal=w8.causal, seed=w8.seed)


def test_fp8_rows_equal_bf16_rows_with_pow2_scales(oracle_mod):
    """FP8 row format: 512 e4m3 bytes x per-128-tile scale, then 64 bf16 RoPE
    values.  With power-of-two scales (different per tile) the dequantised
    row is exact in bf16, so the fp8 and the equivalent bf16 cache must give
    identical results (catches a wrong scale-tile index, RoPE byte order or
    row stride)."""
    w8 = make_workload("t", 2, 1, 4, [130, 64], seed=9, fp8=True)
    rng = np.random.default_rng(1)
    w8.kv_scales = (2.0 ** rng.integers(-2, 3, size=w8.kv_scales.shape)).astype(np.float32)
    wb = _fp8_as_bf16_workload(w8)
    o8, l8 = oracle_mod.decode_all(w8)
    ob, lb = oracle_mod.decode_all(wb)
    np.testing.assert_allclose(o8, ob, atol=1e-14, rtol=0)
    np.testing.assert_allclose(l8, lb, atol=1e-14, rtol=0)


def test_fp8_dequant_is_product_with_scale(oracle_mod):
    """Arbitrary scales: the oracle dequantises to the exact float64 product,
    so its result equals library attention on K built from torch's e4m3
    decode times the scale in float64."""
    w8 = make_workload("t", 1, 1, 3, [100], seed=4, fp8=True)
    out, lse = oracle_mod.decode_all(w8)
    n = 100
    pages = w8.block_table[0, np.arange(n) // 64]
    slots = np.arange(n) % 64
    rows = w8.kv[pages, slots]
    nope = torch.from_numpy(np.ascontiguousarray(rows[:, :D_V])).view(torch.float8_e4m3fn).double()
    sc = torch.from_numpy(w8.kv_scales[pages, slots]).double().repeat_interleave(128, dim=1)
    rope = torch.from_numpy(np.ascontiguousarray(rows[:, D_V:])).view(torch.bfloat16).double()
    K = torch.cat([nope * sc, rope], dim=1)
    ro, rl = _sdpa(_bf16_bits_to_f64(w8.q[0, 0]), K, w8.softmax_scale)
    np.testing.assert_allclose(out[0, 0], ro, atol=1e-12, rtol=0)
    np.testing.assert_allclose(lse[0, :, 0], rl, atol=1e-12, rtol=0)


def test_per_tensor_fp8_rows_equal_bf16_rows_with_pow2_scale(oracle_mod):
    """Per-tensor FP8 rows (576 e4m3 bytes, RoPE included, one scale): with a
    power-of-two scale every dequantised value is exact in bf16, so the cache
    and its bf16 image give identical results (catches a wrong row stride,
    a RoPE part read as bf16, or a missing scale)."""
    w8 = make_workload("tt", 2, 1, 4, [130, 64], seed=19, fp8_tensor=True)
    w8.kv_scales = np.array([0.25], dtype=np.float32)
    vals = torch.from_numpy(np.ascontiguousarray(w8.kv)).view(torch.float8_e4m3fn).double() * 0.25
    kv = vals.to(torch.bfloat16)
    assert torch.equal(kv.double(), vals)  # exact in bf16
    wb = workloads.Workload(
        name="as_bf16", B=w8.B, T=w8.T, H=w8.H, q=w8.q,
        kv=kv.view(torch.int16).numpy().view(np.uint16), kv_format=workloads.KV_BF16,
        kv_scales=None, block_table=w8.block_table, cache_seqlens=w8.cache_seqlens,
        topk=w8.topk, softmax_scale=w8.softmax_scale, causal=w8.causal, seed=w8.seed)
    o8, l8 = oracle_mod.decode_all(w8)
    ob, lb = oracle_mod.decode_all(wb)
    np.testing.assert_allclose(o8, ob, atol=1e-14, rtol=0)
    np.testing.assert_allclose(l8, lb, atol=1e-14, rtol=0)


def test_per_tensor_fp8_dequant_is_product_with_scale(oracle_mod):
    """Arbitrary scale: library attention on K = torch's e4m3 decode x the
    scale in float64, all 576 values."""
    w8 = make_workload("tt", 1, 1, 3, [100], seed=14, fp8_tensor=True)
    out, lse = oracle_mod.decode_all(w8)
    n = 100
    pages = w8.block_table[0, np.arange(n) // 64]
    rows = w8.kv[pages, np.arange(n) % 64]
    K = torch.from_numpy(np.ascontiguousarray(rows)).view(torch.float8_e4m3fn).double() * float(w8.kv_scales[0])
    ro, rl = _sdpa(_bf16_bits_to_f64(w8.q[0, 0]), K, w8.softmax_scale)
    np.testing.assert_allclose(out[0, 0], ro, atol=1e-12, rtol=0)
    np.testing.assert_allclose(lse[0, :, 0], rl, atol=1e-12, rtol=0)


# --- invariants and closed forms ------------------------------------------------------

def _set_rows(w, b, n_keys, rows_bits):
    for n in range(n_keys):
        w.kv[w.block_table[b, n // 64], n % 64] = rows_bits[n]


def test_identical_keys_give_mean_of_v(oracle_mod):
    """All keys equal: O = V (the mean of identical rows) and
    LSE = s + ln|N| (closed form)."""
    sk = 77
    w = make_workload("t", 1, 1, 5, [sk], seed=12)
    row = w.kv[w.block_table[0, 0], 0].copy()
    _set_rows(w, 0, sk, [row] * sk)
    out, lse = oracle_mod.decode_all(w)
    K = _bf16_bits_to_f64(row).numpy()
    for h in range(w.H):
        q = _bf16_bits_to_f64(w.q[0, 0, h]).numpy()
        s = w.softmax_scale * math.fsum(q * K)
        np.testing.assert_allclose(out[0, 0, h], K[:D_V], atol=1e-14, rtol=0)
        assert abs(lse[0, h, 0] - (s + math.log(sk))) < 1e-12


def test_dominant_logit_selects_one_row(oracle_mod):
    """One key with a logit far above the rest: O = its V row and LSE = its
    logit, to within exp(-gap) (catches a wrong max or sign)."""
    sk = 50
    w = make_workload("t", 1, 1, 1, [sk], seed=13, softmax_scale=1.0)
    one = workloads._round_bf16_bits(np.array([1.0], dtype=np.float32))[0]
    w.q[0, 0, 0, :] = 0
    w.q[0, 0, 0, 3] = one
    j = 31
    big = workloads._round_bf16_bits(np.array([80.0], dtype=np.float32))[0]
    for n in range(sk):
        w.kv[w.block_table[0, n // 64], n % 64, 3] = 0
    w.kv[w.block_table[0, j // 64], j % 64, 3] = big
    out, lse = oracle_mod.decode_all(w)
    V = _bf16_bits_to_f64(w.kv[w.block_table[0, j // 64], j % 64]).numpy()[:D_V]
    np.testing.assert_allclose(out[0, 0, 0], V, atol=1e-30, rtol=1e-30)
    assert abs(lse[0, 0, 0] - 80.0) < 1e-30 + 60 * math.exp(-80.0)


def test_closed_form_three_keys(oracle_mod):
    """q = e_0, scale 1, logits 0, 1, 2 on three keys with one-hot V rows:
    O = softmax weights (1, e, e^2)/(1+e+e^2) placed at V's hot columns and
    LSE = ln(1+e+e^2)."""
    w = make_workload("t", 1, 1, 1, [3], seed=14, softmax_scale=1.0)
    w.q[0, 0, 0, :] = 0
    w.q[0, 0, 0, 0] = workloads._round_bf16_bits(np.array([1.0], dtype=np.float32))[0]
    for n, logit in enumerate([0.0, 1.0, 2.0]):
        r = np.zeros(D_QK, dtype=np.float32)
        r[0] = logit
        r[10 + n] = 1.0
        w.kv[w.block_table[0, 0], n] = workloads._round_bf16_bits(r)
    out, lse = oracle_mod.decode_all(w)
    Z = 1 + math.e + math.e ** 2
    exp_o = np.zeros(D_V)
    exp_o[0] = (0 * 1 + 1 * math.e + 2 * math.e ** 2) / Z
    exp_o[10:13] = np.array([1, math.e, math.e ** 2]) / Z
    np.testing.assert_allclose(out[0, 0, 0], exp_o, atol=1e-15, rtol=0)
    assert abs(lse[0, 0, 0] - math.log(Z)) < 1e-15


def test_empty_key_set(oracle_mod):
    """s_k = 0, or a top-k row of only -1: O = 0 and LSE = -inf."""
    w = make_workload("t", 2, 1, 2, [0, 5], seed=15)
    out, lse = oracle_mod.decode_all(w)
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(lse[1]))
    ws = make_workload("t", 1, 1, 2, [70], seed=16, topk=8)
    ws.topk[:] = -1
    out, lse = oracle_mod.decode_all(ws)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def test_kv_order_does_not_matter(oracle_mod):
    """Non-causal: permuting the token order of a sequence (rows moved
    between pages and slots) leaves O and LSE unchanged."""
    sk = 192                                   # whole pages, so the page map can be permuted too
    w = make_workload("t", 1, 1, 4, [sk], seed=17)
    o0, l0 = oracle_mod.decode_all(w)
    perm = np.random.default_rng(2).permutation(sk)
    rows = [w.kv[w.block_table[0, n // 64], n % 64].copy() for n in range(sk)]
    _set_rows(w, 0, sk, [rows[perm[n]] for n in range(sk)])
    w.block_table[0] = w.block_table[0][::-1].copy()       # and a different page map
    rows2 = [w.kv[w.block_table[0, n // 64], n % 64].copy() for n in range(sk)]
    assert sorted(map(bytes, rows2)) == sorted(map(bytes, rows))
    o1, l1 = oracle_mod.decode_all(w)
    np.testing.assert_allclose(o1, o0, atol=1e-14, rtol=0)
    np.testing.assert_allclose(l1, l0, atol=1e-13, rtol=0)


def test_split_and_lse_combine_equals_unsplit(oracle_mod):
    """Cut the key set in pieces, attend each, merge by LSE:
    L = ln sum_i exp(L_i), O = sum_i exp(L_i - L) O_i  ==  unsplit result."""
    sk = 300
    w = make_workload("t", 1, 1, 3, [sk], seed=18)
    for h in range(w.H):
        ref_o, ref_l = oracle_mod.attend_key_list(w, 0, 0, h, np.arange(sk))
        cuts = [0, 1, 64, 65, 200, sk]
        parts = [oracle_mod.attend_key_list(w, 0, 0, h, np.arange(a, b))
                 for a, b in zip(cuts[:-1], cuts[1:])]
        parts.append(oracle_mod.attend_key_list(w, 0, 0, h, np.arange(0)))  # empty piece
        ls = np.array([p[1] for p in parts])
        m = ls.max()
        L = m + math.log(math.fsum(math.exp(x - m) for x in ls))
        O = sum(math.exp(p[1] - L) * p[0] for p in parts)
        np.testing.assert_allclose(O, ref_o, atol=1e-14, rtol=0)
        assert abs(L - ref_l) < 1e-12


def test_lse_is_log_sum_exp_bruteforce(oracle_mod):
    """Tiny case: LSE = ln sum_n exp(s_n) with s_n from exact bf16 products
    summed by math.fsum, and O by the same brute force."""
    sk = 6
    w = make_workload("t", 1, 1, 2, [sk], seed=19, value_std=0.05)
    out, lse = oracle_mod.decode_all(w)
    for h in range(w.H):
        q = [float(x) for x in _bf16_bits_to_f64(w.q[0, 0, h])]
        Ks = [[float(x) for x in _bf16_bits_to_f64(w.kv[w.block_table[0, 0], n])] for n in range(sk)]
        s = [w.softmax_scale * math.fsum(a * b for a, b in zip(q, K)) for K in Ks]
        L = math.log(math.fsum(math.exp(x) for x in s))
        assert abs(lse[0, h, 0] - L) < 1e-13
        for j in (0, 1, 255, 511):
            o = math.fsum(math.exp(s[n] - L) * Ks[n][j] for n in range(sk))
            assert abs(out[0, 0, h, j] - o) < 1e-15


# --- valid sets ---------------------------------------------------------------------

def test_valid_keys_bruteforce(oracle_mod):
    """The gathered-index set: dense = range(s_k), causal = range(s_k-T+t+1),
    top-k = the sorted distinct non-negative indices below s_k."""
    w = make_workload("t", 2, 3, 1, [10, 2], seed=20, causal=True)
    for b in range(2):
        for t in range(3):
            sk = int(w.cache_seqlens[b])
            exp = [n for n in range(sk) if n <= sk - 3 + t]
            assert list(oracle_mod.valid_keys(w, b, t)) == exp
    ws = make_workload("t", 2, 2, 1, [40, 30], seed=22, topk=12, topk_pad_count=3)
    for b in range(2):
        for t in range(2):
            exp = sorted(set(int(i) for i in ws.topk[b, t] if i >= 0))
            assert list(oracle_mod.valid_keys(ws, b, t)) == exp
            assert len(exp) == 9


def test_repeated_topk_position_is_refused(oracle_mod):
    """The indices of one query token are distinct cache positions (a top-k
    selection); a list that names one position twice is outside the
    definition, so both the valid-set query and the decode refuse it instead
    of quietly counting it once or twice.  -1 slots may repeat freely, and a
    position repeated in another query token's list is fine."""
    ws = make_workload("t", 2, 2, 4, [40, 30], seed=23, topk=12, topk_pad_count=3)
    rows = [(b, t, h) for b in range(2) for t in range(2) for h in range(4)]
    oracle_mod.decode_rows(ws, rows)                 # distinct: accepted
    assert (ws.topk[0, 0] == -1).sum() == 3          # -1 repeats within a list
    ws.topk[0, 1] = ws.topk[0, 0]                    # same positions, other token
    oracle_mod.decode_rows(ws, rows)
    valid = ws.topk[1, 1][ws.topk[1, 1] >= 0]
    ws.topk[1, 1, int(np.argmax(ws.topk[1, 1] >= 0)) ] = valid[-1]  # a repeat
    with pytest.raises(ValueError, match="repeats a position"):
        oracle_mod.valid_keys(ws, 1, 1)
    with pytest.raises(ValueError, match="repeats a position"):
        oracle_mod.decode_rows(ws, rows)
    assert list(oracle_mod.valid_keys(ws, 1, 0)) == sorted(int(i) for i in ws.topk[1, 0] if i >= 0)


def test_golden_regression(oracle_mod):
    """The oracle's result on the tiny dense workload, as recorded by
    tests/golden/make_golden.py (a regression record, not a pin)."""
    import json
    import os
    with open(os.path.join(os.path.dirname(__file__), "golden", "tiny_dense_oracle.json")) as f:
        rec = json.load(f)
    w = workloads.config(1)
    out, lse = oracle_mod.decode_all(w)
    np.testing.assert_allclose(lse[:, :, 0], np.array(rec["lse"]), atol=1e-12, rtol=0)
    for key, vals in rec["o_rows"].items():
        b, h = map(int, key.split(","))
        np.testing.assert_allclose(out[b, 0, h, :8], vals, atol=1e-14, rtol=0)
    assert abs(abs(out).sum() - rec["o_abs_sum"]) < 1e-9

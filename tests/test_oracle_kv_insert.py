"""Pins of the KV insert oracle (oracle/kv_insert.py) to facts outside it:
the rounding definitions checked by exact rational arithmetic and against
torch's own casts, closed forms of RMSNorm, and the layout rules of the
insert (vLLM kimi_k3 specialized-decode ``mla.query`` page, MlaQuery.insert)."""
import math
import os
import sys
from fractions import Fraction

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from oracle import kv_insert as K  # noqa: E402
import workloads as W  # noqa: E402


def bf16(x):
    return K.f64_to_bf16_bits(np.asarray(x, dtype=np.float64))


def bf16_val(bits):
    return K.bf16_bits_to_f64(bits)


# --- float -> bf16 -------------------------------------------------------------

def test_bf16_matches_torch_cast_on_float32_values():
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(3.0),
        (rng.standard_normal(5000) * 1e-39).astype(np.float32),      # float32 subnormals
        (rng.standard_normal(5000) * 1e37).astype(np.float32),
        rng.integers(0, 2**32, 20000, dtype=np.uint64).astype(np.uint32).view(np.float32),
    ])
    x = x[np.isfinite(x)]
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = K.f64_to_bf16_bits(x.astype(np.float64))
    np.testing.assert_array_equal(got, want)


def _nearest_even_bf16(v: Fraction) -> int:
    """Brute force: scan the bf16 neighbours of v and keep the nearest, ties to
    the even code."""
    lo = int(np.float32(float(v)).view(np.uint32) >> 16)
    best = None
    for c in range(max(lo - 2, 0), lo + 3):
        for sign in (0, 0x8000):
            code = c | sign
            f = float(bf16_val(np.array([code], np.uint16))[0])
            if not math.isfinite(f):
                continue
            d = abs(Fraction(f) - v)
            key = (d, code & 1)
            if best is None or key < best[0]:
                best = (key, code)
    return best[1]


def test_bf16_from_float64_is_nearest_with_ties_to_even():
    rng = np.random.default_rng(2)
    vals = list(rng.standard_normal(400) * np.exp2(rng.integers(-20, 20, 400)))
    # exact ties between two bf16 neighbours, both parities
    for base in (1.0, 1.0078125, 3.5, 200.0, 2.0 ** -100):
        vals.append(base + base * 2.0 ** -8)
        vals.append(-(base + base * 2.0 ** -8))
    for v in vals:
        got = int(K.f64_to_bf16_bits(np.array([v]))[0])
        assert got == _nearest_even_bf16(Fraction(v)), v


# --- exact sum of squares, rational -> fp32 -------------------------------------

def test_fraction_to_f32_matches_float32_cast_of_doubles():
    """A float64 value is an exact rational, and numpy's float64 -> float32
    cast rounds it correctly: the two must agree everywhere, subnormals and
    overflow included."""
    rng = np.random.default_rng(9)
    vals = np.concatenate([rng.standard_normal(3000) * np.exp2(rng.integers(-160, 130, 3000)),
                           [3.4028235677973366e38, 3.4028235677973366e38 * (1 + 2.0 ** -25), 2.0 ** -150,
                            2.0 ** -150 * 1.5, 1.5 * 2.0 ** -149, 2.0 ** -149]])
    with np.errstate(over="ignore"):
        want = vals.astype(np.float32)
    got = np.array([K.fraction_to_f32(Fraction(v)) for v in vals], dtype=np.float32)
    np.testing.assert_array_equal(got.view(np.uint32), want.view(np.uint32))


def test_fraction_to_f32_ties_to_even_beyond_float64():
    """Ties and near-ties that a float64 intermediate could not hold."""
    one = Fraction(1)
    ulp = Fraction(1, 2 ** 23)
    assert K.fraction_to_f32(one + ulp / 2) == np.float32(1.0)                  # tie -> even
    assert K.fraction_to_f32(one + ulp * 3 / 2) == np.float32(1 + 2.0 ** -22)   # tie -> even
    assert K.fraction_to_f32(one + ulp / 2 + Fraction(1, 2 ** 200)) == np.float32(1 + 2.0 ** -23)
    assert K.fraction_to_f32(one + ulp / 2 - Fraction(1, 2 ** 200)) == np.float32(1.0)
    assert K.fraction_to_f32(-(one + ulp / 2 + Fraction(1, 2 ** 200))) == np.float32(-(1 + 2.0 ** -23))


def test_exact_sum_sq_is_the_correctly_rounded_sum():
    """math.fsum returns the correctly rounded float64 of an exact sum of
    floats; the squares of bf16 values are exact floats."""
    rng = np.random.default_rng(10)
    for k in range(30):
        spread = [0, 10, 40, 120][k % 4]
        x = bf16_val(bf16(rng.standard_normal(512) * np.exp2(rng.uniform(-spread, 0, 512))))
        assert float(K.exact_sum_sq(x)) == math.fsum(v * v for v in x)
    assert K.exact_sum_sq(np.array([3.0, -4.0, 0.0])) == 25
    assert K.exact_sum_sq(np.zeros(4)) == 0


# --- float -> e4m3 -------------------------------------------------------------

FINITE_CODES = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)


def test_e4m3_decode_matches_torch():
    want = torch.from_numpy(FINITE_CODES.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(K.e4m3_bits_to_f64(FINITE_CODES), want)


def test_e4m3_round_trip_of_every_finite_code():
    np.testing.assert_array_equal(K.f64_to_e4m3_bits(K.e4m3_bits_to_f64(FINITE_CODES)), FINITE_CODES)


def test_e4m3_midpoints_round_to_even_and_saturate():
    pos = np.sort(np.unique(K.e4m3_bits_to_f64(FINITE_CODES[FINITE_CODES < 0x80])))
    for a, b in zip(pos[:-1], pos[1:]):
        mid = (a + b) / 2
        ca, cb = K.f64_to_e4m3_bits(np.array([a, b]))
        want = ca if (ca & 1) == 0 else cb
        assert K.f64_to_e4m3_bits(np.array([mid]))[0] == want, (a, b)
        assert K.f64_to_e4m3_bits(np.array([-mid]))[0] == want | 0x80
    assert list(K.f64_to_e4m3_bits(np.array([448.0, 464.0, 465.0, 1e9, -500.0, -1e30]))) == \
        [0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE]
    assert list(K.f64_to_e4m3_bits(np.array([2.0 ** -9, 2.0 ** -10, 2.0 ** -10 * 1.0001, 0.0, -0.0]))) == \
        [0x01, 0x00, 0x01, 0x00, 0x80]


def test_e4m3_matches_torch_cast_inside_range():
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.uniform(-448, 448, 20000), rng.standard_normal(20000) * 0.01,
                        rng.standard_normal(5000) * 2.0 ** -8]).astype(np.float32)
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(K.f64_to_e4m3_bits(x.astype(np.float64)), want)


# --- RMSNorm closed forms ------------------------------------------------------

ONES = bf16(np.ones(512))


def test_constant_row_normalises_to_sign():
    for c in (0.3125, -0.3125, 7.0, -1e-3, 1234.5):
        n = bf16_val(K.rms_norm_row(bf16(np.full(512, c)), ONES, 0.0))
        assert np.all(n == math.copysign(1.0, c)), c


def test_single_spike_is_sqrt_512():
    x = np.zeros(512)
    x[77] = -3.0
    n = bf16_val(K.rms_norm_row(bf16(x), ONES, 0.0))
    assert n[77] == -22.625  # bf16(-sqrt(512)) = -181/128 * 16
    assert np.count_nonzero(n) == 1


def test_power_of_two_scaling_invariance_and_weight_linearity():
    rng = np.random.default_rng(4)
    xb = bf16(rng.standard_normal(512))
    wb = bf16(1 + 0.25 * rng.standard_normal(512))
    n0 = K.rms_norm_row(xb, wb, 0.0)
    for k in (-20, -3, 5, 40):
        xk = bf16(bf16_val(xb) * 2.0 ** k)
        np.testing.assert_array_equal(K.rms_norm_row(xk, wb, 0.0), n0)
    n2 = bf16_val(K.rms_norm_row(xb, bf16(bf16_val(wb) * 2.0), 0.0))
    np.testing.assert_array_equal(n2, 2.0 * bf16_val(n0))


def test_rmsnorm_is_correctly_rounded_exact_value_away_from_ties():
    """n_i is the bf16 nearest to the exact x_i w_i / sqrt(mean) (mean summed
    with rationals), except within 2^-12 bf16 ulp of a rounding tie, where the
    two float32 steps of the definition (r and the product) may decide."""
    rng = np.random.default_rng(5)
    exempt = total = 0
    for trial in range(24):
        scale = 2.0 ** rng.uniform(-8, 6)
        xb = bf16(rng.standard_normal(512) * scale)
        wb = bf16(1 + 0.25 * rng.standard_normal(512))
        eps = [0.0, 1e-6, 0.5][trial % 3]
        x, w = bf16_val(xb), bf16_val(wb)
        S = sum(Fraction(v) ** 2 for v in x)
        mean = S / 512 + Fraction(float(np.float32(eps)))
        exact = x * w / math.sqrt(float(mean))  # float64: error ~2^-52, far below the margin
        got = K.rms_norm_row(xb, wb, eps)
        _, e = np.frexp(exact)
        ulp = np.ldexp(1.0, np.maximum(e - 1, -126) - 7)
        frac = np.abs(exact / ulp) % 1.0
        near_tie = np.abs(frac - 0.5) < 2.0 ** -12
        want = K.f64_to_bf16_bits(exact)
        assert np.array_equal(got[~near_tie], want[~near_tie]), trial
        exempt += int(near_tie.sum())
        total += 512
    assert exempt < total // 200


def test_eps_dominates_small_rows():
    xb = bf16(np.full(512, 1e-3))
    n = bf16_val(K.rms_norm_row(xb, ONES, 100.0))
    want = 1e-3 / math.sqrt(1e-6 + float(np.float32(100.0)))
    assert np.allclose(n, want, rtol=2 ** -8)


def test_all_zero_row_gives_zeros_even_without_eps():
    z = np.zeros(512, np.uint16)
    for eps in (0.0, 1e-6):
        np.testing.assert_array_equal(K.rms_norm_row(z, ONES, eps), z)


# --- row formats ---------------------------------------------------------------

def test_fp8_tile_scales_codes_and_error_bound():
    rng = np.random.default_rng(6)
    xb = bf16(rng.standard_normal(512) * np.repeat([0.01, 1.0, 50.0, 3.0], 128))
    xb[256:384] = bf16(np.zeros(128))  # an all-zero tile
    pe = bf16(rng.standard_normal(64))
    row, sc = K.insert_row(K.FMT_FP8_TILE, xb, pe, ONES, 1e-6)
    assert row.shape == (640,) and sc.dtype == np.float32
    n = bf16_val(K.rms_norm_row(xb, ONES, 1e-6))
    deq = K.e4m3_bits_to_f64(row[:512]) * np.repeat(sc.astype(np.float64), 128)
    for t in range(4):
        tile = n[128 * t:128 * (t + 1)]
        if not tile.any():
            assert sc[t] == 1.0 and not row[128 * t:128 * (t + 1)].any()
            continue
        assert sc[t] == max(np.float32(np.float32(np.abs(tile).max()) / np.float32(448)), np.float32(2.0 ** -126))
        vals = K.e4m3_bits_to_f64(row[128 * t:128 * (t + 1)])
        assert np.abs(vals).max() == 448.0
        d = deq[128 * t:128 * (t + 1)]
        # 3 mantissa bits: half an ulp is 2^-4 relative (normals), 2^-10 * s below 2^-6 * s
        assert np.all(np.abs(d - tile) <= np.maximum(2.0 ** -4 * np.abs(tile), 2.0 ** -10 * sc[t]) * (1 + 1e-6))
    np.testing.assert_array_equal(row[512:].view("<u2"), pe)


def test_extreme_rows_stay_finite_and_follow_the_limits():
    """The generator's edge rows: a 2^172 span (tile scales down to the
    smallest normal), a sum of squares beyond fp32 (r = 0: zeros), a row of
    bf16 subnormals (the sum underflows: r = 1 / sqrt(eps))."""
    inp = W.make_insert_inputs(8, 1, seed=3)
    lat = inp.qkv[:, W.KV_C_COL:W.KV_C_COL + 512]
    pe = inp.qkv[:, W.K_PE_COL:W.K_PE_COL + 64]
    for r in (4, 5, 6):
        row, sc = K.insert_row(K.FMT_FP8_TILE, lat[r], pe[r], inp.w_kva, inp.eps)
        assert np.all((row[:512] & 0x7F) != 0x7F), r  # no NaN code
        assert np.all(np.isfinite(sc)) and np.all(sc >= 2.0 ** -126), r
    assert np.isinf(K.fraction_to_f32(K.exact_sum_sq(bf16_val(lat[5]))))
    assert not bf16_val(K.rms_norm_row(lat[5], inp.w_kva, inp.eps)).any()  # +-0
    assert K.fraction_to_f32(K.exact_sum_sq(bf16_val(lat[6]))) == 0
    n6 = bf16_val(K.rms_norm_row(lat[6], ONES, inp.eps))
    r6 = np.float32(1) / np.sqrt(np.float32(inp.eps))
    np.testing.assert_array_equal(n6, bf16_val(bf16((bf16_val(lat[6]).astype(np.float32) * r6).astype(np.float64))))
    _, sc4 = K.insert_row(K.FMT_FP8_TILE, lat[4], pe[4], inp.w_kva, inp.eps)
    assert sc4[3] == np.float32(2.0 ** -126)


def test_fp8_tensor_codes_with_unit_and_power_of_two_scale():
    rng = np.random.default_rng(7)
    xb = bf16(rng.standard_normal(512))
    pe = bf16(rng.standard_normal(64))
    n = bf16_val(K.rms_norm_row(xb, ONES, 0.0))
    allv = np.concatenate([n, bf16_val(pe)])
    row1, _ = K.insert_row(K.FMT_FP8_TENSOR, xb, pe, ONES, 0.0, ksi=1.0)
    np.testing.assert_array_equal(row1, K.f64_to_e4m3_bits(allv))
    row8, _ = K.insert_row(K.FMT_FP8_TENSOR, xb, pe, ONES, 0.0, ksi=8.0)
    np.testing.assert_array_equal(row8, K.f64_to_e4m3_bits(allv * 8.0))


def test_bf16_row_layout():
    rng = np.random.default_rng(8)
    xb = bf16(rng.standard_normal(512))
    pe = bf16(rng.standard_normal(64))
    row, sc = K.insert_row(K.FMT_BF16, xb, pe, ONES, 1e-6)
    assert sc is None and row.shape == (1152,)
    u = row.view("<u2")
    np.testing.assert_array_equal(u[:512], K.rms_norm_row(xb, ONES, 1e-6))
    np.testing.assert_array_equal(u[512:], pe)


def test_slots_map_to_page_and_offset_and_skip():
    inp = W.make_insert_inputs(40, 3, page_size=16, seed=11)
    slots = inp.slots.copy()
    slots[5] = 3 * 16        # one past the end: bad
    slots[6] = -7            # negative other than -1: bad
    cache = np.full((3, 16, 640), 0xAB, np.uint8)
    scales = np.full((3, 16, 4), -1.0, np.float32)
    kv = inp.qkv[:, W.KV_C_COL:]
    pe = inp.qkv[:, W.K_PE_COL:]
    bad = K.kv_insert(K.FMT_FP8_TILE, kv, pe, inp.w_kva, inp.eps, slots, cache, scales)
    assert bad == 2
    written = set()
    for j, s in enumerate(slots):
        if 0 <= s < 48:
            p, o = divmod(int(s), 16)
            row, sc = K.insert_row(K.FMT_FP8_TILE, kv[j, :512], pe[j, :64], inp.w_kva, inp.eps)
            np.testing.assert_array_equal(cache[p, o], row)
            np.testing.assert_array_equal(scales[p, o], sc)
            written.add(int(s))
    for s in range(48):
        if s not in written:
            p, o = divmod(s, 16)
            assert np.all(cache[p, o] == 0xAB) and np.all(scales[p, o] == -1.0)


def test_generator_special_rows():
    inp = W.make_insert_inputs(8, 2, seed=3)
    lat = inp.qkv[:, W.KV_C_COL:W.KV_C_COL + 512]
    assert not lat[0].any()
    assert not lat[2, 128:256].any()
    assert np.all(lat[3] == lat[3, 0])
    assert len(set(inp.slots[inp.slots >= 0].tolist())) == int((inp.slots >= 0).sum())

"""Three arithmetic shortcuts of the KV insert kernel, checked on the CPU.

1. FP8 tile scales.  For a tile maximum amax (a bf16 value m * 2^E, m its
   8-bit significand) the kernel takes s = max(fp32(amax / 448), 2^-126) and
   1 / s from tables of fp32(m / 448) and fp32(1 / fp32(m / 448)), moving
   only the exponent.  That is exact because scaling by a power of two
   commutes with round-to-nearest while the result stays normal; here it is
   checked for every positive finite bf16 amax with IEEE float32 division.

2. The one-window exact sum of squares.  A row whose nonzero bf16 values lie
   within 2^15 of the largest puts every square m^2 * 2^(2e) at bit
   2 (e - e_max) + 31 of one 64-bit integer; the integer is rounded to fp32
   (correctly rounded u64 -> f32, then e added to the exponent when the
   result is normal, else one rounding at the subnormal quantum).  Restated
   here in integer steps and compared with the oracle's exact sum
   (oracle/kv_insert.py) on rows scaled across the whole fp32 range.

3. The packed range check that picks the branch: the largest and the
   smallest nonzero magnitude of a row, two bf16 values per 32-bit word.
"""
import os
import sys
from fractions import Fraction

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from oracle import kv_insert as K  # noqa: E402
import workloads as W  # noqa: E402

F32 = np.float32


def test_tile_scale_tables_match_division_for_every_bf16_amax():
    bits = np.arange(1, 0x7F80, dtype=np.uint32) << 16          # every positive finite bf16
    amax = bits.view(np.float32)
    with np.errstate(all="ignore"):
        sc_ref = np.maximum((amax / F32(448.0)).astype(np.float32), F32(2.0 ** -126))
        inv_ref = (F32(1.0) / sc_ref).astype(np.float32)
        m = np.arange(256, dtype=np.float32)
        sc_tab = (m / F32(448.0)).astype(np.float32).view(np.uint32).astype(np.int64)
        inv_tab = (F32(1.0) / sc_tab.astype(np.uint32).view(np.float32)).astype(np.float32)
    inv_tab = inv_tab.view(np.uint32).astype(np.int64)
    e = (bits >> 23) & 0xFF
    mm = np.where(e == 0, (bits >> 16) & 0x7F, 0x80 | ((bits >> 16) & 0x7F))
    E = np.where(e == 0, -133, e.astype(np.int64) - 134)
    normal = ((sc_tab[mm] >> 23) & 0xFF) + E >= 1
    sc = np.where(normal, sc_tab[mm] + (E << 23), 0x00800000).astype(np.uint32)
    inv = np.where(normal, inv_tab[mm] - (E << 23), 0x7E800000).astype(np.uint32)
    np.testing.assert_array_equal(sc, sc_ref.view(np.uint32))
    np.testing.assert_array_equal(inv, inv_ref.view(np.uint32))
    assert (~normal).sum() > 1000  # the 2^-126 floor is exercised


def _one_window_sum(bits):
    """The kernel's narrow-window branch in integer steps; None when the row
    takes another branch."""
    bits = np.asarray(bits, dtype=np.uint32)
    mag = bits & 0x7FFF
    amax = int(mag.max())
    if amax == 0:
        return np.float32(0.0)
    amin = int(mag[mag != 0].min())
    emax = amax >> 7
    if emax < 32 or (amin >> 7) < emax - 15:
        return None
    base = 31 - 2 * emax
    hi = 0
    for h in bits.tolist():
        s = 2 * ((h >> 7) & 0xFF) + base
        if 0 <= s <= 31:                                            # shl gives 0 outside [0, 31]
            hi += (((h & 0x7F) | 0x80) ** 2) << s
        else:
            assert h & 0x7FFF == 0
    e = 2 * emax - 299                                              # value = hi * 2^e
    f = int(np.float32(K.fraction_to_f32(Fraction(hi))).view(np.uint32))
    re = (f >> 23) + e
    if re >= 255:
        return np.float32(np.inf)
    if re >= 1:
        return np.uint32((f + (e << 23)) & 0xFFFFFFFF).view(np.float32)
    return K.fraction_to_f32(Fraction(hi) * Fraction(2) ** e)


def test_one_window_sum_of_squares_matches_exact_rounding():
    rng = np.random.default_rng(11)
    inp = W.make_insert_inputs(200, 8, seed=12)
    rows = [inp.qkv[i, W.KV_C_COL:W.KV_C_COL + 512] for i in range(inp.N)]
    for k in range(160):                                            # fp32-range scalings: underflow to overflow
        x = (rng.standard_normal(512) * 2.0 ** rng.uniform(-140, 125)).astype(np.float32)
        rows.append((x.view(np.uint32) >> 16).astype(np.uint16))
    taken = 0
    for r in rows:
        got = _one_window_sum(r)
        if got is None:
            continue
        taken += 1
        want = K.fraction_to_f32(K.exact_sum_sq(K.bf16_bits_to_f64(r)))
        assert np.float32(got).view(np.uint32) == np.float32(want).view(np.uint32)
    assert taken > 300


def test_packed_smallest_nonzero_magnitude():
    """The range check reads two bf16 values per 32-bit word: with bit 15
    set in both halves, subtracting 0x00010001 never borrows across them, so
    per half ((w | 0x80008000) - 0x00010001) & 0x7FFF7FFF is magnitude - 1
    for a nonzero value and 0x7FFF for a zero; the minimum over the row plus
    one is the smallest nonzero magnitude (0x8000 when every value is zero)."""
    rng = np.random.default_rng(3)
    for trial in range(200):
        n = 16
        halves = rng.integers(0, 1 << 16, size=2 * n, dtype=np.uint32)
        halves[rng.random(2 * n) < 0.3] &= 0x8000          # zeros of either sign
        if trial % 50 == 0:
            halves &= 0x8000                                 # an all-zero row
        words = halves[0::2] | (halves[1::2] << 16)
        t = (((words | 0x80008000) - 0x00010001) & 0x7FFF7FFF).astype(np.uint32)
        got = int(min((t & 0xFFFF).min(), (t >> 16).min())) + 1
        mags = halves & 0x7FFF
        want = int(mags[mags != 0].min()) if (mags != 0).any() else 0x8000
        assert got == want
        amax = int(max(((words & 0x7FFF7FFF) & 0xFFFF).max(), ((words & 0x7FFF7FFF) >> 16).max()))
        assert amax == int(mags.max())

"""Pins of the query-absorption oracle (oracle/query_absorb.py) to facts
outside it: RMSNorm closed forms over 1536 values, one-hot weights whose
result is known element by element (a transposed operand, a wrong head
offset or swapped no-PE / RoPE rows all break them), power-of-two scaling,
and exact brute-force dot products (vLLM kimi_k3 specialized-decode
``mla.query`` page, MlaQuery)."""
import math
import os
import sys
from fractions import Fraction

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from oracle import kv_insert as K  # noqa: E402
from oracle import query_absorb as Q  # noqa: E402
import workloads as W  # noqa: E402


def bf16(x):
    return K.f64_to_bf16_bits(np.asarray(x, dtype=np.float64))


def val(bits):
    return K.bf16_bits_to_f64(bits)


ONES = bf16(np.ones(Q.D_QA))


def test_rmsnorm_constant_row_and_spike():
    for c in (0.375, -2.5, 1e-3):
        assert np.all(val(Q.rms_norm_qa(bf16(np.full(Q.D_QA, c)), ONES, 0.0)) == math.copysign(1.0, c))
    x = np.zeros(Q.D_QA)
    x[1000] = 5.0
    n = val(Q.rms_norm_qa(bf16(x), ONES, 0.0))
    assert n[1000] == 39.25  # bf16(sqrt(1536)) = 39.19... -> 39.25
    assert np.count_nonzero(n) == 1


def test_rmsnorm_power_of_two_invariance_and_eps():
    rng = np.random.default_rng(1)
    xb = bf16(rng.standard_normal(Q.D_QA))
    wb = bf16(1 + 0.25 * rng.standard_normal(Q.D_QA))
    n0 = Q.rms_norm_qa(xb, wb, 0.0)
    for k in (-30, 7):
        np.testing.assert_array_equal(Q.rms_norm_qa(bf16(val(xb) * 2.0 ** k), wb, 0.0), n0)
    small = bf16(np.full(Q.D_QA, 1e-3))
    assert np.allclose(val(Q.rms_norm_qa(small, ONES, 4.0)), 1e-3 / 2.0, rtol=2 ** -8)


def test_rmsnorm_is_correctly_rounded_exact_value_away_from_ties():
    """xq_i is the bf16 nearest to the exact x_i w_i / sqrt(sum x^2 / 1536 +
    eps), except within 2^-12 bf16 ulp of a rounding tie, where the fp32 steps
    of the definition may decide."""
    rng = np.random.default_rng(3)
    exempt = total = 0
    for trial in range(12):
        xb = bf16(rng.standard_normal(Q.D_QA) * 2.0 ** rng.uniform(-8, 6))
        wb = bf16(1 + 0.25 * rng.standard_normal(Q.D_QA))
        eps = [0.0, 1e-6, 0.25][trial % 3]
        x, w = val(xb), val(wb)
        mean = sum(Fraction(v) ** 2 for v in x) / 1536 + Fraction(float(np.float32(eps)))
        exact = x * w / math.sqrt(float(mean))
        got = Q.rms_norm_qa(xb, wb, eps)
        _, e = np.frexp(exact)
        ulp = np.ldexp(1.0, np.maximum(e - 1, -126) - 7)
        near_tie = np.abs(np.abs(exact / ulp) % 1.0 - 0.5) < 2.0 ** -12
        want = K.f64_to_bf16_bits(exact)
        assert np.array_equal(got[~near_tie], want[~near_tie]), trial
        exempt += int(near_tie.sum())
        total += Q.D_QA
    assert exempt < total // 200


def _onehot_weights(H):
    w_qb = np.zeros((H * Q.QB_ROWS, Q.D_QA))
    src = np.zeros((H, Q.QB_ROWS), dtype=int)
    for h in range(H):
        for p in range(Q.QB_ROWS):
            k = (7 * h + 3 * p + 11) % Q.D_QA
            w_qb[h * Q.QB_ROWS + p, k] = 1.0
            src[h, p] = k
    w_uk = np.zeros((H, Q.D_NOPE, Q.D_LATENT))
    dst = np.zeros((H, Q.D_NOPE), dtype=int)
    for h in range(H):
        for p in range(Q.D_NOPE):
            l = (4 * p + 5 * h + 1) % Q.D_LATENT
            w_uk[h, p, l] = 2.0
            dst[h, p] = l
    return bf16(w_qb), bf16(w_uk), src, dst


def test_onehot_weights_place_every_value():
    H, N = 3, 2
    inp = W.make_query_inputs(N, H, seed=5)
    w_qb, w_uk, src, dst = _onehot_weights(H)
    r = Q.query_absorb(inp.qkv, inp.w_qa, inp.eps, w_qb, w_uk)
    xq = val(r["xq"])
    q = val(r["q"])
    for n in range(N):
        for h in range(H):
            qb = xq[n, src[h]]                                     # Q_B selects
            np.testing.assert_array_equal(val(r["qb"][n, h]), qb)
            lat = np.zeros(Q.D_LATENT)
            lat[dst[h]] = 2.0 * qb[:Q.D_NOPE]                      # W_UK scatters x 2
            np.testing.assert_array_equal(q[n, h, :Q.D_LATENT], lat)
            np.testing.assert_array_equal(q[n, h, Q.D_LATENT:], qb[Q.D_NOPE:])  # RoPE rows follow
    # the RMSNorm stage is the row-wise definition
    for n in range(N):
        np.testing.assert_array_equal(r["xq"][n], Q.rms_norm_qa(inp.qkv[n, :Q.D_QA], inp.w_qa, inp.eps))


def test_power_of_two_weight_scaling_commutes():
    inp = W.make_query_inputs(2, 2, seed=6)
    r1 = Q.query_absorb(inp.qkv, inp.w_qa, inp.eps, inp.w_qb, inp.w_uk)
    r2 = Q.query_absorb(inp.qkv, inp.w_qa, inp.eps, bf16(val(inp.w_qb) * 4.0), bf16(val(inp.w_uk) * 0.5))
    np.testing.assert_array_equal(val(r2["qb"]), 4.0 * val(r1["qb"]))
    np.testing.assert_array_equal(val(r2["q"][:, :, :512]), 2.0 * val(r1["q"][:, :, :512]))


def _bf16_of_fraction(v: Fraction) -> float:
    """Nearest bf16 (ties to even) of an exact rational, by scanning the two
    neighbours around the float value."""
    f = float(v)
    lo = int(np.float32(f).view(np.uint32) >> 16)
    best = None
    for c in range(max(lo - 2, 0), lo + 3):
        for s in (0, 0x8000):
            code = c | s
            x = float(val(np.array([code], np.uint16))[0])
            if not math.isfinite(x):
                continue
            key = (abs(Fraction(x) - v), code & 1)
            if best is None or key < best[0]:
                best = (key, x)
    return best[1]


def test_brute_force_dot_products():
    """A few outputs from exact rational dot products, independent of the
    oracle's matrix routines."""
    inp = W.make_query_inputs(2, 2, seed=7)
    r = Q.query_absorb(inp.qkv, inp.w_qa, inp.eps, inp.w_qb, inp.w_uk)
    xq = val(r["xq"])
    wqb = val(inp.w_qb)
    wuk = val(inp.w_uk)
    rng = np.random.default_rng(0)
    for _ in range(6):
        n, h, p = int(rng.integers(2)), int(rng.integers(2)), int(rng.integers(Q.QB_ROWS))
        exact = sum(Fraction(a) * Fraction(b) for a, b in zip(xq[n], wqb[h * Q.QB_ROWS + p]))
        assert val(r["qb"][n, h, p]) == _bf16_of_fraction(exact)
    qb = val(r["qb"])
    for _ in range(6):
        n, h, l = int(rng.integers(2)), int(rng.integers(2)), int(rng.integers(Q.D_LATENT))
        exact = sum(Fraction(qb[n, h, p]) * Fraction(wuk[h, p, l]) for p in range(Q.D_NOPE))
        assert val(r["q"][n, h, l]) == _bf16_of_fraction(exact)

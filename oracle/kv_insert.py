"""KV insert, restated plainly (test infrastructure: only tests/, smoke() and
bench.py's cpu_baseline / reference arm use it).

Source: vLLM kimi_k3 specialized-decode ``mla.query`` page, ``MlaQuery.insert``:
for each new token with a slot >= 0, RMSNorm the 512 latent KV values with the
weight ``w_kva``, round to bf16, and write them with ``k_pe`` into cache row
``[slot // page_size, slot % page_size]``; per-tensor FP8 rows hold
``e4m3(value * k_scale_inv)`` for all 576 values.

Arithmetic (the library's definition, written one value at a time with
numpy; every step after S is one IEEE fp32 operation, ties to even):
  S    = sum_i x_i^2, exact (Python integers), then rounded once to fp32
  mean = fp32(fp32(S * 2^-9) + eps)
  r    = fp32(1 / fp32(sqrt(mean)))    (0 when mean is 0: an all-zero row)
  n_i  = bf16(fp32(fp32(x_i * w_i) * r))
Formats:
  bf16         n (512 bf16) then k_pe (64 bf16)
  fp8 (tile)   per 128-value tile t: s_t = max(fp32(max|n| / 448), 2^-126)
               (1 for an all-zero tile), e4m3(fp32(n_i * fp32(1 / s_t)));
               then k_pe as bf16; scales [page][offset][4]
  fp8 (tensor) e4m3(fp32(n_i * ksi)), e4m3(fp32(pe_i * ksi))

The encoders below (exact rational -> fp32, float -> bf16, float -> OCP FP8
E4M3) are written from
the formats' definitions: round to nearest, ties to even; e4m3 saturates to
+-448 (the format has no infinity; 0x7F / 0xFF are NaN).
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np

D_LATENT = 512
D_ROPE = 64
E4M3_MAX = 448.0

FMT_BF16 = 0
FMT_FP8_TILE = 1
FMT_FP8_TENSOR = 2


def bf16_bits_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> values: a bf16 is the top half of an
    IEEE binary32 word."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def _round_to_quantum(x: np.ndarray, sig_bits: int, min_exp: int) -> np.ndarray:
    """Round finite float64 values to a binary format with ``sig_bits``
    significant bits whose smallest normal is 2**min_exp (gradual underflow
    below it), ties to even.  x / ulp is exact (a power-of-two scaling) and
    np.rint rounds half to even."""
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)  # x = m * 2**e, 0.5 <= |m| < 1: leading bit 2**(e-1)
    e = np.maximum(e - 1, min_exp)  # exponent of the leading bit (or subnormal floor)
    ulp = np.ldexp(1.0, e - (sig_bits - 1))
    return np.rint(x / ulp) * ulp


def f64_to_bf16_bits(x) -> np.ndarray:
    """float64 -> bf16 bits, one rounding (8 significant bits, smallest
    normal 2**-126; overflow -> inf)."""
    x = np.asarray(x, dtype=np.float64)
    r = _round_to_quantum(np.where(np.isfinite(x), x, 0.0), 8, -126)
    r = np.where(np.abs(r) > 3.3895313892515355e38, np.copysign(np.inf, x), r)  # max bf16
    r = np.where(np.isfinite(x), r, x)
    # r is a bf16 value, hence exactly a float32 whose low 16 bits are zero
    # (a NaN keeps only its top half, which stays a NaN: the quiet bit is there).
    return (r.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def f64_to_e4m3_bits(x) -> np.ndarray:
    """float64 -> OCP FP8 E4M3 code, round to nearest even, saturate to
    +-448 (4 significant bits, smallest normal 2**-6, exponent bias 7)."""
    x = np.asarray(x, dtype=np.float64)
    nan = np.isnan(x)
    v = np.where(nan, 0.0, x)
    r = _round_to_quantum(np.clip(v, -E4M3_MAX * 2, E4M3_MAX * 2), 4, -6)
    r = np.clip(r, -E4M3_MAX, E4M3_MAX)
    sign = np.signbit(r).astype(np.uint8) << 7
    a = np.abs(r)
    _, e = np.frexp(a)
    e = e - 1  # a = 1.f * 2**e for normals
    normal = a >= 2.0 ** -6
    exp_field = np.where(normal, e + 7, 0)
    man = np.where(normal, a / np.ldexp(1.0, e) - 1.0, a / 2.0 ** -6) * 8.0
    code = (exp_field.astype(np.int64) << 3) | man.astype(np.int64)
    code = np.where(a == 0.0, 0, code)
    out = (sign | code.astype(np.uint8)).astype(np.uint8)
    return np.where(nan, np.uint8(0x7F) | (np.signbit(x).astype(np.uint8) << 7), out).astype(np.uint8)


def e4m3_bits_to_f64(code) -> np.ndarray:
    """OCP FP8 E4M3 code -> value (0x7F / 0xFF are NaN)."""
    c = np.asarray(code, dtype=np.uint8).astype(np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    v = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.ldexp(1.0, e - 7))
    v = np.where((e == 0xF) & (m == 0x7), np.nan, v)
    return s * v


def fraction_to_f32(v: Fraction) -> np.float32:
    """Exact rational -> the nearest binary32 (24 significant bits, smallest
    subnormal 2^-149, ties to even; overflow -> inf).  Python's round() of a
    Fraction rounds half to even."""
    if v == 0:
        return np.float32(0.0)
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()  # 2^e <= a < 2^(e+1), after the fix-up
    if a < Fraction(2) ** e:
        e -= 1
    q = max(e - 23, -149)
    n = round(a / Fraction(2) ** q)
    mag = float(n) * 2.0 ** q  # exact in float64: n <= 2^24, q >= -149
    if mag >= 2.0 ** 128:
        mag = math.inf
    return np.float32(math.copysign(mag, v))


def exact_sum_sq(x: np.ndarray) -> Fraction:
    """sum x_i^2 of float64 values, exact: x = num / den with den a power of
    two, so the sum is an integer over the largest den^2."""
    ratios = [float(v).as_integer_ratio() for v in x if v != 0.0]
    if not ratios:
        return Fraction(0)
    D = max(d for _, d in ratios) ** 2
    return Fraction(sum(n * n * (D // (d * d)) for n, d in ratios), D)


def f32(x) -> np.ndarray:
    """Round float64 values to binary32 (numpy's cast is IEEE, to nearest even)."""
    return np.asarray(x, dtype=np.float64).astype(np.float32)


def rms_norm_row(x_bits: np.ndarray, w_bits: np.ndarray, eps: float) -> np.ndarray:
    """One latent row (bf16 bits [512]) -> n (bf16 bits [512])."""
    x = bf16_bits_to_f64(x_bits)
    w = bf16_bits_to_f64(w_bits)
    S = fraction_to_f32(exact_sum_sq(x))
    mean = np.float32(S * np.float32(1.0 / D_LATENT)) + np.float32(eps)
    with np.errstate(divide="ignore", over="ignore"):
        r = np.float32(1.0) / np.sqrt(mean) if mean > 0 else np.float32(0.0)
    xw = f32(x) * f32(w)                  # float32 product (exact for bf16 inputs)
    v = (xw * r).astype(np.float64)       # float32 product, correctly rounded
    return f64_to_bf16_bits(v)


def insert_row(fmt: int, x_bits, pe_bits, w_bits, eps: float, ksi: float = 1.0):
    """The cache row bytes (and, for the tile format, its 4 scales) that one
    token writes."""
    n_bits = rms_norm_row(x_bits, w_bits, eps)
    pe_bits = np.asarray(pe_bits, dtype=np.uint16)
    if fmt == FMT_BF16:
        row = np.concatenate([n_bits, pe_bits]).astype("<u2").view(np.uint8)
        return row, None
    n = bf16_bits_to_f64(n_bits)
    if fmt == FMT_FP8_TILE:
        codes = np.empty(D_LATENT, dtype=np.uint8)
        scales = np.empty(4, dtype=np.float32)
        for t in range(4):
            tile = n[128 * t:128 * (t + 1)]
            amax = np.float32(np.max(np.abs(tile)))
            s_t = max(np.float32(amax / np.float32(E4M3_MAX)), np.float32(2.0 ** -126)) if amax > 0 else np.float32(1.0)
            scales[t] = s_t
            inv = np.float32(1.0) / s_t
            q = (f32(tile) * inv).astype(np.float64)  # float32 product, correctly rounded
            codes[128 * t:128 * (t + 1)] = f64_to_e4m3_bits(q)
        row = np.concatenate([codes, pe_bits.astype("<u2").view(np.uint8)])
        return row, scales
    if fmt == FMT_FP8_TENSOR:
        k = np.float32(ksi)
        pe = bf16_bits_to_f64(pe_bits)
        codes = f64_to_e4m3_bits((f32(np.concatenate([n, pe])) * k).astype(np.float64))
        return codes.astype(np.uint8), None
    raise ValueError(f"unknown format {fmt}")


ROW_BYTES = {FMT_BF16: 1152, FMT_FP8_TILE: 640, FMT_FP8_TENSOR: 576}


def kv_insert(fmt: int, kv_c_bits: np.ndarray, k_pe_bits: np.ndarray, w_bits: np.ndarray,
              eps: float, slots: np.ndarray, cache: np.ndarray, scales=None, ksi: float = 1.0):
    """Apply the insert of N tokens to ``cache`` (uint8 [pages, page_size,
    row bytes], updated in place) and ``scales`` (float32 [pages, page_size, 4]
    for the tile format).  kv_c_bits [N, >=512] and k_pe_bits [N, >=64] are
    bf16 bit patterns (only the first 512 / 64 columns are read).  Returns the
    number of slots that were neither -1 nor inside the cache."""
    pages, page_size, rb = cache.shape
    if rb != ROW_BYTES[fmt]:
        raise ValueError("cache row size does not match the format")
    bad = 0
    for j, slot in enumerate(np.asarray(slots, dtype=np.int64)):
        slot = int(slot)
        if slot < 0 or slot >= pages * page_size:
            bad += int(slot != -1)
            continue
        page, off = slot // page_size, slot % page_size
        row, sc = insert_row(fmt, kv_c_bits[j, :D_LATENT], k_pe_bits[j, :D_ROPE], w_bits, eps, ksi)
        cache[page, off, :] = row
        if sc is not None:
            scales[page, off, :] = sc
    return bad

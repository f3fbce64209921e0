"""Query absorption, restated plainly (test infrastructure: only tests/,
smoke() and bench.py's cpu_baseline / reference arm use it).

Source: vLLM kimi_k3 specialized-decode ``mla.query`` page, ``MlaQuery``
(the small-batch ``kernel`` and the wide ``tiled`` form compute the same
thing): the query part of the fused projection row is RMSNorm-ed with
``w_qa`` and rounded to bf16; ``W_QB`` maps it to 192 rows per head (128
no-PE rows, then 64 RoPE rows), each rounded to bf16; the no-PE rows of a
head go through that head's ``W_UK`` (128 x 512) to the 512 latent columns,
rounded to bf16; the RoPE rows follow them, so each head's query row has the
576 values the decode reads.

Arithmetic: the RMSNorm as this library defines it (the KV insert's, over
1536 values: exact sum of squares rounded once to fp32, mean =
fp32(fp32(S / 1536) + eps), r = fp32(1 / fp32(sqrt(mean))), xq =
bf16(fp32(fp32(x * w) * r))); each dot product is taken in float64 (every
product of two bf16 values is exact in float64) and rounded to bf16 once.
"""
from __future__ import annotations

import numpy as np

from .kv_insert import bf16_bits_to_f64, exact_sum_sq, f32, f64_to_bf16_bits, fraction_to_f32

D_QA = 1536
QB_ROWS = 192
D_NOPE = 128
D_LATENT = 512


def rms_norm_qa(x_bits: np.ndarray, w_bits: np.ndarray, eps: float) -> np.ndarray:
    """One q_a row (bf16 bits [1536]) -> xq (bf16 bits [1536])."""
    x = bf16_bits_to_f64(x_bits)
    w = bf16_bits_to_f64(w_bits)
    S = fraction_to_f32(exact_sum_sq(x))
    mean = np.float32(S / np.float32(D_QA)) + np.float32(eps)
    with np.errstate(divide="ignore", over="ignore"):
        r = np.float32(1.0) / np.sqrt(mean) if mean > 0 else np.float32(0.0)
    return f64_to_bf16_bits(((f32(x) * f32(w)) * r).astype(np.float64))


def q_b(xq_bits: np.ndarray, w_qb_bits: np.ndarray, H: int):
    """xq bits [N, 1536], W_QB bits [H*192, 1536] -> (qb bits [N, H, 192],
    sum of |products| [N, H, 192] for the accumulation bound)."""
    x = bf16_bits_to_f64(xq_bits)
    w = bf16_bits_to_f64(w_qb_bits)
    dot = x @ w.T
    mag = np.abs(x) @ np.abs(w).T
    N = x.shape[0]
    return f64_to_bf16_bits(dot).reshape(N, H, QB_ROWS), mag.reshape(N, H, QB_ROWS)


def w_uk_latent(qb_bits: np.ndarray, w_uk_bits: np.ndarray):
    """qb bits [N, H, 192], W_UK bits [H, 128, 512] -> (latent bits
    [N, H, 512], sum of |products| [N, H, 512])."""
    qn = bf16_bits_to_f64(qb_bits[:, :, :D_NOPE])
    w = bf16_bits_to_f64(w_uk_bits)
    # per head h: [N, 128] @ [128, 512]
    dot = np.matmul(qn.transpose(1, 0, 2), w).transpose(1, 0, 2)
    mag = np.matmul(np.abs(qn).transpose(1, 0, 2), np.abs(w)).transpose(1, 0, 2)
    return f64_to_bf16_bits(dot), mag


def query_absorb(q_a_bits: np.ndarray, w_qa_bits: np.ndarray, eps: float, w_qb_bits: np.ndarray,
                 w_uk_bits: np.ndarray) -> dict:
    """All stages for N tokens: q_a bits [N, >=1536] (columns 0..1535 read).
    Returns bf16 bits of xq [N, 1536], qb [N, H, 192] and q [N, H, 576], and
    the two magnitude sums."""
    H = w_uk_bits.shape[0]
    xq = np.stack([rms_norm_qa(row[:D_QA], w_qa_bits, eps) for row in q_a_bits])
    qb, qb_mag = q_b(xq, w_qb_bits, H)
    lat, lat_mag = w_uk_latent(qb, w_uk_bits)
    q = np.concatenate([lat, qb[:, :, D_NOPE:]], axis=2)
    return dict(xq=xq, qb=qb, q=q, qb_mag=qb_mag, lat_mag=lat_mag)

"""Seeded synthetic inputs for MLA decode.

This module only draws random numbers and lays them out in the byte formats
the decode path consumes.  It holds none of the attention arithmetic, so both
the float64 oracle (``oracle/``) and the CUDA path read the very same inputs
without sharing any code that computes the result.

Shapes follow the workloads the source pages discuss: one compressed latent KV
row of 576 values per token (512 no-RoPE latent + 64 RoPE, FlashMLA issue #169,
the ``D_NOPE``/``D_ROPE`` blocks of the quoted kernel), 64 or 128 query heads
sharing it (STAGE_D2.md, "DSV4 is MQA"), 64-token pages addressed by a block
table, and a paged slot ``page = slot // page_size`` (vLLM MlaQuery.insert).

Generation order inside one workload (all from one numpy ``SeedSequence``
with ``seed``; big arrays in seeded chunks): cache_seqlens, block_table, q, KV pool, fp8 scales, top-k.

Formats (all little-endian, raw bits):
  q            uint16 bf16 bits  [B, T, H, 576]
  kv (bf16)    uint16 bf16 bits  [num_pages, 64, 576]
  kv (fp8)     uint8             [num_pages, 64, 640]: bytes 0..511 are e4m3
               no-RoPE latent, bytes 512..639 are the 64 bf16 RoPE values
  kv_scales    float32           [num_pages, 64, 4]: one scale per 128-wide
               tile of the no-RoPE latent; the dequantised value is
               e4m3(byte) * scale
  kv (per-tensor fp8)  uint8     [num_pages, 64, 576]: all 576 values e4m3,
               with kv_scales float32 [1], value = e4m3(byte) * scale
  block_table  int32             [B, max_pages]
  cache_seqlens int32            [B]
  topk         int32             [B, T, topk] token positions within the
               sequence, -1 for an unused slot
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np
import torch

D_QK = 576
D_V = 512
D_ROPE = 64
PAGE = 64
FP8_ROW_BYTES = 640
KV_BF16 = 0
KV_FP8 = 1
KV_FP8_TENSOR = 2     # 576 e4m3 bytes per row (RoPE included), one scale for the whole cache


@dataclasses.dataclass
class Workload:
    name: str
    B: int
    T: int
    H: int
    q: np.ndarray                 # uint16 [B,T,H,576]
    kv: np.ndarray                # uint16 [P,64,576] or uint8 [P,64,640]
    kv_format: int                # KV_BF16 | KV_FP8
    kv_scales: Optional[np.ndarray]
    block_table: np.ndarray       # int32 [B, max_pages]
    cache_seqlens: np.ndarray     # int32 [B]
    topk: Optional[np.ndarray]    # int32 [B,T,k] or None
    softmax_scale: float
    causal: bool
    seed: int

    @property
    def num_pages(self) -> int:
        return int(self.kv.shape[0])

    @property
    def topk_len(self) -> int:
        return 0 if self.topk is None else int(self.topk.shape[2])

    @property
    def max_pages(self) -> int:
        return int(self.block_table.shape[1])


_CHUNK = 1 << 24
_POOL = None


def _pool():
    global _POOL
    if _POOL is None:
        import concurrent.futures
        import os
        _POOL = concurrent.futures.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1))
    return _POOL


class _Rng:
    """One seeded stream of draws.  Large arrays are split into fixed 16M-value
    chunks, each with its own child seed, and drawn on a thread pool; the
    values depend only on the seed and the order of calls."""

    def __init__(self, seed: int):
        self.ss = np.random.SeedSequence(seed)
        self.g = np.random.Generator(np.random.PCG64(self.ss.spawn(1)[0]))

    def integers(self, lo, hi, size=None):
        return self.g.integers(lo, hi, size=size)

    def permutation(self, n):
        return self.g.permutation(n)

    def uniform(self, lo, hi, size):
        return self.g.uniform(lo, hi, size=size)

    def normal_f32(self, n: int, std: float) -> np.ndarray:
        out = np.empty(n, dtype=np.float32)
        starts = list(range(0, n, _CHUNK))
        kids = self.ss.spawn(len(starts))

        def fill(i):
            s = starts[i]
            e = min(n, s + _CHUNK)
            gi = np.random.Generator(np.random.PCG64(kids[i]))
            gi.standard_normal(e - s, dtype=np.float32, out=out[s:e])
            out[s:e] *= np.float32(std)

        list(_pool().map(fill, range(len(starts))))
        return out

    def bytes_u8(self, n: int) -> np.ndarray:
        out = np.empty(n, dtype=np.uint8)
        starts = list(range(0, n, _CHUNK * 4))
        kids = self.ss.spawn(len(starts))

        def fill(i):
            s = starts[i]
            e = min(n, s + _CHUNK * 4)
            gi = np.random.Generator(np.random.PCG64(kids[i]))
            out[s:e] = gi.integers(0, 256, size=e - s, dtype=np.uint8)

        list(_pool().map(fill, range(len(starts))))
        return out


def _round_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bits, round to nearest even (the inputs are finite)."""
    v = x.view(np.uint32)
    v = v + (np.uint32(0x7FFF) + ((v >> np.uint32(16)) & np.uint32(1)))
    return (v >> np.uint32(16)).astype(np.uint16)


def _bf16_normal(g: "_Rng", shape, std: float = 0.5) -> np.ndarray:
    """N(0,1)*std rounded to bf16, returned as raw uint16 bits."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    starts = list(range(0, n, _CHUNK))
    kids = g.ss.spawn(len(starts))

    def fill(i):
        s = starts[i]
        e = min(n, s + _CHUNK)
        gi = np.random.Generator(np.random.PCG64(kids[i]))
        x = gi.standard_normal(e - s, dtype=np.float32)
        x *= np.float32(std)
        out[s:e] = _round_bf16_bits(x)

    list(_pool().map(fill, range(len(starts))))
    return out.reshape(shape)


def _to_e4m3_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> OCP e4m3 bits, rounded by torch's float8_e4m3fn cast."""
    b = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    if np.any((b & 0x7F) == 0x7F):
        raise ValueError("e4m3 NaN code generated")
    return b


def make_workload(
    name: str,
    B: int,
    T: int,
    H: int,
    seqlens: Sequence[int] | str,
    *,
    seed: int,
    num_pages: Optional[int] = None,
    identity_pages: bool = False,
    topk: int = 0,
    topk_pad_frac: float = 0.0,
    topk_pad_count: Optional[int] = None,
    fp8: bool = False,
    fp8_tensor: bool = False,
    causal: bool = False,
    softmax_scale: float = 1.0 / math.sqrt(192.0),
    seqlen_range: tuple = (1024, 32768),
    value_std: float = 0.5,
) -> Workload:
    """Build one seeded workload.

    seqlens: a list of B lengths, or "uniform" (each drawn from
    ``randint(lo, hi+1)`` with ``seqlen_range = (lo, hi)``).
    num_pages: pool size; default = the pages the sequences need.
    identity_pages: block_table[b, j] = b * pages_per_seq + j (unpaged cache).
    topk: indices per query token; they are distinct positions in [0, s_k[b]).
    """
    g = _Rng(seed)
    if isinstance(seqlens, str):
        assert seqlens == "uniform"
        lo, hi = seqlen_range
        sk = g.integers(lo, hi + 1, size=B).astype(np.int32)
    else:
        sk = np.asarray(seqlens, dtype=np.int32)
        assert sk.shape == (B,)
    pages_per = [max(1, -(-int(s) // PAGE)) for s in sk]
    max_pages = max(pages_per)
    need = int(sum(pages_per))
    if num_pages is None:
        num_pages = B * max_pages if identity_pages else need
    assert num_pages >= need, "pool too small"
    bt = np.full((B, max_pages), -1, dtype=np.int32)
    if identity_pages:
        assert num_pages >= B * max_pages
        for b in range(B):
            bt[b, :] = np.arange(b * max_pages, (b + 1) * max_pages, dtype=np.int32)
    else:
        perm = g.permutation(num_pages).astype(np.int32)
        off = 0
        for b in range(B):
            bt[b, : pages_per[b]] = perm[off: off + pages_per[b]]
            off += pages_per[b]
    q = _bf16_normal(g, (B, T, H, D_QK), value_std)

    scales = None
    topk_arr = None
    if topk:
        topk_arr = np.empty((B, T, topk), dtype=np.int32)
        n_pad = topk_pad_count if topk_pad_count is not None else int(round(topk_pad_frac * topk))
        for b in range(B):
            for t in range(T):
                assert topk <= int(sk[b]), "top-k longer than the sequence"
                idx = g.permutation(int(sk[b]))[:topk].astype(np.int32)
                if n_pad:
                    pos = g.permutation(topk)[:n_pad]
                    idx[pos] = -1
                topk_arr[b, t] = idx

    if fp8_tensor:
        # per-tensor FP8 rows (the layout of vLLM's MlaQuery.insert): every
        # value, RoPE included, is e4m3(x / scale) for one scale
        fmt = KV_FP8_TENSOR
        scale = np.float32(g.uniform(0.5, 2.0, 1)[0])
        x = g.normal_f32(num_pages * PAGE * D_QK, value_std).reshape(num_pages, PAGE, D_QK)
        kv = _to_e4m3_bits(x / scale).reshape(num_pages, PAGE, D_QK)
        scales = np.array([scale], dtype=np.float32)
    elif not fp8:
        kv = _bf16_normal(g, (num_pages, PAGE, D_QK), value_std)
        fmt = KV_BF16
    else:
        fmt = KV_FP8
        kv = np.empty((num_pages, PAGE, FP8_ROW_BYTES), dtype=np.uint8)
        scales = g.uniform(0.5, 2.0, (num_pages, PAGE, 4)).astype(np.float32)
        if topk_arr is None:
            # dense fp8 cache: every row drawn from the stated distribution
            x = g.normal_f32(num_pages * PAGE * D_V, value_std).reshape(num_pages, PAGE, 4, 128)
            kv[:, :, :D_V] = _to_e4m3_bits(x / scales[..., None]).reshape(num_pages, PAGE, D_V)
            kv[:, :, D_V:] = _bf16_normal(g, (num_pages, PAGE, D_ROPE), value_std).view(np.uint8).reshape(num_pages, PAGE, 2 * D_ROPE)
        else:
            # Rows no top-k index names are never read by the method: they get
            # random finite filler (e4m3 codes with exponent <= 14, bf16 RoPE
            # with |v| < 2); the named rows get the stated distribution.
            kv.reshape(-1)[:] = g.bytes_u8(kv.size)
            kv[:, :, :D_V] &= 0x77
            rope16 = kv[:, :, D_V:].view(np.uint16)
            rope16 &= 0xBFFF
            rows = set()
            for b in range(B):
                for t in range(T):
                    for n in topk_arr[b, t]:
                        if n >= 0:
                            rows.add((b, int(n)))
            rows = sorted(rows)
            if rows:
                pg = np.array([bt[b, n // PAGE] for b, n in rows], dtype=np.int64)
                sl = np.array([n % PAGE for b, n in rows], dtype=np.int64)
                x = g.normal_f32(len(rows) * D_V, value_std).reshape(len(rows), 4, 128)
                kv[pg, sl, :D_V] = _to_e4m3_bits(x / scales[pg, sl][..., None]).reshape(len(rows), D_V)
                kv[pg, sl, D_V:] = _bf16_normal(g, (len(rows), D_ROPE), value_std).view(np.uint8).reshape(len(rows), 2 * D_ROPE)

    return Workload(name=name, B=B, T=T, H=H, q=q, kv=kv, kv_format=fmt,
                    kv_scales=scales, block_table=bt, cache_seqlens=sk,
                    topk=topk_arr, softmax_scale=float(softmax_scale),
                    causal=bool(causal), seed=seed)


# --- the five named workloads -------------------------------------------------

CONFIG_NAMES = (
    "tiny_dense_b2_h64_s256",
    "paged_dense_b16_h128_s4096",
    "varlen_split_b64_h128",
    "sparse_fp8_b32_h64_topk2048",
    "multitoken_causal_b32_t4_h64_s16384",
)


def config(i: int) -> Workload:
    """Workload i (1-based) with seed 1000 + i."""
    seed = 1000 + i
    if i == 1:
        # unpaged [2, 256, 576] cache fed as 4 pages per sequence
        return make_workload(CONFIG_NAMES[0], 2, 1, 64, [256, 256], seed=seed,
                             identity_pages=True, num_pages=8)
    if i == 2:
        return make_workload(CONFIG_NAMES[1], 16, 1, 128, [4096] * 16, seed=seed,
                             num_pages=1024)
    if i == 3:
        return make_workload(CONFIG_NAMES[2], 64, 1, 128, "uniform", seed=seed,
                             seqlen_range=(1024, 32768))
    if i == 4:
        return make_workload(CONFIG_NAMES[3], 32, 1, 64, [65536] * 32, seed=seed,
                             num_pages=32768, topk=2048, topk_pad_count=102,
                             fp8=True)
    if i == 5:
        return make_workload(CONFIG_NAMES[4], 32, 4, 64, [16384] * 32, seed=seed,
                             num_pages=8192, causal=True)
    raise ValueError(i)


# --- KV insert inputs ---------------------------------------------------------

QKV_COLS = 2112     # fused projection row: q_a (1536) | latent KV (512) | k_pe (64)
KV_C_COL = 1536
K_PE_COL = 2048


@dataclasses.dataclass
class InsertInputs:
    qkv: np.ndarray      # uint16 bf16 bits [N, 2112]
    w_kva: np.ndarray    # uint16 bf16 bits [512]
    slots: np.ndarray    # int64 [N], -1 = skip
    num_pages: int
    page_size: int
    eps: float
    k_scale_inv: float

    @property
    def N(self) -> int:
        return self.qkv.shape[0]


def make_insert_inputs(N: int, num_pages: int, page_size: int = PAGE, *, seed: int,
                       skip_every: int = 9, eps: float = 1e-6,
                       k_scale_inv: float = 0.75) -> InsertInputs:
    """New-token rows for the cache insert, laid out like the fused projection
    output the insert reads (latent KV at columns 1536..2047, k_pe at
    2048..2111).  Each token's latent row has its own scale (log-uniform over
    2^-6 .. 2^3) so the normalisation matters; w_kva ~ 1 + 0.25 N(0,1).  Slots
    are distinct, drawn without replacement from the whole cache, with every
    ``skip_every``-th token set to -1.  When N >= 4 the first rows are special
    cases: row 0 all zeros, row 1 one large outlier, row 2 with its second
    128-value tile all zeros, row 3 constant; when N >= 8 also row 4 spanning
    2^40 down to bf16 subnormals, row 5 with a sum of squares beyond fp32
    (2^60 values) and row 6 of bf16 subnormals only."""
    g = _Rng(seed)
    scale = np.exp2(g.uniform(-6.0, 3.0, N)).astype(np.float32)
    lat = _bf16_normal(g, (N, D_V), std=1.0)
    lat_f = (lat.astype(np.uint32) << 16).view(np.float32) * scale[:, None]
    lat = _round_bf16_bits(np.ascontiguousarray(lat_f, dtype=np.float32))
    if N >= 4:
        lat[0] = 0
        lat[1, 77] = _round_bf16_bits(np.array([300.0], np.float32))[0]
        lat[2, 128:256] = 0
        lat[3] = _round_bf16_bits(np.full(D_V, -0.3125, np.float32))
    if N >= 8:
        # row 4: values from 2^40 down to bf16 subnormals (a span beyond 2^31)
        span = np.exp2(np.linspace(40.0, -132.0, D_V)).astype(np.float32)
        lat[4] = _round_bf16_bits(span * np.where(np.arange(D_V) % 3 == 0, -1, 1).astype(np.float32))
        # row 5: squares whose sum overflows fp32 (2^60 squared, 512 times)
        lat[5] = _round_bf16_bits(np.full(D_V, 2.0 ** 60, np.float32) * np.where(np.arange(D_V) % 2, -1, 1).astype(np.float32))
        # row 6: bf16 subnormals only (the sum underflows fp32)
        lat[6] = (np.arange(D_V) % 127 + 1).astype(np.uint16)
    qkv_bits = _bf16_normal(g, (N, QKV_COLS), std=1.0)
    qkv_bits[:, KV_C_COL:KV_C_COL + D_V] = lat
    w = 1.0 + 0.25 * g.normal_f32(D_V, 1.0)
    w_bits = _round_bf16_bits(np.ascontiguousarray(w, dtype=np.float32))
    total = num_pages * page_size
    if N > total:
        raise ValueError("more tokens than cache slots")
    slots = g.permutation(total)[:N].astype(np.int64)
    if skip_every > 0:
        slots[skip_every - 1::skip_every] = -1
    return InsertInputs(qkv=qkv_bits, w_kva=w_bits, slots=slots, num_pages=num_pages,
                        page_size=page_size, eps=float(eps), k_scale_inv=float(k_scale_inv))


# --- query-absorption inputs ---------------------------------------------------

@dataclasses.dataclass
class QueryInputs:
    qkv: np.ndarray      # uint16 bf16 bits [N, 2112]; q_a at columns 0..1535
    w_qa: np.ndarray     # uint16 bf16 bits [1536]
    w_qb: np.ndarray     # uint16 bf16 bits [H*192, 1536]
    w_uk: np.ndarray     # uint16 bf16 bits [H, 128, 512]
    eps: float

    @property
    def N(self) -> int:
        return self.qkv.shape[0]

    @property
    def H(self) -> int:
        return self.w_uk.shape[0]


def make_query_inputs(N: int, H: int, *, seed: int, eps: float = 1e-6) -> QueryInputs:
    """Synthetic inputs of the query path: fused projection rows whose q_a part
    (columns 0..1535) has a per-token scale log-uniform over 2^-6 .. 2^3;
    w_qa ~ 1 + 0.25 N(0,1); W_QB ~ N(0,1)/sqrt(1536) and W_UK ~ N(0,1)/sqrt(128)
    (random weights of the layer's shapes: 192 Q_B rows per head, 128 of them
    no-PE, and a 128 x 512 W_UK per head), all rounded to bf16."""
    g = _Rng(seed)
    scale = np.exp2(g.uniform(-6.0, 3.0, N)).astype(np.float32)
    qa = _bf16_normal(g, (N, 1536), std=1.0)
    qa_f = (qa.astype(np.uint32) << 16).view(np.float32) * scale[:, None]
    qkv = _bf16_normal(g, (N, QKV_COLS), std=1.0)
    qkv[:, :1536] = _round_bf16_bits(np.ascontiguousarray(qa_f, dtype=np.float32))
    w_qa = _round_bf16_bits(np.ascontiguousarray(1.0 + 0.25 * g.normal_f32(1536, 1.0), dtype=np.float32))
    w_qb = _bf16_normal(g, (H * 192, 1536), std=1.0 / math.sqrt(1536.0))
    w_uk = _bf16_normal(g, (H, 128, 512), std=1.0 / math.sqrt(128.0))
    return QueryInputs(qkv=qkv, w_qa=w_qa, w_qb=w_qb, w_uk=w_uk, eps=float(eps))


def kv_bytes_per_token(kv_format: int) -> int:
    """Algorithmic bytes of one valid key: 576 bf16, or 512 e4m3 + 4 fp32
    scales + 64 bf16 RoPE."""
    if kv_format == KV_FP8_TENSOR:
        return D_QK
    return 2 * D_QK if kv_format == KV_BF16 else D_V + 16 + 2 * D_ROPE


FLOP_PER_ROW_KEY = 2 * D_QK + 2 * D_V

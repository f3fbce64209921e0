"""MLA decode attention for GB300 (sm_103a): Python binding.

Argument marshalling over the C ABI of ``_lib/libmla_decode.so`` (declared in
``include/mla_decode.h``).  Every step of the computation runs in the
library's CUDA kernels; PyTorch only provides device memory (outputs and
workspace are ``torch.empty``) and the current CUDA stream.  There is no CPU
path: if the library has not been built, importing the binding works but
every call raises.

    import mla_decode_attention_05_gb300 as mla
    tile_md, num_splits = mla.metadata(cache_seqlens, H, T)
    out, lse = mla.decode(q, kv_cache, block_table, cache_seqlens,
                          softmax_scale=192 ** -0.5,
                          tile_md=tile_md, num_splits=num_splits)
    mla.kv_insert(kv_c, k_pe, w_kva, slots, kv_cache, eps=1e-6,
                  kv_scales=kv_scales)   # the cache producer
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libmla_decode.so")

KV_BF16 = 0
KV_FP8_E4M3 = 1
KV_FP8_E4M3_TENSOR = 2
PAGE_SIZE = 64
D_QK = 576
D_V = 512
FP8_ROW_BYTES = 640
STATUS_BAD_PAGE = 1
STATUS_BAD_TOPK = 2
STATUS_BAD_SEQLEN = 4
STATUS_WAIT_TIMEOUT = 8
STATUS_SMEM_ALIGN = 16

_lock = threading.Lock()
_lib = None


class MlaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"mla error {code}: {msg}")
        self.code = code


def lib():
    """The loaded C library (raises if it was never built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                    "or python -m mla_decode_attention_05_gb300.build")
            L = ctypes.CDLL(LIB_PATH)
            P, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
            L.mla_default_num_parts.argtypes = [i]
            L.mla_decode_num_items.argtypes = [i, i, i, i]
            L.mla_decode_metadata_sizes.argtypes = [i, i, i, i, i, ctypes.POINTER(sz), ctypes.POINTER(sz)]
            L.mla_decode_metadata.argtypes = [P, i, i, i, i, i, i, P, P, P]
            L.mla_decode_workspace_bytes.argtypes = [i, i, i, i, i]
            L.mla_decode_workspace_bytes.restype = sz
            L.mla_decode.argtypes = [P, P, i, i, i, P, i, P, P, i, P, P, ctypes.c_float, i,
                                     P, P, i, P, sz, P, P, i, i, i, P]
            L.mla_decode_noalloc.argtypes = [P, P, i, i, i, P, i, P, P, i, P, ctypes.c_float, i,
                                             P, P, i, i, i, P]
            L.mla_kv_insert.argtypes = [P, i, P, i, P, ctypes.c_float, P, i, P, i, i, i, P, P, P]
            L.mla_query_absorb_workspace_bytes.argtypes = [i, i]
            L.mla_query_absorb_workspace_bytes.restype = sz
            L.mla_query_absorb.argtypes = [P, i, P, ctypes.c_float, P, P, i, i, P, P, sz, P]
            L.mla_last_error_string.restype = ctypes.c_char_p
            L.mla_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
            L.mla_profile_events.argtypes = [P, P]
            L.mla_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
            L.mla_set_dual_gemm.argtypes = [ctypes.c_int]
            _lib = L
    return _lib


def _check(rc: int):
    if rc < 0:
        raise MlaError(rc, lib().mla_last_error_string().decode())
    return rc


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need(t, name, dtype, device=None, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims")


def default_num_parts(device=None) -> int:
    idx = None if device is None else torch.device(device).index
    return _check(lib().mla_default_num_parts(torch.cuda.current_device() if idx is None else idx))


def num_items(B: int, H: int, T: int, topk: int = 0) -> int:
    return _check(lib().mla_decode_num_items(B, H, T, topk))


def metadata_sizes(B: int, H: int, T: int, topk: int, num_parts: int):
    """Element counts of the two schedule arrays -> (tile_md, num_splits)."""
    a = ctypes.c_size_t()
    b = ctypes.c_size_t()
    _check(lib().mla_decode_metadata_sizes(B, H, T, topk, num_parts, ctypes.byref(a), ctypes.byref(b)))
    return int(a.value), int(b.value)


def workspace_bytes(B: int, H: int, T: int, topk: int, num_parts: int) -> int:
    n = lib().mla_decode_workspace_bytes(B, H, T, topk, num_parts)
    if n == 0:
        raise MlaError(-1, "bad sizes for workspace query")
    return int(n)


def metadata(cache_seqlens: torch.Tensor, H: int, T: int, *, topk: int = 0,
             causal: bool = False, num_parts: Optional[int] = None):
    """Split-KV schedule on the current stream -> (tile_md, num_splits)."""
    _need(cache_seqlens, "cache_seqlens", torch.int32, ndim=1)
    dev = cache_seqlens.device
    B = cache_seqlens.shape[0]
    if num_parts is None:
        num_parts = default_num_parts(dev)
    a = ctypes.c_size_t()
    b = ctypes.c_size_t()
    _check(lib().mla_decode_metadata_sizes(B, H, T, topk, num_parts, ctypes.byref(a), ctypes.byref(b)))
    tile_md = torch.empty(a.value, dtype=torch.int32, device=dev).view(num_parts, 8)
    num_splits = torch.empty(b.value, dtype=torch.int32, device=dev)
    with torch.cuda.device(dev):
        _check(lib().mla_decode_metadata(_ptr(cache_seqlens), B, H, T, topk, int(bool(causal)),
                                         num_parts, _ptr(tile_md), _ptr(num_splits), _stream(dev)))
    return tile_md, num_splits


def decode(q: torch.Tensor, kv_cache: torch.Tensor, block_table: torch.Tensor,
           cache_seqlens: torch.Tensor, *, softmax_scale: float,
           causal: bool = False, topk_indices: Optional[torch.Tensor] = None,
           kv_scales: Optional[torch.Tensor] = None,
           tile_md: Optional[torch.Tensor] = None,
           num_splits: Optional[torch.Tensor] = None,
           workspace: Optional[torch.Tensor] = None,
           out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
           gathered: Optional[torch.Tensor] = None):
    """MLA decode on the current stream -> (out bf16 [B,T,H,512], lse fp32 [B,H,T]).

    q bf16 [B,T,H,576]; kv_cache bf16 [P,64,576] (bf16 rows), uint8
    [P,64,640] (e4m3 latent + bf16 RoPE rows, with kv_scales fp32 [P,64,4]) or
    uint8 [P,64,576] (all e4m3, with one fp32 scale in kv_scales: the value is
    e4m3 x scale, i.e. the scale is 1 / the k_scale_inv kv_insert used);
    block_table int32 [B,max_pages]; cache_seqlens int32 [B]; topk_indices
    int32 [B,T,topk] or None.  tile_md/num_splits come from metadata() with
    the same arguments (computed here when omitted)."""
    dev, B, T, H, fmt, topk = _decode_args(q, kv_cache, block_table, cache_seqlens, topk_indices, kv_scales)
    if gathered is not None:
        _need(gathered, "gathered", torch.int32, dev, 3)
    if tile_md is None or num_splits is None:
        tile_md, num_splits = metadata(cache_seqlens, H, T, topk=topk, causal=causal)
    _need(tile_md, "tile_md", torch.int32, dev, 2)
    _need(num_splits, "num_splits", torch.int32, dev, 1)
    num_parts = tile_md.shape[0]
    need = workspace_bytes(B, H, T, topk, num_parts)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    _need(workspace, "workspace", workspace.dtype, dev)
    if out is None:
        out = torch.empty((B, T, H, D_V), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((B, H, T), dtype=torch.float32, device=dev)
    _need(out, "out", torch.bfloat16, dev, 4)
    _need(lse, "lse", torch.float32, dev, 3)
    check_decode_shapes(B, T, H, topk, kv_cache.shape[0], out_shape=out.shape, lse_shape=lse.shape,
                        kv_scales_shape=kv_scales.shape if fmt == KV_FP8_E4M3 else None,
                        tile_md_shape=tile_md.shape, num_splits_numel=num_splits.numel(),
                        n_items=num_items(B, H, T, topk),
                        gathered_shape=None if gathered is None else gathered.shape)
    with torch.cuda.device(dev):
        _check(lib().mla_decode(
            _ptr(q), _ptr(kv_cache), fmt, kv_cache.shape[0], kv_cache.shape[1],
            _ptr(block_table), block_table.shape[1], _ptr(cache_seqlens),
            _ptr(topk_indices), topk, _ptr(gathered), _ptr(kv_scales),
            float(softmax_scale), int(bool(causal)), _ptr(tile_md), _ptr(num_splits),
            num_parts, _ptr(workspace), workspace.numel() * workspace.element_size(),
            _ptr(out), _ptr(lse), B, T, H, _stream(dev)))
    return out, lse


def check_decode_shapes(B: int, T: int, H: int, topk: int, num_pages: int, *,
                        out_shape, lse_shape, kv_scales_shape=None, tile_md_shape=None,
                        num_splits_numel=None, n_items=None, gathered_shape=None) -> None:
    """Shape checks of the caller-given decode buffers (the C ABI sees only
    pointers, so a buffer that is too small would be written past its end):
    out [B,T,H,512], lse [B,H,T], per-128 FP8 scales [num_pages,64,4],
    tile_md [parts,8], num_splits with at least n_items + 1 entries, and a
    gathered record shaped like the top-k indices [B,T,topk].  Raises
    ValueError."""
    if tuple(out_shape) != (B, T, H, D_V):
        raise ValueError(f"out must be [{B}, {T}, {H}, {D_V}], got {list(out_shape)}")
    if tuple(lse_shape) != (B, H, T):
        raise ValueError(f"lse must be [{B}, {H}, {T}], got {list(lse_shape)}")
    if kv_scales_shape is not None and tuple(kv_scales_shape) != (num_pages, PAGE_SIZE, 4):
        raise ValueError(f"kv_scales must be [{num_pages}, {PAGE_SIZE}, 4], got {list(kv_scales_shape)}")
    if tile_md_shape is not None:
        if len(tile_md_shape) != 2 or tile_md_shape[1] != 8 or tile_md_shape[0] < 1:
            raise ValueError(f"tile_md must be [num_parts, 8], got {list(tile_md_shape)}")
    if num_splits_numel is not None and (n_items is None or num_splits_numel < n_items + 1):
        raise ValueError(f"num_splits needs {n_items} + 1 entries, got {num_splits_numel}")
    if gathered_shape is not None and tuple(gathered_shape) != (B, T, topk):
        raise ValueError(f"gathered must be [{B}, {T}, {topk}], got {list(gathered_shape)}")


def _decode_args(q, kv_cache, block_table, cache_seqlens, topk_indices, kv_scales):
    """Checks the decode inputs' dtypes, devices and shapes -> (device, B, T,
    H, cache format, topk)."""
    _need(q, "q", torch.bfloat16, ndim=4)
    dev = q.device
    B, T, H, dq = q.shape
    if dq != D_QK:
        raise ValueError("q must be [B, T, H, 576]")
    if not isinstance(kv_cache, torch.Tensor):
        raise TypeError("kv_cache must be a torch.Tensor")
    if kv_cache.dtype == torch.bfloat16:
        fmt = KV_BF16
        if kv_cache.dim() != 3 or kv_cache.shape[2] != D_QK:
            raise ValueError("bf16 kv_cache must be [P, 64, 576]")
    elif kv_cache.dtype == torch.uint8:
        if kv_cache.dim() != 3 or kv_cache.shape[2] not in (FP8_ROW_BYTES, D_QK):
            raise ValueError("fp8 kv_cache must be uint8 [P, 64, 640] (per-128 scales) or [P, 64, 576] (per-tensor)")
        if kv_cache.shape[2] == FP8_ROW_BYTES:
            fmt = KV_FP8_E4M3
            _need(kv_scales, "kv_scales", torch.float32, dev, 3)
        else:
            fmt = KV_FP8_E4M3_TENSOR
            _need(kv_scales, "kv_scales", torch.float32, dev)
            if kv_scales.numel() != 1:
                raise ValueError("a per-tensor fp8 cache takes kv_scales with one fp32 scale")
    else:
        raise TypeError("kv_cache must be bfloat16 or uint8 (fp8 rows)")
    _need(kv_cache, "kv_cache", kv_cache.dtype, dev)
    _need(block_table, "block_table", torch.int32, dev, 2)
    _need(cache_seqlens, "cache_seqlens", torch.int32, dev, 1)
    if block_table.shape[0] != B or cache_seqlens.shape[0] != B:
        raise ValueError("block_table / cache_seqlens batch mismatch")
    topk = 0
    if topk_indices is not None:
        _need(topk_indices, "topk_indices", torch.int32, dev, 3)
        if tuple(topk_indices.shape[:2]) != (B, T):
            raise ValueError("topk_indices must be [B, T, topk]")
        topk = topk_indices.shape[2]
    return dev, B, T, H, fmt, topk


def decode_noalloc(q: torch.Tensor, kv_cache: torch.Tensor, block_table: torch.Tensor,
                   cache_seqlens: torch.Tensor, *, softmax_scale: float, causal: bool = False,
                   topk_indices: Optional[torch.Tensor] = None,
                   kv_scales: Optional[torch.Tensor] = None,
                   out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None):
    """decode() for callers that cannot allocate device memory: schedule and
    workspace live in the library's fixed device scratch (mla_decode_noalloc).
    Only out / lse are created here when not given."""
    dev, B, T, H, fmt, topk = _decode_args(q, kv_cache, block_table, cache_seqlens, topk_indices, kv_scales)
    if out is None:
        out = torch.empty((B, T, H, D_V), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((B, H, T), dtype=torch.float32, device=dev)
    _need(out, "out", torch.bfloat16, dev, 4)
    _need(lse, "lse", torch.float32, dev, 3)
    check_decode_shapes(B, T, H, topk, kv_cache.shape[0], out_shape=out.shape, lse_shape=lse.shape,
                        kv_scales_shape=kv_scales.shape if fmt == KV_FP8_E4M3 else None)
    with torch.cuda.device(dev):
        _check(lib().mla_decode_noalloc(
            _ptr(q), _ptr(kv_cache), fmt, kv_cache.shape[0], kv_cache.shape[1], _ptr(block_table),
            block_table.shape[1], _ptr(cache_seqlens), _ptr(topk_indices), topk, _ptr(kv_scales),
            float(softmax_scale), int(bool(causal)), _ptr(out), _ptr(lse), B, T, H, _stream(dev)))
    return out, lse


_INSERT_ROW = {KV_BF16: 1152, KV_FP8_E4M3: FP8_ROW_BYTES, KV_FP8_E4M3_TENSOR: D_QK}


def _rows_view(t: torch.Tensor, name: str, width: int):
    """A bf16 matrix whose rows may be strided (a column slice of a wider
    row, e.g. the latent part of a fused projection) -> (tensor, ld)."""
    if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or not t.is_cuda:
        raise TypeError(f"{name} must be a bfloat16 CUDA tensor")
    if t.dim() != 2 or t.shape[1] < width or t.stride(1) != 1:
        raise ValueError(f"{name} must be [N, >={width}] with unit column stride")
    return t, t.stride(0) if t.shape[0] > 1 else max(t.shape[1], width)


def kv_insert(kv_c: torch.Tensor, k_pe: torch.Tensor, w_kva: torch.Tensor, slots: torch.Tensor,
              kv_cache: torch.Tensor, *, eps: float, kv_scales: Optional[torch.Tensor] = None,
              k_scale_inv: Optional[torch.Tensor] = None, fp8_per_tensor: bool = False):
    """RMSNorm the new tokens' latent rows and write them, with k_pe, into
    their cache slots, on the current stream (mla_kv_insert).

    kv_c bf16 [N, >=512] (columns 0..511 are read; rows may be a strided
    column slice); k_pe bf16 [N, >=64]; w_kva bf16 [512]; slots int64 [N]
    (-1 = skip).  kv_cache: bf16 [P, page, 576] (bf16 rows), uint8
    [P, page, 640] with kv_scales fp32 [P, page, 4] (the decode's FP8 rows),
    or uint8 [P, page, 576] with fp8_per_tensor=True and k_scale_inv fp32 [1].
    Returns kv_cache."""
    kv_c, ld_kv = _rows_view(kv_c, "kv_c", D_V)
    k_pe, ld_pe = _rows_view(k_pe, "k_pe", 64)
    dev = kv_c.device
    N = kv_c.shape[0]
    if k_pe.shape[0] != N:
        raise ValueError("kv_c / k_pe row counts differ")
    _need(w_kva, "w_kva", torch.bfloat16, dev, 1)
    _need(slots, "slots", torch.int64, dev, 1)
    if slots.shape[0] != N or w_kva.shape[0] != D_V:
        raise ValueError("slots must be [N], w_kva [512]")
    _need(kv_cache, "kv_cache", kv_cache.dtype, dev, 3)
    if kv_cache.dtype == torch.bfloat16:
        fmt = KV_BF16
    elif kv_cache.dtype == torch.uint8:
        fmt = KV_FP8_E4M3_TENSOR if fp8_per_tensor else KV_FP8_E4M3
    else:
        raise TypeError("kv_cache must be bfloat16 or uint8")
    if kv_cache.shape[2] * kv_cache.element_size() != _INSERT_ROW[fmt]:
        raise ValueError(f"kv_cache rows must be {_INSERT_ROW[fmt]} bytes for this format")
    if fmt == KV_FP8_E4M3:
        _need(kv_scales, "kv_scales", torch.float32, dev, 3)
        if tuple(kv_scales.shape) != (kv_cache.shape[0], kv_cache.shape[1], 4):
            raise ValueError("kv_scales must be [P, page, 4]")
    if fmt == KV_FP8_E4M3_TENSOR:
        _need(k_scale_inv, "k_scale_inv", torch.float32, dev)
    with torch.cuda.device(dev):
        _check(lib().mla_kv_insert(
            _ptr(kv_c), ld_kv, _ptr(k_pe), ld_pe, _ptr(w_kva), float(eps), _ptr(slots), N,
            _ptr(kv_cache), fmt, kv_cache.shape[0], kv_cache.shape[1],
            _ptr(kv_scales) if fmt == KV_FP8_E4M3 else None,
            _ptr(k_scale_inv) if fmt == KV_FP8_E4M3_TENSOR else None, _stream(dev)))
    return kv_cache


D_QA = 1536
QB_ROWS = 192


def query_absorb_workspace_bytes(N: int, H: int) -> int:
    n = lib().mla_query_absorb_workspace_bytes(N, H)
    if n == 0:
        raise MlaError(-1, "bad sizes for the query-absorption workspace")
    return int(n)


def query_absorb(q_a: torch.Tensor, w_qa: torch.Tensor, w_qb: torch.Tensor, w_uk: torch.Tensor, *,
                 eps: float, out: Optional[torch.Tensor] = None,
                 workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """The decode's query rows from q_a, on the current stream
    (mla_query_absorb): RMSNorm(q_a) x w_qa -> Q_B (192 rows per head) ->
    W_UK on the 128 no-PE rows; returns q bf16 [N, H, 576] (reshape to
    [B, T, H, 576] for decode()).

    q_a bf16 [N, >=1536] (rows may be a strided column slice of the fused
    projection output); w_qa bf16 [1536]; w_qb bf16 [H*192, 1536]; w_uk bf16
    [H, 128, 512].  A caller-given workspace (uint8, >=
    query_absorb_workspace_bytes(N, H)) keeps xq and qb for inspection."""
    q_a, ld = _rows_view(q_a, "q_a", D_QA)
    dev = q_a.device
    N = q_a.shape[0]
    _need(w_qa, "w_qa", torch.bfloat16, dev, 1)
    _need(w_qb, "w_qb", torch.bfloat16, dev, 2)
    _need(w_uk, "w_uk", torch.bfloat16, dev, 3)
    H = w_uk.shape[0]
    if w_qa.shape[0] != D_QA or tuple(w_qb.shape) != (H * QB_ROWS, D_QA) or tuple(w_uk.shape[1:]) != (128, D_V):
        raise ValueError("expected w_qa [1536], w_qb [H*192, 1536], w_uk [H, 128, 512]")
    if out is None:
        out = torch.empty((N, H, D_QK), dtype=torch.bfloat16, device=dev)
    _need(out, "out", torch.bfloat16, dev, 3)
    if tuple(out.shape) != (N, H, D_QK):
        raise ValueError("out must be [N, H, 576]")
    need = query_absorb_workspace_bytes(N, H)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    _need(workspace, "workspace", workspace.dtype, dev)
    with torch.cuda.device(dev):
        _check(lib().mla_query_absorb(_ptr(q_a), ld, _ptr(w_qa), float(eps), _ptr(w_qb), _ptr(w_uk), N, H,
                                      _ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                      _stream(dev)))
    return out


def device_status() -> int:
    """Read and clear the device status word (synchronises the device)."""
    v = ctypes.c_uint32()
    _check(lib().mla_device_status(ctypes.byref(v)))
    return int(v.value)


def set_dual_gemm(enable: bool):
    """QK of items with at most 64 query rows as the M = 64 dual GEMM
    (weight-stationary MMAs) for later decode calls on this thread; off by
    default (see mla_set_dual_gemm in include/mla_decode.h)."""
    _check(lib().mla_set_dual_gemm(1 if enable else 0))


def set_wait_limit_ns(ns: int = 0):
    """Test hook: the limit of the decode kernel's bounded waits for later
    decode calls on this thread (0 = the default, 2 s); see
    mla_set_wait_limit_ns in include/mla_decode.h."""
    _check(lib().mla_set_wait_limit_ns(int(ns)))


def profile_events(before=None, after=None):
    """Record CUDA events around the decode kernel of later decode() calls on
    this thread (torch.cuda.Event objects), or stop with no arguments."""
    b = ctypes.c_void_p(before.cuda_event) if before is not None else None
    a = ctypes.c_void_p(after.cuda_event) if after is not None else None
    _check(lib().mla_profile_events(b, a))

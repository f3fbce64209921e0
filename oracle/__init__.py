"""Float64 CPU oracle for MLA decode (test infrastructure).

Only tests/, ``__graft_entry__.smoke()`` and the cpu_baseline / reference arm
of ``bench.py`` may import this package.  It shares no code with the CUDA
library (``mla_decode_attention_05_gb300``) and never imports it; both sides
read the same seeded inputs from ``workloads``.

Parts:
  mla_oracle.c   attention definition in double precision (see its header)
  schedule.py    the split-KV work partition, restated in plain Python
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from . import schedule  # noqa: F401  (re-exported)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_OUT_DIR, "libmla_oracle.so")
_lock = threading.Lock()
_handle = None

D_QK = 576
D_V = 512


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP).  Plain C, no ISA flags, so
    the same source builds on x86-64 and aarch64."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_SO)
            and os.path.getmtime(_SO) >= os.path.getmtime(_SRC)):
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared",
                           "-fno-fast-math", "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _SO)
    return _SO


def _lib():
    global _handle
    with _lock:
        if _handle is None:
            build()
            lib = ctypes.CDLL(_SO)
            P = ctypes.c_void_p
            i = ctypes.c_int
            lib.oracle_bf16_to_f64.restype = ctypes.c_double
            lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
            lib.oracle_e4m3_to_f64.restype = ctypes.c_double
            lib.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
            lib.oracle_valid_keys.restype = i
            lib.oracle_valid_keys.argtypes = [i, i, i, P, P, i, i, P, i]
            lib.oracle_mla_decode_rows.restype = i
            lib.oracle_mla_decode_rows.argtypes = [
                P, i, i, i, P, i, i, i, P, P, i, P, P, i, ctypes.c_double, i,
                P, i, P, P]
            lib.oracle_attend_key_list.restype = i
            lib.oracle_attend_key_list.argtypes = [
                P, P, i, i, i, P, P, i, i, P, i, ctypes.c_double, P, P]
            lib.oracle_num_threads.restype = i
            _handle = lib
    return _handle


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return int(_lib().oracle_num_threads())


def bf16_to_f64(bits: int) -> float:
    return float(_lib().oracle_bf16_to_f64(int(bits)))


def e4m3_to_f64(code: int) -> float:
    return float(_lib().oracle_e4m3_to_f64(int(code)))


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def valid_keys(w, b: int, t: int) -> np.ndarray:
    """Sorted valid key positions of query token t of sequence b."""
    lib = _lib()
    sk = _c(w.cache_seqlens, np.int32)
    tk = _c(w.topk, np.int32)
    cap = max(int(sk[b]), w.topk_len, 1)
    out = np.empty(cap, dtype=np.int32)
    n = lib.oracle_valid_keys(b, t, w.T, _ptr(sk), _ptr(tk), w.topk_len,
                              int(w.causal), _ptr(out), cap)
    if n == -2:
        raise ValueError(f"oracle: the top-k list of (b={b}, t={t}) repeats a position "
                         "(the indices of one query token must be distinct)")
    return out[:n].copy()


def decode_rows(w, rows) -> tuple:
    """rows: iterable of (b, t, h).  Returns (out [n,512], lse [n]) float64."""
    lib = _lib()
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 3))
    n = rows.shape[0]
    out = np.empty((n, D_V), dtype=np.float64)
    lse = np.empty(n, dtype=np.float64)
    q = _c(w.q, np.uint16)
    kv = np.ascontiguousarray(w.kv)
    sc = _c(w.kv_scales, np.float32)
    bt = _c(w.block_table, np.int32)
    sk = _c(w.cache_seqlens, np.int32)
    tk = _c(w.topk, np.int32)
    rc = lib.oracle_mla_decode_rows(
        _ptr(q), w.B, w.T, w.H, _ptr(kv), int(w.kv_format), w.num_pages,
        int(kv.shape[1]), _ptr(sc), _ptr(bt), w.max_pages, _ptr(sk), _ptr(tk),
        w.topk_len, float(w.softmax_scale), int(w.causal), _ptr(rows), n,
        _ptr(out), _ptr(lse))
    if rc == -2:
        raise ValueError("oracle: a top-k list repeats a position "
                         "(the indices of one query token must be distinct)")
    if rc != 0:
        raise ValueError("oracle: bad row or page index")
    return out, lse


def decode_all(w) -> tuple:
    """All rows.  Returns out [B,T,H,512] and lse [B,H,T], float64."""
    rows = [(b, t, h) for b in range(w.B) for t in range(w.T) for h in range(w.H)]
    out, lse = decode_rows(w, rows)
    out = out.reshape(w.B, w.T, w.H, D_V)
    lse = lse.reshape(w.B, w.T, w.H).transpose(0, 2, 1).copy()
    return out, lse


def attend_key_list(w, b: int, t: int, h: int, keys) -> tuple:
    """Attention of row (b,t,h) over an explicit key list (no mask rule)."""
    lib = _lib()
    keys = np.ascontiguousarray(np.asarray(keys, dtype=np.int32))
    qrow = np.ascontiguousarray(w.q[b, t, h], dtype=np.uint16)
    kv = np.ascontiguousarray(w.kv)
    out = np.empty(D_V, dtype=np.float64)
    lse = np.empty(1, dtype=np.float64)
    rc = lib.oracle_attend_key_list(
        _ptr(qrow), _ptr(kv), int(w.kv_format), w.num_pages, int(kv.shape[1]),
        _ptr(_c(w.kv_scales, np.float32)), _ptr(_c(w.block_table, np.int32)),
        w.max_pages, b, _ptr(keys), int(keys.size), float(w.softmax_scale),
        _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle: bad page index")
    return out, float(lse[0])

"""The C ABI: the library builds, loads without a GPU and exports every entry
point that include/*.h declares; host-side argument checks reject bad calls
before anything is launched (no compute call is made here)."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from mla_decode_attention_05_gb300 import build
    build.build()
    import mla_decode_attention_05_gb300 as m
    return m.lib()


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w \*]*?\b(mla_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return names


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert {"mla_decode", "mla_decode_metadata", "mla_decode_workspace_bytes"} <= names
    for n in sorted(names):
        assert hasattr(L, n), f"{n} declared in include/ but not exported"


def test_sizes_and_items(L):
    import mla_decode_attention_05_gb300 as m
    assert m.num_items(64, 128, 1) == 64
    assert m.num_items(32, 64, 4) == 64          # T*H = 256 rows -> 2 M tiles
    assert m.num_items(32, 64, 1, topk=2048) == 32
    assert m.num_items(2, 64, 3, topk=10) == 6   # top-k: one item per query token
    a, b = ctypes.c_size_t(), ctypes.c_size_t()
    assert L.mla_decode_metadata_sizes(16, 128, 1, 0, 76, ctypes.byref(a), ctypes.byref(b)) == 0
    assert (a.value, b.value) == (76 * 8, 17)
    ws = m.workspace_bytes(64, 128, 1, 0, 76)
    assert ws % 256 == 0 and ws >= (64 + 76) * 128 * 513 * 4


@pytest.mark.parametrize("args,code", [
    (dict(B=0), -1), (dict(H=129), -1), (dict(T=17), -1), (dict(page_size=32), -2),
    (dict(kv_format=7), -1), (dict(softmax_scale=0.0), -1), (dict(causal=1, topk=8), -1),
    (dict(workspace_bytes=16), -3), (dict(num_parts=0), -1), (dict(q=0), -1),
    (dict(q=8), -1),
])
def test_argument_checks(L, args, code):
    """Each bad argument returns its error code and an explanation; the
    checks run before any CUDA call, so this needs no device."""
    base = dict(q=256, kv=256, kv_format=0, num_pages=4, page_size=64, bt=256, max_pages=4,
                sk=256, topk_ptr=None, topk=0, gathered=None, scales=None,
                softmax_scale=0.07, causal=0, md=256, ns=256, num_parts=4, ws=256,
                workspace_bytes=1 << 30, out=256, lse=256, B=2, T=1, H=64)
    base.update(args)
    if base["topk"] and base["topk_ptr"] is None:
        base["topk_ptr"] = 256
    v = lambda x: None if x is None else ctypes.c_void_p(x)
    rc = L.mla_decode(v(base["q"]), v(base["kv"]), base["kv_format"], base["num_pages"],
                      base["page_size"], v(base["bt"]), base["max_pages"], v(base["sk"]),
                      v(base["topk_ptr"]), base["topk"], v(base["gathered"]), v(base["scales"]),
                      ctypes.c_float(base["softmax_scale"]), base["causal"], v(base["md"]),
                      v(base["ns"]), base["num_parts"], v(base["ws"]), base["workspace_bytes"],
                      v(base["out"]), v(base["lse"]), base["B"], base["T"], base["H"], None)
    assert rc == code
    assert len(L.mla_last_error_string()) > 0


@pytest.mark.parametrize("args,code", [
    (dict(N=-1), -1), (dict(kv_format=3), -1), (dict(num_pages=0), -1), (dict(page_size=0), -1),
    (dict(ld_kv=500), -1), (dict(ld_kv=516), -1), (dict(ld_pe=60), -1), (dict(eps=-1.0), -1),
    (dict(eps=float("nan")), -1), (dict(kv_c=0), -1), (dict(kv_c=264), -1), (dict(slots=260), -1),
    (dict(kv_format=1, scales=None), -1), (dict(kv_format=1, scales=264), -1),
    (dict(kv_format=2, ksi=None), -1), (dict(kv_format=2, ksi=258), -1),
    (dict(N=0, kv_c=0, slots=0, kv=0), 0),
])
def test_kv_insert_argument_checks(L, args, code):
    """mla_kv_insert rejects each bad argument before any CUDA call; N = 0 is
    a valid empty call that launches nothing."""
    base = dict(kv_c=256, ld_kv=2112, k_pe=256, ld_pe=2112, w=256, eps=1e-6, slots=256, N=4,
                kv=256, kv_format=0, num_pages=4, page_size=64, scales=256, ksi=256)
    base.update(args)
    v = lambda x: None if x is None else ctypes.c_void_p(x)
    rc = L.mla_kv_insert(v(base["kv_c"]), base["ld_kv"], v(base["k_pe"]), base["ld_pe"], v(base["w"]),
                         ctypes.c_float(base["eps"]), v(base["slots"]), base["N"], v(base["kv"]),
                         base["kv_format"], base["num_pages"], base["page_size"], v(base["scales"]),
                         v(base["ksi"]), None)
    assert rc == code
    if code:
        assert len(L.mla_last_error_string()) > 0


@pytest.mark.parametrize("args,code", [
    (dict(N=-1), -1), (dict(H=0), -1), (dict(H=129), -1), (dict(ld=1535), -1), (dict(ld=1540), -1),
    (dict(eps=-1.0), -1), (dict(eps=float("inf")), -1), (dict(q_a=0), -1), (dict(w_qb=264), -1),
    (dict(ws=272), -1), (dict(ws_bytes=64), -3), (dict(N=0, q_a=0, ws=0), 0),
])
def test_query_absorb_argument_checks(L, args, code):
    """mla_query_absorb rejects each bad argument before any CUDA call; N = 0
    is a valid empty call."""
    base = dict(q_a=256, ld=2112, w_qa=256, eps=1e-6, w_qb=256, w_uk=256, N=4, H=128, q=256, ws=512,
                ws_bytes=1 << 30)
    base.update(args)
    v = lambda x: None if x is None else ctypes.c_void_p(x)
    rc = L.mla_query_absorb(v(base["q_a"]), base["ld"], v(base["w_qa"]), ctypes.c_float(base["eps"]),
                            v(base["w_qb"]), v(base["w_uk"]), base["N"], base["H"], v(base["q"]), v(base["ws"]),
                            base["ws_bytes"], None)
    assert rc == code
    if code:
        assert len(L.mla_last_error_string()) > 0


def test_query_absorb_workspace_size(L):
    import mla_decode_attention_05_gb300 as m
    n = m.query_absorb_workspace_bytes(64, 128)
    assert n >= 64 * 1536 * 2 + 64 * 128 * 192 * 2
    assert L.mla_query_absorb_workspace_bytes(-1, 128) == 0 and L.mla_query_absorb_workspace_bytes(4, 0) == 0


def test_library_missing_fails_loudly(tmp_path, monkeypatch):
    """No silent fallback: without the built library every call raises."""
    import mla_decode_attention_05_gb300 as m
    monkeypatch.setattr(m, "LIB_PATH", str(tmp_path / "nope.so"))
    monkeypatch.setattr(m, "_lib", None)
    with pytest.raises(RuntimeError):
        m.num_items(1, 64, 1)


@pytest.mark.parametrize("kw,msg", [
    (dict(out_shape=(2, 1, 64, 256)), "out must be"),
    (dict(out_shape=(2, 1, 32, 512)), "out must be"),
    (dict(lse_shape=(2, 1, 64)), "lse must be"),
    (dict(lse_shape=(2, 64)), "lse must be"),
    (dict(kv_scales_shape=(8, 64, 1)), "kv_scales must be"),
    (dict(kv_scales_shape=(4, 64, 4)), "kv_scales must be"),
    (dict(tile_md_shape=(76, 4)), "tile_md must be"),
    (dict(tile_md_shape=(608,)), "tile_md must be"),
    (dict(num_splits_numel=2, n_items=2), "num_splits needs"),
    (dict(gathered_shape=(2, 1, 7), topk=8), "gathered must be"),
])
def test_binding_rejects_wrong_buffer_shapes(kw, msg):
    """The C ABI receives only pointers, so the binding checks the shapes of
    caller-given buffers: an output, scale array, schedule or gathered record
    of the wrong shape raises ValueError before any call (a short buffer
    would otherwise be written past its end)."""
    import mla_decode_attention_05_gb300 as m
    args = dict(out_shape=(2, 1, 64, 512), lse_shape=(2, 64, 1), kv_scales_shape=(8, 64, 4),
                tile_md_shape=(76, 8), num_splits_numel=3, n_items=2, gathered_shape=None, topk=0)
    m.check_decode_shapes(2, 1, 64, 0, 8, **{k: v for k, v in args.items() if k != "topk"})
    args.update(kw)
    topk = args.pop("topk")
    with pytest.raises(ValueError, match=msg):
        m.check_decode_shapes(2, 1, 64, topk, 8, **args)

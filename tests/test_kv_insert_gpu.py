"""GPU parity of the KV insert (mla_kv_insert) against the oracle: every cache
byte and every scale bit-exact, in all three row formats; skipped and bad
slots; and decode reading the cache the insert wrote."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import kv_insert as K

pytestmark = pytest.mark.gpu

SENTINEL = 0xAB


def _dev_inputs(inp):
    qkv = torch.from_numpy(inp.qkv.view(np.int16)).view(torch.bfloat16).cuda()
    kv_c = qkv[:, W.KV_C_COL:W.KV_C_COL + 512]
    k_pe = qkv[:, W.K_PE_COL:W.K_PE_COL + 64]
    w = torch.from_numpy(inp.w_kva.view(np.int16)).view(torch.bfloat16).cuda()
    slots = torch.from_numpy(inp.slots).cuda()
    return kv_c, k_pe, w, slots


def _oracle(inp, fmt, slots=None):
    rb = K.ROW_BYTES[fmt]
    cache = np.full((inp.num_pages, inp.page_size, rb), SENTINEL, np.uint8)
    scales = np.full((inp.num_pages, inp.page_size, 4), -1.0, np.float32)
    bad = K.kv_insert(fmt, inp.qkv[:, W.KV_C_COL:], inp.qkv[:, W.K_PE_COL:], inp.w_kva, inp.eps,
                      inp.slots if slots is None else slots, cache, scales, inp.k_scale_inv)
    return cache, scales, bad


def _gpu(inp, fmt, slots=None):
    import mla_decode_attention_05_gb300 as mla
    kv_c, k_pe, w, sl = _dev_inputs(inp)
    if slots is not None:
        sl = torch.from_numpy(slots).cuda()
    rb = K.ROW_BYTES[fmt]
    raw = torch.full((inp.num_pages, inp.page_size, rb), SENTINEL, dtype=torch.uint8, device="cuda")
    scales = torch.full((inp.num_pages, inp.page_size, 4), -1.0, dtype=torch.float32, device="cuda")
    ksi = torch.tensor([inp.k_scale_inv], dtype=torch.float32, device="cuda")
    cache = raw.view(torch.bfloat16) if fmt == K.FMT_BF16 else raw
    mla.device_status()  # clear
    mla.kv_insert(kv_c, k_pe, w, sl, cache, eps=inp.eps, kv_scales=scales, k_scale_inv=ksi,
                  fp8_per_tensor=(fmt == K.FMT_FP8_TENSOR))
    torch.cuda.synchronize()
    return raw.cpu().numpy(), scales.cpu().numpy(), mla.device_status()


FMTS = [K.FMT_BF16, K.FMT_FP8_TILE, K.FMT_FP8_TENSOR]


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("N,pages,page_size", [(1, 1, 64), (7, 2, 64), (203, 8, 64), (300, 40, 16)])
def test_insert_bit_exact(fmt, N, pages, page_size):
    inp = W.make_insert_inputs(N, pages, page_size, seed=100 + N)
    want_c, want_s, bad = _oracle(inp, fmt)
    got_c, got_s, status = _gpu(inp, fmt)
    assert bad == 0 and status == 0
    np.testing.assert_array_equal(got_c, want_c)
    if fmt == K.FMT_FP8_TILE:
        np.testing.assert_array_equal(got_s.view(np.uint32), want_s.view(np.uint32))
    else:
        assert np.all(got_s == -1.0)  # untouched


@pytest.mark.parametrize("fmt", FMTS)
def test_bad_slots_skip_and_set_status(fmt):
    import mla_decode_attention_05_gb300 as mla
    inp = W.make_insert_inputs(50, 2, seed=9)
    slots = inp.slots.copy()
    slots[4] = 2 * 64          # one past the end
    slots[10] = -2
    slots[11] = 1 << 40
    want_c, want_s, bad = _oracle(inp, fmt, slots)
    got_c, got_s, status = _gpu(inp, fmt, slots)
    assert bad == 3
    assert status == mla.STATUS_BAD_PAGE
    np.testing.assert_array_equal(got_c, want_c)
    np.testing.assert_array_equal(got_s.view(np.uint32), want_s.view(np.uint32))


def test_all_skipped_and_empty_calls_write_nothing():
    import mla_decode_attention_05_gb300 as mla
    inp = W.make_insert_inputs(16, 1, seed=12)
    got_c, got_s, status = _gpu(inp, K.FMT_FP8_TILE, np.full(16, -1, np.int64))
    assert status == 0 and np.all(got_c == SENTINEL) and np.all(got_s == -1.0)
    kv_c, k_pe, w, sl = _dev_inputs(inp)
    cache = torch.full((1, 64, 640), SENTINEL, dtype=torch.uint8, device="cuda")
    sc = torch.zeros((1, 64, 4), dtype=torch.float32, device="cuda")
    mla.kv_insert(kv_c[:0], k_pe[:0], w, sl[:0], cache, eps=1e-6, kv_scales=sc)
    torch.cuda.synchronize()
    assert torch.all(cache == SENTINEL)


def test_contiguous_rows_and_large_batch():
    """kv_c / k_pe as their own contiguous arrays (ld 512 / 64), a full cache
    of 4096 slots written by 4096 tokens."""
    import mla_decode_attention_05_gb300 as mla
    inp = W.make_insert_inputs(4096, 64, seed=21, skip_every=0)
    want_c, want_s, _ = _oracle(inp, K.FMT_FP8_TILE)
    kv_c, k_pe, w, sl = _dev_inputs(inp)
    kv_c, k_pe = kv_c.contiguous(), k_pe.contiguous()
    cache = torch.full((64, 64, 640), SENTINEL, dtype=torch.uint8, device="cuda")
    sc = torch.full((64, 64, 4), -1.0, dtype=torch.float32, device="cuda")
    mla.kv_insert(kv_c, k_pe, w, sl, cache, eps=inp.eps, kv_scales=sc)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(cache.cpu().numpy(), want_c)
    np.testing.assert_array_equal(sc.cpu().numpy().view(np.uint32), want_s.view(np.uint32))


def test_decode_reads_what_insert_wrote():
    """Insert every token of two sequences into an FP8 cache on the GPU, then
    decode from it: the cache bytes equal the oracle's, and the decode output
    matches the oracle's attention over the oracle-inserted cache."""
    import mla_decode_attention_05_gb300 as mla
    from oracle import decode_rows
    from _gpu import TOL_LSE, TOL_O

    w = W.make_workload("insert_then_decode", 2, 1, 64, [300, 129], seed=77, num_pages=12, fp8=True)
    # token position p of sequence b lives at slot block_table[b, p // 64] * 64 + p % 64
    slots = np.concatenate([w.block_table[b, np.arange(n) // 64].astype(np.int64) * 64 + np.arange(n) % 64
                            for b, n in enumerate(w.cache_seqlens)])
    inp = W.make_insert_inputs(len(slots), w.num_pages, seed=78, skip_every=0)
    inp.slots = slots
    cache = w.kv.copy()
    scales = w.kv_scales.copy()
    K.kv_insert(K.FMT_FP8_TILE, inp.qkv[:, W.KV_C_COL:], inp.qkv[:, W.K_PE_COL:], inp.w_kva, inp.eps,
                slots, cache, scales)
    w.kv, w.kv_scales = cache, scales

    kv_c, k_pe, wk, sl = _dev_inputs(inp)
    d_cache = torch.from_numpy(np.full_like(cache, SENTINEL)).cuda()
    d_scales = torch.full(scales.shape, -1.0, dtype=torch.float32, device="cuda")
    mla.kv_insert(kv_c, k_pe, wk, sl, d_cache, eps=inp.eps, kv_scales=d_scales)
    q = torch.from_numpy(w.q.view(np.int16)).view(torch.bfloat16).cuda()
    bt = torch.from_numpy(w.block_table).cuda()
    sk = torch.from_numpy(w.cache_seqlens).cuda()
    out, lse = mla.decode(q, d_cache, bt, sk, softmax_scale=w.softmax_scale, kv_scales=d_scales)
    torch.cuda.synchronize()
    live = np.zeros(cache.shape[:2], bool)
    live.reshape(-1)[slots] = True
    np.testing.assert_array_equal(d_cache.cpu().numpy()[live], cache[live])
    np.testing.assert_array_equal(d_scales.cpu().numpy()[live].view(np.uint32), scales[live].view(np.uint32))
    rows = [(b, 0, h) for b in range(2) for h in (0, 17, 63)]
    ref_o, ref_l = decode_rows(w, rows)
    got_o = np.stack([out[b, t, h].float().cpu().numpy() for b, t, h in rows])
    got_l = np.array([lse[b, h, t].item() for b, t, h in rows])
    assert np.abs(got_o - ref_o).max() <= TOL_O
    assert np.abs(got_l - ref_l).max() <= TOL_LSE


def test_bench_size_insert_sampled():
    """The bench's insert (262144 tokens filling a 4096-page FP8 cache):
    3000 sampled tokens' rows and scales bit-exact against the oracle."""
    import mla_decode_attention_05_gb300 as mla
    inp = W.make_insert_inputs(262144, 4096, seed=4242, skip_every=0)
    kv_c, k_pe, w, sl = _dev_inputs(inp)
    cache = torch.zeros((4096, 64, 640), dtype=torch.uint8, device="cuda")
    sc = torch.zeros((4096, 64, 4), dtype=torch.float32, device="cuda")
    mla.device_status()
    mla.kv_insert(kv_c, k_pe, w, sl, cache, eps=inp.eps, kv_scales=sc)
    torch.cuda.synchronize()
    assert mla.device_status() == 0
    rng = np.random.default_rng(1)
    pick = rng.choice(inp.N, 3000, replace=False)
    got_c = cache.view(-1, 640)[torch.from_numpy(inp.slots[pick]).cuda()].cpu().numpy()
    got_s = sc.view(-1, 4)[torch.from_numpy(inp.slots[pick]).cuda()].cpu().numpy()
    for k, j in enumerate(pick):
        row, scl = K.insert_row(K.FMT_FP8_TILE, inp.qkv[j, W.KV_C_COL:W.KV_C_COL + 512],
                                inp.qkv[j, W.K_PE_COL:W.K_PE_COL + 64], inp.w_kva, inp.eps)
        np.testing.assert_array_equal(got_c[k], row)
        np.testing.assert_array_equal(got_s[k].view(np.uint32), scl.view(np.uint32))


def test_decode_reads_per_tensor_fp8_insert():
    """The page's own cache layout end to end: insert every token of two
    sequences as per-tensor FP8 rows (e4m3(v * k_scale_inv), RoPE included),
    decode with the scale 1 / k_scale_inv: bytes equal the oracle's and the
    attention matches the oracle's over the oracle-inserted cache."""
    import mla_decode_attention_05_gb300 as mla
    from oracle import decode_rows
    from _gpu import TOL_LSE, TOL_O

    w = W.make_workload("tensor_insert_decode", 2, 1, 64, [300, 129], seed=81, num_pages=12, fp8_tensor=True)
    slots = np.concatenate([w.block_table[b, np.arange(n) // 64].astype(np.int64) * 64 + np.arange(n) % 64
                            for b, n in enumerate(w.cache_seqlens)])
    inp = W.make_insert_inputs(len(slots), w.num_pages, seed=82, skip_every=0, k_scale_inv=4.0)
    inp.slots = slots
    cache = w.kv.copy()
    K.kv_insert(K.FMT_FP8_TENSOR, inp.qkv[:, W.KV_C_COL:], inp.qkv[:, W.K_PE_COL:], inp.w_kva, inp.eps,
                slots, cache, None, inp.k_scale_inv)
    w.kv = cache
    w.kv_scales = np.array([np.float32(1.0) / np.float32(inp.k_scale_inv)], dtype=np.float32)

    kv_c, k_pe, wk, sl = _dev_inputs(inp)
    d_cache = torch.from_numpy(np.full_like(cache, SENTINEL)).cuda()
    ksi = torch.tensor([inp.k_scale_inv], dtype=torch.float32, device="cuda")
    mla.kv_insert(kv_c, k_pe, wk, sl, d_cache, eps=inp.eps, k_scale_inv=ksi, fp8_per_tensor=True)
    q = torch.from_numpy(w.q.view(np.int16)).view(torch.bfloat16).cuda()
    out, lse = mla.decode(q, d_cache, torch.from_numpy(w.block_table).cuda(),
                          torch.from_numpy(w.cache_seqlens).cuda(), softmax_scale=w.softmax_scale,
                          kv_scales=torch.from_numpy(w.kv_scales).cuda())
    torch.cuda.synchronize()
    live = np.zeros(cache.shape[:2], bool)
    live.reshape(-1)[slots] = True
    np.testing.assert_array_equal(d_cache.cpu().numpy()[live], cache[live])
    rows = [(b, 0, h) for b in range(2) for h in (0, 17, 63)]
    ref_o, ref_l = decode_rows(w, rows)
    got_o = np.stack([out[b, t, h].float().cpu().numpy() for b, t, h in rows])
    got_l = np.array([lse[b, h, t].item() for b, t, h in rows])
    assert np.abs(got_o - ref_o).max() <= TOL_O
    assert np.abs(got_l - ref_l).max() <= TOL_LSE

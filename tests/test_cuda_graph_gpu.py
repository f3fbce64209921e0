"""The library's calls inside a captured CUDA graph.

A serving loop replays one captured graph per step instead of issuing each
launch from the host.  That works only if no call synchronises with the host,
allocates device memory or reads an input on the host while it is captured,
and if each replay reads the inputs' current contents: the split-KV schedule,
in particular, has to be recomputed on the device from the sequence lengths
of that step.  These tests capture (1) schedule -> decode -> combine and (2) a
whole layer step -- query absorption, KV insert of the new tokens, schedule,
decode -- change the inputs in place between replays, and require the
replayed results to equal, bit for bit, the same calls issued eagerly on the
same inputs (and, for the layer step, the oracle's attention on sampled rows).
"""
import numpy as np
import pytest
import torch

import workloads as W
import _gpu as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mla():
    from mla_decode_attention_05_gb300 import build
    build.build()
    import mla_decode_attention_05_gb300 as m
    m.device_status()
    return m


def _capture(fn):
    """Two warm-up runs on a side stream, then one capture of fn."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(2):
            fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def _full_rows(w):
    """Every sequence gets a full block-table row (so any length up to
    max_pages * 64 is valid), its pages scattered over the pool."""
    perm = np.random.default_rng(w.seed).permutation(w.num_pages).astype(np.int32)
    w.block_table = perm[w.block_table]
    return w


def test_decode_step_graph_follows_new_lengths_and_queries(mla):
    """schedule + decode + combine captured once; replayed for three sets of
    sequence lengths and queries written into the captured input buffers."""
    w = _full_rows(W.make_workload("graph_decode", 5, 1, 128, [3000, 64, 1, 4000, 129], seed=61,
                                   identity_pages=True))
    d = G.to_device(w)
    B, T, H = w.B, w.T, w.H
    out = torch.empty((B, T, H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H, T), dtype=torch.float32, device="cuda")
    parts = mla.default_num_parts()
    ws = torch.empty(mla.workspace_bytes(B, H, T, 0, parts), dtype=torch.uint8, device="cuda")

    def step():
        md, ns = mla.metadata(d["sk"], H, T, num_parts=parts)
        mla.decode(d["q"], d["kv"], d["bt"], d["sk"], softmax_scale=w.softmax_scale,
                   tile_md=md, num_splits=ns, workspace=ws, out=out, lse=lse)

    g = _capture(step)
    cap = w.block_table.shape[1] * 64       # 63 pages: 4032 tokens
    assert cap == 4032
    rng = np.random.default_rng(5)
    for trial, lens in enumerate(([3000, 64, 1, 4000, 129], [1, 2048, 0, 64, 4032], None)):
        if lens is None:
            lens = rng.integers(0, cap + 1, size=B)
        lens = np.asarray(lens)
        d["sk"].copy_(torch.from_numpy(lens.astype(np.int32)))
        d["q"].normal_(0.0, 0.5, generator=torch.Generator("cuda").manual_seed(100 + trial))
        g.replay()
        torch.cuda.synchronize()
        got_o, got_l = out.clone(), lse.clone()
        step()
        torch.cuda.synchronize()
        assert torch.equal(got_o, out), trial
        assert torch.equal(got_l.view(torch.int32), lse.view(torch.int32)), trial
        assert torch.isneginf(got_l).any().item() == bool((lens == 0).any()), trial
    assert mla.device_status() == 0


def test_layer_step_graph_absorb_insert_decode(mla):
    """Query absorption of the new tokens, their KV insert into an FP8 cache,
    the schedule and the decode, captured as one graph.  Between replays the
    projection rows, the new tokens' slots and the sequence lengths change in
    place (each sequence grows by one token)."""
    from oracle import decode_rows

    B, T, H = 4, 1, 128
    base_len = np.array([700, 1500, 63, 2000], dtype=np.int32)
    w = _full_rows(W.make_workload("graph_layer", B, T, H, list(base_len + 3), seed=91, fp8=True,
                                   identity_pages=True))
    qin = W.make_query_inputs(B * T, H, seed=92)
    ins = W.make_insert_inputs(B * T, w.num_pages, seed=93, skip_every=0)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()

    qkv = dev(qin.qkv)                       # fused projection rows [N, 2112]
    w_qa, w_qb, w_uk, w_kva = dev(qin.w_qa), dev(qin.w_qb), dev(qin.w_uk), dev(ins.w_kva)
    cache0 = torch.from_numpy(w.kv).cuda()
    scales0 = torch.from_numpy(w.kv_scales).cuda()
    cache, scales = cache0.clone(), scales0.clone()
    bt = torch.from_numpy(w.block_table).cuda()
    sk = torch.empty(B, dtype=torch.int32, device="cuda")
    slots = torch.empty(B * T, dtype=torch.int64, device="cuda")
    q = torch.empty((B * T, H, 576), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((B, T, H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H, T), dtype=torch.float32, device="cuda")
    parts = mla.default_num_parts()
    ws_q = torch.empty(mla.query_absorb_workspace_bytes(B * T, H), dtype=torch.uint8, device="cuda")
    ws_d = torch.empty(mla.workspace_bytes(B, H, T, 0, parts), dtype=torch.uint8, device="cuda")

    def set_lengths(lens):
        pos = lens - 1                        # the new token's position
        sl = w.block_table[np.arange(B), pos // 64].astype(np.int64) * 64 + pos % 64
        sk.copy_(torch.from_numpy(lens.astype(np.int32)))
        slots.copy_(torch.from_numpy(sl))

    def step():
        mla.query_absorb(qkv[:, :1536], w_qa, w_qb, w_uk, eps=qin.eps, out=q, workspace=ws_q)
        mla.kv_insert(qkv[:, W.KV_C_COL:W.KV_C_COL + 512], qkv[:, W.K_PE_COL:W.K_PE_COL + 64], w_kva,
                      slots, cache, eps=ins.eps, kv_scales=scales)
        md, ns = mla.metadata(sk, H, T, num_parts=parts)
        mla.decode(q.view(B, T, H, 576), cache, bt, sk, softmax_scale=w.softmax_scale, kv_scales=scales,
                   tile_md=md, num_splits=ns, workspace=ws_d, out=out, lse=lse)

    set_lengths(base_len + 1)
    g = _capture(step)
    for trial in range(3):
        lens = base_len + 1 + trial
        set_lengths(lens)
        if trial:
            qkv.normal_(0.0, 1.0, generator=torch.Generator("cuda").manual_seed(200 + trial))
        cache.copy_(cache0)
        scales.copy_(scales0)
        g.replay()
        torch.cuda.synchronize()
        res = [t.clone() for t in (q, cache, scales, out, lse)]
        cache.copy_(cache0)
        scales.copy_(scales0)
        step()
        torch.cuda.synchronize()
        for name, a, b in zip(("q", "cache", "scales", "out", "lse"), res, (q, cache, scales, out, lse)):
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), (trial, name)
        # the replay's attention against the oracle on its own query rows and cache
        w.q = res[0].view(B, T, H, 576).view(torch.int16).cpu().numpy().view(np.uint16)
        w.kv = res[1].cpu().numpy()
        w.kv_scales = res[2].cpu().numpy()
        w.cache_seqlens = lens.astype(np.int32)
        rows = [(b, 0, h) for b in range(B) for h in (0, 77, 127)]
        ref_o, ref_l = decode_rows(w, rows)
        got_o = np.stack([res[3][b, t, h].float().cpu().numpy() for b, t, h in rows])
        got_l = np.array([res[4][b, h, t].item() for b, t, h in rows])
        assert np.abs(got_o - ref_o).max() <= G.TOL_O
        assert np.abs(got_o - ref_o).max() <= G.TOL_O_REL * np.abs(ref_o).max()
        assert np.abs(got_l - ref_l).max() <= G.TOL_LSE
    assert mla.device_status() == 0

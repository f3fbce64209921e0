"""GPU parity of query absorption (mla_query_absorb) against the oracle,
stage by stage through the caller's workspace: the RMSNorm output bit-exact,
each bf16 dot product within one bf16 ulp of the exactly rounded value plus
the fp32 accumulation bound 2^-12 * sum |products|, the RoPE rows copied
bit for bit."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import kv_insert as K
from oracle import query_absorb as Q

pytestmark = pytest.mark.gpu


def _val(bits):
    return K.bf16_bits_to_f64(bits)


def _ulp(v):
    _, e = np.frexp(np.abs(v))
    return np.ldexp(1.0, np.maximum(e - 1, -126) - 7)


def _bf16_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def _run(inp, strided=True):
    import mla_decode_attention_05_gb300 as mla
    qkv = _bf16_dev(inp.qkv)
    q_a = qkv[:, :1536] if strided else qkv[:, :1536].contiguous()
    N, H = inp.N, inp.H
    ws = torch.zeros(mla.query_absorb_workspace_bytes(N, H), dtype=torch.uint8, device="cuda")
    q = mla.query_absorb(q_a, _bf16_dev(inp.w_qa), _bf16_dev(inp.w_qb), _bf16_dev(inp.w_uk), eps=inp.eps,
                         workspace=ws)
    torch.cuda.synchronize()
    xq_bytes = N * 1536 * 2
    off = (xq_bytes + 255) // 256 * 256
    xq = ws[:xq_bytes].cpu().numpy().view(np.uint16).reshape(N, 1536)
    qb = ws[off:off + N * H * 192 * 2].cpu().numpy().view(np.uint16).reshape(N, H, 192)
    return xq, qb, q.cpu().view(torch.int16).numpy().view(np.uint16)


def _check(inp, strided=True):
    xq, qb, q = _run(inp, strided)
    ref = Q.query_absorb(inp.qkv, inp.w_qa, inp.eps, inp.w_qb, inp.w_uk)
    np.testing.assert_array_equal(xq, ref["xq"])                       # exact definition
    # Q_B from the same xq
    got, want = _val(qb), _val(ref["qb"])
    bound = _ulp(want) + 2.0 ** -12 * ref["qb_mag"]
    assert np.all(np.abs(got - want) <= bound), float(np.max(np.abs(got - want) - bound))
    # W_UK from the GPU's own qb
    lat_ref, lat_mag = Q.w_uk_latent(qb, inp.w_uk)
    got_l, want_l = _val(q[:, :, :512]), _val(lat_ref)
    bound_l = _ulp(want_l) + 2.0 ** -12 * lat_mag
    assert np.all(np.abs(got_l - want_l) <= bound_l), float(np.max(np.abs(got_l - want_l) - bound_l))
    np.testing.assert_array_equal(q[:, :, 512:], qb[:, :, 128:])       # RoPE rows copied
    # end to end against the oracle alone: most values equal, all close
    full = _val(ref["q"])
    err = np.abs(_val(q) - full)
    assert np.mean(err <= _ulp(full)) > 0.98
    assert err.max() <= 0.02 * np.abs(full).max()


@pytest.mark.parametrize("N,H", [(1, 1), (5, 16), (37, 64), (64, 128), (129, 32), (300, 8)])
def test_query_absorb_stages(N, H):
    _check(W.make_query_inputs(N, H, seed=300 + N))


def test_contiguous_q_a_and_empty_call():
    import mla_decode_attention_05_gb300 as mla
    _check(W.make_query_inputs(9, 8, seed=41), strided=False)
    inp = W.make_query_inputs(1, 2, seed=42)
    out = torch.full((0, 2, 576), 7, dtype=torch.bfloat16, device="cuda")
    q = mla.query_absorb(_bf16_dev(inp.qkv)[:0, :1536], _bf16_dev(inp.w_qa), _bf16_dev(inp.w_qb),
                         _bf16_dev(inp.w_uk), eps=inp.eps, out=out)
    assert q.shape == (0, 2, 576)


def test_absorbed_query_feeds_decode():
    """q from the absorption, reshaped [B, T, H, 576], decoded: the decode's
    output matches the oracle's attention for that q."""
    import mla_decode_attention_05_gb300 as mla
    from oracle import decode_rows
    from _gpu import TOL_LSE, TOL_O
    w = W.make_workload("absorbed_q", 2, 1, 64, [300, 129], seed=51)
    inp = W.make_query_inputs(2, 64, seed=52)
    q = mla.query_absorb(_bf16_dev(inp.qkv)[:, :1536], _bf16_dev(inp.w_qa), _bf16_dev(inp.w_qb),
                         _bf16_dev(inp.w_uk), eps=inp.eps).view(2, 1, 64, 576)
    w.q = q.cpu().view(torch.int16).numpy().view(np.uint16)
    kv = torch.from_numpy(w.kv.view(np.int16)).view(torch.bfloat16).cuda()
    out, lse = mla.decode(q, kv, torch.from_numpy(w.block_table).cuda(), torch.from_numpy(w.cache_seqlens).cuda(),
                          softmax_scale=w.softmax_scale)
    torch.cuda.synchronize()
    rows = [(b, 0, h) for b in range(2) for h in (0, 31, 63)]
    ref_o, ref_l = decode_rows(w, rows)
    got_o = np.stack([out[b, t, h].float().cpu().numpy() for b, t, h in rows])
    got_l = np.array([lse[b, h, t].item() for b, t, h in rows])
    assert np.abs(got_o - ref_o).max() <= TOL_O
    assert np.abs(got_l - ref_l).max() <= TOL_LSE

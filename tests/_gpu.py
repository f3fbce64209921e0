"""Helpers of the GPU parity tests: move a seeded workload to the device, run
the library through its binding, compare with the oracle."""
import numpy as np
import torch

TOL_O = 2e-2      # max-abs on bf16 O
TOL_LSE = 1e-3    # max-abs on fp32 LSE
TOL_O_REL = 2e-2  # max-abs relative to max |O*| (keeps the absolute bound honest)


def to_device(w, device="cuda"):
    d = {}
    d["q"] = torch.from_numpy(w.q.view(np.int16)).view(torch.bfloat16).to(device)
    if w.kv_format == 0:
        d["kv"] = torch.from_numpy(w.kv.view(np.int16)).view(torch.bfloat16).to(device)
        d["scales"] = None
    else:
        d["kv"] = torch.from_numpy(w.kv).to(device)
        d["scales"] = torch.from_numpy(w.kv_scales).to(device)
    d["bt"] = torch.from_numpy(w.block_table).to(device)
    d["sk"] = torch.from_numpy(w.cache_seqlens).to(device)
    d["topk"] = None if w.topk is None else torch.from_numpy(w.topk).to(device)
    return d


def run(w, num_parts=None, record=False, dev=None):
    import mla_decode_attention_05_gb300 as mla
    d = dev if dev is not None else to_device(w)
    md, ns = mla.metadata(d["sk"], w.H, w.T, topk=w.topk_len, causal=w.causal,
                          num_parts=num_parts)
    gathered = None
    if record and w.topk is not None:
        gathered = torch.full(tuple(w.topk.shape), -7, dtype=torch.int32, device=d["q"].device)
    out, lse = mla.decode(d["q"], d["kv"], d["bt"], d["sk"], softmax_scale=w.softmax_scale,
                          causal=w.causal, topk_indices=d["topk"], kv_scales=d["scales"],
                          tile_md=md, num_splits=ns, gathered=gathered)
    torch.cuda.synchronize()
    res = dict(out=out.float().cpu().numpy().astype(np.float64),
               lse=lse.cpu().numpy().astype(np.float64), tile_md=md.cpu().numpy(),
               num_splits=ns.cpu().numpy())
    if gathered is not None:
        res["gathered"] = gathered.cpu().numpy()
    return res


def compare_rows(w, res, rows, oracle):
    """Element-by-element comparison of the given (b, t, h) rows."""
    ref_o, ref_l = oracle.decode_rows(w, rows)
    got_o = np.stack([res["out"][b, t, h] for b, t, h in rows])
    got_l = np.array([res["lse"][b, h, t] for b, t, h in rows])
    ninf = np.isneginf(ref_l)
    assert np.array_equal(np.isneginf(got_l), ninf), "empty-set rows must have LSE = -inf"
    assert np.all(got_o[ninf] == 0), "empty-set rows must have O = 0"
    err_o = np.abs(got_o - ref_o).max() if got_o.size else 0.0
    err_l = np.abs(got_l[~ninf] - ref_l[~ninf]).max() if (~ninf).any() else 0.0
    scale = max(np.abs(ref_o).max(), 1e-30) if ref_o.size else 1.0
    assert np.all(np.isfinite(got_o)), "non-finite output"
    assert err_o <= TOL_O, f"O max-abs error {err_o}"
    assert err_l <= TOL_LSE, f"LSE max-abs error {err_l}"
    if (~ninf).any():
        assert err_o / scale <= TOL_O_REL, f"O relative error {err_o / scale}"
    return err_o, err_l


def all_rows(w):
    return [(b, t, h) for b in range(w.B) for t in range(w.T) for h in range(w.H)]

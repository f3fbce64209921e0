"""Failure detection on the GPU without a fault: the decode kernel's waits
are bounded, and a wait that runs out sets MLA_STATUS_WAIT_TIMEOUT, makes
every role of the kernel give up at its next wait, drains the copies and MMAs
in flight, frees tensor memory and returns.  The tests shorten the limit of
every wait to a microsecond through the library's test hook, so that real
waits of an ordinary call run out (nothing is broken on purpose: inputs and
launch are valid), then check the status word, that the device is still
usable, and that a normal call right after gives the oracle's result."""
import numpy as np
import pytest
import torch

from workloads import make_workload

import _gpu as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mla():
    from mla_decode_attention_05_gb300 import build
    build.build()
    import mla_decode_attention_05_gb300 as m
    m.device_status()
    return m


CASES = [
    dict(name="dense", B=4, T=1, H=128, seqlens=[6000, 5000, 7000, 4000], kw={}),
    dict(name="gather_fp8", B=4, T=1, H=64, seqlens=[5000, 3000, 6000, 4000],
         kw=dict(topk=2048, topk_pad_count=100, fp8=True)),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c["name"])
def test_waits_run_out_then_next_call_is_correct(mla, oracle_mod, case):
    w = make_workload("timeout_" + case["name"], case["B"], case["T"], case["H"], case["seqlens"],
                      seed=41, **case["kw"])
    d = G.to_device(w)
    assert mla.device_status() == 0
    mla.set_wait_limit_ns(1000)          # 1 us: the pipeline's ordinary waits are longer
    try:
        md, ns = mla.metadata(d["sk"], w.H, w.T, topk=w.topk_len, causal=w.causal)
        mla.decode(d["q"], d["kv"], d["bt"], d["sk"], softmax_scale=w.softmax_scale,
                   causal=w.causal, topk_indices=d["topk"], kv_scales=d["scales"],
                   tile_md=md, num_splits=ns)
    finally:
        mla.set_wait_limit_ns(0)         # back to the default for everything after
    torch.cuda.synchronize()             # the kernel returned: no fault, no hang
    st = mla.device_status()
    assert st & mla.STATUS_WAIT_TIMEOUT, f"status {st}: no wait ran out"
    assert st & ~(mla.STATUS_WAIT_TIMEOUT) == 0
    # the same call with the default limit: a clean status and the oracle's answer
    res = G.run(w, dev=d, record=w.topk is not None)
    assert mla.device_status() == 0
    G.compare_rows(w, res, G.all_rows(w), oracle_mod)
    if w.topk is not None:
        for b in range(w.B):
            got = res["gathered"][b, 0]
            assert np.array_equal(np.sort(got[got >= 0]), oracle_mod.valid_keys(w, b, 0))

"""MLA decode benchmark: one JSON line on rank 0.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                    [--config I]

A step is one pass of the whole decode path over one batch: the split-KV
metadata kernel, the decode kernel and the LSE combine kernel, on the
variable-length workload (batch 64, one query token, 128 heads, cache
lengths uniform in [1024, 32768], 64-token pages, bf16) unless --config picks
another of the five named workloads.  `value` is KV-cache GB/s: the
algorithmic bytes (1152 per valid key for bf16 rows, 656 for e4m3 + scales +
bf16 RoPE) of the step divided by its device time, summed over ranks.
TFLOP/s counts 2*576 + 2*512 flops per (query row, valid key).

--impl reference times the float64 CPU oracle on the host cores on a
bounded, rotating sample of the same workload (one sequence per step, all
heads) and reports the same metric.

--op kv_insert times the cache producer instead (mla_kv_insert: RMSNorm of
each new token's latent row, per-128 FP8 quantisation, paged write) on
--tokens new tokens filling a cache of as many slots; `value` is its
algorithmic GB/s (1160 bytes read and 656 written per token).

--op query_absorb times the query path (mla_query_absorb: q_a RMSNorm, Q_B,
W_UK) for --tokens tokens (default 64) and 128 heads, with L2 flushed before
each call; `value` is GB/s of weights + q_a + q bytes.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "MLA decode KV-cache GB/s + TFLOP/s at B=64,H=128; % of HBM/tensor roofline"
DEFAULT_CONFIG = 3
L2_BYTES = 129 * 1024 * 1024


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def valid_counts(w):
    """Valid keys per (sequence, query token): the bench's own bookkeeping of
    algorithmic work (dense: s_k; causal: s_k - T + t + 1; top-k: slots that
    are not -1)."""
    c = np.zeros((w.B, w.T), dtype=np.int64)
    for b in range(w.B):
        sk = int(w.cache_seqlens[b])
        for t in range(w.T):
            if w.topk is not None:
                ids = w.topk[b, t]
                c[b, t] = len(set(int(i) for i in ids if 0 <= i < sk))
            elif w.causal:
                c[b, t] = min(max(sk - w.T + t + 1, 0), sk)
            else:
                c[b, t] = sk
    return c


def work_of(w, batches=None):
    """(KV bytes, flops) of the given sequences (all by default).  A key read
    once serves every head and, for dense/causal, every query token of the
    sequence, so KV bytes count each distinct key row once."""
    c = valid_counts(w)
    idx = range(w.B) if batches is None else batches
    per_key = workloads.kv_bytes_per_token(w.kv_format)
    kv = 0
    fl = 0
    for b in idx:
        if w.topk is not None:
            rows = set()
            for t in range(w.T):
                rows |= set(int(i) for i in w.topk[b, t] if 0 <= i < int(w.cache_seqlens[b]))
            kv += len(rows) * per_key
        else:
            kv += int(c[b].max()) * per_key
        fl += int(c[b].sum()) * w.H * workloads.FLOP_PER_ROW_KEY
    return kv, fl


class Clocks:
    """nvidia-smi sampling (every 10 ms) around the timed region."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.t0 = self.t1 = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(index), "-lms", "10"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def finish(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        return summarise_clocks(out, self.t0, self.t1)


def summarise_clocks(text: str, t0, t1) -> dict:
    """The `clocks` entry from nvidia-smi CSV rows (Clocks.FIELDS, no header,
    no units): median and maximum SM clock and the throttle reasons seen
    during [t0, t1] (local time, 50 ms of slack), or the sample nearest t0
    when none falls inside."""
    rows = []
    for line in text.strip().splitlines():
        parts = [x.strip() for x in line.split(",")]
        if len(parts) < 10:
            continue
        try:
            ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
            ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
            rows.append((ts, float(parts[2]), float(parts[3]), parts[5:]))
        except Exception:
            continue
    if not rows:
        return {"samples": 0}
    inside = [r for r in rows if t0 is not None and t0 - 0.05 <= r[0] <= t1 + 0.05]
    used = inside if inside else [min(rows, key=lambda r: abs(r[0] - (t0 or r[0])))]
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    reasons = set()
    for r in used:
        for n, v in zip(names, r[3][1:5]):
            if v.strip().lower() == "active":
                reasons.add(n)
    return {"sm_mhz": statistics.median(r[1] for r in used), "sm_max_mhz": max(r[2] for r in used),
            "reasons": sorted(reasons), "samples": len(used),
            "in_timed_region": bool(inside)}


def traffic_record(kernel_hash: str):
    """DRAM bytes per decode launch from the committed ncu summary, if it was
    taken on the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "decode_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("kernel_source_sha256") != kernel_hash:
        return None
    return d


# The sources the decode kernel is compiled from (its translation unit and
# the headers it includes): the traffic record holds only while they are
# unchanged.
DECODE_KERNEL_SOURCES = ("common.cuh", "decode_tc.cu", "ptx.cuh")


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mla_decode_attention_05_gb300", "csrc")
    for name in DECODE_KERNEL_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()


def device_parts(local: int) -> int:
    """Workers of the split-KV partition on this device: one cluster of two
    CTAs per two SMs (the library's default; 76 on a 152-SM GB300 when no
    device is visible)."""
    try:
        import torch
        n = int(torch.cuda.get_device_properties(local).multi_processor_count)
        return max(n // 2, 1)
    except Exception:
        return 76


def decode_config(w, steps: int, world: int, parts: int, l2_bytes: int):
    """The `config` object of a decode line, identical for the library's arm
    and the reference (oracle) arm: the workload and how the timed steps
    treat L2.  Returns (config, flush_l2)."""
    kv_bytes, flops = work_of(w)
    touched = step_bytes(w, kv_bytes)
    flush = touched < 2 * l2_bytes
    cfg = {"workload": w.name, "B": w.B, "T": w.T, "H": w.H,
           "kv_format": "bf16" if w.kv_format == 0 else "fp8_e4m3",
           "causal": w.causal, "topk": w.topk_len, "page_size": 64, "num_parts": parts,
           "kv_bytes": kv_bytes, "flops": flops, "seed": w.seed,
           "l2": l2_label(touched, l2_bytes, flush),
           "parallelism": f"weak, {world} independent replica(s)",
           "kernel_timing": f"decode kernel duration from a second {steps}-step loop with CUDA events around "
                            "each decode launch"}
    return cfg, flush


def insert_config(N: int, num_pages: int, world: int) -> dict:
    """The `config` of a KV-insert line (both arms)."""
    return {"workload": f"kv_insert_fp8_tile_n{N}", "tokens": N, "page_size": 64,
            "num_pages": num_pages, "bytes_per_token": INSERT_BYTES_PER_TOKEN,
            "l2": f"{N * INSERT_BYTES_PER_TOKEN / 1e6:.0f} MB touched per step vs {L2_BYTES / 1e6:.0f} MB L2; no flush",
            "parallelism": f"weak, {world} independent replica(s)"}


def query_config(N: int, H: int, world: int) -> dict:
    """The `config` of a query-absorption line (both arms)."""
    return {"workload": f"query_absorb_n{N}_h{H}", "tokens": N, "H": H, "bytes": query_bytes(N, H),
            "l2": "256 MB written before every timed call (weights 92 MB would otherwise stay in L2)",
            "gemms": "Q_B and W_UK: this library's tcgen05 kernels (bf16, fp32 accumulate in TMEM)",
            "parallelism": f"weak, {world} independent replica(s)"}


def device_l2_bytes(local: int) -> int:
    """L2 size of the device (the nominal GB300 figure if torch does not
    report it)."""
    try:
        import torch
        n = int(getattr(torch.cuda.get_device_properties(local), "L2_cache_size", 0))
        return n if n > 0 else L2_BYTES
    except Exception:
        return L2_BYTES


def step_bytes(w, kv_bytes: int) -> int:
    """Bytes one decode step touches in memory: the KV rows it reads (each
    distinct row once), the query rows, and the output and LSE it writes."""
    rows = w.B * w.T * w.H
    return int(kv_bytes) + rows * 576 * 2 + rows * 512 * 2 + rows * 4


def l2_label(touched: int, l2_bytes: int, flushed: bool) -> str:
    """The `config.l2` entry: what a step touches against the L2, and whether
    the L2 was flushed between timed steps."""
    head = f"{touched / 1e6:.1f} MB touched per step vs {l2_bytes / 1e6:.1f} MB L2"
    if flushed:
        return head + f"; L2 flushed before every timed step ({2 * l2_bytes / 1e6:.0f} MB written, outside the timed events)"
    return head + "; inputs larger than twice the L2, no flush"


def subset(w, nb: int):
    """The first nb sequences of a workload (the page pool is kept whole)."""
    import dataclasses
    nb = min(nb, w.B)
    return dataclasses.replace(
        w, name=f"{w.name}[:{nb}]", B=nb, q=w.q[:nb].copy(), block_table=w.block_table[:nb].copy(),
        cache_seqlens=w.cache_seqlens[:nb].copy(), topk=None if w.topk is None else w.topk[:nb].copy())


def dist_setup(gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def cpu_baseline(w, budget_s: float = 12.0):
    """The oracle as it stands on the host cores: whole sequences (all heads)
    in order until about budget_s seconds of work; GB/s of their KV bytes."""
    import oracle
    done = []
    t0 = time.perf_counter()
    for b in range(w.B):
        rows = [(b, t, h) for t in range(w.T) for h in range(w.H)]
        oracle.decode_rows(w, rows)
        done.append(b)
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    kv, fl = work_of(w, done)
    return {"value": kv / dt / 1e9, "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"sequences 0..{done[-1]} of {w.B} ({len(done)} x {w.T * w.H} rows, "
                      f"{kv / 1e6:.1f} MB of KV) in {dt:.1f} s, float64",
            "tflops": fl / dt / 1e12}


def run_gpu(args, w, world, rank, local, l2_bytes):
    import torch
    import mla_decode_attention_05_gb300 as mla
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    # nvidia-smi takes a moment to start sampling: start it before the
    # inputs are uploaded so that it is running through the timed region
    clocks = Clocks(local) if rank == 0 else None
    stream = torch.cuda.current_stream(dev)
    q_h = torch.from_numpy(w.q.view(np.int16)).view(torch.bfloat16)
    if w.kv_format == workloads.KV_BF16:
        kv_h = torch.from_numpy(w.kv.view(np.int16)).view(torch.bfloat16)
        sc_h = None
    else:
        kv_h = torch.from_numpy(w.kv)
        sc_h = torch.from_numpy(w.kv_scales)
    bt_h = torch.from_numpy(w.block_table)
    sk_h = torch.from_numpy(w.cache_seqlens)
    tk_h = None if w.topk is None else torch.from_numpy(w.topk)
    host = [x for x in (q_h, kv_h, sc_h, bt_h, sk_h, tk_h) if x is not None]
    q, kv, bt, sk = (x.to(dev) for x in (q_h, kv_h, bt_h, sk_h))
    sc = None if sc_h is None else sc_h.to(dev)
    tk = None if tk_h is None else tk_h.to(dev)
    parts = mla.default_num_parts(dev)
    topk = w.topk_len
    ws = torch.empty(mla.workspace_bytes(w.B, w.H, w.T, topk, parts), dtype=torch.uint8, device=dev)
    out = torch.empty((w.B, w.T, w.H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.H, w.T), dtype=torch.float32, device=dev)
    md = torch.empty((parts, 8), dtype=torch.int32, device=dev)
    nitems = mla.num_items(w.B, w.H, w.T, topk)
    ns = torch.empty(nitems + 1, dtype=torch.int32, device=dev)
    L = mla.lib()
    import ctypes
    P = ctypes.c_void_p
    sptr = P(stream.cuda_stream)

    def step(qq, kk, bb, ss, ss_sc, tt, oo, ll):
        rc = L.mla_decode_metadata(P(ss.data_ptr()), w.B, w.H, w.T, topk, int(w.causal), parts,
                                   P(md.data_ptr()), P(ns.data_ptr()), sptr)
        if rc != 0:
            raise RuntimeError(L.mla_last_error_string().decode())
        rc = L.mla_decode(P(qq.data_ptr()), P(kk.data_ptr()), w.kv_format, w.num_pages, 64,
                          P(bb.data_ptr()), w.max_pages, P(ss.data_ptr()),
                          None if tt is None else P(tt.data_ptr()), topk, None,
                          None if ss_sc is None else P(ss_sc.data_ptr()),
                          ctypes.c_float(w.softmax_scale), int(w.causal), P(md.data_ptr()),
                          P(ns.data_ptr()), parts, P(ws.data_ptr()), ws.numel(),
                          P(oo.data_ptr()), P(ll.data_ptr()), w.B, w.T, w.H, sptr)
        if rc != 0:
            raise RuntimeError(L.mla_last_error_string().decode())

    launches_per_step = 3  # metadata, decode, combine
    # A step that touches less than twice the L2 would find its inputs in L2
    # from the step before: write a buffer of twice the L2 before each such
    # timed step (outside the timed events) so that they come from HBM.
    flush = torch.empty(2 * l2_bytes, dtype=torch.uint8, device=dev) if args.flush_l2 else None
    for _ in range(args.warmup):
        step(q, kv, bt, sk, sc, tk, out, lse)
    torch.cuda.synchronize()
    K = args.steps
    ev_b = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev_a = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    st_b = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    st_a = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    for e in ev_b + ev_a + st_b + st_a:   # create the underlying events before handing them over
        e.record(stream)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    if clocks:
        clocks.mark_start()
    # 1. the steps as a user runs them: nothing between the three kernels
    #    (with the L2 flush: events around each step, the flush between)
    start.record(stream)
    for i in range(K):
        if flush is not None:
            flush.fill_(i & 0xFF)
            st_b[i].record(stream)
        step(q, kv, bt, sk, sc, tk, out, lse)
        if flush is not None:
            st_a[i].record(stream)
    end.record(stream)
    # 2. the same steps with events around each decode kernel (an event
    #    between two kernels stops the second one from starting early, so
    #    this loop only serves the kernel's own duration)
    for i in range(K):
        if flush is not None:
            flush.fill_(i & 0xFF)
        mla.profile_events(ev_b[i], ev_a[i])
        step(q, kv, bt, sk, sc, tk, out, lse)
    mla.profile_events()
    torch.cuda.synchronize()
    if clocks:
        clocks.mark_end()
    barrier(world)
    if flush is not None:
        total_ms = sum(b.elapsed_time(a) for b, a in zip(st_b, st_a))
    else:
        total_ms = start.elapsed_time(end)
    kern_ms = [b.elapsed_time(a) for b, a in zip(ev_b, ev_a)]
    status = mla.device_status()
    clk = clocks.finish() if clocks else None

    # end to end through the C ABI with host buffers: pinned host -> device
    # copies of every input, the three kernels, device -> host of out + lse
    pinned = [x.pin_memory() for x in host]
    dev_bufs = [torch.empty_like(x, device=dev) for x in host]
    o_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    l_h = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    h2d = sum(x.numel() * x.element_size() for x in host)
    d2h = out.numel() * out.element_size() + lse.numel() * lse.element_size()
    names = [n for n, x in zip(("q", "kv", "sc", "bt", "sk", "tk"), (q_h, kv_h, sc_h, bt_h, sk_h, tk_h)) if x is not None]
    D = dict(zip(names, dev_bufs))

    def e2e_step():
        for hb, db in zip(pinned, dev_bufs):
            db.copy_(hb, non_blocking=True)
        step(D["q"], D["kv"], D["bt"], D["sk"], D.get("sc"), D.get("tk"), out, lse)
        o_h.copy_(out, non_blocking=True)
        l_h.copy_(lse, non_blocking=True)

    Ke = max(3, min(K, 20))
    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s2.record(stream)
    for _ in range(Ke):
        e2e_step()
    e2.record(stream)
    torch.cuda.synchronize()
    e2e_ms = s2.elapsed_time(e2) / Ke
    return dict(total_ms=total_ms, kern_ms=kern_ms, status=status, clocks=clk, parts=parts,
                e2e_ms=e2e_ms, h2d=h2d, d2h=d2h, launches=launches_per_step * K,
                kernel_timing_steps=K)


# --- KV insert ------------------------------------------------------------------

INSERT_METRIC = "MLA KV insert GB/s (RMSNorm + per-128 FP8 quantise + paged write); % of HBM roofline"
INSERT_BYTES_PER_TOKEN = 1024 + 128 + 8 + 640 + 16  # latent + k_pe + slot read; FP8 row + 4 scales written


def insert_workload(n_tokens: int):
    """n_tokens new tokens, one per slot of a cache of exactly n_tokens slots
    (64-token pages), FP8 rows with per-128 scales."""
    pages = (n_tokens + 63) // 64
    return workloads.make_insert_inputs(n_tokens, pages, 64, seed=4242, skip_every=0)


def insert_cpu_baseline(inp, budget_s: float = 10.0):
    from oracle import kv_insert as OK
    kv = inp.qkv[:, workloads.KV_C_COL:]
    pe = inp.qkv[:, workloads.K_PE_COL:]
    t0 = time.perf_counter()
    done = 0
    while time.perf_counter() - t0 < budget_s and done < inp.N:
        OK.insert_row(OK.FMT_FP8_TILE, kv[done, :512], pe[done, :64], inp.w_kva, inp.eps)
        done += 1
    dt = time.perf_counter() - t0
    return {"value": done * INSERT_BYTES_PER_TOKEN / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"tokens 0..{done - 1} of {inp.N} ({done} rows) in {dt:.1f} s, one row at a time"}


def run_insert(args, world, rank, local, hbm, peak_src):
    import ctypes
    import torch
    import mla_decode_attention_05_gb300 as mla
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    clocks = Clocks(local) if rank == 0 else None
    inp = insert_workload(args.tokens)
    N = inp.N
    stream = torch.cuda.current_stream(dev)
    qkv_h = torch.from_numpy(inp.qkv.view(np.int16)).view(torch.bfloat16)
    qkv = qkv_h.to(dev)
    w_kva = torch.from_numpy(inp.w_kva.view(np.int16)).view(torch.bfloat16).to(dev)
    slots_h = torch.from_numpy(inp.slots)
    slots = slots_h.to(dev)
    cache = torch.zeros((inp.num_pages, 64, 640), dtype=torch.uint8, device=dev)
    scales = torch.zeros((inp.num_pages, 64, 4), dtype=torch.float32, device=dev)
    L = mla.lib()
    P = ctypes.c_void_p
    sptr = P(stream.cuda_stream)
    ld = qkv.stride(0)

    def step(src, sl, ld_):
        rc = L.mla_kv_insert(P(src.data_ptr() + 2 * workloads.KV_C_COL), ld_, P(src.data_ptr() + 2 * workloads.K_PE_COL),
                             ld_, P(w_kva.data_ptr()), ctypes.c_float(inp.eps), P(sl.data_ptr()), N,
                             P(cache.data_ptr()), mla.KV_FP8_E4M3, inp.num_pages, 64, P(scales.data_ptr()),
                             None, sptr)
        if rc != 0:
            raise RuntimeError(L.mla_last_error_string().decode())

    for _ in range(args.warmup):
        step(qkv, slots, ld)
    torch.cuda.synchronize()
    K = args.steps
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(K + 1)]
    barrier(world)
    torch.cuda.synchronize()
    if clocks:
        clocks.mark_start()
    for i in range(K):
        evs[i].record(stream)
        step(qkv, slots, ld)
    evs[K].record(stream)
    torch.cuda.synchronize()
    if clocks:
        clocks.mark_end()
    barrier(world)
    per = [evs[i].elapsed_time(evs[i + 1]) for i in range(K)]
    total_ms = evs[0].elapsed_time(evs[K])
    status = mla.device_status()
    clk = clocks.finish() if clocks else None

    # end to end: the token rows (latent + k_pe, 1152 bytes) and slots from
    # pinned host memory, the insert, the written cache and scales back
    rows_h = torch.cat([qkv_h[:, workloads.KV_C_COL:workloads.KV_C_COL + 512],
                        qkv_h[:, workloads.K_PE_COL:workloads.K_PE_COL + 64]], dim=1).contiguous().pin_memory()
    sl_pin = slots_h.pin_memory()
    rows_d = torch.empty_like(rows_h, device=dev)
    sl_d = torch.empty_like(sl_pin, device=dev)
    cache_h = torch.empty(cache.shape, dtype=cache.dtype).pin_memory()
    scales_h = torch.empty(scales.shape, dtype=scales.dtype).pin_memory()

    def e2e_step():
        rows_d.copy_(rows_h, non_blocking=True)
        sl_d.copy_(sl_pin, non_blocking=True)
        rc = L.mla_kv_insert(P(rows_d.data_ptr()), 576, P(rows_d.data_ptr() + 1024), 576, P(w_kva.data_ptr()),
                             ctypes.c_float(inp.eps), P(sl_d.data_ptr()), N, P(cache.data_ptr()),
                             mla.KV_FP8_E4M3, inp.num_pages, 64, P(scales.data_ptr()), None, sptr)
        if rc != 0:
            raise RuntimeError(L.mla_last_error_string().decode())
        cache_h.copy_(cache, non_blocking=True)
        scales_h.copy_(scales, non_blocking=True)

    Ke = max(3, min(K, 20))
    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s2.record(stream)
    for _ in range(Ke):
        e2e_step()
    e2.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(s2.elapsed_time(e2) / Ke, world)
    step_ms = max_over_ranks(total_ms / K, world)
    kern_ms = max_over_ranks(statistics.mean(per), world)
    if rank != 0:
        return
    nbytes = N * INSERT_BYTES_PER_TOKEN + 1024
    k_gbs = nbytes / (kern_ms * 1e-3) / 1e9
    line = {
        "metric": INSERT_METRIC, "value": world * nbytes / (step_ms * 1e-3) / 1e9, "unit": "GB/s",
        "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16->e4m3", "data": "synthetic",
        "tokens_per_s": world * N / (step_ms * 1e-3),
        "config": insert_config(N, inp.num_pages, world),
        "roofline": {"bound": "hbm", "achieved": k_gbs, "peak": hbm, "unit": "GB/s", "frac": k_gbs / hbm,
                     "traffic": None, "kernel_ms": kern_ms,
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured" else peak_src},
        "e2e": {"value": world * nbytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": rows_h.numel() * 2 + sl_pin.numel() * 8,
                "d2h_bytes_per_step": cache.numel() + scales.numel() * 4},
        "gpu_launches": K, "device_status": status, "clocks": clk,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = insert_cpu_baseline(inp)
    print(json.dumps(line), flush=True)


# --- query absorption --------------------------------------------------------------

QUERY_METRIC = "MLA query absorption GB/s (q_a RMSNorm + Q_B + W_UK, B=64 tokens, H=128); % of HBM roofline"


def query_bytes(N: int, H: int) -> int:
    """Algorithmic bytes of one call: the two weight matrices, w_qa, the q_a
    rows read and the query rows written."""
    return H * 192 * 1536 * 2 + H * 128 * 512 * 2 + 1536 * 2 + N * 1536 * 2 + N * H * 576 * 2


def query_cpu_baseline(inp, budget_s: float = 10.0):
    from oracle import query_absorb as OQ
    t0 = time.perf_counter()
    done = 0
    while time.perf_counter() - t0 < budget_s and done < inp.N:
        OQ.query_absorb(inp.qkv[done:done + 1], inp.w_qa, inp.eps, inp.w_qb, inp.w_uk)
        done += 1
    dt = time.perf_counter() - t0
    per_token = query_bytes(1, inp.H)
    return {"value": done * per_token / dt / 1e9, "unit": "GB/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"tokens 0..{done - 1} of {inp.N}, one call per token (all weights each), {dt:.1f} s, float64"}


def run_query(args, world, rank, local, hbm, peak_src):
    import ctypes
    import torch
    import mla_decode_attention_05_gb300 as mla
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    clocks = Clocks(local) if rank == 0 else None
    N, H = args.tokens, 128
    inp = workloads.make_query_inputs(N, H, seed=4343)
    stream = torch.cuda.current_stream(dev)
    t16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    qkv_h = t16(inp.qkv)
    qkv = qkv_h.to(dev)
    w_qa, w_qb, w_uk = (t16(a).to(dev) for a in (inp.w_qa, inp.w_qb, inp.w_uk))
    q = torch.empty((N, H, 576), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(mla.query_absorb_workspace_bytes(N, H), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)  # > L2: weights come from HBM
    L = mla.lib()
    P = ctypes.c_void_p
    sptr = P(stream.cuda_stream)

    def step(src, ld, out):
        rc = L.mla_query_absorb(P(src.data_ptr()), ld, P(w_qa.data_ptr()), ctypes.c_float(inp.eps),
                                P(w_qb.data_ptr()), P(w_uk.data_ptr()), N, H, P(out.data_ptr()), P(ws.data_ptr()),
                                ws.numel(), sptr)
        if rc != 0:
            raise RuntimeError(L.mla_last_error_string().decode())

    for _ in range(args.warmup):
        flush.zero_()
        step(qkv, qkv.stride(0), q)
    torch.cuda.synchronize()
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    barrier(world)
    torch.cuda.synchronize()
    if clocks:
        clocks.mark_start()
    for i in range(K):
        flush.zero_()
        ev[i][0].record(stream)
        step(qkv, qkv.stride(0), q)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    if clocks:
        clocks.mark_end()
    barrier(world)
    per = [a.elapsed_time(b) for a, b in ev]
    status = mla.device_status()
    clk = clocks.finish() if clocks else None

    # end to end: q_a rows from pinned host memory, the call, q back
    qa_h = qkv_h[:, :1536].contiguous().pin_memory()
    qa_d = torch.empty_like(qa_h, device=dev)
    q_h = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    Ke = max(3, min(K, 20))
    times = []
    for i in range(Ke + 2):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        qa_d.copy_(qa_h, non_blocking=True)
        step(qa_d, 1536, q)
        q_h.copy_(q, non_blocking=True)
        b.record(stream)
        torch.cuda.synchronize()
        if i >= 2:
            times.append(a.elapsed_time(b))
    step_ms = max_over_ranks(statistics.mean(per), world)
    e2e_ms = max_over_ranks(statistics.mean(times), world)
    if rank != 0:
        return
    nbytes = query_bytes(N, H)
    gbs = nbytes / (step_ms * 1e-3) / 1e9
    line = {
        "metric": QUERY_METRIC, "value": world * gbs, "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (random weights of the layer's shapes)",
        "config": query_config(N, H, world),
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                     "traffic": None, "kernel_ms": step_ms,
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured" else peak_src},
        "e2e": {"value": world * nbytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": qa_h.numel() * 2, "d2h_bytes_per_step": q_h.numel() * 2},
        "gpu_launches": 2 * K, "device_status": status, "clocks": clk,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = query_cpu_baseline(inp)
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--config", type=int, default=DEFAULT_CONFIG)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch", type=int, default=0,
                    help="keep only the first BATCH sequences of the workload (same values; "
                         "used for small profiling cases)")
    ap.add_argument("--op", default="decode", choices=["decode", "kv_insert", "query_absorb"],
                    help="decode: the attention path (default); kv_insert: the cache producer; "
                         "query_absorb: the query rows from q_a")
    ap.add_argument("--tokens", type=int, default=None,
                    help="new tokens per step (kv_insert: 262144; query_absorb: 64)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    world, rank, local = dist_setup(args.gpus)
    hbm, tf_burst, tf_sust, peak_src = load_peaks()

    if args.tokens is None:
        args.tokens = 64 if args.op == "query_absorb" else 262144
    if args.op == "query_absorb":
        if args.impl == "reference":
            if rank != 0:
                return
            inp = workloads.make_query_inputs(args.tokens, 128, seed=4343)
            cb = query_cpu_baseline(inp, budget_s=min(60.0, 1.0 * (args.steps + args.warmup)))
            print(json.dumps({"impl": "reference", "metric": QUERY_METRIC, "value": cb["value"], "unit": "GB/s",
                              "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                              "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                              "data": "synthetic", "config": query_config(inp.N, 128, args.gpus),
                              "cpu_baseline": cb,
                              "e2e": {"value": cb["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                                      "d2h_bytes_per_step": 0}}), flush=True)
            return
        run_query(args, world, rank, local, hbm, peak_src)
        return
    if args.op == "kv_insert":
        if args.impl == "reference":
            if rank != 0:
                return
            inp = insert_workload(args.tokens)
            cb = insert_cpu_baseline(inp, budget_s=min(60.0, 0.5 * (args.steps + args.warmup)))
            print(json.dumps({"impl": "reference", "metric": INSERT_METRIC, "value": cb["value"], "unit": "GB/s",
                              "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                              "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
                              "data": "synthetic", "config": insert_config(inp.N, inp.num_pages, args.gpus),
                              "cpu_baseline": cb,
                              "e2e": {"value": cb["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                                      "d2h_bytes_per_step": 0}}), flush=True)
            return
        run_insert(args, world, rank, local, hbm, peak_src)
        return

    if args.impl == "reference":
        if rank != 0:
            return
        w = workloads.config(args.config)
        import oracle
        order = list(range(w.B))
        per = []
        done_kv = 0
        for i in range(args.warmup + args.steps):
            b = order[i % w.B]
            rows = [(b, t, h) for t in range(w.T) for h in range(w.H)]
            t0 = time.perf_counter()
            oracle.decode_rows(w, rows)
            dt = time.perf_counter() - t0
            if i >= args.warmup:
                kvb, _ = work_of(w, [b])
                per.append((dt, kvb))
        tot_t = sum(p[0] for p in per)
        tot_kv = sum(p[1] for p in per)
        val = tot_kv / tot_t / 1e9
        line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "GB/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_t / len(per),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic",
                "config": decode_config(w, args.steps, args.gpus, device_parts(local), device_l2_bytes(local))[0],
                "cpu_baseline": {"value": val, "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
                                 "sample": f"one sequence (all {w.T * w.H} query rows) per step, rotating over the {w.B} sequences"},
                "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    w = workloads.config(args.config)
    if args.batch:
        w = subset(w, args.batch)
    kv_bytes, flops = work_of(w)
    l2_bytes = device_l2_bytes(local)
    config, args.flush_l2 = decode_config(w, args.steps, world, device_parts(local), l2_bytes)
    r = run_gpu(args, w, world, rank, local, l2_bytes)
    step_ms = max_over_ranks(r["total_ms"] / args.steps, world)
    kern_ms = statistics.mean(r["kern_ms"])
    kern_ms_max = max_over_ranks(kern_ms, world)
    e2e_ms = max_over_ranks(r["e2e_ms"], world)
    if rank != 0:
        return
    gbs = world * kv_bytes / (step_ms * 1e-3) / 1e9
    tflops = world * flops / (step_ms * 1e-3) / 1e12
    roof_us = max(kv_bytes / (hbm * 1e9), flops / (tf_burst * 1e12)) * 1e6
    bound = "hbm" if kv_bytes / hbm >= flops / (tf_burst * 1e3) else "tensor"
    k_gbs = kv_bytes / (kern_ms_max * 1e-3) / 1e9
    k_tf = flops / (kern_ms_max * 1e-3) / 1e12
    tr = traffic_record(kernel_source_hash())
    if bound == "hbm":
        roof = {"bound": "hbm", "achieved": k_gbs, "peak": hbm, "unit": "GB/s", "frac": k_gbs / hbm,
                "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured" else peak_src}
    else:
        roof = {"bound": "tensor", "achieved": k_tf, "peak": tf_burst, "unit": "TFLOP/s", "frac": k_tf / tf_burst,
                "peak_source": f"{peak_src} bf16 burst"}
    roof["traffic"] = None if tr is None else tr["dram_bytes_per_launch"]
    roof["kernel_ms"] = kern_ms_max
    roof["tflops"] = k_tf
    roof["frac_of_roofline_time"] = (roof_us * 1e-3) / kern_ms_max
    line = {
        "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "tflops": tflops, "roofline_time_us": roof_us, "frac_of_roofline": (roof_us * 1e-3) / step_ms,
        "config": config,
        "roofline": roof,
        "e2e": {"value": world * kv_bytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"]},
        "gpu_launches": r["launches"],
        "device_status": r["status"],
        "clocks": r["clocks"],
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w)
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()

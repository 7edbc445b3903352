"""Helpers for the GPU parity tests: move a workload to the device behind the
C ABI, and run the fp64 oracle on (a sample of) the same inputs."""
from __future__ import annotations

import numpy as np
import torch

import workloads
from oracle import oracle as O

PAGE = 16
TOL = {torch.bfloat16: 2e-3, torch.float32: 1e-5}


def device_cache(pkv, w, canary: bool = False, first_valid=None):
    """PagedKVCache over copies of w's pools on cuda.  With canary=True each
    pool is a slice of a larger buffer whose margins hold a sentinel, so an
    out-of-range write shows up in check_canaries()."""
    dev = torch.device("cuda")
    ks, vs, guards = [], [], []
    for t in w.k + w.v:
        if canary:
            n = t.numel()
            buf = torch.full((n + 2 * 4096,), 7.0, dtype=t.dtype, device=dev)
            view = buf[4096:4096 + n].view(t.shape)
            view.copy_(t)
            guards.append(buf)
        else:
            view = t.to(dev).contiguous()
        (ks if len(ks) < len(w.k) else vs).append(view)
    fv = None if first_valid is None else torch.as_tensor(first_valid, dtype=torch.int32).to(dev)
    cache = pkv.PagedKVCache(ks, vs, w.block_table.to(dev), ring_rows=w.ring_rows, bucket=w.bucket,
                             first_valid=fv)
    cache._guards = guards
    return cache


def check_canaries(cache):
    for buf in getattr(cache, "_guards", []):
        head, tail = buf[:4096], buf[-4096:]
        assert bool((head == 7.0).all()) and bool((tail == 7.0).all()), "write outside a pool"


def guarded_out(rows, hq, d):
    buf = torch.full((rows * hq * d + 2048,), 5.0, device="cuda")
    return buf, buf[1024:1024 + rows * hq * d].view(rows, hq, d)


def check_guarded(buf):
    assert bool((buf[:1024] == 5.0).all()) and bool((buf[-1024:] == 5.0).all()), "write outside the output"


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def compact_ids(w, segs, num_blocks: int):
    """Pool page ids the segments `segs` reach, in order, and per segment its
    relabelled table row (-1 for a page the table does not list)."""
    bt = w.block_table.cpu().numpy()
    si = w.seq_info.cpu().numpy()
    ids, rows = [], []
    for s in segs:
        q0, ql, col, kend = (int(x) for x in si[s])
        span = w.ring_rows if w.ring_rows else kend
        npg = (span + PAGE - 1) // PAGE
        row = []
        for pg in range(npg):
            b = int(bt[col, pg])
            if 0 <= b < num_blocks:
                row.append(len(ids))
                ids.append(b)
            else:          # a page the table does not list (e.g. a ring not yet grown to it)
                row.append(-1)
        rows.append(row)
    return ids, rows


def compact(w, layer: int, segs, k_pool: torch.Tensor, v_pool: torch.Tensor):
    """Pool, table and segment table holding only the pages `segs` reach, so
    the oracle runs on a small input.  Block ids are relabelled; the gather
    through the table (and hence the result) is unchanged."""
    si = w.seq_info.cpu().numpy()
    ids, rows = compact_ids(w, segs, k_pool.shape[0])
    mb = max(len(r) for r in rows) if rows else 1
    new_bt = np.full((len(segs), max(mb, 1)), -1, np.int32)
    for i, r in enumerate(rows):
        new_bt[i, :len(r)] = r
    sel = torch.tensor(ids, dtype=torch.long, device=k_pool.device)
    kp = k_pool.index_select(0, sel)
    vp = v_pool.index_select(0, sel)
    new_si = []
    for i, s in enumerate(segs):
        q0, ql, col, kend = (int(x) for x in si[s])
        new_si.append([q0, ql, i, kend])
    return kp, vp, new_bt, np.array(new_si, np.int32)


def oracle_pools(w, layer: int):
    """The pools of layer `layer` after the oracle's own append of this step
    (host tensors).  Oracle inputs never come from the device."""
    kp, vp, err = oracle_append_pools(w, layer)
    assert err == 0
    kt, vt = torch.from_numpy(kp), torch.from_numpy(vp)
    if w.dtype == torch.bfloat16:
        kt, vt = kt.view(torch.bfloat16), vt.view(torch.bfloat16)
    return kt, vt


def oracle_attend(w, layer: int, segs=None, causal=None, window=None, first_valid=None):
    """fp64 oracle on layer `layer` for the segments `segs` (all by default),
    over the oracle-appended pools.  Returns (out, lse) over all rows; rows of
    other segments are zero.  first_valid is indexed by the table row."""
    si = w.seq_info.cpu().numpy()
    segs = list(range(si.shape[0])) if segs is None else list(segs)
    k_pool, v_pool = oracle_pools(w, layer)
    kp, vp, bt, sub = compact(w, layer, segs, k_pool, v_pool)
    fv = None
    if first_valid is not None:   # compact() renumbers the table rows 0..len(segs)-1
        fv = np.array([int(first_valid[int(si[s, 2])]) for s in segs], np.int32)
    out, lse, err = O.attend(f64(w.q[layer]), f64(kp), f64(vp), bt, sub, w.scale,
                             causal=w.causal if causal is None else causal,
                             window=w.window if window is None else window, ring_rows=w.ring_rows,
                             first_valid=fv)
    assert err == 0, f"oracle rejected the workload: {err:#x}"
    return out, lse


def rows_of(w, segs):
    si = w.seq_info.cpu().numpy()
    rows = []
    for s in segs:
        q0, ql = int(si[s, 0]), int(si[s, 1])
        rows.extend(range(q0, q0 + ql))
    return rows


def oracle_append_pools(w, layer: int):
    """Byte copies of the pools after the oracle's append of layer `layer`."""
    kp = w.k[layer].cpu().numpy().copy() if w.dtype != torch.bfloat16 else \
        w.k[layer].cpu().view(torch.int16).numpy().copy()
    vp = w.v[layer].cpu().numpy().copy() if w.dtype != torch.bfloat16 else \
        w.v[layer].cpu().view(torch.int16).numpy().copy()
    kn = w.k_new[layer].cpu()
    vn = w.v_new[layer].cpu()
    if w.dtype == torch.bfloat16:
        kn, vn = kn.view(torch.int16), vn.view(torch.int16)
    err = O.append(kp, vp, w.block_table.cpu().numpy(), w.seq_info.cpu().numpy(), kn.numpy(), vn.numpy(),
                   ring_rows=w.ring_rows, window=w.window, causal=w.causal)
    return kp, vp, err


def pool_bytes(t: torch.Tensor) -> bytes:
    if t.dtype == torch.bfloat16:
        t = t.view(torch.int16)
    return t.cpu().numpy().tobytes()


def nan_tails(w):
    workloads.nan_fill_unused(w)
    return w

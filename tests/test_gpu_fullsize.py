"""Parity at the sizes the benchmark times.

Every workload of the benchmark's scope-table list (batched varlen, the two
speculative-verify calls, the two long-context calls) is drawn with the
benchmark's own generator, seed and sizes and run once through the fused
append + attention call in the benchmark's launch configuration (max_q_len
and max_kv as the benchmark passes them, automatic split count, cluster
merge).  The oracle cannot run a whole call at these sizes in seconds, so:

* every row of a few sampled segments (the longest key range, the most rows,
  a seeded random one) is compared element by element with the fp64 oracle
  run on just the pages those segments reach;
* for every segment, the pages its new rows land in are compared byte for
  byte with the oracle's append applied to the same pages.

Slots no segment may read hold NaN, as in the reduced parity tests.
"""
import numpy as np
import pytest
import torch

import bench
import workloads
from oracle import oracle as O
from tests import gpu_util as U

pytestmark = pytest.mark.gpu

PAGE = 16


@pytest.fixture(scope="module")
def pkv():
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_decode_13_gb300 as m
    return m


def _sampled(si: np.ndarray, k: int) -> list:
    """The segment with the longest key range, the one with the most rows and
    a seeded random other, without repeats (at most k)."""
    S = si.shape[0]
    picks = [int(np.argmax(si[:, 3])), int(np.argmax(si[:, 1]))]
    rng = np.random.default_rng(1234)
    picks.append(int(rng.integers(0, S)))
    out = []
    for s in picks:
        if s not in out:
            out.append(s)
    return out[:k]


def _bytes(t: torch.Tensor) -> np.ndarray:
    return t.cpu().view(torch.int16).numpy().copy()


def _touched(w) -> tuple:
    """Pages the step's new rows land in, per segment: (pool ids in order, a
    table of the same shape as w's whose only valid entries are those pages,
    relabelled)."""
    bt = w.block_table.cpu().numpy()
    si = w.seq_info.cpu().numpy()
    ids, where = [], {}
    small = np.full(bt.shape, -1, np.int32)
    for q0, ql, col, kend in si.tolist():
        for pos in range(kend - ql, kend):
            r = pos % w.ring_rows if w.ring_rows else pos
            pg = r // PAGE
            b = int(bt[col, pg])
            if b not in where:
                where[b] = len(ids)
                ids.append(b)
            small[col, pg] = where[b]
    return ids, small


# Every workload with the default kernels, and the other kernels a caller can
# pick by flag at the same sizes: the CUDA-core decode variant (PKV_FLAG_SIMT,
# head_dim 128 and 256) and the mma.sync tile for wide groups
# (PKV_FLAG_MMA_SYNC).
CASES = [(c[0], 0) for c in bench.CONFIGS] + [("batched", 1), ("long_context_ring", 1), ("verify_causal", 8)]


@pytest.mark.parametrize("key,flags", CASES)
def test_benched_workload_matches_oracle(pkv, key, flags):
    _, name, gen, kw = next(c for c in bench.CONFIGS if c[0] == key)
    dev = torch.device("cuda")
    w = getattr(workloads, gen)(seed=0, device=dev, **kw)
    workloads.nan_fill_unused(w)
    k_pre, v_pre = w.k[0].clone(), w.v[0].clone()

    cache = pkv.PagedKVCache(w.k, w.v, w.block_table, ring_rows=w.ring_rows, bucket=w.bucket)
    out = torch.full((w.total_rows, w.q_heads, w.head_dim), 5.0, device=dev)
    lse = torch.full((w.total_rows, w.q_heads), 5.0, device=dev)
    err = pkv.new_err_flags(dev)
    max_kv = int(w.seq_info[:, 3].max().item())
    pkv.append_attend(cache, 0, w.q[0], w.k_new[0], w.v_new[0], w.seq_info, out, err, w.max_q_len, max_kv, w.scale,
                      w.causal, w.window, lse=lse, flags=flags)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"{name}: device error flags {int(err.item()):#x}"
    assert bool(torch.isfinite(out).all())

    kn = _bytes(w.k_new[0])
    vn = _bytes(w.v_new[0])
    si = w.seq_info.cpu().numpy()

    # Appended slots of every segment: the pages they land in, byte for byte.
    ids, small = _touched(w)
    sel = torch.tensor(ids, dtype=torch.long, device=dev)
    kp, vp = _bytes(k_pre.index_select(0, sel)), _bytes(v_pre.index_select(0, sel))
    assert O.append(kp, vp, small, si, kn, vn, ring_rows=w.ring_rows, window=w.window, causal=w.causal) == 0
    assert _bytes(w.k[0].index_select(0, sel)).tobytes() == kp.tobytes(), f"{name}: K pages differ from the oracle"
    assert _bytes(w.v[0].index_select(0, sel)).tobytes() == vp.tobytes(), f"{name}: V pages differ from the oracle"

    # Sampled segments: every row against the oracle over the pages they reach.
    segs = _sampled(si, 2 if gen == "long_context" else 3)
    q64 = U.f64(w.q[0])
    for s in segs:
        kc, vc, bt, sub = U.compact(w, 0, [s], k_pre, v_pre)
        kb, vb = _bytes(kc), _bytes(vc)
        del kc, vc
        assert O.append(kb, vb, bt, sub, kn, vn, ring_rows=w.ring_rows, window=w.window, causal=w.causal) == 0
        kd = torch.from_numpy(kb).view(torch.bfloat16).double().numpy()
        vd = torch.from_numpy(vb).view(torch.bfloat16).double().numpy()
        ref, ref_lse, e = O.attend(q64, kd, vd, bt, sub, w.scale, causal=w.causal, window=w.window,
                                   ring_rows=w.ring_rows)
        assert e == 0
        rows = U.rows_of(w, [s])
        got = U.f64(out)[rows]
        diff = float(np.abs(got - ref[rows]).max())
        assert diff <= U.TOL[torch.bfloat16], f"{name}, segment {s}: max abs error {diff}"
        gl = U.f64(lse)[rows]
        assert float(np.abs(gl - ref_lse[rows]).max()) <= U.TOL[torch.bfloat16]
        del kd, vd

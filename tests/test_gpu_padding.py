"""Left padding on the GPU against the fp64 oracle.

Each table row's first valid position hides the keys before it from every
query row of that sequence, and a query row whose own position lies before
it (a padding row) attends to its own key alone ([tiny-llm kv_cache.py]
SlotKVCache, padded_causal_mask).  The hidden keys carry NaN in both pools,
so a kernel that reads one fails the finite-output check.
"""
import numpy as np
import pytest
import torch

import workloads
from tests import gpu_util as U
from tests.test_gpu_parity import check_against_oracle, check_append, run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_decode_13_gb300 as m
    return m


def poison_hidden(w, first_valid):
    """NaN in every cached slot below both the sequence's first valid
    position and the step's first row (no row of the step may read them)."""
    if w.ring_rows:
        return w
    si, bt = w.seq_info.numpy(), w.block_table.numpy()
    for q0, ql, col, kend in si:
        hidden = min(max(int(first_valid[col]), 0), int(kend - ql))
        for p in range(hidden):
            b, o = int(bt[col, p // U.PAGE]), p % U.PAGE
            for t in w.k + w.v:
                t[b, o] = float("nan")
    return w


def padded_run(pkv, w, fv, **kw):
    w = poison_hidden(w, fv)
    out, lse, err, cache = run(pkv, w, first_valid=fv, **kw)
    assert err == 0
    check_append(w, 0, cache)
    return check_against_oracle(w, 0, out, lse, cache, first_valid=fv)


DECODE_LENGTHS = [40, 300, 3000, 2000, 17, 900, 1500, 2500, 64, 1]
# 0; inside the first page; mid-range; the step's own row (its key alone);
# kv_end (the row is padding); past kv_end; negative (counts as 0); near the
# end of a long range; the last key of a short one; a one-token sequence
DECODE_FIRST = [0, 5, 1500, 1999, 17, 1000, -3, 2400, 63, 0]


@pytest.mark.parametrize("flags", [0, 1])
def test_padded_decode_batch(pkv, flags):
    # G = 4, one row per sequence: the decode kernel, solo and split ranges (flags 1: CUDA-core kernel)
    w = workloads.batched(S=10, max_len=3072, seed=41, lengths=DECODE_LENGTHS)
    padded_run(pkv, w, np.array(DECODE_FIRST, np.int32), flags=flags, max_kv=3072)


def test_padded_decode_batch_workspace_merge(pkv):
    w = workloads.batched(S=10, max_len=3072, seed=42, lengths=DECODE_LENGTHS)
    padded_run(pkv, w, np.array(DECODE_FIRST, np.int32), workspace=True, max_kv=3072)


def test_padded_decode_fp32(pkv):
    w = workloads.batched(S=10, max_len=3072, seed=43, lengths=DECODE_LENGTHS, dtype=torch.float32, q_heads=8,
                          kv_heads=2, head_dim=64)
    padded_run(pkv, w, np.array(DECODE_FIRST, np.int32), max_kv=3072)


def _verify_first(w, offsets):
    # first valid position relative to each segment's first new row
    si = w.seq_info.numpy()
    fv = np.zeros(w.max_seqs, np.int32)
    for s, (q0, ql, col, kend) in enumerate(si):
        fv[col] = max(0, int(kend - ql) + offsets[s % len(offsets)])
    return fv


@pytest.mark.parametrize("q_heads,causal", [(8, True), (8, False), (64, True), (64, False)])
def test_padded_verify_rows(pkv, q_heads, causal):
    # q_len up to 4 (q_heads 8: G = 1, decode kernel) or up to 16 rows of G = 8 (the general kernel);
    # first valid at, inside and past the step's rows, so some rows are padding
    max_q = 4 if q_heads == 8 else 16
    w = workloads.spec_verify(S=8, max_q=max_q, len_lo=100, len_hi=2000, causal=causal, seed=44 + q_heads,
                              q_heads=q_heads, kv_heads=8)
    fv = _verify_first(w, [-50, 0, 1, 2, 3, 10, -1000, 5])
    padded_run(pkv, w, fv, max_kv=2000)


@pytest.mark.parametrize("ring_rows", [0, 1024])
def test_padded_window(pkv, ring_rows):
    # a sliding window of 500 over flat or ring storage; first valid below, inside and past the window
    w = workloads.long_context(S=4, kv_len=3000, window=500, ring_rows=ring_rows, seed=45, q_heads=32,
                               kv_heads=4, head_dim=256)
    padded_run(pkv, w, np.array([0, 2200, 2800, 3500], np.int32), max_kv=3000)


def test_zero_first_valid_equals_no_padding(pkv):
    w = workloads.batched(S=6, max_len=2048, seed=46, lengths=[2000, 30, 700, 1200, 5, 1600])
    a, _, e1, _ = run(pkv, w, max_kv=2048)
    b, _, e2, _ = run(pkv, w, max_kv=2048, first_valid=np.zeros(6, np.int32))
    assert e1 == e2 == 0
    assert torch.equal(a, b)

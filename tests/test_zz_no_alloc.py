"""pkv_append_attend_noalloc: the fused call with its split-merge scratch in
the library's fixed device array, against pkv_append_attend with a caller
workspace, on the same inputs over two successive steps."""
import ctypes
import math

import numpy as np
import pytest
import torch

import workloads
from oracle import oracle as O
from tests import gpu_util as U


@pytest.fixture(scope="module")
def pkv():
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_decode_13_gb300 as m
    return m


def _oversize_args(pkv):
    # 8 sequences x 8 kv heads x 64 splits of head_dim 128 rows: 16 MiB of partials
    return dict(num_q_heads=32, num_segments=8, max_q_len=1, max_kv=8192, num_splits=64)


def test_oversize_rejected_before_launch(pkv):
    from paged_kv_decode_13_gb300 import _lib
    fake = (ctypes.c_void_p * 1)(0x1000)
    d = _lib.CacheDesc(num_layers=1, kv_heads=8, head_dim=128, dtype=_lib.BF16, num_blocks=4096, max_seqs=8,
                       max_blocks_per_seq=512, ring_rows=0, reserved0=0, k=ctypes.cast(fake, ctypes.c_void_p),
                       v=ctypes.cast(fake, ctypes.c_void_p), block_table=0x3000, bucket=8192, generation=0)
    a = _oversize_args(pkv)
    need = _lib.lib.pkv_attend_workspace_bytes(ctypes.byref(d), a["num_q_heads"], a["num_segments"], a["max_q_len"],
                                               a["max_kv"], a["num_splits"], 0)
    assert need > (8 << 20)
    st = _lib.lib.pkv_append_attend_noalloc(ctypes.byref(d), 0, 0x4000, 0x4000, 0x4000, a["num_q_heads"], 8, 0x5000,
                                           a["num_segments"], a["max_q_len"], a["max_kv"], a["num_splits"], 1.0, 0, 0,
                                           0x6000, None, 0x7000, 0, None)
    assert st == -4  # PKV_ECAPACITY


@pytest.mark.gpu
@pytest.mark.parametrize("seqused,bucket,num_splits", [(3000, 4096, 0), (8190, 8192, 19), (200, 512, 3)])
def test_noalloc_matches_workspace_call_over_two_steps(pkv, seqused, bucket, num_splits):
    w = U.nan_tails(workloads.sensenova(seqused, bucket, num_layers=1, seed=seqused))
    dev = torch.device("cuda")
    caches = [U.device_cache(pkv, w), U.device_cache(pkv, w)]
    ws = pkv.new_workspace(caches[0], w.q_heads, 1, 1, bucket, num_splits)
    assert ws is not None  # these launches merge their splits through scratch
    gen = torch.Generator().manual_seed(seqused)
    for step in range(2):
        si = w.seq_info.clone()
        si[0, 3] += step
        q = torch.randn(1, w.q_heads, w.head_dim, generator=gen).to(torch.bfloat16).to(dev)
        kn = (torch.randn(1, w.kv_heads, w.head_dim, generator=gen) / math.sqrt(w.head_dim)).to(torch.bfloat16).to(dev)
        vn = (torch.randn(1, w.kv_heads, w.head_dim, generator=gen) / math.sqrt(w.head_dim)).to(torch.bfloat16).to(dev)
        res = []
        for i, cache in enumerate(caches):
            out = torch.zeros(1, w.q_heads, w.head_dim, device=dev)
            lse = torch.zeros(1, w.q_heads, device=dev)
            err = pkv.new_err_flags()
            if i == 0:
                pkv.append_attend(cache, 0, q, kn, vn, si.to(dev), out, err, 1, bucket, w.scale, lse=lse,
                                  num_splits=num_splits, workspace=ws)
            else:
                pkv.append_attend_noalloc(cache, 0, q, kn, vn, si.to(dev), out, err, 1, bucket, w.scale, lse=lse,
                                          num_splits=num_splits)
            torch.cuda.synchronize()
            assert int(err.item()) == 0
            res.append((out, lse))
        assert torch.equal(res[0][0], res[1][0]) and torch.equal(res[0][1], res[1][1])
        assert U.pool_bytes(caches[0].k[0]) == U.pool_bytes(caches[1].k[0])
        assert U.pool_bytes(caches[0].v[0]) == U.pool_bytes(caches[1].v[0])
        assert np.isfinite(U.f64(res[1][0])).all()


@pytest.mark.gpu
def test_noalloc_oversize_launches_nothing(pkv):
    w = workloads.batched(S=8, max_len=8192, seed=3, lengths=[8192] * 8)
    cache = U.device_cache(pkv, w)
    dev = torch.device("cuda")
    out = torch.full((8, w.q_heads, w.head_dim), 4.0, device=dev)
    err = pkv.new_err_flags()
    with pytest.raises(pkv.PkvError):
        pkv.append_attend_noalloc(cache, 0, w.q[0].to(dev), w.k_new[0].to(dev), w.v_new[0].to(dev),
                                  w.seq_info.to(dev), out, err, 1, 8192, w.scale, num_splits=64)
    torch.cuda.synchronize()
    assert bool((out == 4.0).all()) and int(err.item()) == 0


@pytest.mark.gpu
def test_noalloc_batch_of_32_matches_oracle_over_two_steps(pkv):
    """32 sequences of different lengths, four splits per (sequence, kv head)
    range, so the library's scratch holds 256 ranges' partials and arrival
    counters at once.  Both steps match the fp64 oracle (the second over the
    pools the first appended to) and, bit for bit, the workspace call."""
    rng = np.random.default_rng(41)
    lengths = [int(x) for x in rng.integers(200, 3999, 32)]
    lengths = [L - 1 if L % 16 == 0 else L for L in lengths]   # the second step stays in the last page
    w = U.nan_tails(workloads.batched(S=32, max_len=4000, seed=41, lengths=lengths))
    dev = torch.device("cuda")
    caches = [U.device_cache(pkv, w), U.device_cache(pkv, w)]
    splits = 4
    ws = pkv.new_workspace(caches[0], w.q_heads, 32, 1, 4000, splits)
    assert ws is not None and ws.numel() <= (8 << 20)
    kp = w.k[0].view(torch.int16).numpy().copy()
    vp = w.v[0].view(torch.int16).numpy().copy()
    bt = w.block_table.numpy()
    gen = torch.Generator().manual_seed(42)
    for step in range(2):
        si = w.seq_info.clone()
        si[:, 3] += step
        q = torch.randn(32, w.q_heads, w.head_dim, generator=gen).to(torch.bfloat16)
        kn = (torch.randn(32, w.kv_heads, w.head_dim, generator=gen) / math.sqrt(w.head_dim)).to(torch.bfloat16)
        vn = (torch.randn(32, w.kv_heads, w.head_dim, generator=gen) / math.sqrt(w.head_dim)).to(torch.bfloat16)
        res = []
        for i, cache in enumerate(caches):
            out = torch.zeros(32, w.q_heads, w.head_dim, device=dev)
            lse = torch.zeros(32, w.q_heads, device=dev)
            err = pkv.new_err_flags()
            args = (cache, 0, q.to(dev), kn.to(dev), vn.to(dev), si.to(dev), out, err, 1, 4000, w.scale)
            if i == 0:
                pkv.append_attend(*args, lse=lse, num_splits=splits, workspace=ws)
            else:
                pkv.append_attend_noalloc(*args, lse=lse, num_splits=splits)
            torch.cuda.synchronize()
            assert int(err.item()) == 0
            res.append((out, lse))
        assert torch.equal(res[0][0], res[1][0]) and torch.equal(res[0][1], res[1][1])
        sin = si.numpy()
        assert O.append(kp, vp, bt, sin, kn.view(torch.int16).numpy(), vn.view(torch.int16).numpy()) == 0
        assert U.pool_bytes(caches[1].k[0]) == kp.tobytes() and U.pool_bytes(caches[1].v[0]) == vp.tobytes()
        ref, ref_lse, e = O.attend(q.double().numpy(), torch.from_numpy(kp).view(torch.bfloat16).double().numpy(),
                                   torch.from_numpy(vp).view(torch.bfloat16).double().numpy(), bt, sin, w.scale)
        assert e == 0
        diff = float(np.abs(U.f64(res[1][0]) - ref).max())
        assert diff <= U.TOL[torch.bfloat16], (step, diff)
        assert float(np.abs(U.f64(res[1][1]) - ref_lse).max()) <= U.TOL[torch.bfloat16]


@pytest.mark.gpu
@pytest.mark.parametrize("causal", [True, False])
def test_noalloc_wide_groups_match_append_attend(pkv, causal):
    """More than 8 rows per kv head (speculative verify: the tcgen05 tile,
    merged in the cluster): the call needs none of the library's scratch,
    and it equals pkv_append_attend bit for bit and the oracle."""
    w = U.nan_tails(workloads.spec_verify(S=6, max_q=16, len_lo=16, len_hi=2500, causal=causal, seed=57,
                                          q_heads=64))
    dev = torch.device("cuda")
    caches = [U.device_cache(pkv, w), U.device_cache(pkv, w)]
    res = []
    for i, cache in enumerate(caches):
        out = torch.zeros(w.total_rows, w.q_heads, w.head_dim, device=dev)
        lse = torch.zeros(w.total_rows, w.q_heads, device=dev)
        err = pkv.new_err_flags()
        args = (cache, 0, w.q[0].to(dev), w.k_new[0].to(dev), w.v_new[0].to(dev), w.seq_info.to(dev), out, err,
                w.max_q_len, 2500, w.scale, causal)
        if i == 0:
            pkv.append_attend(*args, lse=lse)
        else:
            pkv.append_attend_noalloc(*args, lse=lse)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        res.append((out, lse))
    assert torch.equal(res[0][0], res[1][0]) and torch.equal(res[0][1], res[1][1])
    assert U.pool_bytes(caches[0].k[0]) == U.pool_bytes(caches[1].k[0])
    ref, ref_lse = U.oracle_attend(w, 0)
    assert float(np.abs(U.f64(res[1][0]) - ref).max()) <= U.TOL[torch.bfloat16]

"""Batched-sequence cache operations on the GPU against the oracle:
seq_clone (device copy of a sequence's prefix) and rewind (kv_end back,
bounded by the ring floor), after ExecuTorch #24073's CudaBatchedSequenceCache."""
import numpy as np
import pytest
import torch

import workloads
from oracle import oracle as O
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_decode_13_gb300 as m
    return m


def _host_pools(w):
    return [t.view(torch.int16).numpy().copy() for t in w.k], [t.view(torch.int16).numpy().copy() for t in w.v]


@pytest.mark.parametrize("n", [1, 17, 300])
def test_seq_clone_matches_oracle_bit_exact(pkv, n):
    w = workloads.batched(S=3, max_len=400, num_layers=2, seed=n, lengths=[300, 40, 320])
    ks, vs = _host_pools(w)
    bt = w.block_table.numpy()
    for layer in range(2):
        assert O.seq_clone(ks[layer], vs[layer], bt, 0, 2, n) == 0
    cache = U.device_cache(pkv, w, canary=True)
    err = pkv.new_err_flags()
    pkv.seq_clone(cache, 0, 2, n, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    U.check_canaries(cache)
    for layer in range(2):
        assert U.pool_bytes(cache.k[layer]) == ks[layer].tobytes()
        assert U.pool_bytes(cache.v[layer]) == vs[layer].tobytes()


def test_seq_clone_ring_matches_oracle(pkv):
    w = workloads.long_context(S=2, kv_len=150, window=40, ring_rows=64, num_layers=2, seed=3, q_heads=8,
                               kv_heads=2, head_dim=64)
    ks, vs = _host_pools(w)
    bt = w.block_table.numpy()
    for layer in range(2):
        assert O.seq_clone(ks[layer], vs[layer], bt, 1, 0, 150, ring_rows=64) == 0
    cache = U.device_cache(pkv, w)
    err = pkv.new_err_flags()
    pkv.seq_clone(cache, 1, 0, 150, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for layer in range(2):
        assert U.pool_bytes(cache.k[layer]) == ks[layer].tobytes()
        assert U.pool_bytes(cache.v[layer]) == vs[layer].tobytes()


def test_seq_clone_bad_page_writes_nothing(pkv):
    w = workloads.batched(S=2, max_len=200, num_layers=1, seed=4, lengths=[180, 190])
    w.block_table[1, 5] = w.num_blocks + 3
    before = U.pool_bytes(w.k[0]), U.pool_bytes(w.v[0])
    cache = U.device_cache(pkv, w)
    err = pkv.new_err_flags()
    pkv.seq_clone(cache, 0, 1, 180, err)
    torch.cuda.synchronize()
    assert int(err.item()) & pkv.ERR_BLOCK
    assert (U.pool_bytes(cache.k[0]), U.pool_bytes(cache.v[0])) == before


def test_clone_then_attention_equals_source(pkv):
    # two sequences in the bf16 decode shape; the clone's attention equals the source's
    w = workloads.batched(S=2, max_len=1200, num_layers=1, seed=8, lengths=[1000, 1100])
    w.seq_info[1, 3] = 1000
    w.q[0][1] = w.q[0][0]
    w.k_new[0][1] = w.k_new[0][0]
    w.v_new[0][1] = w.v_new[0][0]
    cache = U.device_cache(pkv, w)
    dev = torch.device("cuda")
    err = pkv.new_err_flags()
    pkv.seq_clone(cache, 0, 1, 1000, err)
    out = torch.zeros(2, w.q_heads, w.head_dim, device=dev)
    pkv.append_attend(cache, 0, w.q[0].to(dev), w.k_new[0].to(dev), w.v_new[0].to(dev), w.seq_info.to(dev), out,
                      err, 1, 1200, w.scale)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(out[0], out[1])
    ref, _ = U.oracle_attend(w, 0, segs=[0])
    assert float(np.abs(U.f64(out[0]) - ref[0]).max()) <= U.TOL[w.dtype]


def test_rewind_matches_oracle(pkv):
    si = np.array([[0, 1, 0, 100], [1, 1, 1, 5], [2, 1, 2, 50], [3, 1, 3, 8], [4, 1, 4, 30]], np.int32)
    amount = np.array([10, 6, 0, -1, 30], np.int32)
    w = workloads.batched(S=5, max_len=128, num_layers=1, seed=1, lengths=[100, 5, 50, 8, 30])
    cache = U.device_cache(pkv, w)
    dev = torch.device("cuda")
    for ring, window in ((0, 0),):
        exp, bits = O.rewind(si, amount, ring_rows=ring, window=window)
        d_si = torch.from_numpy(si.copy()).to(dev)
        err = pkv.new_err_flags()
        pkv.rewind(cache, d_si, torch.from_numpy(amount).to(dev), err, window=window)
        torch.cuda.synchronize()
        assert np.array_equal(d_si.cpu().numpy(), exp)
        assert bool(int(err.item()) & pkv.ERR_SEGMENT) == bool(bits & (1 << 1))


def test_rewind_ring_floor(pkv):
    w = workloads.long_context(S=2, kv_len=300, window=40, ring_rows=64, num_layers=1, seed=2, q_heads=8,
                               kv_heads=2, head_dim=64)
    cache = U.device_cache(pkv, w)
    dev = torch.device("cuda")
    si = np.array([[0, 1, 0, 300], [1, 1, 1, 300]], np.int32)
    amount = np.array([25, 26], np.int32)     # 64 - 40 + 1 = 25 is the most a ring of 64 allows
    exp, bits = O.rewind(si, amount, ring_rows=64, window=40)
    d_si = torch.from_numpy(si.copy()).to(dev)
    err = pkv.new_err_flags()
    pkv.rewind(cache, d_si, torch.from_numpy(amount).to(dev), err, window=40)
    torch.cuda.synchronize()
    assert np.array_equal(d_si.cpu().numpy(), exp) and exp[:, 3].tolist() == [275, 300]
    assert int(err.item()) & pkv.ERR_RING and bits == 1 << 3


def test_verify_then_rewind_then_decode_matches_oracle(pkv):
    # a verify step appends 4 draft rows (causal), 3 are rejected, the next
    # decode step writes one row at the rewound length and attends over it
    w = workloads.spec_verify(S=1, max_q=4, len_lo=500, len_hi=500, causal=True, seed=12, q_heads=8, kv_heads=8)
    w.seq_info[0] = torch.tensor([0, 4, 0, 504], dtype=torch.int32)
    w.q[0] = torch.randn(4, 8, 128).to(torch.bfloat16)
    w.k_new[0] = (torch.randn(4, 8, 128) / 11.3).to(torch.bfloat16)
    w.v_new[0] = (torch.randn(4, 8, 128) / 11.3).to(torch.bfloat16)
    cache = U.device_cache(pkv, w)
    dev = torch.device("cuda")
    err = pkv.new_err_flags()
    si = w.seq_info.to(dev)
    out4 = torch.zeros(4, 8, 128, device=dev)
    pkv.append_attend(cache, 0, w.q[0].to(dev), w.k_new[0].to(dev), w.v_new[0].to(dev), si, out4, err, 4, 512,
                      w.scale, causal=True)
    pkv.rewind(cache, si, torch.tensor([3], dtype=torch.int32, device=dev), err)
    torch.cuda.synchronize()
    assert si.cpu().tolist() == [[0, 4, 0, 501]]
    # next step: one row at position 501
    q1 = torch.randn(1, 8, 128).to(torch.bfloat16)
    k1 = (torch.randn(1, 8, 128) / 11.3).to(torch.bfloat16)
    v1 = (torch.randn(1, 8, 128) / 11.3).to(torch.bfloat16)
    si1 = torch.tensor([[0, 1, 0, 502]], dtype=torch.int32, device=dev)
    out1 = torch.zeros(1, 8, 128, device=dev)
    pkv.append_attend(cache, 0, q1.to(dev), k1.to(dev), v1.to(dev), si1, out1, err, 1, 512, w.scale)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    # oracle: the same three operations on host pools
    kp = w.k[0].view(torch.int16).numpy().copy()
    vp = w.v[0].view(torch.int16).numpy().copy()
    bt = w.block_table.numpy()
    assert O.append(kp, vp, bt, np.array([[0, 4, 0, 504]], np.int32), w.k_new[0].view(torch.int16).numpy(),
                    w.v_new[0].view(torch.int16).numpy(), causal=True) == 0
    assert O.append(kp, vp, bt, np.array([[0, 1, 0, 502]], np.int32), k1.view(torch.int16).numpy(),
                    v1.view(torch.int16).numpy()) == 0
    assert U.pool_bytes(cache.k[0]) == kp.tobytes() and U.pool_bytes(cache.v[0]) == vp.tobytes()
    kpf = torch.from_numpy(kp).view(torch.bfloat16).double().numpy()
    vpf = torch.from_numpy(vp).view(torch.bfloat16).double().numpy()
    ref, _, e = O.attend(q1.double().numpy(), kpf, vpf, bt, np.array([[0, 1, 0, 502]], np.int32), w.scale)
    assert e == 0
    assert float(np.abs(U.f64(out1) - ref).max()) <= U.TOL[torch.bfloat16]


def test_growable_ring_table_lists_only_filled_pages(pkv):
    # before a ring layer wraps, its table may list only the pages filled so far
    w = workloads.long_context(S=3, kv_len=70, window=100, ring_rows=128, num_layers=1, seed=31, q_heads=16,
                               kv_heads=2, head_dim=128)
    w.block_table[:, (70 + 15) // 16:] = -1
    w = U.nan_tails(w)
    dev = torch.device("cuda")
    cache = U.device_cache(pkv, w)
    out = torch.zeros(w.total_rows, w.q_heads, w.head_dim, device=dev)
    lse = torch.zeros(w.total_rows, w.q_heads, device=dev)
    err = pkv.new_err_flags()
    pkv.append_attend(cache, 0, w.q[0].to(dev), w.k_new[0].to(dev), w.v_new[0].to(dev), w.seq_info.to(dev), out,
                      err, 1, 128, w.scale, True, 100, lse=lse)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref, ref_lse = U.oracle_attend(w, 0)
    assert float(np.abs(U.f64(out) - ref).max()) <= U.TOL[w.dtype]

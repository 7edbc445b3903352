"""CUDA path against the fp64 oracle, element by element, through the C ABI.

Attention: max-abs error <= 2e-3 for bf16 inputs (fp32 out, fp32
accumulation) and <= 1e-5 for fp32 inputs.  Append, resize and prefix copies:
bit-exact.  Pools carry NaN in every slot no segment may read, and guard
margins around pools and outputs catch out-of-range writes.
"""
import math

import numpy as np
import pytest
import torch

import workloads
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_decode_13_gb300 as m
    return m


def run(pkv, w, layer=0, fused=True, flags=0, num_splits=0, max_q_len=None, max_kv=None, canary=True,
        workspace=False, first_valid=None):
    """Append + attend layer `layer` of w on the GPU.  Returns (out, lse, err, cache).  With
    workspace=True the split merge goes through a workspace (decode kernel) instead of the cluster."""
    cache = U.device_cache(pkv, w, canary=canary, first_valid=first_valid)
    dev = torch.device("cuda")
    q = w.q[layer].to(dev)
    kn = w.k_new[layer].to(dev)
    vn = w.v_new[layer].to(dev)
    si = w.seq_info.to(dev)
    mq = max_q_len or w.max_q_len
    mk = max_kv or max(int(w.seq_info[:, 3].max()) if w.num_segments else 1, 1)
    obuf, out = U.guarded_out(w.total_rows, w.q_heads, w.head_dim)
    lse = torch.full((max(w.total_rows, 1), w.q_heads), 3.0, device=dev)[:w.total_rows]
    err = pkv.new_err_flags()
    ws = None
    if workspace:
        ws = pkv.new_workspace(cache, w.q_heads, w.num_segments, mq, mk, num_splits, flags)
        if ws is not None:  # guard margin: the call must not write past the size it asked for
            n = ws.numel()
            ws_buf = torch.full((n + 1024,), 0x5A, dtype=torch.uint8, device=dev)
            ws_buf[:n].zero_()
            ws = ws_buf[:n]
    if fused:
        pkv.append_attend(cache, layer, q, kn, vn, si, out, err, mq, mk, w.scale, w.causal, w.window, lse=lse,
                          num_splits=num_splits, flags=flags, workspace=ws)
    else:
        pkv.append(cache, layer, kn, vn, si, err, window=w.window)
        pkv.attend_varlen(cache, layer, q, si, out, err, mq, mk, w.scale, w.causal, w.window, lse=lse,
                          num_splits=num_splits, flags=flags, workspace=ws)
    torch.cuda.synchronize()
    U.check_guarded(obuf)
    U.check_canaries(cache)
    if ws is not None:
        assert bool((ws_buf[ws.numel():] == 0x5A).all()), "write past the workspace"
    return out, lse, int(err.item()), cache


def check_against_oracle(w, layer, out, lse, cache, segs=None, tol=None, first_valid=None):
    tol = tol or U.TOL[w.dtype]
    ref, ref_lse = U.oracle_attend(w, layer, segs=segs, first_valid=first_valid)
    rows = U.rows_of(w, segs) if segs is not None else list(range(w.total_rows))
    got = U.f64(out)[rows]
    exp = ref[rows]
    assert np.isfinite(got).all()
    diff = float(np.abs(got - exp).max()) if rows else 0.0
    assert diff <= tol, f"max abs error {diff} > {tol}"
    gl, el = U.f64(lse)[rows], ref_lse[rows]
    same_inf = np.isinf(gl) == np.isinf(el)
    assert same_inf.all()
    fin = np.isfinite(el)
    if fin.any():
        assert float(np.abs(gl[fin] - el[fin]).max()) <= max(tol, 1e-5)
    return diff


def check_append(w, layer, cache):
    kp, vp, err = U.oracle_append_pools(w, layer)
    assert err == 0
    assert U.pool_bytes(cache.k[layer]) == kp.tobytes(), "K pool differs from the oracle's append"
    assert U.pool_bytes(cache.v[layer]) == vp.tobytes(), "V pool differs from the oracle's append"


# ---------------------------------------------------------------- the five workloads, reduced

@pytest.mark.parametrize("fused", [True, False])
def test_tiny_fp32(pkv, fused):
    w = U.nan_tails(workloads.tiny(seed=0))
    out, lse, err, cache = run(pkv, w, fused=fused)
    assert err == 0
    check_append(w, 0, cache)
    check_against_oracle(w, 0, out, lse, cache)


@pytest.mark.parametrize("seqused", [1, 15, 16, 17, 300, 1000, 1024])
@pytest.mark.parametrize("flags", [0, 1])
def test_sensenova_shape(pkv, seqused, flags):
    w = U.nan_tails(workloads.sensenova(seqused, 1024, num_layers=2, seed=seqused))
    for layer in (0, 1):
        out, lse, err, cache = run(pkv, w, layer=layer, flags=flags, max_kv=1024)
        assert err == 0
        check_append(w, layer, cache)
        check_against_oracle(w, layer, out, lse, cache)


@pytest.mark.parametrize("flags,fused", [(0, True), (0, False), (1, True)])
def test_batched_varlen(pkv, flags, fused):
    w = U.nan_tails(workloads.batched(S=8, max_len=3000, seed=3))
    out, lse, err, cache = run(pkv, w, fused=fused, flags=flags, max_kv=3000)
    assert err == 0
    check_append(w, 0, cache)
    check_against_oracle(w, 0, out, lse, cache)


@pytest.mark.parametrize("q_heads", [8, 16, 32, 64])
@pytest.mark.parametrize("causal", [True, False])
def test_spec_verify(pkv, q_heads, causal):
    w = U.nan_tails(workloads.spec_verify(S=6, max_q=16, len_lo=256, len_hi=2000, causal=causal, seed=q_heads,
                                          q_heads=q_heads))
    for flags in (0, 1):
        out, lse, err, cache = run(pkv, w, flags=flags, max_kv=2000)
        assert err == 0
        check_append(w, 0, cache)
        check_against_oracle(w, 0, out, lse, cache)


@pytest.mark.parametrize("q_heads,max_q", [(8, 8), (16, 4), (32, 2), (64, 1)])
@pytest.mark.parametrize("causal", [True, False])
def test_narrow_groups_multi_row(pkv, q_heads, max_q, causal):
    # G * max_q_len <= 8: the decode kernel with several rows per token group
    w = U.nan_tails(workloads.spec_verify(S=6, max_q=max_q, len_lo=1, len_hi=1500, causal=causal,
                                          seed=q_heads + max_q, q_heads=q_heads))
    out, lse, err, cache = run(pkv, w, max_kv=1500)
    assert err == 0
    check_append(w, 0, cache)
    check_against_oracle(w, 0, out, lse, cache)


def _prefetch_workload(kind):
    if kind == "single":
        return workloads.sensenova(1000, 1024, num_layers=3, seed=5)
    if kind == "batched":
        return workloads.batched(S=8, max_len=2000, num_layers=3, seed=6, kv_heads=8, q_heads=32)
    return workloads.long_context(S=2, kv_len=5000, window=300, ring_rows=320, num_layers=3, seed=7, q_heads=16,
                                  kv_heads=4, head_dim=128)


@pytest.mark.parametrize("kind", ["single", "batched", "ring"])
def test_prefetch_next_hint_changes_nothing(pkv, kind):
    # The next-layer L2 warm-up is a hint: results are bitwise those without it,
    # and on the last layer it is ignored.
    w = _prefetch_workload(kind)
    dev = torch.device("cuda")
    max_kv = int(w.seq_info[:, 3].max())
    res = {}
    for flags in (0, pkv.FLAG_PREFETCH_NEXT):
        cache = U.device_cache(pkv, w)
        outs = []
        for layer in range(3):
            out = torch.zeros(w.total_rows, w.q_heads, w.head_dim, device=dev)
            lse = torch.zeros(w.total_rows, w.q_heads, device=dev)
            err = pkv.new_err_flags()
            pkv.append_attend(cache, layer, w.q[layer].to(dev), w.k_new[layer].to(dev), w.v_new[layer].to(dev),
                              w.seq_info.to(dev), out, err, 1, max_kv, w.scale, w.causal, w.window, lse=lse,
                              flags=flags)
            torch.cuda.synchronize()
            assert int(err.item()) == 0
            outs.append((out.clone(), lse.clone()))
        res[flags] = (outs, [U.pool_bytes(t) for t in cache.k + cache.v])
    for (a, la), (b, lb) in zip(res[0][0], res[pkv.FLAG_PREFETCH_NEXT][0]):
        assert torch.equal(a, b) and torch.equal(la, lb)
    assert res[0][1] == res[pkv.FLAG_PREFETCH_NEXT][1]
    for layer in range(3):
        ref, _ = U.oracle_attend(w, layer)
        assert float(np.abs(U.f64(res[0][0][layer][0]) - ref).max()) <= U.TOL[w.dtype]


@pytest.mark.parametrize("seqused", [176, 192, 193, 208, 4099])
@pytest.mark.parametrize("num_splits", [0, 5, 16])
def test_decode_one_cta_or_cluster(pkv, seqused, num_splits):
    # Up to 12 pages a key range runs on one CTA without the cluster merge;
    # from 13 pages on it is split across the cluster (any split count).
    w = U.nan_tails(workloads.sensenova(seqused, pkv.bucket_for(seqused), num_layers=1, seed=seqused))
    out, lse, err, cache = run(pkv, w, max_kv=w.bucket, num_splits=num_splits)
    assert err == 0
    check_append(w, 0, cache)
    check_against_oracle(w, 0, out, lse, cache)


@pytest.mark.parametrize("window", [5, 40, 180, 700])
def test_decode_windows_edge_pages(pkv, window):
    # windows whose first page starts mid-page (stale rows before the window
    # zeroed), with single and clustered ranges
    w = U.nan_tails(workloads.batched(S=6, max_len=3000, seed=window, kv_heads=8, q_heads=32, min_len=100))
    w.causal, w.window = True, window
    # slots before each window hold NaN too: they must never reach the output
    bt, si = w.block_table.numpy(), w.seq_info.numpy()
    for q0, ql, col, kend in si:
        for pos in range(max(0, int(kend) - window)):
            b = int(bt[col, pos // 16])
            for t in w.k + w.v:
                t[b, pos % 16] = float("nan")
    out, lse, err, cache = run(pkv, w, max_kv=3000)
    assert err == 0
    check_against_oracle(w, 0, out, lse, cache)


def _ws_workload(kind):
    if kind == "single_8192":
        return U.nan_tails(workloads.sensenova(8190, 8192, num_layers=1, seed=21))
    if kind == "single_1000":
        return U.nan_tails(workloads.sensenova(1000, 1024, num_layers=1, seed=22))
    if kind == "batched":
        return U.nan_tails(workloads.batched(S=32, max_len=4000, seed=23, num_layers=1))
    if kind == "narrow_rows":
        return U.nan_tails(workloads.spec_verify(S=6, max_q=2, len_lo=1, len_hi=3000, causal=True, seed=24,
                                                 q_heads=32))
    return U.nan_tails(workloads.long_context(S=3, kv_len=20000, window=1000, ring_rows=1024, seed=25, num_layers=1,
                                              q_heads=32, kv_heads=4, head_dim=256))


@pytest.mark.parametrize("kind", ["single_8192", "single_1000", "batched", "narrow_rows", "ring_d256"])
@pytest.mark.parametrize("num_splits", [0, 3, 19, 64])
def test_workspace_merge_matches_oracle(pkv, kind, num_splits):
    # independent CTAs merging through the workspace, any split count up to 64
    w = _ws_workload(kind)
    mk = int(w.seq_info[:, 3].max())
    out, lse, err, cache = run(pkv, w, max_kv=mk, num_splits=num_splits, workspace=True)
    assert err == 0
    check_append(w, 0, cache)
    check_against_oracle(w, 0, out, lse, cache)


def test_workspace_is_reusable_and_poison_zeroes(pkv):
    w = U.nan_tails(workloads.sensenova(3000, 4096, num_layers=1, seed=26))
    dev = torch.device("cuda")
    cache = U.device_cache(pkv, w)
    ws = pkv.new_workspace(cache, w.q_heads, 1, 1, 4096, 0)
    assert ws is not None
    outs = []
    for _ in range(3):  # the counters return to zero: every call merges the same way
        out = torch.zeros(1, w.q_heads, w.head_dim, device=dev)
        err = pkv.new_err_flags()
        pkv.attend_varlen(cache, 0, w.q[0].to(dev), w.seq_info.to(dev), out, err, 1, 4096, w.scale, workspace=ws)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        outs.append(out.clone())
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])
    # a bad block id in one split's range: the merged rows are zero, the flag is set
    bt = cache.block_table
    bt[0, 100] = w.num_blocks + 5
    out = torch.full((1, w.q_heads, w.head_dim), 9.0, device=dev)
    err = pkv.new_err_flags()
    pkv.attend_varlen(cache, 0, w.q[0].to(dev), w.seq_info.to(dev), out, err, 1, 4096, w.scale, workspace=ws)
    torch.cuda.synchronize()
    assert int(err.item()) & pkv.ERR_BLOCK
    assert not out.abs().sum().item()


@pytest.mark.parametrize("window,ring", [(0, 0), (1000, 0), (1024, 1024), (300, 320)])
def test_long_context(pkv, window, ring):
    w = U.nan_tails(workloads.long_context(S=2, kv_len=20000, window=window, ring_rows=ring, seed=5))
    out, lse, err, cache = run(pkv, w, max_kv=20000)
    assert err == 0
    check_append(w, 0, cache)
    check_against_oracle(w, 0, out, lse, cache)


# ---------------------------------------------------------------- shapes, splits, modes

@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("head_dim", [8, 40, 64, 72, 96, 136, 192, 256])
def test_head_dims(pkv, dtype, head_dim):
    w = U.nan_tails(workloads.batched(S=3, max_len=700, seed=head_dim, q_heads=8, kv_heads=2, head_dim=head_dim,
                                      dtype=dtype))
    out, lse, err, cache = run(pkv, w, max_kv=700)
    assert err == 0
    check_append(w, 0, cache)
    check_against_oracle(w, 0, out, lse, cache)


@pytest.mark.parametrize("num_splits", [1, 2, 3, 16, 0])
def test_split_count_does_not_change_result(pkv, num_splits):
    w = U.nan_tails(workloads.sensenova(2500, 4096, num_layers=1, seed=9))
    out, lse, err, cache = run(pkv, w, num_splits=num_splits, max_kv=4096)
    assert err == 0
    check_against_oracle(w, 0, out, lse, cache)


@pytest.mark.parametrize("q_heads,max_q,flags", [(64, 16, 0), (64, 8, 0), (32, 8, 0), (16, 8, 0), (64, 16, 1)])
@pytest.mark.parametrize("num_splits", [1, 3])
def test_long_ranges_per_cta(pkv, q_heads, max_q, flags, num_splits):
    # one or three CTAs per range of 2000..5000 keys: each key group copies
    # far more pages than its stages and its L2 warm-up hold, through several
    # page-id windows, and the last pass of a 4-page loop may hold 1..4 pages
    # (every row class of the general kernel; flags 1: the CUDA-core kernel)
    w = U.nan_tails(workloads.spec_verify(S=4, max_q=max_q, len_lo=2000, len_hi=5000, seed=70 + q_heads + max_q,
                                          q_heads=q_heads, kv_heads=8))
    out, lse, err, cache = run(pkv, w, num_splits=num_splits, max_kv=5000, flags=flags)
    assert err == 0
    check_append(w, 0, cache)
    check_against_oracle(w, 0, out, lse, cache)


def _simt_workload(kind):
    if kind == "single_1000":
        return U.nan_tails(workloads.sensenova(1000, 1024, num_layers=1, seed=81))
    if kind == "single_4099":
        return U.nan_tails(workloads.sensenova(4099, 8192, num_layers=1, seed=82))
    if kind == "batched_d64":
        return U.nan_tails(workloads.batched(S=8, max_len=2000, seed=83, q_heads=16, kv_heads=2, head_dim=64))
    if kind == "batched_d96":  # head_dim below its padded width: zero-filled columns
        return U.nan_tails(workloads.batched(S=5, max_len=1500, seed=84, q_heads=8, kv_heads=1, head_dim=96))
    if kind == "window_d128":
        w = U.nan_tails(workloads.batched(S=6, max_len=3000, seed=85, kv_heads=8, q_heads=32, min_len=100))
        w.causal, w.window = True, 180
        return w
    if kind == "two_rows":  # q_len 2 x 4 heads: 8 rows per kv head, causal inside the step
        return U.nan_tails(workloads.spec_verify(S=6, max_q=2, len_lo=1, len_hi=3000, causal=True, seed=86,
                                                 q_heads=32))
    return U.nan_tails(workloads.long_context(S=3, kv_len=20000, window=1000, ring_rows=1024, seed=87, num_layers=1,
                                              q_heads=32, kv_heads=4, head_dim=256))


@pytest.mark.parametrize("kind", ["single_1000", "single_4099", "batched_d64", "batched_d96", "window_d128",
                                  "two_rows", "ring_d256"])
@pytest.mark.parametrize("workspace", [False, True])
def test_cuda_core_decode_variant(pkv, kind, workspace):
    # PKV_FLAG_SIMT with at most 8 rows per kv head: the decode kernel with
    # fp32 FMA dot products, merging its splits in the cluster or through the
    # workspace, at head_dim 64 / 96 / 128 / 256
    w = _simt_workload(kind)
    mk = int(w.seq_info[:, 3].max())
    out, lse, err, cache = run(pkv, w, max_kv=mk, flags=pkv.FLAG_SIMT, workspace=workspace)
    assert err == 0
    check_append(w, 0, cache)
    check_against_oracle(w, 0, out, lse, cache)


def test_fused_equals_two_calls_bitwise(pkv):
    w = U.nan_tails(workloads.spec_verify(S=5, max_q=8, len_lo=100, len_hi=900, seed=11, q_heads=16))
    a, la, ea, ca = run(pkv, w, fused=True, max_kv=900)
    b, lb, eb, cb = run(pkv, w, fused=False, max_kv=900)
    assert ea == eb == 0
    assert torch.equal(a, b) and torch.equal(la, lb)
    assert U.pool_bytes(ca.k[0]) == U.pool_bytes(cb.k[0])


@pytest.mark.parametrize("window", [1, 7, 33, 500])
def test_causal_window_flat(pkv, window):
    w = U.nan_tails(workloads.spec_verify(S=4, max_q=12, len_lo=40, len_hi=800, seed=window, q_heads=16))
    w.window = window
    out, lse, err, cache = run(pkv, w, max_kv=800)
    assert err == 0
    check_against_oracle(w, 0, out, lse, cache)


def test_ring_wraps_many_times(pkv):
    # kv_end far past the ring: the window keys sit at slots p % R after many wraps.
    w = workloads.long_context(S=3, kv_len=50_001, window=64, ring_rows=80, seed=13, q_heads=8, kv_heads=2,
                               head_dim=64)
    w = U.nan_tails(w)
    out, lse, err, cache = run(pkv, w, max_kv=50_001)
    assert err == 0
    check_append(w, 0, cache)
    check_against_oracle(w, 0, out, lse, cache)


# ---------------------------------------------------------------- edge cases

def _single(kend, ql=1, D=64, dtype=torch.bfloat16, seed=0, nblocks=None, Hq=4, Hkv=2):
    g = torch.Generator().manual_seed(seed)
    nb = nblocks or max((kend + 15) // 16, 1) + 1
    k = [torch.randn(nb, 16, Hkv, D, generator=g).to(dtype)]
    v = [torch.randn(nb, 16, Hkv, D, generator=g).to(dtype)]
    rows = max(ql, 1)
    q = [torch.randn(rows, Hq, D, generator=g).to(dtype)]
    kn = [torch.randn(rows, Hkv, D, generator=g).to(dtype)]
    vn = [torch.randn(rows, Hkv, D, generator=g).to(dtype)]
    bt = torch.arange(nb, dtype=torch.int32).unsqueeze(0)
    si = torch.tensor([[0, ql, 0, kend]], dtype=torch.int32)
    return workloads.Workload("edge", dtype, 1, Hq, Hkv, D, nb, bt, si, k, v, q, kn, vn, causal=True,
                              bucket=nb * 16, max_q_len=max(ql, 1))


def test_single_key_returns_new_value(pkv):
    w = _single(1)
    out, lse, err, cache = run(pkv, w, max_kv=16)
    assert err == 0
    for h in range(4):
        assert torch.equal(out[0, h].cpu(), w.v_new[0][0, h // 2].float())


def test_zero_length_segments_and_uncovered_rows(pkv):
    w = U.nan_tails(workloads.spec_verify(S=4, max_q=4, len_lo=20, len_hi=200, seed=21, q_heads=8))
    si = w.seq_info.clone()
    si[1, 1] = 0                     # an empty segment
    si[:, 0] += 2                    # two leading rows no segment covers
    w.seq_info = si
    extra = 5
    for lst in (w.q, w.k_new, w.v_new):
        lst[0] = torch.cat([lst[0], lst[0][:extra]], 0)
    out, lse, err, cache = run(pkv, w, max_kv=200)
    assert err == 0
    covered = set(U.rows_of(w, range(4)))
    for t in range(w.total_rows):
        if t not in covered:
            assert not out[t].abs().sum().item() and bool(torch.isinf(lse[t]).all())
    check_against_oracle(w, 0, out, lse, cache, segs=[0, 2, 3])


def test_no_segments_zeroes_every_row(pkv):
    w = _single(10, ql=1)
    w.seq_info = torch.zeros(0, 4, dtype=torch.int32)
    w.q[0] = torch.cat([w.q[0]] * 3)
    w.k_new[0] = torch.cat([w.k_new[0]] * 3)
    w.v_new[0] = torch.cat([w.v_new[0]] * 3)
    out, lse, err, cache = run(pkv, w, max_q_len=1, max_kv=16)
    assert err == 0 and not out.abs().sum().item() and bool(torch.isinf(lse).all())


@pytest.mark.parametrize("seg,window,ring,bit", [
    ([0, 2, 0, 1], 0, 0, 1),        # kv_end < q_len
    ([0, 1, 3, 10], 0, 0, 1),       # col past max_seqs
    ([0, 3, 0, 10], 0, 0, 1),       # rows past total_rows
    ([0, 1, 0, 100000], 0, 0, 2),   # past the table's capacity
    ([0, 1, 0, 40], 0, 32, 4),      # ring without a window
    ([0, 2, 0, 40], 32, 32, 4),     # window + q_len - 1 > ring rows
])
def test_invalid_segment_sets_error_and_zeroes(pkv, seg, window, ring, bit):
    w = _single(40, ql=2, nblocks=6)
    w.seq_info = torch.tensor([seg], dtype=torch.int32)
    w.window, w.ring_rows, w.causal = window, ring, True
    before = U.pool_bytes(w.k[0])
    out, lse, err, cache = run(pkv, w, max_q_len=2, max_kv=64)
    assert err & bit, f"expected bit {bit}, got {err:#x}"
    assert not out.abs().sum().item()
    assert U.pool_bytes(cache.k[0]) == before          # nothing appended


def test_bad_block_id_in_range(pkv):
    w = _single(100, ql=1, nblocks=8)
    bt = w.block_table.clone()
    bt[0, 2] = 1 << 20
    w.block_table = bt
    out, lse, err, cache = run(pkv, w, max_kv=128, num_splits=3)
    assert err & 8 and not out.abs().sum().item()
    assert bool(torch.isinf(lse).all())


def test_q_len_above_launch_bound(pkv):
    w = _single(50, ql=4)
    out, lse, err, cache = run(pkv, w, max_q_len=2, max_kv=64)
    assert err & 16 and not out.abs().sum().item()


def test_overlapping_segments_flagged(pkv):
    w = U.nan_tails(workloads.spec_verify(S=2, max_q=4, len_lo=50, len_hi=60, seed=3, q_heads=8))
    si = w.seq_info.clone()
    si[1, 0] = si[0, 0]
    w.seq_info = si
    _, _, err, _ = run(pkv, w, max_kv=64)
    assert err & 32


# ---------------------------------------------------------------- table helpers, resize, prefix

def test_seqinfo_from_seqused_and_advance(pkv):
    cu = torch.tensor([0, 1, 4, 4, 9], dtype=torch.int32, device="cuda")
    used = torch.tensor([7, 30, 2, 500], dtype=torch.int32, device="cuda")
    si = torch.zeros(4, 4, dtype=torch.int32, device="cuda")
    pkv.seqinfo_from_seqused(cu, used, si)
    pkv.advance(si)
    torch.cuda.synchronize()
    expect = [[0, 1, 0, 8], [1, 3, 1, 33], [4, 0, 2, 2], [4, 5, 3, 505]]
    assert si.cpu().tolist() == expect


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_resize_keeps_prefix_and_bumps_generation(pkv, dtype):
    old = pkv.PagedKVCache.allocate(3, 4, 64, 512, dtype=dtype)
    for t in old.k + old.v:
        t.copy_(torch.randn(t.shape, device="cuda").to(dtype))
    n = pkv.bucket_for(700)
    new = pkv.PagedKVCache.allocate(3, 4, 64, n, dtype=dtype)
    assert pkv.resize_bucket(old, new, 333) == 0
    torch.cuda.synchronize()
    assert new.generation == old.generation + 1
    for a, b in zip(old.k + old.v, new.k + new.v):
        fa, fb = a.view(-1, 4, 64), b.view(-1, 4, 64)
        assert torch.equal(fa[:333], fb[:333])
        assert not fb[333:].abs().sum().item()
    same = pkv.PagedKVCache.allocate(3, 4, 64, 512, dtype=dtype)
    assert pkv.resize_bucket(old, same, 10) == 2 and same.generation == 0


def test_load_prefix_and_write_back(pkv):
    L, H, S, D = 2, 4, 77, 64
    cache = pkv.PagedKVCache.allocate(L, H, D, 512)
    keys = [torch.randn(1, H, S, D, device="cuda").to(torch.bfloat16) for _ in range(L)]
    vals = [torch.randn(1, H, S, D, device="cuda").to(torch.bfloat16) for _ in range(L)]
    # [B, H, S, D] -> [S, H, D] views, as PagedDecodeCache.load_prefix does
    assert pkv.load_prefix(cache, [k[0].transpose(0, 1) for k in keys], [v[0].transpose(0, 1) for v in vals])
    assert not pkv.load_prefix(cache, [keys[0][0, :, :0].transpose(0, 1)] * L,
                               [vals[0][0, :, :0].transpose(0, 1)] * L)
    for layer in range(L):
        ko = torch.empty(H, S, D, dtype=torch.bfloat16, device="cuda")
        vo = torch.empty_like(ko)
        pkv.to_contiguous(cache, layer, S, ko, vo)
        torch.cuda.synchronize()
        assert torch.equal(ko, keys[layer][0]) and torch.equal(vo, vals[layer][0])
        flat = cache.k[layer].view(-1, H, D)
        assert torch.equal(flat[:S], keys[layer][0].transpose(0, 1))


@pytest.mark.parametrize("q_heads,q_len", [(32, 1), (64, 2)])
def test_thousands_of_segments_with_gaps(pkv, q_heads, q_len):
    """2048 segments (the decode kernel at q_len 1, the general kernel at 2)
    over an output with a gap row after every 16th segment: the check of rows
    no segment covers is spread over many CTAs, the gaps come back zero with
    lse = -inf, every covered row matches the oracle, and making two segments
    claim one row sets the overlap bit."""
    S = 2048
    w = workloads.batched(S=S, max_len=48, seed=q_heads + q_len, q_heads=q_heads, kv_heads=8, min_len=q_len)
    q0 = [s * q_len + s // 16 for s in range(S)]
    rows = q0[-1] + q_len + 3
    gen = torch.Generator().manual_seed(5)
    w.q[0] = torch.randn(rows, q_heads, w.head_dim, generator=gen).to(torch.bfloat16)
    w.k_new[0] = (torch.randn(rows, 8, w.head_dim, generator=gen) / math.sqrt(w.head_dim)).to(torch.bfloat16)
    w.v_new[0] = (torch.randn(rows, 8, w.head_dim, generator=gen) / math.sqrt(w.head_dim)).to(torch.bfloat16)
    si = w.seq_info.clone()
    si[:, 0] = torch.tensor(q0, dtype=torch.int32)
    si[:, 1] = q_len
    w.seq_info = si
    w.causal, w.max_q_len = True, q_len
    w = U.nan_tails(w)
    out, lse, err, cache = run(pkv, w, max_kv=48)
    assert err == 0
    covered = set(U.rows_of(w, range(S)))
    gaps = [t for t in range(rows) if t not in covered]
    assert len(gaps) == S // 16 - 1 + 3
    g = torch.tensor(gaps, device=out.device)
    assert not out[g].abs().sum().item() and bool(torch.isinf(lse[g]).all())
    check_append(w, 0, cache)
    check_against_oracle(w, 0, out, lse, cache)
    si2 = si.clone()
    si2[1000, 0] = si2[999, 0]          # two segments claim the same rows
    w.seq_info = si2
    _, _, err, _ = run(pkv, w, max_kv=48)
    assert err & pkv.ERR_OVERLAP


@pytest.mark.parametrize("q_heads,max_q", [(64, 16), (64, 32), (16, 8), (8, 16)])
@pytest.mark.parametrize("causal", [True, False])
def test_tcgen05_and_mma_sync_tiles_match_oracle(pkv, q_heads, max_q, causal):
    """Wide bf16 groups with head_dim 128 (more than 8 rows per kv head) run
    on the tcgen05 tile by default and on the mma.sync tile with
    PKV_FLAG_MMA_SYNC; both match the oracle for one CTA per range, a split
    that does not divide the pages, and the automatic split.  64 heads x 32
    rows is 256 rows per kv head: two 128-row tiles."""
    w = U.nan_tails(workloads.spec_verify(S=5, max_q=max_q, len_lo=1, len_hi=2500, causal=causal,
                                          seed=q_heads * 3 + max_q, q_heads=q_heads))
    for flags in (0, pkv.FLAG_MMA_SYNC):
        for splits in (0, 1, 5):
            out, lse, err, cache = run(pkv, w, flags=flags, num_splits=splits, max_kv=2500)
            assert err == 0
            check_append(w, 0, cache)
            check_against_oracle(w, 0, out, lse, cache)


@pytest.mark.parametrize("kv_len", [1472, 1536, 1537, 1600])
@pytest.mark.parametrize("num_splits", [0, 2, 4])
def test_tcgen05_solo_threshold(pkv, kv_len, num_splits):
    """Ranges of at most 24 groups of 64 keys (1536 keys) run on the
    cluster's first CTA alone, the other CTAs leaving before any cluster
    barrier; one page more splits the range.  Equal lengths also exercise
    the longest-first ranking's tie order."""
    w = U.nan_tails(workloads.spec_verify(S=3, max_q=16, len_lo=kv_len, len_hi=kv_len, causal=True,
                                          seed=kv_len + num_splits, q_heads=64))
    out, lse, err, cache = run(pkv, w, num_splits=num_splits, max_kv=kv_len)
    assert err == 0
    check_append(w, 0, cache)
    check_against_oracle(w, 0, out, lse, cache)


@pytest.mark.parametrize("S", [2, 64, 65])
def test_tcgen05_longest_first_order(pkv, S):
    """Up to 64 segments the CTAs take the ranges longest first (a
    permutation of blockIdx.z computed on the device); beyond, in segment
    order.  Either way every row matches the oracle."""
    # kv_end >= q_len (= at most 8), so every segment is valid
    w = U.nan_tails(workloads.spec_verify(S=S, max_q=8, len_lo=8, len_hi=2200, causal=S % 2 == 0, seed=90 + S,
                                          q_heads=16))
    out, lse, err, cache = run(pkv, w, max_kv=2200)
    assert err == 0
    check_append(w, 0, cache)
    check_against_oracle(w, 0, out, lse, cache)


@pytest.mark.parametrize("kv_len,page", [(2000, 40), (2000, 100), (1000, 30)])
def test_tcgen05_bad_block_poisons_only_its_segment(pkv, kv_len, page):
    """A block id out of range inside one segment's key range (in one CTA of
    a range split over a cluster, or in a range run by one CTA alone):
    that segment's rows are zero with lse -inf and PKV_ERR_BLOCK is set; the
    other segments still match the oracle."""
    w = U.nan_tails(workloads.spec_verify(S=3, max_q=16, len_lo=kv_len, len_hi=kv_len, causal=True, seed=page,
                                          q_heads=64))
    bt = w.block_table.clone()
    bt[1, page] = 1 << 20
    w.block_table = bt
    out, lse, err, cache = run(pkv, w, max_kv=kv_len)
    assert err & pkv.ERR_BLOCK
    rows = U.rows_of(w, [1])
    assert not out[rows].abs().sum().item()
    assert bool(torch.isinf(lse[rows]).all())
    check_against_oracle(w, 0, out, lse, cache, segs=[0, 2])


def test_tcgen05_tile_ring_window_and_padding(pkv):
    """The tcgen05 tile over ring storage with a window, and with left padding."""
    w = U.nan_tails(workloads.long_context(S=3, kv_len=9000, window=700, ring_rows=720, seed=31, q_heads=64,
                                           kv_heads=8, head_dim=128))
    w.max_q_len = 2
    out, lse, err, cache = run(pkv, w, max_kv=9000, max_q_len=2)
    assert err == 0
    check_append(w, 0, cache)
    check_against_oracle(w, 0, out, lse, cache)
    w = U.nan_tails(workloads.spec_verify(S=4, max_q=16, len_lo=200, len_hi=1200, seed=32, q_heads=64))
    first = [150, 0, 1199, 37]
    out, lse, err, cache = run(pkv, w, max_kv=1200, first_valid=first)
    assert err == 0
    check_against_oracle(w, 0, out, lse, cache, first_valid=first)

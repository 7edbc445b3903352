"""Pins for the fp64 CPU oracle (no GPU).

Each test checks the oracle against something other than itself: a value the
pages print, a closed form, an invariant the pages state, a library routine
on a special case, or an independent brute-force twin on tiny inputs.
"""
import math
import os

import numpy as np
import pytest
import torch

from oracle import oracle as O
from oracle import brute

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
PAGE = 16


# ---------------------------------------------------------------- helpers

def identity_case(rng, kend, Hq=4, Hkv=2, D=8, nblocks=None, rows=1, q0=0):
    nb = nblocks or (kend + PAGE - 1) // PAGE + 1
    q = rng.standard_normal((rows, Hq, D))
    kp = rng.standard_normal((nb, PAGE, Hkv, D))
    vp = rng.standard_normal((nb, PAGE, Hkv, D))
    bt = np.arange(nb, dtype=np.int32)[None, :]
    return q, kp, vp, bt


def flat_keys(pool, kend, g):
    """Keys 0..kend-1 of kv head g from a pool behind an identity table."""
    return pool.reshape(-1, pool.shape[2], pool.shape[3])[:kend, g, :]


def sdpa_dense(q, k, v, scale, mask=None):
    """torch SDPA in fp64 on CPU: q (R, D), k/v (N, D), mask (R, N) bool."""
    qt = torch.from_numpy(q)[None, None]
    kt = torch.from_numpy(k)[None, None]
    vt = torch.from_numpy(v)[None, None]
    m = None if mask is None else torch.from_numpy(mask)[None, None]
    return torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=m, scale=scale)[0, 0].numpy()


def random_paged(rng, lens, qlens, Hq, Hkv, D, ring_rows=0, spare=3):
    """Segments over a shuffled page pool; unused table entries are -1."""
    span = [ring_rows if ring_rows else L for L in lens]
    need = [(s + PAGE - 1) // PAGE for s in span]
    mbps = max(need) + 1
    nb = sum(need) + spare
    perm = rng.permutation(nb).astype(np.int32)
    bt = np.full((len(lens), mbps), -1, dtype=np.int32)
    at = 0
    for s, n in enumerate(need):
        bt[s, :n] = perm[at:at + n]
        at += n
    rows = sum(qlens)
    q = rng.standard_normal((rows, Hq, D))
    kp = rng.standard_normal((nb, PAGE, Hkv, D))
    vp = rng.standard_normal((nb, PAGE, Hkv, D))
    si, r = [], 0
    for s in range(len(lens)):
        si.append([r, qlens[s], s, lens[s]])
        r += qlens[s]
    return q, kp, vp, bt, np.array(si, dtype=np.int32)


# ---------------------------------------------------------------- bucket schedule

def test_bucket_for_golden():
    rows = []
    with open(os.path.join(GOLDEN, "bucket_for.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                rows.append(tuple(int(x) for x in line.split()))
    assert len(rows) > 10
    for length, bucket in rows:
        assert O.bucket_for(length) == bucket, (length, bucket)


def test_tail_step_reservation_matches_page_ratio():
    # vllm-omni paged_decode.py, comment on TAIL_STEP: at a 9,100-token request
    # doubling the last bucket would leave 766 MiB unused against 118 MiB with
    # the tail step.  Unused tokens must stand in about that ratio.
    L = 9100
    tail_unused = O.bucket_for(L) - L
    doubling_unused = 16384 - L
    assert abs(doubling_unused / tail_unused - 766 / 118) / (766 / 118) < 0.03


# ---------------------------------------------------------------- closed forms

def test_single_key_returns_v_exactly():
    rng = np.random.default_rng(1)
    q, kp, vp, bt = identity_case(rng, 1)
    si = np.array([[0, 1, 0, 1]], np.int32)
    out, lse, err = O.attend(q, kp, vp, bt, si, 0.3)
    assert err == 0
    for h in range(4):
        g = h // 2
        assert np.array_equal(out[0, h], vp[0, 0, g])
        assert lse[0, h] == pytest.approx(0.3 * float(q[0, h] @ kp[0, 0, g]), abs=1e-14)


def test_equal_keys_give_mean_v():
    rng = np.random.default_rng(2)
    n = 37
    q, kp, vp, bt = identity_case(rng, n)
    kp[:] = kp[0, 0]          # every key identical -> uniform weights
    si = np.array([[0, 1, 0, n]], np.int32)
    out, lse, _ = O.attend(q, kp, vp, bt, si, 0.5)
    for h in range(4):
        g = h // 2
        np.testing.assert_allclose(out[0, h], flat_keys(vp, n, g).mean(0), rtol=0, atol=1e-14)
        s = 0.5 * float(q[0, h] @ kp[0, 0, g])
        assert lse[0, h] == pytest.approx(s + math.log(n), abs=1e-12)


def test_one_dominant_score_selects_its_value():
    rng = np.random.default_rng(3)
    n = 50
    q, kp, vp, bt = identity_case(rng, n, Hq=2, Hkv=2)
    q[:] = 0.0
    q[0, :, 0] = 1.0
    kp[..., 0] = 0.0
    flat = kp.reshape(-1, 2, 8)
    flat[17, :, 0] = 1000.0   # score gap 1000 * scale: weight of the rest < e^-500
    si = np.array([[0, 1, 0, n]], np.int32)
    out, _, _ = O.attend(q, kp, vp, bt, si, 1.0)
    for h in range(2):
        np.testing.assert_allclose(out[0, h], vp.reshape(-1, 2, 8)[17, h], atol=1e-15)


# ---------------------------------------------------------------- library special case

@pytest.mark.parametrize("kend,Hq,Hkv,D", [(1, 4, 4, 8), (33, 8, 2, 16), (300, 8, 2, 64)])
def test_identity_table_equals_dense_sdpa(kend, Hq, Hkv, D):
    rng = np.random.default_rng(kend)
    q, kp, vp, bt = identity_case(rng, kend, Hq, Hkv, D)
    si = np.array([[0, 1, 0, kend]], np.int32)
    sc = 1 / math.sqrt(D)
    out, lse, _ = O.attend(q, kp, vp, bt, si, sc)
    G = Hq // Hkv
    for h in range(Hq):
        k = flat_keys(kp, kend, h // G)
        v = flat_keys(vp, kend, h // G)
        ref = sdpa_dense(q[0, h][None], k, v, sc)[0]
        np.testing.assert_allclose(out[0, h], ref, rtol=0, atol=1e-13)
        ref_lse = np.log(np.sum(np.exp(sc * (k @ q[0, h]))))
        assert lse[0, h] == pytest.approx(ref_lse, abs=1e-12)


def test_gqa_equals_repeated_kv_heads():
    # Contiguous head groups: q head h reads kv head h // (Hq/Hkv), i.e. the
    # result equals plain multi-head attention over K/V repeated per group.
    rng = np.random.default_rng(5)
    kend, Hq, Hkv, D = 45, 6, 2, 8
    q, kp, vp, bt = identity_case(rng, kend, Hq, Hkv, D)
    si = np.array([[0, 1, 0, kend]], np.int32)
    out, _, _ = O.attend(q, kp, vp, bt, si, 0.4)
    kt = torch.from_numpy(flat_keys(kp, kend, slice(None)).transpose(1, 0, 2).copy())
    vt = torch.from_numpy(flat_keys(vp, kend, slice(None)).transpose(1, 0, 2).copy())
    kt = kt.repeat_interleave(Hq // Hkv, dim=0)[None]
    vt = vt.repeat_interleave(Hq // Hkv, dim=0)[None]
    qt = torch.from_numpy(q[0])[None, :, None, :]
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=0.4)[0, :, 0].numpy()
    np.testing.assert_allclose(out[0], ref, atol=1e-13)


def test_causal_rows_match_tinyllm_mask_dense():
    # tiny-llm kv_cache.py causal_kwargs: T new queries at start..start+T-1 over
    # start+T keys; query i sees keys 0..start+i (bottom-right alignment).
    rng = np.random.default_rng(6)
    T, start, Hq, Hkv, D = 5, 23, 4, 2, 8
    kend = start + T
    q, kp, vp, bt = identity_case(rng, kend, Hq, Hkv, D, rows=T)
    si = np.array([[0, T, 0, kend]], np.int32)
    out, _, _ = O.attend(q, kp, vp, bt, si, 0.35, causal=True)
    qpos = np.arange(start, start + T)[:, None]
    kpos = np.arange(kend)[None, :]
    mask = kpos <= qpos
    for h in range(Hq):
        ref = sdpa_dense(q[:, h], flat_keys(kp, kend, h // 2), flat_keys(vp, kend, h // 2), 0.35, mask)
        np.testing.assert_allclose(out[:, h], ref, atol=1e-13)


def test_causal_single_row_equals_non_causal():
    rng = np.random.default_rng(7)
    q, kp, vp, bt = identity_case(rng, 70)
    si = np.array([[0, 1, 0, 70]], np.int32)
    a, la, _ = O.attend(q, kp, vp, bt, si, 0.3, causal=True)
    b, lb, _ = O.attend(q, kp, vp, bt, si, 0.3, causal=False)
    assert np.array_equal(a, b) and np.array_equal(la, lb)


def test_causal_row_reduces_to_single_token_decode():
    rng = np.random.default_rng(8)
    T, kend = 6, 90
    q, kp, vp, bt = identity_case(rng, kend, rows=T)
    si = np.array([[0, T, 0, kend]], np.int32)
    full, lfull, _ = O.attend(q, kp, vp, bt, si, 0.3, causal=True, window=20)
    for i in range(T):
        one = np.array([[0, 1, 0, kend - T + i + 1]], np.int32)
        o, l, _ = O.attend(q[i:i + 1], kp, vp, bt, one, 0.3, causal=True, window=20)
        assert np.array_equal(full[i], o[0]) and np.array_equal(lfull[i], l[0])


def test_non_causal_rows_all_see_every_key():
    rng = np.random.default_rng(9)
    T, kend = 4, 40
    q, kp, vp, bt = identity_case(rng, kend, rows=T)
    si = np.array([[0, T, 0, kend]], np.int32)
    out, _, _ = O.attend(q, kp, vp, bt, si, 0.3, causal=False)
    for h in range(4):
        ref = sdpa_dense(q[:, h], flat_keys(kp, kend, h // 2), flat_keys(vp, kend, h // 2), 0.3)
        np.testing.assert_allclose(out[:, h], ref, atol=1e-13)


# ---------------------------------------------------------------- window and ring

def test_window_at_least_kend_equals_no_window():
    rng = np.random.default_rng(10)
    q, kp, vp, bt = identity_case(rng, 77, rows=3)
    si = np.array([[0, 3, 0, 77]], np.int32)
    a, la, _ = O.attend(q, kp, vp, bt, si, 0.3, causal=True, window=77)
    b, lb, _ = O.attend(q, kp, vp, bt, si, 0.3, causal=True, window=0)
    assert np.array_equal(a, b) and np.array_equal(la, lb)


@pytest.mark.parametrize("causal", [True, False])
def test_window_equals_dense_over_last_keys(causal):
    rng = np.random.default_rng(11)
    T, kend, W = 3, 100, 17
    q, kp, vp, bt = identity_case(rng, kend, rows=T)
    si = np.array([[0, T, 0, kend]], np.int32)
    out, _, _ = O.attend(q, kp, vp, bt, si, 0.3, causal=causal, window=W)
    for i in range(T):
        newest = (kend - T + i) if causal else kend - 1
        lo = newest - W + 1
        for h in range(4):
            k = flat_keys(kp, kend, h // 2)[lo:newest + 1]
            v = flat_keys(vp, kend, h // 2)[lo:newest + 1]
            ref = sdpa_dense(q[i, h][None], k, v, 0.3)[0]
            np.testing.assert_allclose(out[i, h], ref, atol=1e-13)


@pytest.mark.parametrize("causal,T", [(True, 1), (True, 4), (False, 3)])
def test_ring_equals_flat_with_same_window(causal, T):
    # ExecuTorch #24074: ring slot = position % rows; #24073: a ring of
    # window + max_write - 1 rows suffices.  Same keys, ring or flat storage,
    # must give the same result.
    rng = np.random.default_rng(12)
    Hkv, D, W, kend = 2, 8, 29, 211
    R = 32 * ((W + T - 1 + 31) // 32)   # rounded up to whole pages
    Rtight = W + T - 1
    keys = rng.standard_normal((kend, Hkv, D))
    vals = rng.standard_normal((kend, Hkv, D))
    q = rng.standard_normal((T, 4, D))
    si = np.array([[0, T, 0, kend]], np.int32)
    nb = (kend + PAGE - 1) // PAGE
    kf = np.full((nb, PAGE, Hkv, D), np.nan)
    vf = np.full((nb, PAGE, Hkv, D), np.nan)
    kf.reshape(-1, Hkv, D)[:kend] = keys
    vf.reshape(-1, Hkv, D)[:kend] = vals
    flat, lflat, e1 = O.attend(q, kf, vf, np.arange(nb, dtype=np.int32)[None], si, 0.3,
                               causal=causal, window=W)
    for rr in (R, Rtight):
        nbr = (rr + PAGE - 1) // PAGE
        perm = rng.permutation(nbr + 2).astype(np.int32)
        kr = np.full((nbr + 2, PAGE, Hkv, D), np.nan)
        vr = np.full((nbr + 2, PAGE, Hkv, D), np.nan)
        # store positions kend-rr..kend-1 at slot p % rr through the table
        for p in range(kend - rr, kend):
            r = p % rr
            kr[perm[r // PAGE], r % PAGE] = keys[p]
            vr[perm[r // PAGE], r % PAGE] = vals[p]
        ring, lring, e2 = O.attend(q, kr, vr, perm[None, :nbr], si, 0.3, causal=causal, window=W,
                                   ring_rows=rr)
        assert e1 == e2 == 0
        assert np.array_equal(flat, ring) and np.array_equal(lflat, lring)


# ---------------------------------------------------------------- paging invariants

def test_permuted_block_table_is_bit_identical():
    rng = np.random.default_rng(13)
    kend, Hkv, D = 150, 2, 8
    q, kp, vp, bt = identity_case(rng, kend, Hkv=Hkv, D=D)
    si = np.array([[0, 1, 0, kend]], np.int32)
    ref, lref, _ = O.attend(q, kp, vp, bt, si, 0.3)
    nb = kp.shape[0]
    perm = rng.permutation(nb).astype(np.int32)
    kq = np.empty_like(kp)
    vq = np.empty_like(vp)
    kq[perm] = kp          # logical page i now lives in physical page perm[i]
    vq[perm] = vp
    out, lse, _ = O.attend(q, kq, vq, perm[None], si, 0.3)
    assert np.array_equal(out, ref) and np.array_equal(lse, lref)


def test_nan_tail_and_unused_pages_are_ignored():
    # vllm-omni paged_decode.py, load_prefix: only the first seqused rows are
    # read; the tail keeps whatever the previous request wrote.
    rng = np.random.default_rng(14)
    kend = 45
    q, kp, vp, bt = identity_case(rng, kend, nblocks=8)
    si = np.array([[0, 1, 0, kend]], np.int32)
    ref, lref, _ = O.attend(q, kp, vp, bt, si, 0.3)
    kn, vn = kp.copy(), vp.copy()
    kn.reshape(-1, 2, 8)[kend:] = np.nan
    vn.reshape(-1, 2, 8)[kend:] = np.nan
    bt2 = bt.copy()
    bt2[0, 3:] = -1          # pages past the live prefix are not even listed
    out, lse, err = O.attend(q, kn, vn, bt2, si, 0.3)
    assert err == 0 and np.isfinite(out).all()
    assert np.array_equal(out, ref) and np.array_equal(lse, lref)


def test_empty_and_uncovered_rows_are_zero():
    rng = np.random.default_rng(15)
    q, kp, vp, bt = identity_case(rng, 40, rows=5)
    # rows 0, 3, 4: not covered; segment 2 has q_len 0.
    si = np.array([[1, 2, 0, 40], [3, 0, 0, 10]], np.int32)
    out, lse, err = O.attend(q, kp, vp, bt, si, 0.3, causal=True)
    assert err == 0
    for t in (0, 3, 4):
        assert not out[t].any() and np.all(lse[t] == -np.inf)
    assert np.abs(out[1:3]).sum() > 0


# ---------------------------------------------------------------- brute force

@pytest.mark.parametrize("seed", range(8))
def test_matches_brute_force_twin(seed):
    rng = np.random.default_rng(100 + seed)
    S = int(rng.integers(1, 4))
    Hkv = int(rng.choice([1, 2]))
    Hq = Hkv * int(rng.choice([1, 2, 3]))
    D = int(rng.choice([4, 8, 16]))
    causal = bool(seed % 2)
    ring = seed in (2, 3, 6)
    window = int(rng.integers(1, 20)) if (ring or seed in (4, 5)) else 0
    qlens = [int(rng.integers(0 if seed == 7 else 1, 5)) for _ in range(S)]
    lens = [int(rng.integers(max(q, 1), 40)) for q in qlens]
    R = 0
    if ring:
        R = PAGE * ((window + max(qlens) - 1 + PAGE - 1) // PAGE)
    q, kp, vp, bt, si = random_paged(rng, lens, qlens, Hq, Hkv, D, ring_rows=R)
    out, lse, err = O.attend(q, kp, vp, bt, si, 0.37, causal=causal, window=window, ring_rows=R)
    assert err == 0
    bo, bl = brute.attend(q.tolist(), kp.tolist(), vp.tolist(), bt.tolist(), si.tolist(), 0.37,
                          causal=causal, window=window, ring_rows=R)
    np.testing.assert_allclose(out, np.array(bo), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, np.array(bl), rtol=0, atol=1e-12)


# ---------------------------------------------------------------- append

@pytest.mark.parametrize("ring", [False, True])
def test_append_scatters_bit_exact(ring):
    rng = np.random.default_rng(20)
    lens, qlens = [37, 5, 64], [3, 1, 4]
    R = 32 if ring else 0
    _, kp, vp, bt, si = random_paged(rng, lens, qlens, 4, 2, 8, ring_rows=R)
    kp = kp.astype(np.float32)
    vp = vp.astype(np.float32)
    rows = sum(qlens) + 2                    # two trailing rows no segment covers
    kn = rng.standard_normal((rows, 2, 8)).astype(np.float32)
    vn = rng.standard_normal((rows, 2, 8)).astype(np.float32)
    k0, v0 = kp.copy(), vp.copy()
    err = O.append(kp, vp, bt, si, kn, vn, ring_rows=R, window=8 if ring else 0, causal=True)
    assert err == 0
    expect_k, expect_v = k0.copy(), v0.copy()
    written = set()
    for t, b, o in brute.append_slots(bt.tolist(), si.tolist(), ring_rows=R):
        expect_k[b, o] = kn[t]
        expect_v[b, o] = vn[t]
        written.add((b, o))
    assert kp.tobytes() == expect_k.tobytes() and vp.tobytes() == expect_v.tobytes()
    assert len(written) == sum(qlens)


def test_append_identity_table_writes_flat_row_length_minus_one():
    # vllm-omni paged_decode.py, PagedDecodeCache.attend: with the identity
    # table the new token lands at flat row length - 1.
    nb, n = 8, 77
    kp = np.zeros((nb, PAGE, 2, 4), np.uint16)
    vp = np.zeros_like(kp)
    kn = np.arange(8, dtype=np.uint16).reshape(1, 2, 4) + 1
    vn = kn + 100
    bt = np.arange(nb, dtype=np.int32)[None]
    O.append(kp, vp, bt, np.array([[0, 1, 0, n]], np.int32), kn, vn)
    flat = kp.reshape(-1, 2, 4)
    assert np.array_equal(flat[n - 1], kn[0]) and flat.sum() == kn.sum()
    assert np.array_equal(vp.reshape(-1, 2, 4)[n - 1], vn[0])


def test_append_ring_wraps_position_modulo_rows():
    nb, R = 4, 64
    bt = np.array([[2, 0, 3, 1]], np.int32)
    for pos in (5, 5 + R, 5 + 3 * R):
        kp = np.zeros((nb, PAGE, 1, 2), np.int32)
        vp = np.zeros_like(kp)
        kn = np.array([[[7, 9]]], np.int32)
        O.append(kp, vp, bt, np.array([[0, 1, 0, pos + 1]], np.int32), kn, kn, ring_rows=R,
                 window=16, causal=True)
        assert np.array_equal(kp[2, 5, 0], [7, 9]) and kp.sum() == 16


# ---------------------------------------------------------------- validation

@pytest.mark.parametrize("seg,ring,window,bit", [
    ([0, 2, 0, 1], 0, 0, 1),      # kv_end < q_len
    ([0, 1, 5, 10], 0, 0, 1),     # col past max_seqs
    ([1, 1, 0, 10], 0, 0, 1),     # rows past total_rows
    ([-1, 1, 0, 10], 0, 0, 1),    # negative q_start
    ([0, 1, 0, 200], 0, 0, 2),    # kv_end beyond 8 pages
    ([0, 1, 0, 50], 64, 0, 3),    # ring without a window
    ([0, 1, 0, 50], 64, 65, 3),   # window + q_len - 1 > ring rows
    ([0, 1, 0, 120], 0, 0, 4),    # reaches a page id out of range
])
def test_invalid_segments_write_nothing(seg, ring, window, bit):
    rng = np.random.default_rng(30)
    q = rng.standard_normal((1, 2, 4))
    kp = rng.standard_normal((8, PAGE, 1, 4))
    vp = rng.standard_normal((8, PAGE, 1, 4))
    bt = np.arange(8, dtype=np.int32)[None].copy()
    bt[0, 7] = 99
    si = np.array([seg], np.int32)
    out, lse, err = O.attend(q, kp, vp, bt, si, 0.3, window=window, ring_rows=ring)
    assert err == 1 << bit
    assert not out.any() and np.all(lse == -np.inf)
    k0 = kp.copy()
    err2 = O.append(kp, vp, bt, si, q[:, :1].copy(), q[:, :1].copy(), ring_rows=ring, window=window)
    assert err2 == 1 << bit and np.array_equal(kp, k0)


def test_append_gated_only_by_written_slots():
    # A bad page before the written slot blocks the attention (it would be
    # read) but not the append (it is never written).
    q = np.ones((1, 2, 4))
    kp = np.zeros((8, PAGE, 1, 4))
    vp = np.zeros_like(kp)
    bt = np.arange(8, dtype=np.int32)[None].copy()
    bt[0, 2] = -5
    si = np.array([[0, 1, 0, 100]], np.int32)
    _, _, err = O.attend(q, kp, vp, bt, si, 0.3)
    assert err == 1 << 4
    kn = np.full((1, 1, 4), 3.0)
    assert O.append(kp, vp, bt, si, kn, kn) == 0
    assert np.array_equal(kp.reshape(-1, 1, 4)[99], kn[0])


# ---------------------------------------------------------------- batched-sequence cache operations
# (ExecuTorch #24073, CudaBatchedSequenceCache: seq_clone copies the source
# prefix on the device; rewind is bounded by the ring floor)

def _two_seq_pool(rng, n_src, ring_rows=0, Hkv=2, D=8):
    span = ring_rows if ring_rows else max(n_src, 1)
    need = (span + PAGE - 1) // PAGE
    nb = 2 * need + 3
    perm = rng.permutation(nb).astype(np.int32)
    bt = np.full((2, need + 1), -1, dtype=np.int32)
    bt[0, :need] = perm[:need]
    bt[1, :need] = perm[need:2 * need]
    kp = rng.standard_normal((nb, PAGE, Hkv, D))
    vp = rng.standard_normal((nb, PAGE, Hkv, D))
    return kp, vp, bt


def _slot(bt, col, pos, ring_rows=0):
    r = pos % ring_rows if ring_rows else pos
    return int(bt[col, r // PAGE]), r % PAGE


@pytest.mark.parametrize("n", [0, 1, 15, 16, 40])
def test_seq_clone_copies_the_prefix_bit_exact(n):
    rng = np.random.default_rng(n + 1)
    kp, vp, bt = _two_seq_pool(rng, 48)
    k0, v0 = kp.copy(), vp.copy()
    assert O.seq_clone(kp, vp, bt, 0, 1, n) == 0
    for pos in range(48):
        bs, os_ = _slot(bt, 0, pos)
        bd, od = _slot(bt, 1, pos)
        if pos < n:   # the destination's slot now holds the source's row
            assert np.array_equal(kp[bd, od], k0[bs, os_]) and np.array_equal(vp[bd, od], v0[bs, os_])
        else:         # untouched past n
            assert np.array_equal(kp[bd, od], k0[bd, od]) and np.array_equal(vp[bd, od], v0[bd, od])
    # the source never changes
    for pos in range(48):
        bs, os_ = _slot(bt, 0, pos)
        assert np.array_equal(kp[bs, os_], k0[bs, os_])


def test_seq_clone_then_attention_matches_the_source():
    rng = np.random.default_rng(7)
    kp, vp, bt = _two_seq_pool(rng, 37, Hkv=2, D=16)
    assert O.seq_clone(kp, vp, bt, 0, 1, 37) == 0
    q = rng.standard_normal((2, 4, 16))
    si = np.array([[0, 1, 0, 37], [1, 1, 1, 37]], np.int32)
    q[1] = q[0]
    out, lse, err = O.attend(q, kp, vp, bt, si, 0.25)
    assert err == 0
    assert np.array_equal(out[0], out[1]) and np.array_equal(lse[0], lse[1])


def test_seq_clone_ring_copies_only_the_last_rows():
    rng = np.random.default_rng(9)
    R = 32
    kp, vp, bt = _two_seq_pool(rng, 0, ring_rows=R)
    k0 = kp.copy()
    assert O.seq_clone(kp, vp, bt, 0, 1, 75, ring_rows=R) == 0
    # positions 43..74 live in the ring; each one's slot holds the source row of the same slot
    for pos in range(75 - R, 75):
        bs, os_ = _slot(bt, 0, pos, R)
        bd, od = _slot(bt, 1, pos, R)
        assert np.array_equal(kp[bd, od], k0[bs, os_])
    # and a windowed attention on the clone equals the source's
    q = rng.standard_normal((1, 4, 8))
    for col in (0, 1):
        si = np.array([[0, 1, col, 75]], np.int32)
        o, l, e = O.attend(q, kp, vp, bt, si, 0.3, causal=True, window=20, ring_rows=R)
        assert e == 0
        if col == 0:
            ref = o
        else:
            assert np.array_equal(o, ref)


def test_seq_clone_all_or_nothing_on_bad_pages():
    rng = np.random.default_rng(11)
    kp, vp, bt = _two_seq_pool(rng, 40)
    bt[1, 2] = -1     # the destination's third page is missing
    k0, v0 = kp.copy(), vp.copy()
    assert O.seq_clone(kp, vp, bt, 0, 1, 40) == 1 << 4
    assert np.array_equal(kp, k0) and np.array_equal(vp, v0)
    assert O.seq_clone(kp, vp, bt, 0, 5, 4) == 1 << 1      # no such sequence
    assert O.seq_clone(kp, vp, bt, 0, 1, 10_000) == 1 << 2  # beyond the table's capacity


def test_rewind_arithmetic_and_ring_floor():
    si = np.array([[0, 1, 0, 100], [1, 1, 1, 5], [2, 1, 2, 50], [3, 1, 3, 8]], np.int32)
    new, err = O.rewind(si, np.array([10, 6, 0, -1]))
    assert new[:, 3].tolist() == [90, 5, 50, 8] and err == 1 << 1
    # ring of 64 rows with a window of 40: at most 64 - 40 + 1 = 25 positions back
    new, err = O.rewind(si[:1], np.array([25]), ring_rows=64, window=40)
    assert new[0, 3] == 75 and err == 0
    new, err = O.rewind(si[:1], np.array([26]), ring_rows=64, window=40)
    assert new[0, 3] == 100 and err == 1 << 3


def test_rewind_then_rewrite_restores_the_state():
    # a verify step appends 4 draft rows and rejects 3 of them: attending over
    # the accepted length equals having appended the one accepted row alone
    rng = np.random.default_rng(5)
    kp, vp, bt = _two_seq_pool(rng, 64, Hkv=2, D=8)
    kn = rng.standard_normal((4, 2, 8))
    vn = rng.standard_normal((4, 2, 8))
    a_k, a_v = kp.copy(), vp.copy()
    assert O.append(a_k, a_v, bt, np.array([[0, 4, 0, 24]], np.int32), kn, vn) == 0
    si, err = O.rewind(np.array([[0, 4, 0, 24]], np.int32), np.array([3]))
    assert err == 0 and si[0, 3] == 21
    b_k, b_v = kp.copy(), vp.copy()
    assert O.append(b_k, b_v, bt, np.array([[0, 1, 0, 21]], np.int32), kn[:1], vn[:1]) == 0
    q = rng.standard_normal((1, 4, 8))
    one = np.array([[0, 1, 0, 21]], np.int32)
    oa, _, _ = O.attend(q, a_k, a_v, bt, one, 0.5)
    ob, _, _ = O.attend(q, b_k, b_v, bt, one, 0.5)
    assert np.array_equal(oa, ob)


def test_growable_ring_reads_only_filled_pages():
    # ExecuTorch #24076: a ring layer grows with the flat layers until it holds
    # all its rows, so before the first wrap its table may list only the pages
    # filled so far; the result equals the flat layout with the same window
    rng = np.random.default_rng(21)
    R, W, kend = 128, 100, 70            # 70 < R: no wrap yet, 5 of 8 pages filled
    q, kp, vp, bt, si = random_paged(rng, [kend], [1], 4, 2, 8, ring_rows=R)
    bt[0, (kend + PAGE - 1) // PAGE:] = -1
    out_r, lse_r, err = O.attend(q, kp, vp, bt, si, 0.3, causal=True, window=W, ring_rows=R)
    assert err == 0
    out_f, lse_f, err = O.attend(q, kp, vp, bt, si, 0.3, causal=True, window=W)
    assert err == 0
    assert np.array_equal(out_r, out_f) and np.array_equal(lse_r, lse_f)


# ---------------------------------------------------------------- left padding (tiny-llm kv_cache.py, SlotKVCache:
# slot b holds keys at positions first[b] .. lens[b]-1; padded_causal_mask hides keys before first_valid[b] and
# always keeps the diagonal)

def test_first_valid_zero_is_no_padding():
    rng = np.random.default_rng(40)
    q, kp, vp, bt, si = random_paged(rng, [37, 90], [3, 1], 4, 2, 8)
    a = O.attend(q, kp, vp, bt, si, 0.3, causal=True)
    b = O.attend(q, kp, vp, bt, si, 0.3, causal=True, first_valid=np.zeros(2, np.int32))
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]) and a[2] == b[2] == 0


@pytest.mark.parametrize("causal", [True, False])
def test_left_padding_decode_equals_dense_over_valid_keys(causal):
    rng = np.random.default_rng(41)
    kend, first = 70, 23
    q, kp, vp, bt = identity_case(rng, kend, Hq=4, Hkv=2, D=16)
    si = np.array([[0, 1, 0, kend]], np.int32)
    out, lse, err = O.attend(q, kp, vp, bt, si, 0.25, causal=causal, first_valid=np.array([first], np.int32))
    assert err == 0
    for h in range(4):
        g = h // 2
        ref = sdpa_dense(q[0, h][None], flat_keys(kp, kend, g)[first:], flat_keys(vp, kend, g)[first:], 0.25)
        assert np.abs(out[0, h] - ref[0]).max() < 1e-12


def test_padded_rows_see_only_themselves():
    # rows at positions before first_valid read exactly their own value
    rng = np.random.default_rng(42)
    kend, ql, first = 40, 6, 37          # rows at 34..39: 34, 35, 36 are padding
    q, kp, vp, bt = identity_case(rng, kend, Hq=2, Hkv=1, D=8, rows=ql)
    si = np.array([[0, ql, 0, kend]], np.int32)
    out, lse, err = O.attend(q, kp, vp, bt, si, 0.5, causal=True, first_valid=np.array([first], np.int32))
    assert err == 0
    for i in range(3):
        pos = kend - ql + i
        for h in range(2):
            assert np.array_equal(out[i, h], flat_keys(vp, kend, 0)[pos])
            assert lse[i, h] == pytest.approx(0.5 * float(q[i, h] @ flat_keys(kp, kend, 0)[pos]), abs=1e-12)


def test_left_padding_matches_tinyllm_mask_dense():
    # multi-row causal step with padding: SDPA with the page's padded_causal_mask rule
    rng = np.random.default_rng(43)
    kend, ql, first = 30, 8, 25
    q, kp, vp, bt = identity_case(rng, kend, Hq=2, Hkv=2, D=8, rows=ql)
    si = np.array([[0, ql, 0, kend]], np.int32)
    out, _, err = O.attend(q, kp, vp, bt, si, 0.35, causal=True, first_valid=np.array([first], np.int32))
    assert err == 0
    start = kend - ql
    qpos = np.arange(start, kend)[:, None]
    kpos = np.arange(kend)[None, :]
    mask = (kpos <= qpos) & ((kpos >= first) | (kpos == qpos))
    for h in range(2):
        ref = sdpa_dense(q[:, h], flat_keys(kp, kend, h), flat_keys(vp, kend, h), 0.35, mask=mask)
        assert np.abs(out[:, h] - ref).max() < 1e-12


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_left_padding_matches_brute_force_twin(seed):
    rng = np.random.default_rng(100 + seed)
    lens, qlens = [33, 20, 47], [2, 1, 3]
    q, kp, vp, bt, si = random_paged(rng, lens, qlens, 4, 2, 8)
    fv = np.array([rng.integers(0, L + 2) for L in lens], np.int32)
    for causal in (True, False):
        out, lse, err = O.attend(q, kp, vp, bt, si, 0.37, causal=causal, window=9, first_valid=fv)
        assert err == 0
        bo, bl = brute.attend(q.tolist(), kp.tolist(), vp.tolist(), bt.tolist(), si.tolist(), 0.37, causal=causal,
                              window=9, first_valid=fv.tolist())
        assert np.abs(out - np.array(bo)).max() < 1e-12
        fin = np.isfinite(lse)
        assert np.array_equal(fin, np.isfinite(np.array(bl)))
        assert np.abs(lse[fin] - np.array(bl)[fin]).max() < 1e-12

"""Randomised agreement of the C oracle with its pure-Python twin over the
whole configuration space (GQA ratio, head_dim, causal or not, window, ring
storage, left padding, empty segments), drawn by hypothesis.  The twin tests
each key against a visibility predicate; the oracle computes a key range."""
import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

from oracle import brute  # noqa: E402
from oracle import oracle as O  # noqa: E402
from tests.test_oracle import PAGE, random_paged  # noqa: E402


@st.composite
def configs(draw):
    S = draw(st.integers(1, 3))
    Hkv = draw(st.sampled_from([1, 2]))
    G = draw(st.sampled_from([1, 2, 3]))
    D = draw(st.sampled_from([4, 8, 16]))
    causal = draw(st.booleans())
    ring = draw(st.booleans())
    window = draw(st.integers(1, 24)) if ring or draw(st.booleans()) else 0
    qlens = [draw(st.integers(1 if s == 0 else 0, 4)) for s in range(S)]  # at least one row
    lens = [draw(st.integers(max(q, 1), 48)) for q in qlens]
    R = PAGE * ((window + max(max(qlens), 1) - 1 + PAGE - 1) // PAGE) if ring else 0
    padded = draw(st.booleans())
    first = [draw(st.integers(-2, L + 2)) for L in lens] if padded else None
    seed = draw(st.integers(0, 2 ** 31 - 1))
    return S, Hkv, G, D, causal, window, qlens, lens, R, first, seed


@settings(max_examples=150, deadline=None, derandomize=True, database=None)
@given(configs())
def test_oracle_matches_twin_everywhere(cfg):
    S, Hkv, G, D, causal, window, qlens, lens, R, first, seed = cfg
    rng = np.random.default_rng(seed)
    q, kp, vp, bt, si = random_paged(rng, lens, qlens, Hkv * G, Hkv, D, ring_rows=R)
    fv = None if first is None else np.array(first, np.int32)
    out, lse, err = O.attend(q, kp, vp, bt, si, 0.41, causal=causal, window=window, ring_rows=R, first_valid=fv)
    assert err == 0
    bo, bl = brute.attend(q.tolist(), kp.tolist(), vp.tolist(), bt.tolist(), si.tolist(), 0.41, causal=causal,
                          window=window, ring_rows=R, first_valid=None if fv is None else fv.tolist())
    np.testing.assert_allclose(out, np.array(bo), rtol=0, atol=1e-12)
    bl = np.array(bl)
    assert np.array_equal(np.isfinite(lse), np.isfinite(bl))
    fin = np.isfinite(lse)
    np.testing.assert_allclose(lse[fin], bl[fin], rtol=0, atol=1e-12)

"""bench.py's byte and flop accounting, checked on the CPU: the general
per-workload count against the single-sequence per-layer formula, and the
flop count against a key-by-key visibility enumeration."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads  # noqa: E402
from oracle import brute  # noqa: E402


@pytest.mark.parametrize("L", [1, 300, 4096, 8192])
def test_workload_bytes_match_per_layer_formula(L):
    w = workloads.sensenova(L, max(512, L), num_layers=1)
    nbytes, flops = bench.workload_bytes_flops(w)
    assert nbytes == bench.algorithmic_bytes_per_layer(L)
    assert flops == 4 * w.q_heads * w.head_dim * L


@pytest.mark.parametrize("causal,window", [(True, 0), (False, 0), (True, 37), (False, 37)])
def test_workload_flops_match_visibility_count(causal, window):
    w = workloads.spec_verify(S=5, max_q=6, len_lo=20, len_hi=200, causal=causal, seed=3, q_heads=16, kv_heads=4,
                              head_dim=32)
    w.window = window
    _, flops = bench.workload_bytes_flops(w)
    visible = 0
    for q0, ql, col, kend in w.seq_info.tolist():
        for i in range(ql):
            pos = kend - ql + i
            visible += sum(brute._visible(j, pos, kend, causal, window) for j in range(kend))
    assert flops == 4 * w.q_heads * w.head_dim * visible

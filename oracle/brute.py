"""Brute-force twin of the oracle, pure Python loops -- test infrastructure only.

Written independently of pkv_oracle.c: instead of a key range it tests each
position 0..kv_end-1 against a visibility predicate, finds each key by
walking the block table page by page, and uses math.exp / math.log.  Only
for tiny inputs (a few segments, tens of keys, head_dim <= 16).
"""
from __future__ import annotations

import math

PAGE = 16


def _visible(j: int, pos: int, kend: int, causal: bool, window: int, first: int = 0) -> bool:
    """Is key position j visible to the query row sitting at position pos?
    Keys before `first` (left padding) are hidden, except the row's own key."""
    if j >= kend:
        return False
    if j == pos and pos < first:
        return True
    if j < first or pos < first:
        return False
    if causal and j > pos:
        return False
    newest = pos if causal else kend - 1
    if window > 0 and j <= newest - window:
        return False
    return True


def _slot(block_table, col: int, j: int, ring_rows: int):
    r = j % ring_rows if ring_rows else j
    page, off = divmod(r, PAGE)
    return int(block_table[col][page]), off


def attend(q, k_pool, v_pool, block_table, seq_info, scale, causal=False, window=0, ring_rows=0, first_valid=None):
    """Same contract as oracle.attend for valid inputs; returns (out, lse) as nested lists."""
    rows, hq, d = len(q), len(q[0]), len(q[0][0])
    hkv = len(k_pool[0][0])
    group = hq // hkv
    out = [[[0.0] * d for _ in range(hq)] for _ in range(rows)]
    lse = [[-math.inf] * hq for _ in range(rows)]
    for q0, ql, col, kend in seq_info:
        for i in range(ql):
            t, pos = q0 + i, kend - ql + i
            for h in range(hq):
                g = h // group
                first = max(0, int(first_valid[col])) if first_valid is not None else 0
                keys = [j for j in range(kend) if _visible(j, pos, kend, causal, window, first)]
                if not keys:
                    continue
                scores = []
                for j in keys:
                    b, o = _slot(block_table, col, j, ring_rows)
                    dot = 0.0
                    for e in range(d):
                        dot += float(q[t][h][e]) * float(k_pool[b][o][g][e])
                    scores.append(scale * dot)
                top = max(scores)
                ws = [math.exp(x - top) for x in scores]
                tot = sum(ws)
                for e in range(d):
                    acc = 0.0
                    for w, j in zip(ws, keys):
                        b, o = _slot(block_table, col, j, ring_rows)
                        acc += w * float(v_pool[b][o][g][e])
                    out[t][h][e] = acc / tot
                lse[t][h] = top + math.log(tot)
    return out, lse


def append_slots(block_table, seq_info, ring_rows=0):
    """List of (row t, block, offset) the append writes, one per covered row."""
    res = []
    for q0, ql, col, kend in seq_info:
        for i in range(ql):
            b, o = _slot(block_table, col, kend - ql + i, ring_rows)
            res.append((q0 + i, b, o))
    return res

"""Seeded synthetic inputs for paged decode attention.

This module only draws random numbers and lays them out in the shapes the
paged cache uses; it holds none of the attention arithmetic.  Both the CPU
oracle (through the tests) and the CUDA path consume what it returns.

Shapes follow the pages:
  * K/V pool per layer: (num_blocks, 16, kv_heads, head_dim), the layout the
    vLLM-Omni SenseNova-U1 ``PagedDecodeCache`` docstring gives;
  * block table: int32 (max_seqs, max_blocks_per_seq);
  * segment table: int32 (S, 4) = (q_start, q_len, col, kv_end), the
    ``seq_info`` table of ExecuTorch PR #24072 (``triton::sdpa_varlen``);
  * q: (total_rows, q_heads, head_dim); k_new / v_new: (total_rows,
    kv_heads, head_dim).

Values: q ~ N(0, 1); K/V ~ N(0, 1) / sqrt(head_dim) for bf16 workloads and
N(0, 1) for the fp32 tiny case, cast to the workload dtype.  Every draw comes
from one ``torch.Generator`` seeded by the caller, on the device the caller
names.  The bucket size of a single-sequence workload is an input here: it
is computed by the code under test (and, separately, by the oracle).
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import torch

BLOCK = 16  # tokens per page, fixed by the page layout


@dataclasses.dataclass
class Workload:
    """One batch of synthetic decode inputs (all tensors on ``device``)."""

    name: str
    dtype: torch.dtype
    num_layers: int
    q_heads: int
    kv_heads: int
    head_dim: int
    num_blocks: int
    block_table: torch.Tensor          # int32 (max_seqs, max_blocks_per_seq)
    seq_info: torch.Tensor             # int32 (S, 4)
    k: List[torch.Tensor]              # per layer (num_blocks, 16, Hkv, D)
    v: List[torch.Tensor]
    q: List[torch.Tensor]              # per layer (total_rows, Hq, D)
    k_new: List[torch.Tensor]          # per layer (total_rows, Hkv, D)
    v_new: List[torch.Tensor]
    causal: bool = False
    window: int = 0
    ring_rows: int = 0
    bucket: int = 0                    # tokens the per-sequence table spans
    max_q_len: int = 1

    @property
    def total_rows(self) -> int:
        return int(self.q[0].shape[0])

    @property
    def num_segments(self) -> int:
        return int(self.seq_info.shape[0])

    @property
    def max_seqs(self) -> int:
        return int(self.block_table.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    def to(self, device) -> "Workload":
        mv = lambda ts: [t.to(device) for t in ts]  # noqa: E731
        return dataclasses.replace(
            self, block_table=self.block_table.to(device), seq_info=self.seq_info.to(device),
            k=mv(self.k), v=mv(self.v), q=mv(self.q), k_new=mv(self.k_new), v_new=mv(self.v_new))


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal(shape, g, device, std: float, dtype) -> torch.Tensor:
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def _pools(g, device, num_layers, num_blocks, kv_heads, head_dim, std, dtype, nan_fill):
    shape = (num_blocks, BLOCK, kv_heads, head_dim)
    ks, vs = [], []
    for _ in range(num_layers):
        ks.append(_normal(shape, g, device, std, dtype))
        vs.append(_normal(shape, g, device, std, dtype))
    return ks, vs


def _step_rows(g, device, num_layers, rows, q_heads, kv_heads, head_dim, kv_std, dtype):
    q, kn, vn = [], [], []
    for _ in range(num_layers):
        q.append(_normal((rows, q_heads, head_dim), g, device, 1.0, dtype))
        kn.append(_normal((rows, kv_heads, head_dim), g, device, kv_std, dtype))
        vn.append(_normal((rows, kv_heads, head_dim), g, device, kv_std, dtype))
    return q, kn, vn


def nan_fill_unused(w: Workload) -> None:
    """Write NaN into every pool slot no segment's key range reaches.

    A slot is 'live' when it lies in a block the table lists for a segment's
    column, at an in-block offset below that segment's kv_end.  Anything else
    (stale tails, blocks no table row lists) becomes NaN, so a kernel that
    reads past the live prefix produces NaN and fails parity.  Ring layouts
    keep every slot of a listed block (all of them can be live).
    """
    if not w.dtype.is_floating_point:
        return
    live = torch.zeros(w.num_blocks * BLOCK, dtype=torch.bool)
    bt = w.block_table.cpu()
    si = w.seq_info.cpu()
    for s in range(si.shape[0]):
        _, _, col, kend = [int(x) for x in si[s]]
        if not (0 <= col < bt.shape[0]):
            continue
        span = w.ring_rows if w.ring_rows else kend
        span = min(span, bt.shape[1] * BLOCK)
        j = torch.arange(max(span, 0), dtype=torch.long)
        b = bt[col, j // BLOCK].long()
        ok = (b >= 0) & (b < w.num_blocks)
        live[(b * BLOCK + j % BLOCK)[ok]] = True
    dead = (~live).to(w.k[0].device)
    for t in w.k + w.v:
        flat = t.view(-1, t.shape[2], t.shape[3])
        flat[dead] = float("nan")


def tiny(seed: int = 0, device="cpu", bucket: int = 512, seqused: int = 300) -> Workload:
    """1 layer, 8 q / 2 kv heads, head_dim 64, fp32, identity table, one token."""
    g = _gen(seed, device)
    Hq, Hkv, D = 8, 2, 64
    nblocks = bucket // BLOCK
    k, v = _pools(g, device, 1, nblocks, Hkv, D, 1.0, torch.float32, False)
    q, kn, vn = _step_rows(g, device, 1, 1, Hq, Hkv, D, 1.0, torch.float32)
    bt = torch.arange(nblocks, dtype=torch.int32, device=device).unsqueeze(0)
    si = torch.tensor([[0, 1, 0, seqused]], dtype=torch.int32, device=device)
    return Workload("tiny", torch.float32, 1, Hq, Hkv, D, nblocks, bt, si, k, v, q, kn, vn,
                    bucket=bucket)


def sensenova(seqused: int, bucket: int, num_layers: int = 42, seed: int = 0, device="cpu",
              q_heads: int = 32, kv_heads: int = 8, head_dim: int = 128,
              dtype=torch.bfloat16) -> Workload:
    """Single-sequence decode behind an identity table, one token per step."""
    g = _gen(seed, device)
    nblocks = bucket // BLOCK
    std = 1.0 / math.sqrt(head_dim)
    k, v = _pools(g, device, num_layers, nblocks, kv_heads, head_dim, std, dtype, False)
    q, kn, vn = _step_rows(g, device, num_layers, 1, q_heads, kv_heads, head_dim, std, dtype)
    bt = torch.arange(nblocks, dtype=torch.int32, device=device).unsqueeze(0)
    si = torch.tensor([[0, 1, 0, seqused]], dtype=torch.int32, device=device)
    return Workload("sensenova", dtype, num_layers, q_heads, kv_heads, head_dim, nblocks, bt, si,
                    k, v, q, kn, vn, bucket=bucket)


def _shared_pool_tables(g, lengths: List[int], max_blocks_per_seq: int, extra_blocks: int = 0):
    """Per-sequence block tables drawn from one shuffled pool of pages."""
    need = [(L + BLOCK - 1) // BLOCK for L in lengths]
    total = sum(need) + extra_blocks
    perm = torch.randperm(total, generator=g, device=g.device).to("cpu", torch.int32)
    bt = torch.full((len(lengths), max_blocks_per_seq), -1, dtype=torch.int32)
    at = 0
    for s, n in enumerate(need):
        bt[s, :n] = perm[at:at + n]
        at += n
    return bt, total


def batched(S: int = 32, max_len: int = 16384, seed: int = 0, device="cpu", num_layers: int = 1,
            q_heads: int = 32, kv_heads: int = 8, head_dim: int = 128, dtype=torch.bfloat16,
            min_len: int = 1, lengths: Optional[List[int]] = None) -> Workload:
    """S sequences with lengths U[min_len, max_len], pages shuffled over a shared pool."""
    g = _gen(seed, device)
    if lengths is None:
        lengths = torch.randint(min_len, max_len + 1, (S,), generator=g, device=device).tolist()
    mbps = (max_len + BLOCK - 1) // BLOCK
    bt, nblocks = _shared_pool_tables(g, lengths, mbps)
    std = 1.0 / math.sqrt(head_dim)
    k, v = _pools(g, device, num_layers, nblocks, kv_heads, head_dim, std, dtype, False)
    q, kn, vn = _step_rows(g, device, num_layers, S, q_heads, kv_heads, head_dim, std, dtype)
    si = torch.tensor([[s, 1, s, lengths[s]] for s in range(S)], dtype=torch.int32)
    return Workload("batched", dtype, num_layers, q_heads, kv_heads, head_dim, nblocks,
                    bt.to(device), si.to(device), k, v, q, kn, vn, bucket=mbps * BLOCK)


def spec_verify(S: int = 16, max_q: int = 16, len_lo: int = 256, len_hi: int = 8192,
                causal: bool = True, seed: int = 0, device="cpu", num_layers: int = 1,
                q_heads: int = 64, kv_heads: int = 8, head_dim: int = 128,
                dtype=torch.bfloat16) -> Workload:
    """S segments of q_len U[1, max_q] rows packed back to back; kv_end U[len_lo, len_hi]."""
    g = _gen(seed, device)
    qlens = torch.randint(1, max_q + 1, (S,), generator=g, device=device).tolist()
    lengths = torch.randint(len_lo, len_hi + 1, (S,), generator=g, device=device).tolist()
    mbps = (len_hi + BLOCK - 1) // BLOCK
    bt, nblocks = _shared_pool_tables(g, lengths, mbps)
    std = 1.0 / math.sqrt(head_dim)
    rows = sum(qlens)
    k, v = _pools(g, device, num_layers, nblocks, kv_heads, head_dim, std, dtype, False)
    q, kn, vn = _step_rows(g, device, num_layers, rows, q_heads, kv_heads, head_dim, std, dtype)
    si, at = [], 0
    for s in range(S):
        si.append([at, qlens[s], s, lengths[s]])
        at += qlens[s]
    return Workload("spec_verify", dtype, num_layers, q_heads, kv_heads, head_dim, nblocks,
                    bt.to(device), torch.tensor(si, dtype=torch.int32, device=device),
                    k, v, q, kn, vn, causal=causal, bucket=mbps * BLOCK, max_q_len=max_q)


def long_context(S: int = 4, kv_len: int = 131072, window: int = 0, ring_rows: int = 0,
                 seed: int = 0, device="cpu", num_layers: int = 1, q_heads: int = 32,
                 kv_heads: int = 4, head_dim: int = 256, dtype=torch.bfloat16) -> Workload:
    """Few very long sequences; optionally a sliding window over ring storage of ring_rows."""
    g = _gen(seed, device)
    span = ring_rows if ring_rows else kv_len
    mbps = (span + BLOCK - 1) // BLOCK
    bt, nblocks = _shared_pool_tables(g, [span] * S, mbps)
    std = 1.0 / math.sqrt(head_dim)
    k, v = _pools(g, device, num_layers, nblocks, kv_heads, head_dim, std, dtype, False)
    q, kn, vn = _step_rows(g, device, num_layers, S, q_heads, kv_heads, head_dim, std, dtype)
    si = torch.tensor([[s, 1, s, kv_len] for s in range(S)], dtype=torch.int32, device=device)
    return Workload("long_context", dtype, num_layers, q_heads, kv_heads, head_dim, nblocks,
                    bt.to(device), si, k, v, q, kn, vn, causal=True, window=window,
                    ring_rows=ring_rows, bucket=mbps * BLOCK)

"""CUDA-graph decode step over the paged cache: one capture per bucket.

Mirrors vLLM-Omni's SenseNova-U1 DecodeGraphRunner without a model: every
input a step varies (the new rows' q/k/v and the segment table holding the
live lengths) sits in static device tensors, so one captured graph of
`num_layers` append+attend launches serves every length in the bucket.  A
capture is keyed on (bucket, generation); a resize bumps the generation and
the next step captures again.  Warm-up runs three times on a side stream
before capture (it rewrites the same rows to the same slots, so it is
idempotent), and every capture shares one graph memory pool: a private pool
per runner grew device memory without bound in the page's measurement.
"""
from __future__ import annotations

import math
from typing import Dict, List, Optional, Tuple

import torch

from . import _lib
from .api import PagedKVCache, append, append_attend, attend_varlen, new_err_flags, new_workspace
from .api import advance as advance_lengths

_SHARED_POOL = None


def shared_pool():
    global _SHARED_POOL
    if _SHARED_POOL is None:
        _SHARED_POOL = torch.cuda.graph_pool_handle()
    return _SHARED_POOL


def _carve(spec, device) -> Tuple[torch.Tensor, List[torch.Tensor]]:
    """One zeroed uint8 buffer holding tensors of the given (shape, dtype)
    back to back, each at a 16-byte offset; returns it and the typed views."""
    sizes = [math.prod(shape) * torch.empty((), dtype=dt).element_size() for shape, dt in spec]
    offs, total = [], 0
    for n in sizes:
        offs.append(total)
        total += (n + 15) // 16 * 16
    buf = torch.zeros(max(total, 16), dtype=torch.uint8, device=device)
    views = [buf[o:o + n].view(dt).view(shape) for (shape, dt), o, n in zip(spec, offs, sizes)]
    return buf, views


class DecodeStep:
    """Static buffers and launches of one decode step over all layers.

    Every input a step varies (per layer q, k_new, v_new; then the segment
    table) lives in one device buffer, `inputs`, and every output (per layer
    out, then lse) in another, `outputs`; the per-layer tensors are views of
    them, so a step's host round trip is one copy each way.

    With advance=True the step ends with `kv_end += q_len` for every segment
    on the device (tiny-llm kv_cache.py, SlotKVCache.end_step), so a replay
    leaves the segment table ready for the next step and the host writes it
    only once: per step it copies q, k_new and v_new (`step_inputs`) and
    keeps its own copy of the lengths in step (advance_host).
    """

    def __init__(self, cache: PagedKVCache, num_q_heads: int, rows: int = 1, num_segments: int = 1,
                 max_q_len: int = 1, max_kv: Optional[int] = None, scale: Optional[float] = None,
                 causal: bool = False, window: int = 0, fused: bool = True, pdl: bool = True,
                 flags: int = 0, num_splits: int = 0, with_lse: bool = False, prefetch_next: bool = True,
                 workspace: bool = False, advance: bool = False):
        dev = cache.k[0].device
        L, Hkv, D = cache.num_layers, cache.kv_heads, cache.head_dim
        self.cache = cache
        self.num_q_heads = num_q_heads
        self.max_q_len = max_q_len
        self.max_kv = int(max_kv if max_kv is not None else cache.bucket)
        self.scale = scale if scale is not None else 1.0 / math.sqrt(D)
        self.causal, self.window = causal, window
        self.fused, self.pdl, self.flags, self.num_splits = fused, pdl, flags, num_splits
        self.prefetch_next = prefetch_next
        spec_in = ([((rows, num_q_heads, D), cache.dtype)] * L + [((rows, Hkv, D), cache.dtype)] * (2 * L)
                   + [((num_segments, 4), torch.int32)])
        self.inputs, views = _carve(spec_in, dev)
        self.q, self.k_new, self.v_new = views[:L], views[L:2 * L], views[2 * L:3 * L]
        self.seq_info = views[3 * L]
        # the per-step part of `inputs` (q, k_new, v_new of every layer): the
        # segment table sits after it
        self.step_inputs = self.inputs[:self.seq_info.data_ptr() - self.inputs.data_ptr()]
        self.advance = advance
        spec_out = [((rows, num_q_heads, D), torch.float32)] * L
        if with_lse:
            spec_out += [((rows, num_q_heads), torch.float32)] * L
        self.outputs, views = _carve(spec_out, dev)
        self.out = views[:L]
        self.lse = views[L:] if with_lse else [None] * L
        self.err = new_err_flags(dev)
        self.use_workspace = workspace
        self.ws = None
        self.size_workspace()

    def size_workspace(self) -> None:
        """(Re)allocate the split-merge workspace for the current cache and bounds (None when not needed)."""
        self.ws = None
        if self.use_workspace:
            self.ws = new_workspace(self.cache, self.num_q_heads, int(self.seq_info.shape[0]), self.max_q_len,
                                    self.max_kv, self.num_splits, self.flags)

    def launch_count(self) -> int:
        return self.cache.num_layers * (1 if self.fused else 2) + (1 if self.advance else 0)

    def run(self, stream=None, advance: Optional[bool] = None) -> None:
        """Enqueue every layer's append + attention on the current stream,
        then (advance=True, by default the step's setting) the on-device
        length advance."""
        c = self.cache
        for layer in range(c.num_layers):
            flags = self.flags
            if self.pdl and layer > 0 and self.fused:
                flags |= _lib.FLAG_PDL
            if self.prefetch_next and layer + 1 < c.num_layers:
                flags |= _lib.FLAG_PREFETCH_NEXT  # the next call attends layer + 1 over the same segments
            if self.fused:
                append_attend(c, layer, self.q[layer], self.k_new[layer], self.v_new[layer], self.seq_info,
                              self.out[layer], self.err, self.max_q_len, self.max_kv, self.scale, self.causal,
                              self.window, lse=self.lse[layer], num_splits=self.num_splits, flags=flags,
                              stream=stream, workspace=self.ws)
            else:
                append(c, layer, self.k_new[layer], self.v_new[layer], self.seq_info, self.err,
                       window=self.window, stream=stream)
                attend_varlen(c, layer, self.q[layer], self.seq_info, self.out[layer], self.err, self.max_q_len,
                              self.max_kv, self.scale, self.causal, self.window, lse=self.lse[layer],
                              num_splits=self.num_splits, flags=flags, stream=stream, workspace=self.ws)
        if self.advance if advance is None else advance:
            advance_lengths(self.seq_info, stream=stream)


class DecodeGraphRunner:
    """One captured DecodeStep per (bucket, generation), replayed for every length."""

    def __init__(self, step: DecodeStep):
        self.step_bufs = step
        self._graphs: Dict[Tuple[int, int], torch.cuda.CUDAGraph] = {}
        self.captures = 0

    def _capture(self, key):
        st = self.step_bufs
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            # Warm-up leaves the lengths alone (a warm-up that advanced them
            # would move the step three tokens on); the advance kernel is
            # warmed on a scratch row instead.
            for _ in range(3):
                st.run(advance=False)
            if st.advance:
                advance_lengths(torch.zeros(1, 4, dtype=torch.int32, device=st.seq_info.device))
        torch.cuda.current_stream().wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, pool=shared_pool()):
            st.run()
        self.captures += 1
        self._graphs[key] = graph
        return graph

    def rebind(self, cache: PagedKVCache) -> None:
        """Point the step at a resized cache; captures of older buffers are dropped."""
        st = self.step_bufs
        st.cache = cache
        st.max_kv = cache.bucket
        st.size_workspace()
        self._graphs = {k: g for k, g in self._graphs.items() if k == (cache.bucket, cache.generation)}

    def graph_for(self) -> torch.cuda.CUDAGraph:
        c = self.step_bufs.cache
        key = (c.bucket, c.generation)
        return self._graphs.get(key) or self._capture(key)

    def step(self) -> None:
        """Replay the step for whatever lengths the segment table holds now."""
        self.graph_for().replay()

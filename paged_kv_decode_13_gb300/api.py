"""Python binding of libpkv: the C entry points under the same names.

Only argument marshalling happens here (tensor pointers, the current CUDA
stream, status checks).  Every step of the computation runs in the library's
CUDA kernels; torch supplies device memory and streams.
"""
from __future__ import annotations

import ctypes
from typing import List, Optional, Sequence

import torch

from . import _lib
from ._lib import lib

_DTYPES = {torch.bfloat16: _lib.BF16, torch.float32: _lib.F32}


def _stream(stream=None) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    return t.data_ptr()


def _contig(t: torch.Tensor, name: str) -> torch.Tensor:
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


class PagedKVCache:
    """Per-layer paged K/V pools plus one block table, and their descriptor.

    Pools are (num_blocks, 16, kv_heads, head_dim) tensors of bf16 or fp32
    (the layout of vLLM-Omni's SenseNova-U1 PagedDecodeCache); the block
    table is int32 (max_seqs, max_blocks_per_seq).  first_valid, optional
    int32 (max_seqs,), is each sequence's first non-padding position for
    left-padded batches (tiny-llm kv_cache.py, SlotKVCache): the attention
    calls hide earlier keys and let a padding row see only its own key.  The
    tensors are owned by this object; the descriptor only points at them.
    """

    def __init__(self, k: Sequence[torch.Tensor], v: Sequence[torch.Tensor], block_table: torch.Tensor,
                 ring_rows: int = 0, bucket: Optional[int] = None, generation: int = 0,
                 first_valid: Optional[torch.Tensor] = None):
        if len(k) != len(v) or not k:
            raise ValueError("k and v need one tensor per layer")
        shape, dtype = k[0].shape, k[0].dtype
        if dtype not in _DTYPES:
            raise ValueError(f"unsupported dtype {dtype}")
        for t in list(k) + list(v):
            if t.shape != shape or t.dtype != dtype or not t.is_contiguous():
                raise ValueError("every pool must be contiguous with the same shape and dtype")
        if len(shape) != 4 or shape[1] != _lib.BLOCK_SIZE:
            raise ValueError("pools are (num_blocks, 16, kv_heads, head_dim)")
        if block_table.dtype != torch.int32 or block_table.dim() != 2:
            raise ValueError("block_table is int32 (max_seqs, max_blocks_per_seq)")
        self.k: List[torch.Tensor] = list(k)
        self.v: List[torch.Tensor] = list(v)
        self.block_table = _contig(block_table, "block_table")
        if first_valid is not None and (first_valid.dtype != torch.int32 or first_valid.dim() != 1
                                        or first_valid.shape[0] != block_table.shape[0]):
            raise ValueError("first_valid is int32 (max_seqs,)")
        self.first_valid = None if first_valid is None else _contig(first_valid, "first_valid")
        self.ring_rows = int(ring_rows)
        self.generation = int(generation)
        nb = shape[0]
        self.bucket = int(bucket) if bucket is not None else int(block_table.shape[1]) * _lib.BLOCK_SIZE
        self._kp = (ctypes.c_void_p * len(k))(*[t.data_ptr() for t in self.k])
        self._vp = (ctypes.c_void_p * len(v))(*[t.data_ptr() for t in self.v])
        self.desc = _lib.CacheDesc(
            num_layers=len(k), kv_heads=shape[2], head_dim=shape[3], dtype=_DTYPES[dtype], num_blocks=nb,
            max_seqs=block_table.shape[0], max_blocks_per_seq=block_table.shape[1], ring_rows=self.ring_rows,
            reserved0=0, k=ctypes.cast(self._kp, ctypes.c_void_p), v=ctypes.cast(self._vp, ctypes.c_void_p),
            block_table=block_table.data_ptr(), bucket=self.bucket, generation=self.generation,
            first_valid=_ptr(self.first_valid))

    @classmethod
    def allocate(cls, num_layers: int, kv_heads: int, head_dim: int, bucket: int, dtype=torch.bfloat16,
                 device="cuda", generation: int = 0) -> "PagedKVCache":
        """Zeroed single-sequence cache behind an identity table (one bucket)."""
        nb = (bucket + _lib.BLOCK_SIZE - 1) // _lib.BLOCK_SIZE
        shape = (nb, _lib.BLOCK_SIZE, kv_heads, head_dim)
        k = [torch.zeros(shape, dtype=dtype, device=device) for _ in range(num_layers)]
        v = [torch.zeros(shape, dtype=dtype, device=device) for _ in range(num_layers)]
        bt = torch.arange(nb, dtype=torch.int32, device=device).unsqueeze(0)
        return cls(k, v, bt, bucket=bucket, generation=generation)

    @property
    def num_layers(self) -> int:
        return len(self.k)

    @property
    def kv_heads(self) -> int:
        return int(self.k[0].shape[2])

    @property
    def head_dim(self) -> int:
        return int(self.k[0].shape[3])

    @property
    def dtype(self) -> torch.dtype:
        return self.k[0].dtype

    def ref(self):
        return ctypes.byref(self.desc)

    def reusable_for(self, num_layers, kv_heads, head_dim, dtype, length) -> bool:
        """Same shape and the length fits the current bucket (PagedDecodeCache.reusable_for)."""
        return (self.num_layers == num_layers and self.kv_heads == kv_heads and self.head_dim == head_dim
                and self.dtype == dtype and bucket_for(length) <= self.bucket)


def bucket_for(length: int) -> int:
    return int(lib.pkv_bucket_for(int(length)))


def new_err_flags(device="cuda") -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device)


def append(cache: PagedKVCache, layer: int, k_new: torch.Tensor, v_new: torch.Tensor, seq_info: torch.Tensor,
           err: torch.Tensor, window: int = 0, stream=None) -> None:
    rows = int(k_new.shape[0])
    _lib.check("pkv_append", lib.pkv_append(
        cache.ref(), layer, _ptr(_contig(k_new, "k_new")), _ptr(_contig(v_new, "v_new")), rows,
        _ptr(_contig(seq_info, "seq_info")), int(seq_info.shape[0]), int(window), _ptr(err), _stream(stream)))


def _attend(fn_name, cache, layer, q, k_new, v_new, seq_info, out, lse, err, max_q_len, max_kv, scale, causal,
            window, num_splits, flags, stream, workspace):
    rows, hq = int(q.shape[0]), int(q.shape[1])
    args = [cache.ref(), layer, _ptr(_contig(q, "q"))]
    if fn_name == "pkv_append_attend":
        args += [_ptr(_contig(k_new, "k_new")), _ptr(_contig(v_new, "v_new"))]
    ws_bytes = int(workspace.numel() * workspace.element_size()) if workspace is not None else 0
    args += [hq, rows, _ptr(_contig(seq_info, "seq_info")), int(seq_info.shape[0]), int(max_q_len), int(max_kv),
             int(num_splits), float(scale), int(bool(causal)), int(window), _ptr(_contig(out, "out")),
             _ptr(lse), _ptr(workspace), ws_bytes, _ptr(err), int(flags), _stream(stream)]
    _lib.check(fn_name, getattr(lib, fn_name)(*args))


def attend_varlen(cache: PagedKVCache, layer: int, q: torch.Tensor, seq_info: torch.Tensor, out: torch.Tensor,
                  err: torch.Tensor, max_q_len: int, max_kv: int, scale: float, causal: bool = False,
                  window: int = 0, lse: Optional[torch.Tensor] = None, num_splits: int = 0, flags: int = 0,
                  stream=None, workspace: Optional[torch.Tensor] = None) -> None:
    _attend("pkv_attend_varlen", cache, layer, q, None, None, seq_info, out, lse, err, max_q_len, max_kv, scale,
            causal, window, num_splits, flags, stream, workspace)


def append_attend(cache: PagedKVCache, layer: int, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                  seq_info: torch.Tensor, out: torch.Tensor, err: torch.Tensor, max_q_len: int, max_kv: int,
                  scale: float, causal: bool = False, window: int = 0, lse: Optional[torch.Tensor] = None,
                  num_splits: int = 0, flags: int = 0, stream=None, workspace: Optional[torch.Tensor] = None) -> None:
    _attend("pkv_append_attend", cache, layer, q, k_new, v_new, seq_info, out, lse, err, max_q_len, max_kv, scale,
            causal, window, num_splits, flags, stream, workspace)


def append_attend_noalloc(cache: PagedKVCache, layer: int, q: torch.Tensor, k_new: torch.Tensor,
                          v_new: torch.Tensor, seq_info: torch.Tensor, out: torch.Tensor, err: torch.Tensor,
                          max_q_len: int, max_kv: int, scale: float, causal: bool = False, window: int = 0,
                          lse: Optional[torch.Tensor] = None, num_splits: int = 0, flags: int = 0,
                          stream=None) -> None:
    """pkv_append_attend_noalloc: append_attend merging its splits in the library's fixed scratch."""
    rows, hq = int(q.shape[0]), int(q.shape[1])
    _lib.check("pkv_append_attend_noalloc", lib.pkv_append_attend_noalloc(
        cache.ref(), layer, _ptr(_contig(q, "q")), _ptr(_contig(k_new, "k_new")), _ptr(_contig(v_new, "v_new")),
        hq, rows, _ptr(_contig(seq_info, "seq_info")), int(seq_info.shape[0]), int(max_q_len), int(max_kv),
        int(num_splits), float(scale), int(bool(causal)), int(window), _ptr(_contig(out, "out")), _ptr(lse),
        _ptr(err), int(flags), _stream(stream)))


def attend_workspace_bytes(cache: PagedKVCache, num_q_heads: int, num_segments: int, max_q_len: int, max_kv: int,
                           num_splits: int = 0, flags: int = 0) -> int:
    """pkv_attend_workspace_bytes: workspace the attention calls need for these bounds (0: none)."""
    n = int(lib.pkv_attend_workspace_bytes(cache.ref(), int(num_q_heads), int(num_segments), int(max_q_len),
                                           int(max_kv), int(num_splits), int(flags)))
    if n < 0:
        _lib.check("pkv_attend_workspace_bytes", n)
    return n


def new_workspace(cache: PagedKVCache, num_q_heads: int, num_segments: int, max_q_len: int, max_kv: int,
                  num_splits: int = 0, flags: int = 0) -> Optional[torch.Tensor]:
    """A zero-filled workspace for these bounds on the cache's device, or None if none is needed."""
    n = attend_workspace_bytes(cache, num_q_heads, num_segments, max_q_len, max_kv, num_splits, flags)
    return torch.zeros(n, dtype=torch.uint8, device=cache.k[0].device) if n > 0 else None


def seq_clone(cache: PagedKVCache, src_col: int, dst_col: int, n: int, err: torch.Tensor, stream=None) -> None:
    """pkv_seq_clone: copy positions 0..n-1 of block-table row src_col to dst_col in every layer."""
    _lib.check("pkv_seq_clone", lib.pkv_seq_clone(cache.ref(), int(src_col), int(dst_col), int(n), _ptr(err),
                                                  _stream(stream)))


def rewind(cache: PagedKVCache, seq_info: torch.Tensor, amount: torch.Tensor, err: torch.Tensor, window: int = 0,
           stream=None) -> None:
    """pkv_rewind: kv_end -= amount per segment on the device, bounded by the ring floor."""
    _lib.check("pkv_rewind", lib.pkv_rewind(cache.ref(), _ptr(_contig(seq_info, "seq_info")), int(seq_info.shape[0]),
                                            _ptr(_contig(amount, "amount")), int(window), _ptr(err),
                                            _stream(stream)))


def seqinfo_from_seqused(cu_seqlens_q: torch.Tensor, seqused_k: torch.Tensor, out: torch.Tensor,
                         stream=None) -> None:
    n = int(seqused_k.shape[0])
    _lib.check("pkv_seqinfo_from_seqused", lib.pkv_seqinfo_from_seqused(
        _ptr(cu_seqlens_q), _ptr(seqused_k), n, _ptr(out), _stream(stream)))


def advance(seq_info: torch.Tensor, stream=None) -> None:
    _lib.check("pkv_advance", lib.pkv_advance(_ptr(seq_info), int(seq_info.shape[0]), _stream(stream)))


def resize_bucket(old: PagedKVCache, new: PagedKVCache, old_len: int, stream=None) -> int:
    """Copy the first old_len tokens of every layer; bumps new.generation on success."""
    st = _lib.check("pkv_resize_bucket", lib.pkv_resize_bucket(old.ref(), new.ref(), int(old_len),
                                                                 _stream(stream)), (_lib.OK, _lib.SAME_BUCKET))
    new.generation = int(new.desc.generation)
    return st


def load_prefix(cache: PagedKVCache, keys: Sequence[torch.Tensor], values: Sequence[torch.Tensor],
                stream=None) -> bool:
    """keys/values: per layer [S, H, D] views (any strides with D contiguous).  False if empty."""
    if not keys or keys[0] is None or keys[0].shape[0] == 0:
        return False
    n = int(keys[0].shape[0])
    ss, sh, sd = keys[0].stride()
    if sd != 1:
        raise ValueError("head_dim must be contiguous")
    for t in list(keys) + list(values):
        if t.stride() != (ss, sh, 1) or t.shape != keys[0].shape or t.dtype != cache.dtype:
            raise ValueError("all prefix tensors need the same shape, strides and dtype")
    kp = (ctypes.c_void_p * len(keys))(*[t.data_ptr() for t in keys])
    vp = (ctypes.c_void_p * len(values))(*[t.data_ptr() for t in values])
    st = lib.pkv_load_prefix(cache.ref(), ctypes.cast(kp, ctypes.c_void_p), ctypes.cast(vp, ctypes.c_void_p), n,
                             ss, sh, _stream(stream))
    return _lib.check("pkv_load_prefix", st, (_lib.OK, _lib.EMPTY)) == _lib.OK


def to_contiguous(cache: PagedKVCache, layer: int, n: int, keys_out: torch.Tensor, values_out: torch.Tensor,
                  stream=None) -> None:
    """keys_out / values_out: contiguous [kv_heads, n, head_dim]."""
    _lib.check("pkv_to_contiguous", lib.pkv_to_contiguous(cache.ref(), layer, int(n), _ptr(keys_out),
                                                          _ptr(values_out), _stream(stream)))

"""ctypes loader for libpkv.so and the pkv_cache descriptor mirror.

The library is built in-tree (``build.py``).  Importing this module without
it raises ImportError: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpkv.so")

# pkv_status
OK, EMPTY, SAME_BUCKET = 0, 1, 2
EINVAL, EUNSUPPORTED, ECUDA, ECAPACITY, ESTALE = -1, -2, -3, -4, -5
# pkv_dtype
BF16, F32 = 0, 1
# device error bits
ERR_SEGMENT, ERR_CAPACITY, ERR_RING, ERR_BLOCK, ERR_QLEN, ERR_OVERLAP, ERR_TIMEOUT = 1, 2, 4, 8, 16, 32, 64
# attention flags
FLAG_SIMT, FLAG_PDL, FLAG_PREFETCH_NEXT, FLAG_MMA_SYNC = 1, 2, 4, 8
BLOCK_SIZE = 16


class CacheDesc(ctypes.Structure):
    """Mirror of ``struct pkv_cache`` in include/pkv.h."""

    _fields_ = [
        ("num_layers", ctypes.c_int32),
        ("kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("num_blocks", ctypes.c_int64),
        ("max_seqs", ctypes.c_int32),
        ("max_blocks_per_seq", ctypes.c_int32),
        ("ring_rows", ctypes.c_int32),
        ("reserved0", ctypes.c_int32),
        ("k", ctypes.c_void_p),
        ("v", ctypes.c_void_p),
        ("block_table", ctypes.c_void_p),
        ("bucket", ctypes.c_int64),
        ("generation", ctypes.c_int64),
        ("first_valid", ctypes.c_void_p),
    ]


def _declare(lib):
    i32, i64, u32, f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32, ctypes.c_float
    p = ctypes.c_void_p
    cp = ctypes.POINTER(CacheDesc)
    sigs = {
        "pkv_bucket_for": (i64, [i64]),
        "pkv_status_str": (ctypes.c_char_p, [ctypes.c_int]),
        "pkv_append": (ctypes.c_int, [cp, i32, p, p, i32, p, i32, i32, p, p]),
        "pkv_attend_varlen": (ctypes.c_int, [cp, i32, p, i32, i32, p, i32, i32, i64, i32, f32, i32, i32,
                                             p, p, p, i64, p, u32, p]),
        "pkv_append_attend": (ctypes.c_int, [cp, i32, p, p, p, i32, i32, p, i32, i32, i64, i32, f32, i32,
                                             i32, p, p, p, i64, p, u32, p]),
        "pkv_attend_workspace_bytes": (i64, [cp, i32, i32, i32, i64, i32, u32]),
        "pkv_append_attend_noalloc": (ctypes.c_int, [cp, i32, p, p, p, i32, i32, p, i32, i32, i64, i32, f32, i32,
                                                     i32, p, p, p, u32, p]),
        "pkv_seqinfo_from_seqused": (ctypes.c_int, [p, p, i32, p, p]),
        "pkv_seq_clone": (ctypes.c_int, [cp, i32, i32, i64, p, p]),
        "pkv_rewind": (ctypes.c_int, [cp, p, i32, p, i32, p, p]),
        "pkv_advance": (ctypes.c_int, [p, i32, p]),
        "pkv_resize_bucket": (ctypes.c_int, [cp, cp, i64, p]),
        "pkv_load_prefix": (ctypes.c_int, [cp, p, p, i64, i64, i64, p]),
        "pkv_to_contiguous": (ctypes.c_int, [cp, i32, i64, p, p, p]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"libpkv.so not found at {LIB_PATH}; build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'` (needs nvcc)")
    return _declare(ctypes.CDLL(LIB_PATH))


lib = load()


class PkvError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        msg = lib.pkv_status_str(status).decode()
        super().__init__(f"{fn} returned {status} ({msg})")


def check(fn: str, status: int, allowed=(OK,)) -> int:
    if status not in allowed:
        raise PkvError(fn, status)
    return status

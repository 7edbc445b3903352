"""ctypes binding of the fp64 C oracle -- test infrastructure only.

Arrays are NumPy.  Floating inputs are widened to float64 by the caller
(bf16 and fp32 widen exactly); the append works on raw bytes so it can be
compared bit for bit with any element type.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_OUT = os.path.join(_HERE, "_build")
_LIB = None
_LOCK = threading.Lock()


def lib_path() -> str:
    # PKV_ORACLE_LIB lets the mutation test load a deliberately broken copy.
    return os.environ.get("PKV_ORACLE_LIB") or os.path.join(_OUT, "liboracle.so")


def build(force: bool = False) -> str:
    """Compile the oracle with the host C compiler (seconds)."""
    path = lib_path()
    if os.environ.get("PKV_ORACLE_LIB"):
        return path
    if force or not os.path.exists(path) or os.path.getmtime(path) < os.path.getmtime(_SRC):
        os.makedirs(_OUT, exist_ok=True)
        tmp = path + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, path)
    return path


def _lib():
    global _LIB
    with _LOCK:
        if _LIB is None:
            lib = ctypes.CDLL(build())
            i32, i64, p = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p
            lib.oracle_bucket_for.argtypes = [i64]
            lib.oracle_bucket_for.restype = i64
            lib.oracle_append.argtypes = [p, p, i32, i64, i32, i32, p, i32, i32, i32, i32, i32,
                                          p, p, i32, p, i32]
            lib.oracle_append.restype = i32
            lib.oracle_attend.argtypes = [p, i32, i32, p, p, i64, i32, i32, p, i32, i32, i32, p, i32,
                                          ctypes.c_double, i32, i32, p, p, p, p]
            lib.oracle_attend.restype = i32
            lib.oracle_seq_clone.argtypes = [p, p, i32, i64, i32, i32, p, i32, i32, i32, i32, i32, i64]
            lib.oracle_seq_clone.restype = i32
            lib.oracle_rewind.argtypes = [p, i32, p, i32, i32]
            lib.oracle_rewind.restype = i32
            _LIB = lib
    return _LIB


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def bucket_for(length: int) -> int:
    return int(_lib().oracle_bucket_for(int(length)))


def append(k_pool: np.ndarray, v_pool: np.ndarray, block_table: np.ndarray, seq_info: np.ndarray,
           k_new: np.ndarray, v_new: np.ndarray, ring_rows: int = 0, window: int = 0,
           causal: bool = False) -> int:
    """Scatter each covered row of k_new / v_new into its slot, in place.

    k_pool, v_pool: (num_blocks, 16, Hkv, D), any element type, C-contiguous.
    Returns the failed-segment bitmask (bit 1 bad segment, 2 capacity,
    3 ring, 4 block id).
    """
    assert k_pool.flags.c_contiguous and v_pool.flags.c_contiguous
    assert k_pool.dtype == k_new.dtype == v_new.dtype == v_pool.dtype
    nb, blk, hkv, d = k_pool.shape
    assert blk == 16
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    si = np.ascontiguousarray(seq_info, dtype=np.int32).reshape(-1, 4)
    kn = np.ascontiguousarray(k_new)
    vn = np.ascontiguousarray(v_new)
    return int(_lib().oracle_append(_ptr(k_pool), _ptr(v_pool), k_pool.itemsize, nb, hkv, d,
                                    _ptr(bt), bt.shape[0], bt.shape[1], int(ring_rows), int(window),
                                    int(bool(causal)), _ptr(kn), _ptr(vn), kn.shape[0], _ptr(si),
                                    si.shape[0]))


def attend(q: np.ndarray, k_pool: np.ndarray, v_pool: np.ndarray, block_table: np.ndarray,
           seq_info: np.ndarray, scale: float, causal: bool = False, window: int = 0,
           ring_rows: int = 0, first_valid=None):
    """fp64 paged attention.  Returns (out, lse, failed-segment bitmask).

    first_valid (optional, int32 [max_seqs]): each sequence's first valid
    position (left padding): earlier keys are hidden, and a row sitting before
    it sees only its own key.

    q: (rows, Hq, D); k_pool / v_pool: (num_blocks, 16, Hkv, D); all widened
    to float64 here.  out: (rows, Hq, D); lse: (rows, Hq), natural log.
    """
    q = np.ascontiguousarray(q, dtype=np.float64)
    kp = np.ascontiguousarray(k_pool, dtype=np.float64)
    vp = np.ascontiguousarray(v_pool, dtype=np.float64)
    rows, hq, d = q.shape
    nb, blk, hkv, d2 = kp.shape
    assert blk == 16 and d2 == d and hq % hkv == 0
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    si = np.ascontiguousarray(seq_info, dtype=np.int32).reshape(-1, 4)
    out = np.zeros((rows, hq, d), dtype=np.float64)
    lse = np.zeros((rows, hq), dtype=np.float64)
    max_keys = int(max([int(s[3]) for s in si] + [1]))
    work = np.zeros(max_keys + 1, dtype=np.float64)
    fv = None if first_valid is None else np.ascontiguousarray(first_valid, dtype=np.int32).reshape(-1)
    assert fv is None or fv.shape[0] == bt.shape[0]
    errs = _lib().oracle_attend(_ptr(q), hq, rows, _ptr(kp), _ptr(vp), nb, hkv, d, _ptr(bt),
                                bt.shape[0], bt.shape[1], int(ring_rows), _ptr(si), si.shape[0],
                                float(scale), int(bool(causal)), int(window),
                                None if fv is None else _ptr(fv), _ptr(out), _ptr(lse), _ptr(work))
    return out, lse, int(errs)


def seq_clone(k_pool: np.ndarray, v_pool: np.ndarray, block_table: np.ndarray, src_col: int, dst_col: int,
              n: int, ring_rows: int = 0) -> int:
    """Copy positions 0..n-1 of sequence src_col to dst_col in place (one layer; ring: the last
    min(n, ring_rows) positions).  Returns 0 or the failure bit (all or nothing)."""
    assert k_pool.flags.c_contiguous and v_pool.flags.c_contiguous
    nb, blk, hkv, d = k_pool.shape
    assert blk == 16
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    return int(_lib().oracle_seq_clone(_ptr(k_pool), _ptr(v_pool), k_pool.itemsize, nb, hkv, d, _ptr(bt),
                                       bt.shape[0], bt.shape[1], int(ring_rows), int(src_col), int(dst_col),
                                       int(n)))


def rewind(seq_info: np.ndarray, amount: np.ndarray, ring_rows: int = 0, window: int = 0):
    """kv_end -= amount per segment where allowed.  Returns (new seq_info, failed-segment bitmask)."""
    si = np.ascontiguousarray(seq_info, dtype=np.int32).reshape(-1, 4).copy()
    am = np.ascontiguousarray(amount, dtype=np.int32).reshape(-1)
    assert am.shape[0] == si.shape[0]
    errs = _lib().oracle_rewind(_ptr(si), si.shape[0], _ptr(am), int(ring_rows), int(window))
    return si, int(errs)

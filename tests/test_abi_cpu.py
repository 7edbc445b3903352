"""C-ABI checks that need no GPU: the library loads, exports every entry
point include/pkv.h declares, and rejects bad arguments on the host before
launching anything."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pkv.h")
GOLDEN = os.path.join(ROOT, "tests", "golden", "bucket_for.txt")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from paged_kv_decode_13_gb300 import _lib
    return _lib


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_four_named_calls():
    names = declared_symbols()
    for n in ("pkv_append", "pkv_attend_varlen", "pkv_resize_bucket", "pkv_load_prefix"):
        assert n in names
    assert len(names) >= 10


def test_every_declared_symbol_is_exported(lib):
    raw = ctypes.CDLL(lib.LIB_PATH)
    missing = [n for n in declared_symbols() if not hasattr(raw, n)]
    assert not missing, missing


def test_struct_layout_matches_header(lib):
    # int32 x4, int64, int32 x4, three pointers, int64 x2, one pointer on LP64.
    assert ctypes.sizeof(lib.CacheDesc) == 4 * 4 + 8 + 4 * 4 + 3 * 8 + 2 * 8 + 8
    assert lib.CacheDesc.k.offset == 40 and lib.CacheDesc.bucket.offset == 64
    assert lib.CacheDesc.first_valid.offset == 80


def test_bucket_for_matches_golden(lib):
    from oracle import oracle as O
    for line in open(GOLDEN):
        line = line.split("#")[0].strip()
        if not line:
            continue
        length, bucket = (int(x) for x in line.split())
        assert lib.lib.pkv_bucket_for(length) == bucket
        assert O.bucket_for(length) == bucket
    for length in range(0, 40000, 37):
        assert lib.lib.pkv_bucket_for(length) == O.bucket_for(length)


def test_status_strings(lib):
    for s in (0, 1, 2, -1, -2, -3, -4, -5):
        assert lib.lib.pkv_status_str(s)
    assert b"unknown" in lib.lib.pkv_status_str(99)


def _desc(lib, **kw):
    fake = (ctypes.c_void_p * 2)(0x1000, 0x2000)
    d = lib.CacheDesc(num_layers=1, kv_heads=2, head_dim=64, dtype=lib.BF16, num_blocks=32, max_seqs=1,
                      max_blocks_per_seq=32, ring_rows=0, reserved0=0, k=ctypes.cast(fake, ctypes.c_void_p),
                      v=ctypes.cast(ctypes.byref(fake, 8), ctypes.c_void_p), block_table=0x3000, bucket=512,
                      generation=0)
    for k, v in kw.items():
        setattr(d, k, v)
    return d, fake


@pytest.mark.parametrize("field,value,status", [
    ("head_dim", 72 + 4, -2),      # not a multiple of 8
    ("head_dim", 264, -2),         # above 256
    ("dtype", 7, -2),
    ("kv_heads", 0, -1),
    ("ring_rows", 24, -1),         # not a multiple of 16
    ("ring_rows", 1024, -1),       # beyond the table's capacity
    ("num_blocks", 0, -1),
])
def test_bad_cache_rejected_before_launch(lib, field, value, status):
    d, keep = _desc(lib, **{field: value})
    L = lib.lib
    st = L.pkv_attend_varlen(ctypes.byref(d), 0, 0x4000, 8, 1, 0x5000, 1, 1, 512, 0, 0.125, 0, 0,
                             0x6000, None, None, 0, 0x7000, 0, None)
    assert st == status
    st = L.pkv_append(ctypes.byref(d), 0, 0x4000, 0x4000, 1, 0x5000, 1, 0, 0x7000, None)
    assert st == status


def test_bad_call_arguments_rejected(lib):
    d, keep = _desc(lib)
    L = lib.lib
    ref = ctypes.byref(d)

    def attend(**kw):
        a = dict(layer=0, q=0x4000, hq=8, rows=1, si=0x5000, S=1, mq=1, mk=512, ns=0, scale=1.0, causal=0,
                 window=0, out=0x6000, lse=None, ws=None, wsb=0, err=0x7000, flags=0)
        a.update(kw)
        return L.pkv_attend_varlen(ref, a["layer"], a["q"], a["hq"], a["rows"], a["si"], a["S"], a["mq"], a["mk"],
                                   a["ns"], a["scale"], a["causal"], a["window"], a["out"], a["lse"], a["ws"],
                                   a["wsb"], a["err"], a["flags"], None)

    assert attend(hq=3) == -1              # q heads not a multiple of kv heads
    assert attend(layer=1) == -1           # layer out of range
    assert attend(q=0x4004) == -1          # misaligned q
    assert attend(si=0x5004) == -1         # misaligned segment table
    assert attend(err=None) == -1          # missing error word
    assert attend(causal=2) == -1
    assert attend(window=-1) == -1
    assert attend(ns=17) == -1             # more splits than a cluster can hold
    assert attend(ns=65, ws=0x8000, wsb=1 << 30) == -1   # more than the workspace mode allows
    assert attend(ns=17, ws=0x8000, wsb=16) == -1        # workspace smaller than the split merge needs
    assert attend(ws=0x8004, wsb=1 << 30) == -1          # misaligned workspace
    assert attend(ns=-1) == -1
    assert attend(mq=0) == -1
    assert attend(mk=0) == -1
    assert attend(S=-1) == -1
    # fused call without k_new / v_new
    assert L.pkv_append_attend(ref, 0, 0x4000, None, None, 8, 1, 0x5000, 1, 1, 512, 0, 1.0, 0, 0, 0x6000,
                               None, None, 0, 0x7000, 0, None) == -1
    # nothing to do: no rows and no segments
    assert attend(rows=0, S=0) == 0


def test_batch_ops_host_rules(lib):
    L = lib.lib
    d, keep = _desc(lib)       # one sequence row, 32 pages of 16
    ref = ctypes.byref(d)
    assert L.pkv_seq_clone(ref, 0, 1, 4, 0x7000, None) == -1      # no row 1
    assert L.pkv_seq_clone(ref, -1, 0, 4, 0x7000, None) == -1
    assert L.pkv_seq_clone(ref, 0, 0, -1, 0x7000, None) == -1
    assert L.pkv_seq_clone(ref, 0, 0, 4, None, None) == -1        # no error word
    assert L.pkv_seq_clone(ref, 0, 0, 513, 0x7000, None) == -4    # beyond 32 pages
    assert L.pkv_seq_clone(ref, 0, 0, 100, 0x7000, None) == 0     # same row: nothing to copy, no launch
    assert L.pkv_rewind(ref, 0x5000, -1, 0x6000, 0, 0x7000, None) == -1
    assert L.pkv_rewind(ref, 0x5004, 1, 0x6000, 0, 0x7000, None) == -1   # misaligned segment table
    assert L.pkv_rewind(ref, 0x5000, 1, 0x6002, 0, 0x7000, None) == -1   # misaligned amounts
    assert L.pkv_rewind(ref, 0x5000, 0, None, 0, 0x7000, None) == 0      # nothing to do


def test_workspace_size_query(lib):
    L = lib.lib
    d, keep = _desc(lib)   # bf16, 2 kv heads, head_dim 64, 512 tokens
    ref = ctypes.byref(d)
    # decode kernel (8 q heads over 2 kv heads, one row each): splits merge through the workspace
    n = L.pkv_attend_workspace_bytes(ref, 8, 1, 1, 512, 0, 0)
    assert n > 0 and n % 256 == 0
    # more segments need more
    assert L.pkv_attend_workspace_bytes(ref, 8, 4, 1, 512, 0, 0) > n
    # one split: nothing to merge
    assert L.pkv_attend_workspace_bytes(ref, 8, 1, 1, 512, 1, 0) == 0
    # 16 query rows per kv head: the wide kernel, which merges in the cluster
    assert L.pkv_attend_workspace_bytes(ref, 8, 1, 4, 512, 0, 0) == 0
    # the CUDA-core variant of the decode kernel merges the same way
    assert L.pkv_attend_workspace_bytes(ref, 8, 1, 1, 512, 0, 1) == n
    # the fp32 tile never uses one
    f, keep32 = _desc(lib, dtype=lib.F32)
    assert L.pkv_attend_workspace_bytes(ctypes.byref(f), 8, 1, 1, 512, 0, 0) == 0
    assert L.pkv_attend_workspace_bytes(ref, 3, 1, 1, 512, 0, 0) == -1


def test_resize_and_prefix_host_rules(lib):
    L = lib.lib
    a, ka = _desc(lib)
    b, kb = _desc(lib, num_layers=1, head_dim=128)
    assert L.pkv_resize_bucket(ctypes.byref(a), ctypes.byref(b), 10, None) == -5   # shapes differ
    c, kc = _desc(lib)
    assert L.pkv_resize_bucket(ctypes.byref(a), ctypes.byref(c), 10, None) == 2    # same bucket
    c.bucket = 1024
    assert L.pkv_resize_bucket(ctypes.byref(a), ctypes.byref(c), 10_000, None) == -4
    assert c.generation == 0
    assert L.pkv_load_prefix(ctypes.byref(a), None, None, 5, 128, 64, None) == 1   # empty
    assert L.pkv_load_prefix(ctypes.byref(a), ctypes.cast(ka, ctypes.c_void_p), ctypes.cast(ka, ctypes.c_void_p),
                             0, 128, 64, None) == 1
    assert L.pkv_load_prefix(ctypes.byref(a), ctypes.cast(ka, ctypes.c_void_p), ctypes.cast(ka, ctypes.c_void_p),
                             10_000, 128, 64, None) == -4


def test_binding_fails_loudly_without_library(tmp_path):
    import subprocess
    import sys
    # A copy of the binding package with no libpkv.so must refuse to import.
    pkg = tmp_path / "paged_kv_decode_13_gb300"
    pkg.mkdir()
    src = os.path.join(ROOT, "paged_kv_decode_13_gb300")
    for f in ("__init__.py", "_lib.py", "api.py", "graph.py"):
        (pkg / f).write_text(open(os.path.join(src, f)).read())
    r = subprocess.run([sys.executable, "-c", "import paged_kv_decode_13_gb300"], cwd=tmp_path,
                       capture_output=True, text=True)
    assert r.returncode != 0 and "libpkv.so not found" in r.stderr


def test_struct_layout_matches_compiled_header(lib, tmp_path):
    # the C compiler's own offsets for include/pkv.h against the ctypes mirror
    src = tmp_path / "layout.c"
    src.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "pkv.h"\n'
                   'int main(void) { printf("%zu", sizeof(pkv_cache));\n'
                   + "".join(f'  printf(" %zu", offsetof(pkv_cache, {n}));\n' for n, _ in lib.CacheDesc._fields_)
                   + "  return 0; }\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    assert got[0] == ctypes.sizeof(lib.CacheDesc)
    assert got[1:] == [getattr(lib.CacheDesc, n).offset for n, _ in lib.CacheDesc._fields_]

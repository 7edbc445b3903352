"""CPU oracle for paged decode attention -- test infrastructure only.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg import this package.  The product path (the CUDA library and its Python
binding) never does.
"""
from .oracle import append, attend, bucket_for, build, lib_path  # noqa: F401

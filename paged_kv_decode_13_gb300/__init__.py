"""pkv: decode attention over a paged KV cache on GB300 (sm_103a).

The compute lives in libpkv.so (CUDA, C ABI, include/pkv.h); this package is
its thin Python binding plus a CUDA-graph decode-step harness.  Importing it
without the built library raises ImportError.
"""
from ._lib import (BF16, BLOCK_SIZE, ERR_BLOCK, ERR_CAPACITY, ERR_OVERLAP, ERR_QLEN, ERR_RING,  # noqa: F401
                   ERR_SEGMENT, ERR_TIMEOUT, F32, FLAG_MMA_SYNC, FLAG_PDL, FLAG_PREFETCH_NEXT, FLAG_SIMT, LIB_PATH,
                   PkvError)
from .api import (PagedKVCache, advance, append, append_attend, append_attend_noalloc,  # noqa: F401
                  attend_varlen, attend_workspace_bytes,
                  bucket_for, load_prefix, new_err_flags, new_workspace, resize_bucket, rewind, seq_clone,
                  seqinfo_from_seqused, to_contiguous)

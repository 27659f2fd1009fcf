"""GB300 (sm_103a) FP8 lightning indexer -> top-k -> sparse MLA prefill.

The compute runs in libsmla.so (hand-written CUDA + inline PTX); this package
holds its ctypes binding (``_lib``), the in-tree build (``build``) and the
seeded synthetic input generators (``workloads``).  Importing the package
does not load the library; the binding's first call does, and raises if the
library is missing.
"""
from ._lib import (  # noqa: F401
    Seqs,
    SmlaError,
    indexer_scores,
    topk_workspace_size,
    topk,
    indexer_topk_workspace_size,
    indexer_topk,
    sparse_prefill,
    sparse_prefill_bf16_cache,
    dense_prefill,
    sparse_decode_workspace_size,
    sparse_decode,
    sparse_decode_noalloc,
    check_device_errors,
    selftest_wait_timeout,
    version,
    load,
)

"""CPU oracle for the FP8 indexer -> top-k -> sparse MLA prefill path.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or
executes this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may use it.

It is a plain, slow, float64 restatement of what the path computes, written
from the pages' definitions (see ``reference.py`` for the passage each
function follows).  It shares no code with the CUDA library or its Python
binding; the only code both sides use is the seeded input generator module,
which holds none of the method's arithmetic.

Pins (tests/test_oracle_*.py) tie every function to something other than
itself: the e4m3 format's closed forms, torch's float8/bfloat16 dtypes,
hand-constructed closed-form cases, invariants, brute force and
torch.nn.functional.scaled_dot_product_attention in float64.
"""
from .reference import (  # noqa: F401
    E4M3_TABLE,
    decode_e4m3,
    decode_bf16,
    token_positions,
    phys_rows_of,
    indexer_scores,
    topk_select,
    topk,
    dequant_rows,
    softmax_weights,
    sparse_prefill,
    dense_prefill,
)

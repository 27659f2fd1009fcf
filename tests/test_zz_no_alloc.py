"""The allocation-free decode entry point (smla_sparse_decode_noalloc).

Some callers cannot allocate device memory where they decode: an
inference-engine plugin whose enqueue step forbids it, or a serving loop
whose device memory all belongs to a pool it may not go around.  For them
the library keeps the decode's split partials in a fixed device array
instead of a caller workspace.  This test calls that entry point through the
C ABI twice in a row, with different shapes, so that the second call runs
over the first call's leftovers in the shared array, and checks each result
against the workspace entry point's output on the same inputs (the same
arithmetic; the two may differ only by the order of the row-sum atomics) and
against the oracle.  It lives in a file of its own that pytest collects last.
"""
import numpy as np
import pytest
import torch

import serving_fp8_indexer_gb300 as smla
from serving_fp8_indexer_gb300 import workloads as wl

from _gpu_helpers import check_prefill, q_attn_tensor, rows_of

pytestmark = pytest.mark.gpu

# same-arithmetic bound used by the other GPU tests (row-sum atomics order)
RUN_TO_RUN = 1e-2


def _inputs(w):
    scales = None if w.scales is None else torch.from_numpy(w.scales).cuda()
    return (q_attn_tensor(w), torch.from_numpy(w.latent).cuda(), scales, w.scale_block_size,
            torch.from_numpy(w.indices).cuda(), torch.from_numpy(w.topk_lengths).cuda(), w.softmax_scale)


def _with_workspace(w, args):
    ws_bytes = smla.sparse_decode_workspace_size(w.seqs.T, w.H, w.indices.shape[1])
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda") if ws_bytes else None
    out = torch.empty((w.seqs.T, w.H, 512), dtype=torch.bfloat16, device="cuda")
    smla.sparse_decode(*args, out, ws)
    smla.check_device_errors()
    return out, ws_bytes


def _no_alloc(w, args):
    out = torch.full((w.seqs.T, w.H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    smla.sparse_decode_noalloc(*args, out)
    smla.check_device_errors()
    return out


def test_no_alloc_decode_matches_workspace_decode_twice():
    # two shapes whose split layouts differ: the second call reads back only
    # what it wrote, never the first call's partials
    cases = [wl.sparse_decode(seed=200, H=128, q_dtype=wl.Q_BF16, sbs=0, L=4096),
             wl.sparse_decode(seed=201, B=4, H=64, q_dtype=wl.Q_E4M3, sbs=576, L=3000)]
    for w in cases:
        args = _inputs(w)
        ref, ws_bytes = _with_workspace(w, args)
        assert ws_bytes > 0, "the case must use split scratch"
        got = _no_alloc(w, args)
        assert float((got.float() - ref.float()).abs().max()) <= RUN_TO_RUN
        toks = np.arange(w.seqs.T)
        check_prefill(w, rows_of(got, toks), w.indices, w.topk_lengths, toks)
    # and the first shape again, right after the second
    w = cases[0]
    args = _inputs(w)
    ref, _ = _with_workspace(w, args)
    got = _no_alloc(w, args)
    assert float((got.float() - ref.float()).abs().max()) <= RUN_TO_RUN

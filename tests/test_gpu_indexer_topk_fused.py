"""GPU parity of the fused indexer + top-k (score rows kept on chip): the
same indices and lengths as the standalone indexer followed by top-k, and
the oracle's sets up to the tie band, through the C ABI."""
import numpy as np
import pytest
import torch

import serving_fp8_indexer_gb300 as smla
from serving_fp8_indexer_gb300 import workloads as wl

from _gpu_helpers import check_topk_against, run_indexer, run_topk, score_stride_for, stratified_tokens

pytestmark = pytest.mark.gpu


def _fused(w, stride=None):
    seqs = smla.Seqs.from_host(w.seqs)
    stride = stride or score_stride_for(w.seqs)
    T = w.seqs.T
    ws_bytes = smla.indexer_topk_workspace_size(T, stride, w.h_idx, w.topk)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda") if ws_bytes else None
    idx = torch.full((T, w.topk), 0x7777, dtype=torch.uint32, device="cuda")
    lens = torch.full((T,), 0x7777, dtype=torch.uint32, device="cuda")
    smla.indexer_topk(torch.from_numpy(w.q_idx).cuda(), torch.from_numpy(w.q_scale).cuda(),
                      torch.from_numpy(w.k_pool).cuda(), torch.from_numpy(w.k_scale).cuda(), seqs, stride, w.topk,
                      idx, lens, ws)
    smla.check_device_errors()
    return idx.cpu().numpy(), lens.cpu().numpy(), ws_bytes


def _unfused(w, stride=None):
    seqs, scores = run_indexer(w, stride)
    idx, lens = run_topk(seqs, scores, w.topk, w.seqs.T)
    return idx.cpu().numpy(), lens.cpu().numpy(), scores


def _same_as_unfused(w, stride=None):
    fi, fl, ws_bytes = _fused(w, stride)
    ui, ul, scores = _unfused(w, stride)
    assert np.array_equal(fl, ul), "topk_lengths differ from the unfused path"
    assert np.array_equal(fi, ui), "indices differ from the unfused path"
    return fi, fl, ws_bytes, scores


@pytest.mark.parametrize("h_idx", [4, 8, 16, 32, 64])
def test_fused_equals_unfused_ragged_paged(h_idx):
    # ragged sequences, a cached prefix, one-token sequences, partial tiles
    w = wl.build("fused_ragged", 300 + h_idx, [37, 1, 130, 5, 64], [300, 1, 480, 5, 512], 16, h_idx=h_idx, topk=50)
    _, _, ws_bytes, _ = _same_as_unfused(w)
    assert ws_bytes == 0


def test_fused_tiny_and_mtp_decode_against_oracle():
    for w in (wl.tiny_prefill(), wl.mtp_decode_indexer()):
        fi, fl, ws_bytes, scores = _same_as_unfused(w)
        assert ws_bytes == 0
        toks = np.arange(w.seqs.T)
        # the kernel's own scores decide exactly; the oracle's up to the tie band
        check_topk_against(w, scores.cpu().numpy().astype(np.float64), fi, fl, toks, w.topk, exact=True)


def test_fused_ties_and_equal_scores():
    """Integer-valued q and k give many exactly equal scores: ties at the
    k-th value must go to the lower keys, as in the unfused path."""
    w = wl.build("fused_ties", 320, [64, 9], [900, 300], 64, h_idx=64, topk=128)
    rng = np.random.default_rng(321)
    w.q_idx = wl.to_e4m3_bytes(rng.integers(-1, 2, size=w.q_idx.shape).astype(np.float32))
    w.k_pool = wl.to_e4m3_bytes(rng.integers(-1, 2, size=w.k_pool.shape).astype(np.float32))
    w.q_scale[:] = 1.0
    w.k_scale[:] = 1.0
    _same_as_unfused(w)


def test_fused_rows_longer_than_on_chip_use_the_workspace():
    """score_stride above 128 * H_idx: the call runs the unfused pair with
    the score buffer in the caller's workspace."""
    w = wl.build("fused_long", 330, [20], [9000], 64, h_idx=64, topk=2048)
    fi, fl, ws_bytes, _ = _same_as_unfused(w)
    assert ws_bytes >= w.seqs.T * 9000 * 4


@pytest.mark.slow
def test_fused_chunk_full_size():
    """The end-to-end chunk (8 x 8192 keys, 16384 tokens, H_idx 64, top-2048)
    in the benchmark's launch configuration: identical to the unfused pair on
    every token."""
    w = wl.e2e_chunk()
    fi, fl, ws_bytes, scores = _same_as_unfused(w)
    assert ws_bytes == 0
    pos = wl.token_positions(w.seqs)
    assert np.array_equal(fl, np.minimum(pos + 1, w.topk).astype(np.uint32))
    toks = stratified_tokens(w.seqs, 64)
    rows = scores[torch.from_numpy(toks).cuda()].cpu().numpy().astype(np.float64)
    check_topk_against(w, rows, fi[toks], fl[toks], toks, w.topk, exact=True)

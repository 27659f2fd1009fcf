"""GPU parity of stage 3 (sparse MLA prefill) and of the whole path against
the float64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

from serving_fp8_indexer_gb300 import workloads as wl

from _gpu_helpers import (check_prefill, q_attn_tensor, rows_of, run_indexer, run_prefill, run_topk)

pytestmark = pytest.mark.gpu


def _sampled(w, tokens=None):
    """Stage 3 alone on the workload's sampled indices."""
    idx = torch.from_numpy(w.indices).cuda()
    lens = torch.from_numpy(w.topk_lengths).cuda()
    out = run_prefill(w, idx, lens)
    toks = np.arange(w.seqs.T) if tokens is None else tokens
    return check_prefill(w, rows_of(out, toks), w.indices[toks], w.topk_lengths[toks], toks)


def _end_to_end(w, tokens=None):
    """indexer -> top-k -> attention on the GPU; attention checked on the
    GPU's own indices."""
    seqs, scores = run_indexer(w)
    idx, lens = run_topk(seqs, scores, w.topk, w.seqs.T)
    out = run_prefill(w, idx, lens)
    toks = np.arange(w.seqs.T) if tokens is None else tokens
    return check_prefill(w, rows_of(out, toks), rows_of(idx, toks), rows_of(lens, toks), toks)


def test_tiny_prefill_end_to_end():
    _end_to_end(wl.tiny_prefill())


def test_bf16_unit_several_blocks_ragged():
    # positions 0..299, k=256: lengths 1..256 (partial last blocks, 1-key rows)
    _sampled(wl.dsv32_prefill(T=300, k=256))


def test_fp8_blockwise_ragged_batch():
    _sampled(wl.blockwise_fp8_prefill(lens=(100, 200, 333), k=256))


def test_fp8_unit_and_tensorwise():
    w = wl.build("fp8_unit", 9, [150], [150], 64, topk=160, H=64, q_dtype=wl.Q_E4M3, sbs=0, sample_indices=True)
    _sampled(w)
    w = wl.build("fp8_row", 10, [150], [150], 64, topk=160, H=64, q_dtype=wl.Q_E4M3, sbs=576, sample_indices=True)
    _sampled(w)


def test_bf16_tensorwise_chunk_end_to_end():
    _end_to_end(wl.e2e_chunk(B=2, L=600, q_len=200, k=256, H=128, h_idx=64))


@pytest.mark.parametrize("H", [16, 32, 48, 192, 256])
def test_head_counts(H):
    w = wl.build(f"h{H}", 40 + H, [70], [200], 64, topk=130, H=H, q_dtype=wl.Q_BF16, sbs=0, sample_indices=True)
    _sampled(w)


@pytest.mark.parametrize("H", [16, 48])
def test_fp8_q_partial_head_group(H):
    # e4m3 q with fewer than 64 heads: the q tile's rows past the group belong
    # to the next token (or lie past the tensor) and must not leak in
    w = wl.build(f"fp8_h{H}", 60 + H, [90, 33], [150, 40], 64, topk=140, H=H, q_dtype=wl.Q_E4M3, sbs=576,
                 sample_indices=True)
    _sampled(w)


def test_two_head_groups_e4m3_and_tensorwise():
    # H = 128: two 64-head work items per token, e4m3 q, unit and row scales
    for sbs, seed in ((0, 50), (576, 51)):
        w = wl.build(f"pair_fp8_{sbs}", seed, [90, 40], [300, 40], 64, topk=200, H=128, q_dtype=wl.Q_E4M3,
                     sbs=sbs, sample_indices=True)
        _sampled(w)


@pytest.mark.parametrize("H", [64, 128])
def test_single_key_rows_are_exact(H):
    """topk_lengths == 1: the softmax weight is exactly 1 and the output is
    the selected row's first 512 values (exact in bf16)."""
    w = wl.build("one", 3, [40], [40], 64, topk=4, H=H, q_dtype=wl.Q_BF16, sbs=0, sample_indices=True)
    lens = np.ones(40, np.uint32)
    out = run_prefill(w, torch.from_numpy(w.indices).cuda(), torch.from_numpy(lens).cuda())
    import oracle
    for t in range(40):
        v = oracle.decode_e4m3(w.latent[w.indices[t, 0]])[:512]
        assert np.array_equal(out[t].float().cpu().numpy(), np.broadcast_to(v, (H, 512)).astype(np.float32))


def test_zero_length_rows_and_wide_stride():
    """topk_lengths == 0 gives zeros; indices_stride wider than the lengths."""
    w = wl.build("zero", 4, [50], [300], 64, topk=200, H=128, q_dtype=wl.Q_BF16, sbs=0, sample_indices=True)
    idx = np.full((50, 256), 0xFFFFFFFF, np.uint32)
    idx[:, :200] = w.indices
    lens = w.topk_lengths.copy()
    lens[::7] = 0
    out = run_prefill(w, torch.from_numpy(idx).cuda(), torch.from_numpy(lens).cuda())
    o = out.float().cpu().numpy()
    assert (o[::7] == 0).all()
    toks = np.array([t for t in range(50) if t % 7])
    check_prefill(w, o[toks], idx[toks], lens[toks], toks)


def test_prefill_repeats_are_stable():
    # Several items per CTA with one- and two-block selections: a pipeline
    # race shows up as a run that differs from the first.  The row-sum
    # atomics may add in another order (a few bf16 ulps).
    w = wl.dsv32_prefill(T=300, k=256)
    idx = torch.from_numpy(w.indices).cuda()
    lens = torch.from_numpy(w.topk_lengths).cuda()
    q = q_attn_tensor(w)
    first = run_prefill(w, idx, lens, q=q).float()
    assert torch.isfinite(first).all()
    for _ in range(100):
        out = run_prefill(w, idx, lens, q=q).float()
        assert torch.isfinite(out).all()
        assert float((out - first).abs().max()) <= 1e-2

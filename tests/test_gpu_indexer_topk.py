"""GPU parity of stage 1 (indexer scores) and stage 2 (top-k) against the
float64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import serving_fp8_indexer_gb300 as smla
from serving_fp8_indexer_gb300 import workloads as wl

from _gpu_helpers import check_scores, check_topk_against, run_indexer, run_topk

pytestmark = pytest.mark.gpu


def _full(w):
    seqs, scores = run_indexer(w)
    stride = scores.shape[1]
    toks = np.arange(w.seqs.T)
    ref, _ = check_scores(w, scores.cpu().numpy(), toks, stride)
    idx, lens = run_topk(seqs, scores, w.topk, w.seqs.T)
    gi, gl = idx.cpu().numpy(), lens.cpu().numpy()
    # same scores in -> same set out (the kernel's own scores, decoded exactly)
    check_topk_against(w, scores.cpu().numpy().astype(np.float64), gi, gl, toks, w.topk, exact=True)
    # against the oracle's scores, up to the tie band
    check_topk_against(w, ref, gi, gl, toks, w.topk, exact=False)


def test_tiny_prefill_indexer_topk():
    _full(wl.tiny_prefill())


def test_mtp_decode_indexer_topk():
    _full(wl.mtp_decode_indexer())


@pytest.mark.parametrize("h_idx", [4, 8, 16, 32, 64])
def test_ragged_paged_indexer(h_idx):
    # ragged sequences, a tail tile, several key tiles, page_size 16
    w = wl.build("ragged", 20 + h_idx, [37, 1, 130, 5], [300, 1, 520, 5], 16, h_idx=h_idx, topk=50)
    _full(w)


@pytest.mark.parametrize("page_size", [8, 64, 256])
def test_page_sizes(page_size):
    w = wl.build("pages", 31, [70, 9], [700, 9], page_size, h_idx=64, topk=130)
    _full(w)


def test_wide_stride_and_small_k():
    w = wl.build("stride", 5, [17], [333], 64, h_idx=16, topk=1)
    seqs, scores = run_indexer(w, stride=512)
    toks = np.arange(w.seqs.T)
    check_scores(w, scores.cpu().numpy(), toks, 512)   # -inf up to the full stride
    idx, lens = run_topk(seqs, scores, 1, w.seqs.T)
    check_topk_against(w, scores.cpu().numpy().astype(np.float64), idx.cpu().numpy(), lens.cpu().numpy(), toks, 1,
                       exact=True)


def test_topk_ties_go_to_lower_keys():
    """Hand-made score rows with many equal values: the GPU must take the
    lowest-keyed ties (the oracle's rule) and report identical sets."""
    w = wl.build("ties", 2, [3], [1000], 64, h_idx=4, topk=100)
    seqs = __import__("serving_fp8_indexer_gb300").Seqs.from_host(w.seqs)
    rng = np.random.default_rng(0)
    sc = np.full((3, 1000), -np.inf, np.float32)
    pos = wl.token_positions(w.seqs)
    for t in range(3):
        sc[t, :pos[t] + 1] = rng.integers(0, 7, pos[t] + 1).astype(np.float32)  # heavy ties
    scores = torch.from_numpy(sc).cuda()
    idx, lens = run_topk(seqs, scores, 100, 3)
    check_topk_against(w, sc.astype(np.float64), idx.cpu().numpy(), lens.cpu().numpy(), np.arange(3), 100, exact=True)


def test_empty_batch_is_noop():
    import serving_fp8_indexer_gb300 as smla
    w = wl.build("empty", 0, [0], [64], 64, h_idx=64, topk=8)
    seqs = smla.Seqs.from_host(w.seqs)
    scores = torch.empty((0, 64), device="cuda")
    smla.indexer_scores(torch.empty((0, 64, 128), dtype=torch.uint8, device="cuda"),
                        torch.empty((0, 64), device="cuda"), torch.from_numpy(w.k_pool).cuda(),
                        torch.from_numpy(w.k_scale).cuda(), seqs, scores)
    smla.topk(scores, seqs, 8, torch.empty((0, 8), dtype=torch.uint32, device="cuda"),
              torch.empty((0,), dtype=torch.uint32, device="cuda"))
    smla.check_device_errors()


@pytest.mark.parametrize("stride", [8192, 12288, 20000])
@pytest.mark.parametrize("dist", ["normal", "ties", "equal"])
def test_topk_paths_on_synthetic_rows(stride, dist):
    """Top-k alone on controlled score rows: each stride picks one kernel path
    (register rows of 16 or 32 keys a thread, or the shared-memory row cache);
    the distributions exercise plain selection, long runs of ties at the k-th
    value (the lowest keys win) and rows whose valid scores are all equal."""
    L = stride - 37
    w = wl.build("topk_paths", 50 + stride % 97, [6], [L], 64, h_idx=4, topk=2048)
    rng = np.random.default_rng(stride)
    pos = wl.token_positions(w.seqs)
    rows = np.full((w.seqs.T, stride), -np.inf, dtype=np.float32)
    for t in range(w.seqs.T):
        n = int(pos[t]) + 1
        if dist == "normal":
            rows[t, :n] = rng.standard_normal(n).astype(np.float32)
        elif dist == "ties":
            rows[t, :n] = rng.integers(0, 4, size=n).astype(np.float32)
        else:
            rows[t, :n] = 1.5
    seqs = smla.Seqs.from_host(w.seqs, "cuda")
    scores = torch.from_numpy(rows).cuda()
    idx, lens = run_topk(seqs, scores, w.topk, w.seqs.T)
    gi, gl = idx.cpu().numpy(), lens.cpu().numpy()
    toks = np.arange(w.seqs.T)
    check_topk_against(w, rows.astype(np.float64), gi, gl, toks, w.topk, exact=True)
    # selected keys come out in ascending logical-key order
    for t in toks:
        g = gi[t, :int(gl[t])].astype(np.int64)
        lk = {int(r): j for j, r in enumerate(wl.logical_to_phys(w.seqs, 0, np.arange(int(pos[t]) + 1)))}
        order = [lk[int(r)] for r in g]
        assert order == sorted(order), f"token {t}: output not in key order"

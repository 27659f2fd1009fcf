"""Edge cases of the sparse attention kernel against the float64 oracle.

* Lazy rescale on later blocks: the kernel keeps one reference maximum per
  head and only raises it when a later 128-key block exceeds it by more
  than 2^8 (log2 units), rescaling the output accumulator and the row sums.
  With N(0,1) inputs and softmax_scale = 1/sqrt(576) no later block gets
  there, so these cases sharpen the logits (softmax_scale x 8) and order
  each token's indices by ascending head-0 logit, so that later blocks
  keep raising the maximum.  The inputs are checked on the CPU to reach
  the path.  Sharp logits also make the softmax peaky: most weights
  underflow and a few keys carry the output.
* One large q component per head (|q| = 100 or 1000 among N(0,1) values):
  the per-head power-of-two scaling of the bf16 q split into two e4m3
  terms then spans a wide range within one row.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from serving_fp8_indexer_gb300 import workloads as wl

from _gpu_helpers import check_prefill, rows_of, run_prefill

pytestmark = pytest.mark.gpu

TAU_LOG2 = 8.0
LOG2E = 1.0 / math.log(2.0)


def _q_f64(w, t):
    return oracle.decode_bf16(w.q_attn[t]) if w.q_dtype == wl.Q_BF16 else oracle.decode_e4m3(w.q_attn[t])


def _logits_log2(w, t, idx_row, n):
    """[H, n] logits of token t in log2 units (exact, float64)."""
    K = oracle.dequant_rows(w.latent, w.scales, w.scale_block_size, idx_row[:n].astype(np.int64))
    return w.softmax_scale * LOG2E * (_q_f64(w, t) @ K.T)


def _order_by_head0_logit(w):
    """Reorders every token's selected indices by ascending head-0 logit."""
    idx = w.indices.copy()
    for t in range(w.seqs.T):
        n = int(w.topk_lengths[t])
        z0 = _logits_log2(w, t, idx[t], n)[0]
        idx[t, :n] = idx[t, :n][np.argsort(z0, kind="stable")]
    w.indices = idx


def _later_block_raises(w, bk=128):
    """(rows where some block j > 0 beats the running reference by more
    than tau, rows) over every (token, head)."""
    hit = rows = 0
    for t in range(w.seqs.T):
        n = int(w.topk_lengths[t])
        z = _logits_log2(w, t, w.indices[t], n)
        for h in range(z.shape[0]):
            m = z[h, :bk].max()
            raised = False
            for j0 in range(bk, n, bk):
                b = z[h, j0:j0 + bk].max()
                if b - m > TAU_LOG2:
                    m, raised = b, True
            hit += raised
            rows += 1
    return hit, rows


RESCALE_CASES = [
    # name, q dtype, scale_block_size, heads
    ("bf16_unit", wl.Q_BF16, 0, 128),
    ("bf16_row", wl.Q_BF16, 576, 64),
    ("e4m3_unit", wl.Q_E4M3, 0, 64),
    ("e4m3_row", wl.Q_E4M3, 576, 64),
    ("e4m3_block", wl.Q_E4M3, 32, 64),
]


@pytest.mark.parametrize("name,qd,sbs,H", RESCALE_CASES, ids=[c[0] for c in RESCALE_CASES])
def test_lazy_rescale_on_later_blocks(name, qd, sbs, H):
    w = wl.build(f"rescale_{name}", 70 + sbs % 7 + qd, [40], [2048], 64, topk=1024, H=H, q_dtype=qd, sbs=sbs,
                 sample_indices=True)
    w.softmax_scale = 8.0 / math.sqrt(576.0)
    _order_by_head0_logit(w)
    hit, rows = _later_block_raises(w)
    assert hit >= rows // 8, f"only {hit} of {rows} (token, head) rows reach a later-block rescale"
    out = run_prefill(w, torch.from_numpy(w.indices).cuda(), torch.from_numpy(w.topk_lengths).cuda())
    toks = np.arange(w.seqs.T)
    check_prefill(w, rows_of(out, toks), w.indices, w.topk_lengths, toks)


@pytest.mark.parametrize("scale_mult", [3.0, 16.0])
def test_peaky_softmax_random_order(scale_mult):
    """Sharp logits in the sampled (random) order: most P underflow to zero in
    e4m3 while the row sums still count them (in f32)."""
    w = wl.build("peaky", 80 + int(scale_mult), [64, 30], [1500, 400], 64, topk=512, H=128, q_dtype=wl.Q_BF16,
                 sbs=576, sample_indices=True)
    w.softmax_scale = scale_mult / math.sqrt(576.0)
    out = run_prefill(w, torch.from_numpy(w.indices).cuda(), torch.from_numpy(w.topk_lengths).cuda())
    toks = np.arange(w.seqs.T)
    check_prefill(w, rows_of(out, toks), w.indices, w.topk_lengths, toks)


@pytest.mark.parametrize("big", [100.0, 1000.0])
def test_bf16_q_outlier_per_head(big):
    """One component of magnitude `big` per (token, head) at a random depth,
    the rest N(0,1), at the usual softmax scale (the outlier makes the
    logits sharp).  The split keeps the small components to about 2^-8
    relative while they lie within about 2^10 of the head's largest |q|;
    further below, the low term falls under e4m3's normal range."""
    w = wl.build("outlier", 90, [50], [1024], 64, topk=512, H=128, q_dtype=wl.Q_BF16, sbs=0, sample_indices=True)
    rng = np.random.default_rng(91)
    q = rng.standard_normal((w.seqs.T, w.H, 576)).astype(np.float32)
    d = rng.integers(0, 576, size=(w.seqs.T, w.H))
    sgn = rng.choice([-1.0, 1.0], size=(w.seqs.T, w.H))
    np.put_along_axis(q, d[..., None], (big * sgn)[..., None].astype(np.float32), axis=2)
    w.q_attn = wl.to_bf16_bits(q)
    out = run_prefill(w, torch.from_numpy(w.indices).cuda(), torch.from_numpy(w.topk_lengths).cuda())
    toks = np.arange(w.seqs.T)
    check_prefill(w, rows_of(out, toks), w.indices, w.topk_lengths, toks)

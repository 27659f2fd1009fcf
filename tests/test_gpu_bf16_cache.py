"""GPU parity of the sparse MLA prefill over a BF16 latent cache (bf16 x bf16
tcgen05 MMAs) against the float64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import serving_fp8_indexer_gb300 as smla
from serving_fp8_indexer_gb300 import workloads as wl

from _gpu_helpers import check_prefill, q_attn_tensor, rows_of

pytestmark = pytest.mark.gpu


def _run(w, lens=None, sink=None, stride=None):
    idx = w.indices if stride is None else np.pad(w.indices, ((0, 0), (0, stride - w.indices.shape[1])),
                                                 constant_values=0xFFFFFFFF)
    lens = w.topk_lengths if lens is None else lens
    out = torch.full((w.seqs.T, w.H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lat = torch.from_numpy(w.latent.view(np.int16)).view(torch.bfloat16).cuda()
    sk = None if sink is None else torch.from_numpy(sink).cuda()
    smla.sparse_prefill_bf16_cache(q_attn_tensor(w), lat, torch.from_numpy(idx).cuda(), torch.from_numpy(lens).cuda(),
                                   w.softmax_scale, out, attn_sink=sk)
    smla.check_device_errors()
    return out, idx, lens


@pytest.mark.parametrize("H", [16, 64, 128, 192])
def test_bf16_cache_matches_oracle(H):
    # positions 0..299 and 1000..1299: lengths 1..256, partial last blocks
    w = wl.build(f"bf16cache_h{H}", 210 + H, [300, 300], [300, 1300], 64, topk=256, H=H, q_dtype=wl.Q_BF16, sbs=0,
                 sample_indices=True, latent_bf16=True)
    out, idx, lens = _run(w)
    toks = np.arange(w.seqs.T)
    check_prefill(w, rows_of(out, toks), idx, lens, toks)


def test_bf16_cache_long_selection_wide_stride_empty_rows_and_sink():
    w = wl.build("bf16cache_long", 230, [64], [4096], 64, topk=2048, H=128, q_dtype=wl.Q_BF16, sbs=0,
                 sample_indices=True, latent_bf16=True)
    lens = w.topk_lengths.copy()
    lens[::5] = 0
    sink = np.random.default_rng(231).standard_normal(128).astype(np.float32)
    out, idx, lens = _run(w, lens=lens, sink=sink, stride=2304)
    o = rows_of(out, np.arange(64))
    assert (o[::5] == 0).all()
    toks = np.array([t for t in range(64) if t % 5])
    ref = oracle.sparse_prefill(w.q_attn, 0, w.latent, None, 0, idx, lens, w.softmax_scale, tokens=toks,
                                attn_sink=sink)
    g = o[toks].astype(np.float64)
    rel = float(np.linalg.norm(g - ref) / np.linalg.norm(ref))
    assert rel <= 1e-2 and float(np.abs(g - ref).max()) <= 3e-2, rel

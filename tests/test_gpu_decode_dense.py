"""GPU parity of the dense causal prefill, the split-K sparse decode and the
attention sink against the float64 oracle, through the C ABI."""
import math

import numpy as np
import pytest
import torch

import oracle
import serving_fp8_indexer_gb300 as smla
from serving_fp8_indexer_gb300 import workloads as wl

from _gpu_helpers import BF16_MAX_ABS, BF16_REL_L2, FP8_REL_L2, check_prefill, q_attn_tensor, rows_of, run_prefill

pytestmark = pytest.mark.gpu


def _compare(w, got, ref, what):
    g = got.astype(np.float64)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    rel = float(np.linalg.norm(g - ref) / max(np.linalg.norm(ref), 1e-300))
    mabs = float(np.abs(g - ref).max())
    print(f"[{what}] {w.name}: rel L2 {rel:.3e}, max abs {mabs:.3e}")
    if w.q_dtype == wl.Q_BF16:
        assert rel <= BF16_REL_L2 and mabs <= BF16_MAX_ABS, f"{what}: rel L2 {rel:.3g}, max abs {mabs:.3g}"
    else:
        assert rel <= FP8_REL_L2, f"{what}: rel L2 {rel:.3g} (max abs {mabs:.3g})"


def _dense(w, sink=None):
    seqs = smla.Seqs.from_host(w.seqs)
    out = torch.full((w.seqs.T, w.H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    scales = None if w.scales is None else torch.from_numpy(w.scales).cuda()
    sk = None if sink is None else torch.from_numpy(sink).cuda()
    smla.dense_prefill(q_attn_tensor(w), torch.from_numpy(w.latent).cuda(), scales, w.scale_block_size, seqs,
                       w.softmax_scale, out, attn_sink=sk)
    smla.check_device_errors()
    return out


DENSE_CASES = [
    ("bf16_unit", wl.Q_BF16, 0, 128, 64),
    ("bf16_row", wl.Q_BF16, 576, 64, 16),
    ("e4m3_unit", wl.Q_E4M3, 0, 64, 64),
    ("e4m3_row", wl.Q_E4M3, 576, 128, 256),
    ("e4m3_block", wl.Q_E4M3, 32, 64, 64),
]


@pytest.mark.parametrize("name,qd,sbs,H,ps", DENSE_CASES, ids=[c[0] for c in DENSE_CASES])
def test_dense_prefill_matches_oracle(name, qd, sbs, H, ps):
    # ragged prompts, some with a cached prefix (q_len < kv_len), one of a single token
    w = wl.build(f"dense_{name}", 100 + sbs % 11 + qd, [130, 1, 77, 300], [130, 40, 200, 300], ps, H=H, q_dtype=qd,
                 sbs=sbs)
    out = _dense(w)
    s = w.seqs
    toks = np.arange(s.T)
    ref = oracle.dense_prefill(w.q_attn, w.q_dtype, w.latent, w.scales, w.scale_block_size, s.cu_q, s.kv_len,
                               s.page_table, s.page_size, w.softmax_scale, tokens=toks)
    _compare(w, rows_of(out, toks), ref, "dense prefill")


# Two launches of the same arithmetic may differ by the order in which the
# four TMEM lane quarters add their f32 shares of a row sum (shared-memory
# atomics): a few bf16 ulps of the output at most.
RUN_TO_RUN = 1e-2


def test_dense_equals_sparse_over_every_key():
    """Dense prefill and sparse prefill given every causal key in order run
    the same arithmetic on the same rows."""
    w = wl.build("dense_vs_sparse", 120, [200, 90], [500, 90], 64, H=128, q_dtype=wl.Q_BF16, sbs=0)
    s = w.seqs
    pos, sid = wl.token_positions(s), wl.token_seq(s)
    L = int(pos.max()) + 1
    idx = np.full((s.T, L), 0xFFFFFFFF, np.uint32)
    for t in range(s.T):
        idx[t, :pos[t] + 1] = wl.logical_to_phys(s, int(sid[t]), np.arange(pos[t] + 1))
    lens = (pos + 1).astype(np.uint32)
    a = _dense(w)
    b = run_prefill(w, torch.from_numpy(idx).cuda(), torch.from_numpy(lens).cuda())
    assert float((a.float() - b.float()).abs().max()) <= RUN_TO_RUN


def _decode(w, sink=None):
    ws_bytes = smla.sparse_decode_workspace_size(w.seqs.T, w.H, w.indices.shape[1])
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda") if ws_bytes else None
    out = torch.full((w.seqs.T, w.H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    scales = None if w.scales is None else torch.from_numpy(w.scales).cuda()
    sk = None if sink is None else torch.from_numpy(sink).cuda()
    smla.sparse_decode(q_attn_tensor(w), torch.from_numpy(w.latent).cuda(), scales, w.scale_block_size,
                       torch.from_numpy(w.indices).cuda(), torch.from_numpy(w.topk_lengths).cuda(), w.softmax_scale,
                       out, ws, attn_sink=sk)
    smla.check_device_errors()
    return out, ws_bytes


DECODE_CASES = [
    ("bf16_unit_h128", wl.Q_BF16, 0, 128),
    ("bf16_row_h64", wl.Q_BF16, 576, 64),
    ("e4m3_unit_h64", wl.Q_E4M3, 0, 64),
    ("e4m3_row_h128", wl.Q_E4M3, 576, 128),
    ("e4m3_block_h64", wl.Q_E4M3, 32, 64),
]


@pytest.mark.parametrize("name,qd,sbs,H", DECODE_CASES, ids=[c[0] for c in DECODE_CASES])
def test_sparse_decode_matches_oracle(name, qd, sbs, H):
    w = wl.sparse_decode(seed=130 + sbs % 7 + qd, L=4096, H=H, q_dtype=qd, sbs=sbs)
    out, ws_bytes = _decode(w)
    assert ws_bytes > 0, "16 decode tokens should be split across CTAs"
    toks = np.arange(w.seqs.T)
    check_prefill(w, rows_of(out, toks), w.indices, w.topk_lengths, toks)


def test_decode_short_and_ragged_selections():
    """Lengths from 1 to the full stride (splits that get no blocks, a single
    block, a partial last block) and an empty selection."""
    w = wl.sparse_decode(seed=140, B=4, q_per_seq=2, L=2048, k=2048, H=64, q_dtype=wl.Q_E4M3, sbs=576)
    lens = np.array([1, 2048, 129, 0, 300, 1000, 128, 2047], np.uint32)
    w.topk_lengths = lens
    out, _ = _decode(w)
    o = rows_of(out, np.arange(8))
    assert (o[3] == 0).all()
    toks = np.array([0, 1, 2, 4, 5, 6, 7])
    check_prefill(w, o[toks], w.indices[toks], lens[toks], toks)


def test_decode_many_tokens_runs_unsplit():
    """Enough (token, head group) pairs to fill the GPU: no workspace, and the
    same result as the prefill entry point."""
    w = wl.build("decode_many", 150, [600], [1200], 64, topk=256, H=64, q_dtype=wl.Q_E4M3, sbs=0,
                 sample_indices=True)
    assert smla.sparse_decode_workspace_size(w.seqs.T, w.H, 256) == 0
    out, _ = _decode(w)
    ref = run_prefill(w, torch.from_numpy(w.indices).cuda(), torch.from_numpy(w.topk_lengths).cuda())
    assert float((out.float() - ref.float()).abs().max()) <= RUN_TO_RUN


SINK_CASES = [("bf16", wl.Q_BF16, 0, 128), ("e4m3_row", wl.Q_E4M3, 576, 64)]


@pytest.mark.parametrize("name,qd,sbs,H", SINK_CASES, ids=[c[0] for c in SINK_CASES])
def test_attention_sink_all_entry_points(name, qd, sbs, H):
    """A per-head sink logit on the sparse prefill, the dense prefill and the
    split-K decode, against the oracle; some heads' sinks dominate."""
    rng = np.random.default_rng(160 + qd)
    sink = (rng.standard_normal(H) * 2.0).astype(np.float32)
    sink[::9] = 6.0
    # sparse prefill
    w = wl.build(f"sink_{name}", 161 + qd, [70], [400], 64, topk=256, H=H, q_dtype=qd, sbs=sbs, sample_indices=True)
    out = torch.empty((w.seqs.T, H, 512), dtype=torch.bfloat16, device="cuda")
    scales = None if w.scales is None else torch.from_numpy(w.scales).cuda()
    smla.sparse_prefill(q_attn_tensor(w), torch.from_numpy(w.latent).cuda(), scales, sbs,
                        torch.from_numpy(w.indices).cuda(), torch.from_numpy(w.topk_lengths).cuda(), w.softmax_scale,
                        out, attn_sink=torch.from_numpy(sink).cuda())
    smla.check_device_errors()
    toks = np.arange(w.seqs.T)
    ref = oracle.sparse_prefill(w.q_attn, qd, w.latent, w.scales, sbs, w.indices, w.topk_lengths, w.softmax_scale,
                                tokens=toks, attn_sink=sink)
    _compare(w, rows_of(out, toks), ref, "sparse prefill + sink")
    # dense prefill
    wd = wl.build(f"sink_dense_{name}", 162 + qd, [50, 20], [300, 20], 64, H=H, q_dtype=qd, sbs=sbs)
    s = wd.seqs
    ref = oracle.dense_prefill(wd.q_attn, qd, wd.latent, wd.scales, sbs, s.cu_q, s.kv_len, s.page_table,
                               s.page_size, wd.softmax_scale, attn_sink=sink)
    _compare(wd, rows_of(_dense(wd, sink), np.arange(s.T)), ref, "dense prefill + sink")
    # split-K decode
    wdec = wl.sparse_decode(seed=163 + qd, L=3000, H=H, q_dtype=qd, sbs=sbs)
    got, ws_bytes = _decode(wdec, sink)
    assert ws_bytes > 0
    toks = np.arange(wdec.seqs.T)
    ref = oracle.sparse_prefill(wdec.q_attn, qd, wdec.latent, wdec.scales, sbs, wdec.indices, wdec.topk_lengths,
                                wdec.softmax_scale, tokens=toks, attn_sink=sink)
    _compare(wdec, rows_of(got, toks), ref, "decode + sink")

"""Shared helpers of the GPU parity tests: upload a workload, run the three
C-ABI stages, and compare with the float64 oracle under the stated rules."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import serving_fp8_indexer_gb300 as smla
from serving_fp8_indexer_gb300 import workloads as wl

# Tolerances (from the method's stated targets).
SCORE_REL = 1e-4          # |gpu - oracle| <= 1e-4 * sum|terms|
TOPK_TIE_REL = 1e-4       # keys within 1e-4 relative of the k-th score may differ
BF16_REL_L2, BF16_MAX_ABS = 1e-2, 3e-2   # bf16-P path (bf16 q)
FP8_REL_L2 = 3e-2                         # native FP8-P path (e4m3 q)


def score_stride_for(seqs: wl.Seqs) -> int:
    m = int(seqs.kv_len.max()) if seqs.B else 4
    return max(4, (m + 3) // 4 * 4)


def run_indexer(w: wl.Workload, stride=None):
    dev = "cuda"
    seqs = smla.Seqs.from_host(w.seqs, dev)
    stride = stride or score_stride_for(w.seqs)
    q = torch.from_numpy(w.q_idx).to(dev)
    qs = torch.from_numpy(w.q_scale).to(dev)
    kp = torch.from_numpy(w.k_pool).to(dev)
    ks = torch.from_numpy(w.k_scale).to(dev)
    scores = torch.full((w.seqs.T, stride), float("nan"), device=dev)
    smla.indexer_scores(q, qs, kp, ks, seqs, scores)
    smla.check_device_errors()
    return seqs, scores


def run_topk(seqs, scores, k, T):
    idx = torch.empty((T, k), dtype=torch.uint32, device="cuda")
    lens = torch.empty((T,), dtype=torch.uint32, device="cuda")
    smla.topk(scores, seqs, k, idx, lens)
    smla.check_device_errors()
    return idx, lens


def check_scores(w: wl.Workload, gpu_rows: np.ndarray, tokens: np.ndarray, stride: int):
    s = w.seqs
    ref, bound = oracle.indexer_scores(w.q_idx, w.q_scale, w.k_pool, w.k_scale, s.cu_q, s.kv_len, s.page_table,
                                       s.page_size, stride, tokens=tokens, with_bound=True)
    g = gpu_rows.astype(np.float64)
    inf = np.isinf(ref)
    assert np.array_equal(np.isneginf(g), inf), "-inf pattern differs (causal fill)"
    err = np.abs(g[~inf] - ref[~inf])
    tol = SCORE_REL * bound[~inf] + 1e-30
    worst = float((err / tol).max()) if err.size else 0.0
    assert worst <= 1.0, f"score error {worst:.3g}x the 1e-4*sum|terms| bound"
    return ref, worst


def check_topk_against(w: wl.Workload, ref_scores: np.ndarray, gpu_idx: np.ndarray, gpu_len: np.ndarray,
                       tokens: np.ndarray, k: int, exact: bool):
    """ref_scores: float64 rows (the oracle's, or the GPU's own scores) of
    `tokens`.  exact=True demands identical sets (same scores in -> same
    selection); otherwise keys within 1e-4 relative of the k-th reference
    score may differ."""
    s = w.seqs
    pos = wl.token_positions(s)
    sid = wl.token_seq(s)
    ref_idx, ref_len = oracle.topk(ref_scores, k, s.cu_q, s.kv_len, s.page_table, s.page_size, tokens=tokens)
    for i, t in enumerate(tokens):
        n = int(ref_len[i])
        assert int(gpu_len[i]) == n, f"token {t}: topk_lengths {gpu_len[i]} != {n}"
        g = gpu_idx[i, :n].astype(np.int64)
        assert (gpu_idx[i, n:] == 0xFFFFFFFF).all(), f"token {t}: tail not filled"
        assert len(np.unique(g)) == n, f"token {t}: duplicate indices"
        valid = wl.logical_to_phys(s, int(sid[t]), np.arange(int(pos[t]) + 1))
        lk = {int(r): j for j, r in enumerate(valid)}
        assert all(int(r) in lk for r in g), f"token {t}: index outside keys 0..pos"
        gs = set(int(r) for r in g)
        rs = set(int(r) for r in ref_idx[i, :n].astype(np.int64))
        if exact:
            assert gs == rs, f"token {t}: top-k set differs on identical scores"
        else:
            kth = ref_scores[i, lk[int(ref_idx[i, n - 1])]] if n else 0.0
            for r in gs ^ rs:
                sc = ref_scores[i, lk[r]]
                assert abs(sc - kth) <= TOPK_TIE_REL * abs(kth), f"token {t}: key {lk[r]} differs beyond the tie band"


def sample_tokens(seqs: wl.Seqs, per_seq: int, seed=0) -> np.ndarray:
    """Deterministic sample: first and last token of every sequence plus
    `per_seq` random ones."""
    rng = np.random.default_rng(seed)
    out = []
    for b in range(seqs.B):
        a, e = int(seqs.cu_q[b]), int(seqs.cu_q[b + 1])
        if e <= a:
            continue
        pick = {a, e - 1}
        if e - a > 2:
            pick |= set(rng.choice(np.arange(a + 1, e - 1), size=min(per_seq, e - a - 2), replace=False).tolist())
        out += sorted(pick)
    return np.array(out, dtype=np.int64)


def stratified_tokens(seqs: wl.Seqs, per_seq: int = 512, seed=0) -> np.ndarray:
    """Deterministic stratified sample of at least `per_seq` tokens of every
    sequence (all of them when it has no more): its first and last token,
    plus one token drawn uniformly from each of per_seq - 2 equal strata of
    the positions in between, so every part of the sequence is covered."""
    rng = np.random.default_rng(seed)
    out = []
    for b in range(seqs.B):
        a, e = int(seqs.cu_q[b]), int(seqs.cu_q[b + 1])
        if e - a <= per_seq:
            out += list(range(a, e))
            continue
        inner = np.arange(a + 1, e - 1)
        strata = np.array_split(inner, per_seq - 2)
        out += [a] + [int(rng.choice(st)) for st in strata] + [e - 1]
    toks = np.array(out, dtype=np.int64)
    assert len(np.unique(toks)) == len(toks)
    return toks


def q_attn_tensor(w: wl.Workload, dev="cuda"):
    if w.q_dtype == wl.Q_BF16:
        return torch.from_numpy(w.q_attn.view(np.int16)).view(torch.bfloat16).to(dev)
    return torch.from_numpy(w.q_attn).to(dev)


def run_prefill(w: wl.Workload, indices: torch.Tensor, lens: torch.Tensor, q=None):
    dev = "cuda"
    q = q_attn_tensor(w) if q is None else q
    latent = torch.from_numpy(w.latent).to(dev)
    scales = None if w.scales is None else torch.from_numpy(w.scales).to(dev)
    out = torch.full((w.seqs.T, w.H, 512), float("nan"), dtype=torch.bfloat16, device=dev)
    smla.sparse_prefill(q, latent, scales, w.scale_block_size, indices, lens, w.softmax_scale, out)
    smla.check_device_errors()
    return out


def check_prefill(w: wl.Workload, gpu_out_rows: np.ndarray, idx_rows: np.ndarray, len_rows: np.ndarray,
                  tokens: np.ndarray):
    """gpu_out_rows: bf16 output rows (as float32) of `tokens`; idx/len rows
    the indices the GPU consumed.  Returns (rel_l2, max_abs)."""
    T = len(tokens)
    idx_full = np.zeros((int(tokens.max()) + 1, idx_rows.shape[1]), np.uint32)
    len_full = np.zeros(int(tokens.max()) + 1, np.uint32)
    idx_full[tokens] = idx_rows
    len_full[tokens] = len_rows
    ref = oracle.sparse_prefill(w.q_attn, w.q_dtype, w.latent, w.scales, w.scale_block_size, idx_full, len_full,
                                w.softmax_scale, tokens=tokens)
    g = gpu_out_rows.astype(np.float64)
    assert np.isfinite(g).all(), "non-finite attention output"
    rel = float(np.linalg.norm(g - ref) / max(np.linalg.norm(ref), 1e-300))
    mabs = float(np.abs(g - ref).max()) if T else 0.0
    print(f"[prefill parity] {w.name}: {T} tokens, rel L2 {rel:.3e}, max abs {mabs:.3e}")
    if w.q_dtype == wl.Q_BF16:
        assert rel <= BF16_REL_L2 and mabs <= BF16_MAX_ABS, f"bf16 path: rel L2 {rel:.3g}, max abs {mabs:.3g}"
    else:
        assert rel <= FP8_REL_L2, f"FP8 path: rel L2 {rel:.3g} (max abs {mabs:.3g})"
    return rel, mabs


def rows_of(t: torch.Tensor, tokens: np.ndarray) -> np.ndarray:
    """Selected rows of a CUDA tensor as numpy (uint32 via an int32 view)."""
    sel = torch.from_numpy(tokens).to(t.device)
    if t.dtype == torch.uint32:
        return t.view(torch.int32)[sel].cpu().numpy().view(np.uint32)
    if t.dtype == torch.bfloat16:
        return t[sel].float().cpu().numpy()
    return t[sel].cpu().numpy()

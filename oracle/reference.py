"""Float64 reference of the sparse MLA prefill path (test infrastructure only).

Sources (Modular "Mojo kernels" API pages):
  * "sparse_index_fp8_sm100" module page -- the lightning-indexer score
    definition (module summary) and its epilogue order (section "Layout
    (crux)"): relu of the per-head dot product, times q_scale, summed over
    heads, times the key's k_scale; causal masking / -inf tail fill happen
    after scoring.
  * "mla_sm100_prefill_sparse_fp8" function page -- the sparse prefill call:
    q [tokens, heads, qk_depth], a paged FP8 latent cache, per-query uint32
    gather indices in physical-row space with a per-query topk_lengths, the
    scale_block_size modes (0 = unit, >= qk_depth = one scale per row,
    smaller = ceil(qk_depth/sbs) block scales per row, V using the first
    ceil(v_depth/sbs)), the softmax scale, and the output [tokens, heads,
    v_depth].
  * "mla_prefill_sparse_qkv_fp8" module page -- K and V share the MLA
    latent: V is the first v_depth columns of the same gathered rows.

Everything is computed in float64 from exactly decoded inputs.  No blocking,
fusion or reordering beyond the definitions; numpy matmul is the only library
step (a plain contraction).
"""
from __future__ import annotations

import math

import numpy as np


# ---------------------------------------------------------------------------
# Element formats.  FP8 e4m3 ("float8_e4m3fn", the cache dtype named on the
# mla_prefill_sparse_qkv_fp8 page): 1 sign bit, 4 exponent bits with bias 7,
# 3 mantissa bits; exponent 0 is subnormal; S.1111.111 is NaN; no infinities.
# ---------------------------------------------------------------------------
def _e4m3_value(byte: int) -> float:
    s = (byte >> 7) & 1
    e = (byte >> 3) & 0xF
    m = byte & 0x7
    if e == 0xF and m == 0x7:
        return math.nan
    if e == 0:
        mag = math.ldexp(m / 8.0, -6)
    else:
        mag = math.ldexp(1.0 + m / 8.0, e - 7)
    return -mag if s else mag


E4M3_TABLE = np.array([_e4m3_value(b) for b in range(256)], dtype=np.float64)


def decode_e4m3(b: np.ndarray) -> np.ndarray:
    """Exact float64 value of e4m3 bytes.  The synthetic inputs never hold the
    NaN encodings; this asserts it."""
    v = E4M3_TABLE[np.asarray(b, dtype=np.uint8)]
    assert not np.isnan(v).any(), "NaN e4m3 byte in an oracle input"
    return v


def decode_bf16(bits: np.ndarray) -> np.ndarray:
    """Exact float64 value of bfloat16 bit patterns (the upper half of an
    IEEE binary32)."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):
        return u.view(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# Ragged, paged sequences.  The pages leave the position of the new tokens
# open; the reading used throughout: sequence b's q_len new tokens are the
# LAST q_len of its kv_len cached positions, so token i of sequence b sits at
# pos = kv_len[b] - q_len + i and may attend to logical keys 0..pos.
# Logical key j of sequence b lives in physical row
#   page_table[b, j // page_size] * page_size + j % page_size
# ("get_tma_row space" on the mla_sm100_prefill_sparse_fp8 page).
# ---------------------------------------------------------------------------
def token_positions(cu_q: np.ndarray, kv_len: np.ndarray):
    cu_q = np.asarray(cu_q, dtype=np.int64)
    kv_len = np.asarray(kv_len, dtype=np.int64)
    T = int(cu_q[-1])
    pos = np.empty(T, dtype=np.int64)
    seq = np.empty(T, dtype=np.int64)
    for b in range(len(kv_len)):
        a, e = int(cu_q[b]), int(cu_q[b + 1])
        pos[a:e] = int(kv_len[b]) - (e - a) + np.arange(e - a)
        seq[a:e] = b
    return pos, seq


def phys_rows_of(page_table: np.ndarray, page_size: int, b: int, keys: np.ndarray) -> np.ndarray:
    keys = np.asarray(keys, dtype=np.int64)
    pages = np.asarray(page_table)[b, keys // page_size].astype(np.int64)
    assert (pages >= 0).all(), "logical key past the sequence's pages"
    return pages * page_size + keys % page_size


# ---------------------------------------------------------------------------
# Stage 1: lightning-indexer score ("sparse_index_fp8_sm100", module summary
# and "Layout (crux)"):
#   score[t, key] = k_scale[key] * sum_h relu(q[t, h] . k[key]) * q_scale[t, h]
# with Q [tokens, H_idx, 128] and paged K [keys, 128] in e4m3.  k_scale is
# per physical cache row.  Keys past the token's position are -inf (the
# causal "-inf tail fill" the page defers to the next stage; fused here).
# ---------------------------------------------------------------------------
def indexer_scores(q_idx, q_scale, k_pool, k_scale, cu_q, kv_len, page_table, page_size,
                   score_stride, tokens=None, with_bound=False):
    """Rows of the score buffer for the requested tokens (all by default),
    float64 [n, score_stride], -inf past each token's position.  With
    with_bound, also returns A[t, key] = k_scale * sum_h q_scale * sum_d
    |q_d k_d|, the absolute mass of the terms (the tolerance's scale)."""
    pos, seq = token_positions(cu_q, kv_len)
    tokens = np.arange(len(pos)) if tokens is None else np.asarray(tokens, dtype=np.int64)
    out = np.full((len(tokens), score_stride), -np.inf, dtype=np.float64)
    bound = np.zeros((len(tokens), score_stride), dtype=np.float64) if with_bound else None
    for i, t in enumerate(tokens):
        b, p = int(seq[t]), int(pos[t])
        keys = np.arange(p + 1)
        rows = phys_rows_of(page_table, page_size, b, keys)
        K = decode_e4m3(k_pool[rows])                     # [p+1, 128]
        Q = decode_e4m3(q_idx[t])                         # [H_idx, 128]
        qs = np.asarray(q_scale[t], dtype=np.float64)     # [H_idx]
        ks = np.asarray(k_scale, dtype=np.float64)[rows]  # [p+1]
        dots = Q @ K.T                                    # [H_idx, p+1]
        out[i, :p + 1] = ks * (qs @ np.maximum(dots, 0.0))
        if with_bound:
            bound[i, :p + 1] = ks * (qs @ (np.abs(Q) @ np.abs(K).T))
    return (out, bound) if with_bound else out


# ---------------------------------------------------------------------------
# Stage 2: per-token top-k over the causally valid keys.  The pages name the
# stage ("top-k set match" test, mla_sm100_prefill_sparse_fp8's per-query
# indices + topk_lengths) without fixing ties or order; the reading used:
# the k largest scores among keys 0..pos, ties to the lower logical key,
# topk_lengths = min(k, pos+1), indices as physical rows, slots past the
# length filled with 0xFFFFFFFF.  Brute force: a full sort per token.
# ---------------------------------------------------------------------------
def topk_select(valid_scores: np.ndarray, k: int) -> np.ndarray:
    """Logical keys of the top-k of one token's valid scores (keys 0..pos),
    ordered by (score descending, key ascending)."""
    s = np.asarray(valid_scores, dtype=np.float64)
    keys = np.arange(len(s))
    order = np.lexsort((keys, -s))
    return keys[order[:min(k, len(s))]]


def topk(scores, k, cu_q, kv_len, page_table, page_size, tokens=None):
    """Returns (indices uint32 [n, k] physical rows with 0xFFFFFFFF tail,
    lengths uint32 [n]) for the requested tokens; ``scores`` holds those
    tokens' rows in the same order."""
    pos, seq = token_positions(cu_q, kv_len)
    tokens = np.arange(len(pos)) if tokens is None else np.asarray(tokens, dtype=np.int64)
    idx = np.full((len(tokens), k), 0xFFFFFFFF, dtype=np.uint32)
    lens = np.zeros(len(tokens), dtype=np.uint32)
    for i, t in enumerate(tokens):
        p = int(pos[t])
        sel = topk_select(scores[i][:p + 1], k)
        rows = phys_rows_of(page_table, page_size, int(seq[t]), sel)
        idx[i, :len(sel)] = rows.astype(np.uint32)
        lens[i] = len(sel)
    return idx, lens


# ---------------------------------------------------------------------------
# Stage 3: sparse MLA prefill ("mla_sm100_prefill_sparse_fp8" arguments;
# "mla_prefill_sparse_qkv_fp8" for K/V sharing the latent).
# ---------------------------------------------------------------------------
def dequant_rows(latent, scales, scale_block_size, rows, qk_depth=576):
    """Dequantised latent rows, float64 [len(rows), qk_depth]:
    e4m3(byte) * scale(row, d) with scale = 1 (sbs == 0), scales[row, 0]
    (sbs >= qk_depth), or scales[row, d // sbs] (0 < sbs < qk_depth).  A
    uint16 latent is a BF16 cache (the mla_sm100_prefill_sparse form the
    FP8 page names as its base), read exactly and unscaled."""
    rows = np.asarray(rows, dtype=np.int64)
    if np.asarray(latent).dtype == np.uint16:
        assert int(scale_block_size) == 0, "a bf16 cache carries no scales"
        return decode_bf16(latent[rows])
    x = decode_e4m3(latent[rows])
    sbs = int(scale_block_size)
    if sbs == 0:
        return x
    sc = np.asarray(scales, dtype=np.float64)[rows]
    if sbs >= qk_depth:
        return x * sc[:, :1]
    blk = np.arange(qk_depth) // sbs
    return x * sc[:, blk]


def softmax_weights(s: np.ndarray, sink=None) -> np.ndarray:
    """Row softmax of a [H, n] logit matrix (max-subtracted, float64).  With
    a per-head sink logit [H] (the attention sink argument of the
    mla_sm100_prefill_sparse_fp8 page, which names it without defining it;
    the reading taken: a logit that joins every denominator and carries no
    value), p_j = exp(s_j) / (exp(sink_h) + sum_i exp(s_i)), so the row sums
    to less than 1."""
    if sink is None:
        m = s.max(axis=1, keepdims=True)
        e = np.exp(s - m)
        return e / e.sum(axis=1, keepdims=True)
    sk = np.asarray(sink, dtype=np.float64)[:, None]
    m = np.maximum(s.max(axis=1, keepdims=True), sk)
    e = np.exp(s - m)
    return e / (e.sum(axis=1, keepdims=True) + np.exp(sk - m))


def _attend(q_row, q_dtype, K, softmax_scale, v_depth, sink):
    """One token's attention over the dequantised key rows K [n, 576]."""
    q = decode_bf16(q_row) if q_dtype == 0 else decode_e4m3(q_row)  # [H, 576]
    s = float(softmax_scale) * (q @ K.T)                              # [H, n]
    return softmax_weights(s, sink) @ K[:, :v_depth]


def sparse_prefill(q_attn, q_dtype, latent, scales, scale_block_size, indices, topk_lengths,
                   softmax_scale, v_depth=512, tokens=None, attn_sink=None):
    """out[t, h, :] = sum_j p_j * V_j with s_j = softmax_scale * q[t,h] . K_j,
    p = softmax(s) over j < topk_lengths[t] (with the per-head sink logit
    attn_sink[h] in the denominator when given), K_j = dequantised latent
    row indices[t, j], V_j = K_j[:v_depth].  float64 [n, H, v_depth]; a token
    with topk_lengths 0 yields zeros (reading: empty softmax contributes
    nothing).  ``q_dtype`` is 0 for bf16 bits, 1 for e4m3 bytes."""
    T, H, D = q_attn.shape
    tokens = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    out = np.zeros((len(tokens), H, v_depth), dtype=np.float64)
    for i, t in enumerate(tokens):
        n = int(topk_lengths[t])
        if n == 0:
            continue
        rows = np.asarray(indices[t, :n], dtype=np.int64)
        K = dequant_rows(latent, scales, scale_block_size, rows, D)   # [n, 576]
        out[i] = _attend(q_attn[t], q_dtype, K, softmax_scale, v_depth, attn_sink)
    return out


# ---------------------------------------------------------------------------
# Dense causal MLA prefill ("SM100MLA" struct page; "mla_sm100_prefill_
# blockscale" for the block-scaled FP8 cache): every query token attends to
# every cached key of its sequence up to its own position, read through the
# page table; the latent dequantisation, softmax scale and sink are those of
# the sparse prefill above.
# ---------------------------------------------------------------------------
def dense_prefill(q_attn, q_dtype, latent, scales, scale_block_size, cu_q, kv_len, page_table, page_size,
                  softmax_scale, v_depth=512, tokens=None, attn_sink=None):
    """out[t, h, :] over the logical keys 0..pos(t) of t's sequence,
    float64 [n, H, v_depth]."""
    pos, seq = token_positions(cu_q, kv_len)
    T, H, D = q_attn.shape
    tokens = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    out = np.zeros((len(tokens), H, v_depth), dtype=np.float64)
    for i, t in enumerate(tokens):
        rows = phys_rows_of(page_table, page_size, int(seq[t]), np.arange(int(pos[t]) + 1))
        K = dequant_rows(latent, scales, scale_block_size, rows, D)
        out[i] = _attend(q_attn[t], q_dtype, K, softmax_scale, v_depth, attn_sink)
    return out

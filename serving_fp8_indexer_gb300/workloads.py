"""Seeded synthetic inputs for the FP8 indexer -> top-k -> sparse MLA prefill path.

This module is shared by the CUDA path's tests/bench and by the CPU oracle's
tests.  It only draws random numbers and stores them in the byte formats the
path consumes (e4m3 bytes, bf16 bits, f32 scales, int32 page tables, uint32
physical row indices).  It contains none of the method's arithmetic: no score,
no selection, no softmax.

Draw order per workload (one ``numpy.random.Generator(PCG64(seed))``):
  1. physical page permutation
  2. indexer q (N(0,1) -> e4m3)           3. q_scale  U(0.5, 1.5)
  4. indexer K pool (N(0,1) -> e4m3)      5. k_scale  U(0.5, 1.5)
  6. MLA latent pool (N(0,1), quantised per the scale mode)
  7. attention Q (N(0,1) -> bf16 or e4m3)
  8. sampled top-k indices (only when the workload samples them)

Quantisation of the synthetic data: values are rounded to e4m3 (round to
nearest even, clamped to +-448) or bf16 (round to nearest even) with torch's
CPU casts.  Blockwise scale = block amax / 448 (1.0 when amax == 0); the
latent byte is e4m3(x / scale).  Tensorwise uses the row amax the same way.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

QK_DEPTH = 576          # 512 nope + 64 rope (MLA latent width)
V_DEPTH = 512
IDX_DEPTH = 128         # lightning-indexer head depth

Q_BF16 = 0
Q_E4M3 = 1


def to_e4m3_bytes(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).clamp_(-448.0, 448.0)
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _normal(rng: np.random.Generator, shape, chunk=1 << 26) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e] = rng.standard_normal(e - s, dtype=np.float32)
    return out.reshape(shape)


def _normal_e4m3(rng, shape, chunk=1 << 26) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint8)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e] = to_e4m3_bytes(rng.standard_normal(e - s, dtype=np.float32))
    return out.reshape(shape)


def _normal_bf16(rng, shape, chunk=1 << 26) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e] = to_bf16_bits(rng.standard_normal(e - s, dtype=np.float32))
    return out.reshape(shape)


@dataclasses.dataclass
class Seqs:
    """Ragged batch over a paged cache.

    cu_q[b]..cu_q[b+1] are sequence b's query tokens; kv_len[b] its cached
    keys; the new tokens are the last q_len of those keys.  page_table[b, i]
    is the physical page of logical page i (-1 past the sequence's pages).
    """
    cu_q: np.ndarray          # int32 [B+1]
    kv_len: np.ndarray        # int32 [B]
    page_table: np.ndarray    # int32 [B, max_pages]
    page_size: int
    phys_rows: int

    @property
    def B(self) -> int:
        return int(self.kv_len.shape[0])

    @property
    def T(self) -> int:
        return int(self.cu_q[-1])

    @property
    def max_pages(self) -> int:
        return int(self.page_table.shape[1])


def make_seqs(rng, q_lens, kv_lens, page_size) -> Seqs:
    q_lens = [int(x) for x in q_lens]
    kv_lens = [int(x) for x in kv_lens]
    assert all(q <= kv for q, kv in zip(q_lens, kv_lens))
    pages = [math.ceil(kv / page_size) for kv in kv_lens]
    total = sum(pages)
    perm = rng.permutation(total).astype(np.int32)
    max_pages = max(pages) if pages else 1
    pt = np.full((len(kv_lens), max(1, max_pages)), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(pages):
        pt[b, :n] = perm[off:off + n]
        off += n
    cu = np.zeros(len(q_lens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(q_lens)
    return Seqs(cu, np.asarray(kv_lens, np.int32), pt, page_size, total * page_size)


def token_positions(seqs: Seqs) -> np.ndarray:
    """Absolute cache position of each query token (input recipe helper)."""
    pos = np.empty(seqs.T, dtype=np.int64)
    for b in range(seqs.B):
        a, e = int(seqs.cu_q[b]), int(seqs.cu_q[b + 1])
        pos[a:e] = int(seqs.kv_len[b]) - (e - a) + np.arange(e - a)
    return pos


def token_seq(seqs: Seqs) -> np.ndarray:
    sid = np.empty(seqs.T, dtype=np.int64)
    for b in range(seqs.B):
        sid[int(seqs.cu_q[b]):int(seqs.cu_q[b + 1])] = b
    return sid


def logical_to_phys(seqs: Seqs, b: int, keys: np.ndarray) -> np.ndarray:
    keys = np.asarray(keys, dtype=np.int64)
    return seqs.page_table[b, keys // seqs.page_size].astype(np.int64) * seqs.page_size + keys % seqs.page_size


@dataclasses.dataclass
class Workload:
    name: str
    seqs: Seqs
    # indexer (None when the workload has no indexer stage)
    h_idx: int = 0
    q_idx: Optional[np.ndarray] = None       # uint8 [T, H_idx, 128]
    q_scale: Optional[np.ndarray] = None     # f32 [T, H_idx]
    k_pool: Optional[np.ndarray] = None      # uint8 [phys_rows, 128]
    k_scale: Optional[np.ndarray] = None     # f32 [phys_rows]
    topk: int = 0
    # sparse attention (None when the workload has no attention stage)
    H: int = 0
    q_dtype: int = Q_BF16
    q_attn: Optional[np.ndarray] = None      # uint16 bf16 bits or uint8 e4m3, [T, H, 576]
    latent: Optional[np.ndarray] = None      # uint8 e4m3 [phys_rows, 576] (uint16 bf16 for a BF16 cache)
    scale_block_size: int = 0
    scales: Optional[np.ndarray] = None      # f32 [phys_rows, ceil(576/sbs)] or None
    indices: Optional[np.ndarray] = None     # uint32 [T, topk] physical rows (sampled workloads)
    topk_lengths: Optional[np.ndarray] = None  # uint32 [T]
    softmax_scale: float = 1.0 / math.sqrt(QK_DEPTH)


def _quantise_latent(rng, rows, sbs):
    x = _normal(rng, (rows, QK_DEPTH))
    if sbs == 0:
        return to_e4m3_bytes(x), None
    width = QK_DEPTH if sbs >= QK_DEPTH else sbs
    nblk = (QK_DEPTH + width - 1) // width
    xb = np.zeros((rows, nblk * width), dtype=np.float32)
    xb[:, :QK_DEPTH] = x
    xb = xb.reshape(rows, nblk, width)
    amax = np.abs(xb).max(axis=2)
    s = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    q = to_e4m3_bytes(xb / s[:, :, None]).reshape(rows, nblk * width)[:, :QK_DEPTH]
    return np.ascontiguousarray(q), s


def sample_causal_indices(rng, seqs: Seqs, k: int):
    """k distinct causally valid keys per token, uniform without replacement
    (all keys 0..pos when pos+1 <= k); returned as physical rows, tail
    0xFFFFFFFF, in sampled order."""
    T = seqs.T
    pos = token_positions(seqs)
    sid = token_seq(seqs)
    idx = np.full((T, k), 0xFFFFFFFF, dtype=np.uint32)
    lens = np.minimum(pos + 1, k).astype(np.uint32)
    for t in range(T):
        n = int(pos[t]) + 1
        if n <= k:
            keys = rng.permutation(n)
        else:
            keys = rng.choice(n, size=k, replace=False)
        idx[t, :len(keys)] = logical_to_phys(seqs, int(sid[t]), keys).astype(np.uint32)
    return idx, lens


def build(name: str, seed: int, q_lens, kv_lens, page_size=64, *, h_idx=0, topk=0,
          H=0, q_dtype=Q_BF16, sbs=0, sample_indices=False, latent_bf16=False) -> Workload:
    rng = np.random.default_rng(seed)
    seqs = make_seqs(rng, q_lens, kv_lens, page_size)
    T, R = seqs.T, seqs.phys_rows
    w = Workload(name=name, seqs=seqs, h_idx=h_idx, topk=topk, H=H, q_dtype=q_dtype,
                 scale_block_size=sbs)
    if h_idx:
        w.q_idx = _normal_e4m3(rng, (T, h_idx, IDX_DEPTH))
        w.q_scale = rng.uniform(0.5, 1.5, size=(T, h_idx)).astype(np.float32)
        w.k_pool = _normal_e4m3(rng, (R, IDX_DEPTH))
        w.k_scale = rng.uniform(0.5, 1.5, size=(R,)).astype(np.float32)
    if H:
        if latent_bf16:  # a BF16 latent cache (no scales): N(0,1) rounded to bf16
            assert sbs == 0
            w.latent, w.scales = _normal_bf16(rng, (R, QK_DEPTH)), None
        else:
            w.latent, w.scales = _quantise_latent(rng, R, sbs)
        if q_dtype == Q_BF16:
            w.q_attn = _normal_bf16(rng, (T, H, QK_DEPTH))
        else:
            w.q_attn = _normal_e4m3(rng, (T, H, QK_DEPTH))
        if sample_indices:
            w.indices, w.topk_lengths = sample_causal_indices(rng, seqs, topk)
    return w


# The five synthetic workloads (seed = workload number - 1).
def tiny_prefill(seed=0) -> Workload:
    """1 sequence, 64 query tokens at positions 192..255 over a 256-token
    cache (4 permuted pages of 64); indexer H_idx=4; top-64; attention H=16,
    bf16 Q, unit-scale e4m3 latent."""
    return build("tiny_prefill_T64_L256", seed, [64], [256], 64, h_idx=4, topk=64, H=16,
                 q_dtype=Q_BF16, sbs=0)


def mtp_decode_indexer(seed=1) -> Workload:
    """batch 8 x 2 query tokens (positions 2046, 2047) over 2048 keys each,
    H_idx=64; top-2048 over all valid keys."""
    return build("mtp_decode_B8x2_L2048_Hidx64", seed, [2] * 8, [2048] * 8, 64, h_idx=64, topk=2048)


def dsv32_prefill(seed=2, T=4096, k=2048, latent_bf16=False) -> Workload:
    """1 sequence of T tokens (positions 0..T-1), H=128 bf16 Q, unit-scale
    e4m3 latent (or a BF16 latent cache), top-k causally sampled indices."""
    return build(f"sparse_prefill_T{T}_H128_bf16_{'bf16cache' if latent_bf16 else 'unit'}_k{k}", seed, [T], [T], 64,
                 topk=k, H=128, q_dtype=Q_BF16, sbs=0, sample_indices=True, latent_bf16=latent_bf16)


def blockwise_fp8_prefill(seed=3, lens=(1024, 2048, 3072, 4096), k=2048) -> Workload:
    """4 ragged sequences (10240 tokens), H=64, e4m3 Q, latent e4m3 with
    32-wide block scales, top-k causally sampled indices."""
    return build(f"sparse_prefill_{'-'.join(map(str, lens))}_H64_fp8_sbs32_k{k}", seed, list(lens),
                 list(lens), 64, topk=k, H=64, q_dtype=Q_E4M3, sbs=32, sample_indices=True)


def e2e_chunk(seed=4, B=8, L=8192, q_len=2048, k=2048, H=128, h_idx=64) -> Workload:
    """B sequences x L cached tokens, q_len new tokens each (the last q_len
    positions); indexer H_idx=64 -> causal top-k -> sparse MLA with H=128,
    bf16 Q, tensorwise-scaled e4m3 latent (one scale per row)."""
    return build(f"e2e_chunk_B{B}_L{L}_q{q_len}_H{H}_k{k}", seed, [q_len] * B, [L] * B, 64,
                 h_idx=h_idx, topk=k, H=H, q_dtype=Q_BF16, sbs=QK_DEPTH)


def sparse_decode(seed=5, B=8, q_per_seq=2, L=8192, k=2048, H=128, q_dtype=Q_BF16, sbs=0) -> Workload:
    """Sparse MLA decode: B sequences of L cached tokens with q_per_seq new
    tokens each (the last positions, as in MTP decode), top-k causally
    sampled indices, H heads."""
    return build(f"sparse_decode_B{B}x{q_per_seq}_L{L}_H{H}_k{k}_{'bf16' if q_dtype == Q_BF16 else 'fp8'}_sbs{sbs}",
                 seed, [q_per_seq] * B, [L] * B, 64, topk=k, H=H, q_dtype=q_dtype, sbs=sbs, sample_indices=True)


def dense_prefill(seed=6, lens=(512, 1024, 2048, 1537), H=128, q_dtype=Q_BF16, sbs=0) -> Workload:
    """Dense causal prefill of short prompts: every token attends to all of
    its sequence's keys 0..pos (no indices), H heads."""
    return build(f"dense_prefill_{'-'.join(map(str, lens))}_H{H}_{'bf16' if q_dtype == Q_BF16 else 'fp8'}_sbs{sbs}",
                 seed, list(lens), list(lens), 64, H=H, q_dtype=q_dtype, sbs=sbs)

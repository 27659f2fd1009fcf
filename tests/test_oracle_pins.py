"""Pins of the float64 oracle to facts outside itself (CPU only).

Each check is chosen so that a plausible slip in the oracle (a dropped relu,
a transposed scale, logical instead of physical k_scale, V taking the rope
columns, a wrong scale block, a missing softmax scale, a wrong tie rule)
fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from serving_fp8_indexer_gb300 import workloads as wl


def _hex(s):
    return int(s, 16)


# --------------------------------------------------------------------------- formats
def test_e4m3_closed_forms(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "e4m3_closed_forms.json")))
    for h, v in g["values"].items():
        got = oracle.E4M3_TABLE[_hex(h)]
        assert got == v and math.copysign(1, got) == math.copysign(1, v), h
    for h in g["nan"]:
        assert math.isnan(oracle.E4M3_TABLE[_hex(h)])


def test_e4m3_matches_torch_float8():
    b = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = b.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = oracle.E4M3_TABLE
    nan = np.isnan(ref)
    assert (nan == np.isnan(ours)).all() and nan.sum() == 2
    assert np.array_equal(ref[~nan], ours[~nan])


def test_bf16_matches_torch():
    bits = np.arange(0, 65536, 7, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    ours = oracle.decode_bf16(bits)
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], ours[ok]) and np.isnan(ours[~ok]).all()


# --------------------------------------------------------------------------- indexer
def _handcase(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "indexer_handcase.json")))
    D, H = g["depth"], g["h_idx"]
    k_pool = np.zeros((g["phys_rows"], D), np.uint8)
    for r, cols in g["k_rows_nonzero"].items():
        for c, h in cols.items():
            k_pool[int(r), int(c)] = _hex(h)
    T = sum(g["q_len"])
    q = np.zeros((T, H, D), np.uint8)
    for t, heads in g["q_nonzero"].items():
        for h, cols in heads.items():
            for c, hx in cols.items():
                q[int(t), int(h), int(c)] = _hex(hx)
    cu = np.array([0] + list(np.cumsum(g["q_len"])), np.int32)
    return g, q, np.array(g["q_scale"], np.float32), k_pool, np.array(g["k_scale"], np.float32), cu


def test_indexer_handcase(golden_dir):
    g, q, qs, kp, ks, cu = _handcase(golden_dir)
    s = oracle.indexer_scores(q, qs, kp, ks, cu, np.array(g["kv_len"]), np.array(g["page_table"]),
                              g["page_size"], g["score_stride"])
    exp = np.array([[float(x) for x in row] for row in g["expected"]])
    assert np.array_equal(s, exp)


def test_indexer_onehot_closed_form():
    """k[key] = v_key * e_{d_key} and q[t,h] = c_{t,h} * (all ones on the
    support) give dot = c_{t,h} * v_key exactly, so
    score = ks[phys(key)] * sum_h qs[t,h] * relu(c_{t,h} * v_key)."""
    rng = np.random.default_rng(7)
    seqs = wl.make_seqs(rng, [5, 3], [40, 20], 8)
    T, R, H, D = seqs.T, seqs.phys_rows, 3, 128
    vals = np.array([0x30, 0x38, 0x3c, 0x40, 0xb0, 0xb8, 0xc0, 0x44], np.uint8)   # +-0.5,1,1.5,2,3
    vkey = rng.choice(vals, size=R)
    dkey = rng.integers(0, D, size=R)
    kp = np.zeros((R, D), np.uint8)
    kp[np.arange(R), dkey] = vkey
    cvals = np.array([0x38, 0xb8, 0x40], np.uint8)                                 # 1, -1, 2
    c = rng.choice(cvals, size=(T, H))
    q = np.repeat(c[:, :, None], D, axis=2).astype(np.uint8)
    qs = rng.uniform(0.5, 1.5, (T, H)).astype(np.float32)
    ks = rng.uniform(0.5, 1.5, R).astype(np.float32)
    out = oracle.indexer_scores(q, qs, kp, ks, seqs.cu_q, seqs.kv_len, seqs.page_table,
                                seqs.page_size, 48)
    dec = {int(b): v for b, v in zip(vals, [0.5, 1, 1.5, 2, -0.5, -1, -2, 3])}
    dec.update({0x38: 1.0, 0xb8: -1.0, 0x40: 2.0})
    pos = wl.token_positions(seqs)
    sid = wl.token_seq(seqs)
    for t in range(T):
        for key in range(48):
            if key > pos[t]:
                assert out[t, key] == -np.inf
                continue
            r = int(wl.logical_to_phys(seqs, int(sid[t]), np.array([key]))[0])
            e = float(ks[r]) * sum(float(qs[t, h]) * max(0.0, dec[int(c[t, h])] * dec[int(vkey[r])])
                                   for h in range(H))
            assert out[t, key] == pytest.approx(e, rel=1e-15, abs=0)


def _random_indexer(seed, q_lens=(3, 4), kv=(30, 17), ps=8, H=4):
    w = wl.build("t", seed, list(q_lens), list(kv), ps, h_idx=H, topk=8)
    return w


def test_indexer_invariants():
    w = _random_indexer(11)
    s = w.seqs
    args = (s.cu_q, s.kv_len, s.page_table, s.page_size, 32)
    base = oracle.indexer_scores(w.q_idx, w.q_scale, w.k_pool, w.k_scale, *args)
    pos = wl.token_positions(s)
    valid = np.arange(32)[None, :] <= pos[:, None]
    assert np.isfinite(base[valid]).all() and (base[valid] >= 0).all()
    assert (base[~valid] == -np.inf).all()
    # linear in k_scale and q_scale
    dbl = oracle.indexer_scores(w.q_idx, w.q_scale, w.k_pool, 2 * w.k_scale, *args)
    assert np.allclose(dbl[valid], 2 * base[valid], rtol=1e-14)
    dbl = oracle.indexer_scores(w.q_idx, 4 * w.q_scale, w.k_pool, w.k_scale, *args)
    assert np.allclose(dbl[valid], 4 * base[valid], rtol=1e-14)
    # the per-head q_scale is not interchangeable across heads
    perm = oracle.indexer_scores(w.q_idx, w.q_scale[:, ::-1].copy(), w.k_pool, w.k_scale, *args)
    assert not np.allclose(perm[valid], base[valid])
    # relayout of physical pages with a matching page table and k_scale
    npages = s.phys_rows // s.page_size
    newpos = np.random.default_rng(3).permutation(npages)
    kp2 = np.zeros_like(w.k_pool)
    ks2 = np.zeros_like(w.k_scale)
    for old, new in enumerate(newpos):
        kp2[new * s.page_size:(new + 1) * s.page_size] = w.k_pool[old * s.page_size:(old + 1) * s.page_size]
        ks2[new * s.page_size:(new + 1) * s.page_size] = w.k_scale[old * s.page_size:(old + 1) * s.page_size]
    pt2 = np.where(s.page_table >= 0, newpos[np.maximum(s.page_table, 0)], -1).astype(np.int32)
    moved = oracle.indexer_scores(w.q_idx, w.q_scale, kp2, ks2, s.cu_q, s.kv_len, pt2, s.page_size, 32)
    assert np.array_equal(moved, base)


def test_indexer_matches_torch_einsum():
    w = _random_indexer(5, q_lens=(6,), kv=(21,), ps=4, H=8)
    s = w.seqs
    out = oracle.indexer_scores(w.q_idx, w.q_scale, w.k_pool, w.k_scale, s.cu_q, s.kv_len,
                                s.page_table, s.page_size, 21)
    f8 = lambda a: torch.from_numpy(a).view(torch.float8_e4m3fn).to(torch.float64)
    rows = wl.logical_to_phys(s, 0, np.arange(21))
    K = f8(w.k_pool[rows])
    Q = f8(w.q_idx)
    dots = torch.einsum("thd,kd->thk", Q, K).clamp_min(0)
    ref = torch.einsum("thk,th->tk", dots, torch.from_numpy(w.q_scale).double()) * \
        torch.from_numpy(w.k_scale[rows]).double()[None, :]
    pos = wl.token_positions(s)
    mask = torch.arange(21)[None, :] > torch.from_numpy(pos)[:, None]
    ref = ref.masked_fill(mask, -math.inf).numpy()
    assert np.allclose(out, ref, rtol=1e-13, atol=0) and np.array_equal(np.isinf(out), np.isinf(ref))


# --------------------------------------------------------------------------- top-k
def test_topk_handcase(golden_dir):
    g, q, qs, kp, ks, cu = _handcase(golden_dir)
    pt = np.array(g["page_table"])
    s = oracle.indexer_scores(q, qs, kp, ks, cu, np.array(g["kv_len"]), pt, g["page_size"], 4)
    idx, lens = oracle.topk(s, 2, cu, np.array(g["kv_len"]), pt, g["page_size"])
    assert list(lens) == g["topk2_expected_lengths"]
    for t, exp in enumerate(g["topk2_expected_phys_sets"]):
        assert sorted(idx[t, :lens[t]].tolist()) == sorted(exp)


def test_topk_tie_rule_and_fill():
    sel = oracle.topk_select(np.array([5.0, 7.0, 7.0, 1.0, 7.0]), 2)
    assert sel.tolist() == [1, 2]                   # ties go to the lower key
    assert oracle.topk_select(np.array([2.0, 9.0]), 8).tolist() == [1, 0]  # k > valid -> all


def test_topk_invariants_and_torch_topk():
    rng = np.random.default_rng(2)
    seqs = wl.make_seqs(rng, [6, 5], [70, 9], 16)
    pos = wl.token_positions(seqs)
    sid = wl.token_seq(seqs)
    k = 12
    scores = np.full((seqs.T, 80), -np.inf)
    for t in range(seqs.T):
        scores[t, :pos[t] + 1] = rng.permutation(pos[t] + 1) * 0.25   # distinct
    idx, lens = oracle.topk(scores, k, seqs.cu_q, seqs.kv_len, seqs.page_table, seqs.page_size)
    for t in range(seqs.T):
        n = int(pos[t]) + 1
        assert lens[t] == min(k, n)
        got = idx[t, :lens[t]].astype(np.int64)
        assert (idx[t, lens[t]:] == 0xFFFFFFFF).all()
        assert len(set(got.tolist())) == len(got)
        valid_rows = wl.logical_to_phys(seqs, int(sid[t]), np.arange(n))
        assert set(got.tolist()) <= set(valid_rows.tolist())
        lk = {int(r): j for j, r in enumerate(valid_rows)}
        chosen = np.array([lk[int(r)] for r in got])
        rest = np.setdiff1d(np.arange(n), chosen)
        if len(rest):
            assert scores[t, chosen].min() >= scores[t, rest].max()
        tk = torch.topk(torch.from_numpy(scores[t, :n]), min(k, n)).indices.numpy()
        assert set(tk.tolist()) == set(chosen.tolist())


# --------------------------------------------------------------------------- attention
def _attn_inputs(rng, T, H, R, n, sbs=0, q_dtype=0):
    latent = wl.to_e4m3_bytes(rng.standard_normal((R, 576)).astype(np.float32))
    if q_dtype == 0:
        q = wl.to_bf16_bits(rng.standard_normal((T, H, 576)).astype(np.float32))
    else:
        q = wl.to_e4m3_bytes(rng.standard_normal((T, H, 576)).astype(np.float32))
    idx = np.stack([rng.choice(R, n, replace=False) for _ in range(T)]).astype(np.uint32)
    return latent, q, idx


def test_attention_handcase(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "attention_handcase.json")))
    lat = np.zeros((2, 576), np.uint8)
    for r, cols in g["latent_rows_nonzero"].items():
        for c, hx in cols.items():
            lat[int(r), int(c)] = _hex(hx)
    qf = np.zeros((1, 1, 576), np.float32)
    for c, v in g["q_bf16_nonzero"].items():
        qf[0, 0, int(c)] = v
    q = wl.to_bf16_bits(qf)
    idx = np.array([g["indices"]], np.uint32)
    out = oracle.sparse_prefill(q, 0, lat, None, 0, idx, np.array([2], np.uint32), g["softmax_scale"])
    pA = 1.0 / (1.0 + math.exp(g["s_B"] - g["s_A"]))
    pB = 1.0 - pA
    exp = np.zeros(512)
    exp[0], exp[10], exp[511] = pA - pB, 3 * pA + pB, 2 * pA
    assert np.allclose(out[0, 0], exp, rtol=1e-14, atol=1e-15)


def test_attention_single_key_and_zero_q():
    rng = np.random.default_rng(4)
    latent, q, idx = _attn_inputs(rng, 3, 4, 50, 7)
    one = oracle.sparse_prefill(q, 0, latent, None, 0, idx, np.array([1, 1, 1], np.uint32), 0.04)
    for t in range(3):
        v = oracle.decode_e4m3(latent[idx[t, 0]])[:512]
        assert np.array_equal(one[t], np.broadcast_to(v, (4, 512)))
    qz = np.zeros_like(q)
    mean = oracle.sparse_prefill(qz, 0, latent, None, 0, idx, np.array([7, 7, 7], np.uint32), 0.04)
    for t in range(3):
        v = oracle.decode_e4m3(latent[idx[t, :7].astype(np.int64)])[:, :512].mean(axis=0)
        assert np.allclose(mean[t], v, rtol=1e-13, atol=1e-15)


def test_attention_index_permutation_invariant():
    rng = np.random.default_rng(8)
    latent, q, idx = _attn_inputs(rng, 2, 8, 300, 130)
    lens = np.array([130, 77], np.uint32)
    a = oracle.sparse_prefill(q, 0, latent, None, 0, idx, lens, 0.05)
    idx2 = idx.copy()
    idx2[0] = idx[0][rng.permutation(130)]
    idx2[1, :77] = idx[1, :77][rng.permutation(77)]
    b = oracle.sparse_prefill(q, 0, latent, None, 0, idx2, lens, 0.05)
    assert np.allclose(a, b, rtol=1e-12, atol=1e-14)


def test_softmax_rows_sum_to_one():
    s = np.random.default_rng(1).standard_normal((16, 333)) * 30
    p = oracle.softmax_weights(s)
    assert np.abs(p.sum(axis=1) - 1).max() < 1e-12 and (p >= 0).all()


def test_attention_all_keys_equals_dense_causal_sdpa():
    """k = every causal key turns the sparse path into dense causal MQA over
    the latent (K = latent[:, :576], V = latent[:, :512] shared by all
    heads); torch's scaled_dot_product_attention in float64 is the
    independent reference."""
    rng = np.random.default_rng(12)
    L, H, ps = 37, 4, 8
    seqs = wl.make_seqs(rng, [L], [L], ps)
    latent = wl.to_e4m3_bytes(rng.standard_normal((seqs.phys_rows, 576)).astype(np.float32))
    q = wl.to_bf16_bits(rng.standard_normal((L, H, 576)).astype(np.float32))
    rows = wl.logical_to_phys(seqs, 0, np.arange(L))
    idx = np.full((L, L), 0xFFFFFFFF, np.uint32)
    for t in range(L):
        idx[t, :t + 1] = rows[:t + 1]
    lens = np.arange(1, L + 1, dtype=np.uint32)
    sc = 1 / math.sqrt(576)
    out = oracle.sparse_prefill(q, 0, latent, None, 0, idx, lens, sc)
    K = torch.from_numpy(latent[rows]).view(torch.float8_e4m3fn).double()
    Q = torch.from_numpy(q.view(np.int16)).view(torch.bfloat16).double().permute(1, 0, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(
        Q[None], K[None, None].expand(1, H, L, 576), K[None, None, :, :512].expand(1, H, L, 512),
        is_causal=True, scale=sc)[0].permute(1, 0, 2).numpy()
    assert np.allclose(out, ref, rtol=1e-11, atol=1e-13)


def test_dequant_scale_modes():
    rng = np.random.default_rng(9)
    R = 6
    lat = wl.to_e4m3_bytes(rng.standard_normal((R, 576)).astype(np.float32))
    base = oracle.decode_e4m3(lat)
    blk = rng.uniform(0.25, 4, (R, 18)).astype(np.float32)
    d = oracle.dequant_rows(lat, blk, 32, np.arange(R))
    for r in range(R):
        for col in (0, 31, 32, 63, 511, 512, 575):
            assert d[r, col] == base[r, col] * float(blk[r, col // 32])
    tw = rng.uniform(0.25, 4, (R, 1)).astype(np.float32)
    d = oracle.dequant_rows(lat, tw, 576, np.arange(R))
    assert np.array_equal(d, base * tw.astype(np.float64))
    assert np.array_equal(oracle.dequant_rows(lat, None, 0, np.arange(R)), base)
    # equal block scales == one row scale, through the whole attention
    q = wl.to_bf16_bits(rng.standard_normal((2, 3, 576)).astype(np.float32))
    idx = np.array([[0, 2, 4, 5], [1, 3, 5, 0]], np.uint32)
    lens = np.array([4, 3], np.uint32)
    c = np.float32(0.75)
    a = oracle.sparse_prefill(q, 0, lat, np.full((R, 18), c, np.float32), 32, idx, lens, 0.1)
    b = oracle.sparse_prefill(q, 0, lat, np.full((R, 1), c, np.float32), 576, idx, lens, 0.1)
    assert np.array_equal(a, b)
    u = oracle.sparse_prefill(q, 0, lat, None, 0, idx, lens, 0.1)
    assert not np.allclose(a, u)   # the scale reaches both the logits and V


def test_two_summation_orders_agree():
    """The whole oracle on the tiny workload, once as written and once with
    a per-(token, head, key) python loop for the logits and the weighted
    sum: agreement to ~1e-12 shows no order-dependent slip."""
    w = wl.tiny_prefill()
    s = w.seqs
    sc = oracle.indexer_scores(w.q_idx, w.q_scale, w.k_pool, w.k_scale, s.cu_q, s.kv_len,
                               s.page_table, s.page_size, 256)
    idx, lens = oracle.topk(sc, w.topk, s.cu_q, s.kv_len, s.page_table, s.page_size)
    out = oracle.sparse_prefill(w.q_attn, 0, w.latent, None, 0, idx, lens, w.softmax_scale)
    for t in (0, 17, 63):
        n = int(lens[t])
        K = oracle.decode_e4m3(w.latent[idx[t, :n].astype(np.int64)])
        q = oracle.decode_bf16(w.q_attn[t])
        for h in (0, 9, 15):
            logits = [w.softmax_scale * math.fsum(q[h] * K[j]) for j in range(n)]
            m = max(logits)
            e = [math.exp(x - m) for x in logits]
            z = math.fsum(e)
            ref = [math.fsum(e[j] * K[j, c] for j in range(n)) / z for c in range(0, 512, 37)]
            assert np.allclose(out[t, h, ::37], ref, rtol=1e-12, atol=1e-14)


def test_attention_e4m3_q_branch():
    """The e4m3-q branch of the oracle, pinned two ways.  (1) Every finite
    e4m3 value is exact in bf16, so the same q given as e4m3 bytes
    (q_dtype 1) and as the bf16 bits of the same values (q_dtype 0) must
    give identical results; a branch that decoded the bytes any other way
    would not.  (2) k = every causal key against torch's float64
    scaled_dot_product_attention with q taken from torch's float8 dtype."""
    rng = np.random.default_rng(21)
    latent, q8, idx = _attn_inputs(rng, 3, 5, 90, 40, q_dtype=1)
    q16 = torch.from_numpy(q8).view(torch.float8_e4m3fn).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.decode_bf16(q16), oracle.decode_e4m3(q8))
    lens = np.array([40, 17, 1], np.uint32)
    a = oracle.sparse_prefill(q8, 1, latent, None, 0, idx, lens, 0.07)
    b = oracle.sparse_prefill(q16, 0, latent, None, 0, idx, lens, 0.07)
    assert np.array_equal(a, b)
    L, H, ps = 29, 3, 8
    seqs = wl.make_seqs(rng, [L], [L], ps)
    lat = wl.to_e4m3_bytes(rng.standard_normal((seqs.phys_rows, 576)).astype(np.float32))
    q = wl.to_e4m3_bytes(rng.standard_normal((L, H, 576)).astype(np.float32))
    rows = wl.logical_to_phys(seqs, 0, np.arange(L))
    ind = np.full((L, L), 0xFFFFFFFF, np.uint32)
    for t in range(L):
        ind[t, :t + 1] = rows[:t + 1]
    sc = 1 / math.sqrt(576)
    out = oracle.sparse_prefill(q, 1, lat, None, 0, ind, np.arange(1, L + 1, dtype=np.uint32), sc)
    K = torch.from_numpy(lat[rows]).view(torch.float8_e4m3fn).double()
    Q = torch.from_numpy(q).view(torch.float8_e4m3fn).double().permute(1, 0, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(
        Q[None], K[None, None].expand(1, H, L, 576), K[None, None, :, :512].expand(1, H, L, 512),
        is_causal=True, scale=sc)[0].permute(1, 0, 2).numpy()
    assert np.allclose(out, ref, rtol=1e-11, atol=1e-13)


def test_attention_sink_closed_forms():
    """The sink reading pinned by closed forms: one key of logit s and sink
    logit z give out = V * e^s / (e^s + e^z) = V * sigmoid(s - z); a sink of
    -inf is no sink; two keys and a sink at the same logit give each key 1/3;
    a very large sink drives the output to 0."""
    rng = np.random.default_rng(31)
    latent, q, idx = _attn_inputs(rng, 2, 3, 40, 6)
    sc = 0.05
    one = np.ones(2, np.uint32)
    z = np.array([0.3, -1.2, 2.5])
    out = oracle.sparse_prefill(q, 0, latent, None, 0, idx, one, sc, attn_sink=z)
    for t in range(2):
        K = oracle.decode_e4m3(latent[idx[t, 0]])
        qf = oracle.decode_bf16(q[t])
        for h in range(3):
            s = sc * math.fsum(qf[h] * K)
            w = 1.0 / (1.0 + math.exp(z[h] - s))
            assert np.allclose(out[t, h], w * K[:512], rtol=1e-13, atol=1e-15)
    lens = np.array([6, 4], np.uint32)
    a = oracle.sparse_prefill(q, 0, latent, None, 0, idx, lens, sc)
    b = oracle.sparse_prefill(q, 0, latent, None, 0, idx, lens, sc, attn_sink=np.full(3, -np.inf))
    assert np.array_equal(a, b)
    big = oracle.sparse_prefill(q, 0, latent, None, 0, idx, lens, sc, attn_sink=np.full(3, 1e4))
    assert np.abs(big).max() == 0.0
    # two identical rows (equal logits) and a sink at that logit: weights 1/3 each
    lat2 = np.zeros((2, 576), np.uint8)
    lat2[0] = lat2[1] = latent[0]
    qz = np.zeros((1, 1, 576), np.uint16)   # q = 0: every logit 0
    o3 = oracle.sparse_prefill(qz, 0, lat2, None, 0, np.array([[0, 1]], np.uint32), np.array([2], np.uint32), sc,
                               attn_sink=np.zeros(1))
    assert np.allclose(o3[0, 0], (2.0 / 3.0) * oracle.decode_e4m3(latent[0])[:512], rtol=1e-14, atol=0)


def test_dense_prefill_equals_causal_sdpa_over_pages():
    """The dense causal oracle on two paged sequences (new tokens at the end
    of each) against float64 scaled_dot_product_attention with the causal
    mask offset by the cached prefix, per sequence."""
    rng = np.random.default_rng(33)
    q_lens, kv_lens, ps, H = [5, 9], [12, 9], 4, 3
    seqs = wl.make_seqs(rng, q_lens, kv_lens, ps)
    lat = wl.to_e4m3_bytes(rng.standard_normal((seqs.phys_rows, 576)).astype(np.float32))
    q = wl.to_bf16_bits(rng.standard_normal((seqs.T, H, 576)).astype(np.float32))
    sc = 1 / math.sqrt(576)
    out = oracle.dense_prefill(q, 0, lat, None, 0, seqs.cu_q, seqs.kv_len, seqs.page_table, ps, sc)
    for b in range(2):
        a, e = int(seqs.cu_q[b]), int(seqs.cu_q[b + 1])
        L = int(seqs.kv_len[b])
        rows = wl.logical_to_phys(seqs, b, np.arange(L))
        K = torch.from_numpy(lat[rows]).view(torch.float8_e4m3fn).double()
        Q = torch.from_numpy(q[a:e].view(np.int16)).view(torch.bfloat16).double().permute(1, 0, 2)
        pos = L - (e - a) + np.arange(e - a)
        mask = torch.from_numpy(np.arange(L)[None, :] <= pos[:, None])
        ref = torch.nn.functional.scaled_dot_product_attention(
            Q[None], K[None, None].expand(1, H, L, 576), K[None, None, :, :512].expand(1, H, L, 512),
            attn_mask=mask, scale=sc)[0].permute(1, 0, 2).numpy()
        assert np.allclose(out[a:e], ref, rtol=1e-11, atol=1e-13)


def test_bf16_cache_reads_exactly():
    """A BF16 cache is read as its exact values: rows holding e4m3-exact
    values give the e4m3 cache's result bit for bit, and k = every causal
    key matches float64 scaled_dot_product_attention with K, V from torch's
    bfloat16."""
    rng = np.random.default_rng(35)
    latent, q, idx = _attn_inputs(rng, 3, 4, 60, 20)
    lat16 = torch.from_numpy(latent).view(torch.float8_e4m3fn).to(torch.bfloat16).view(torch.int16).numpy()
    lat16 = lat16.view(np.uint16)
    lens = np.array([20, 5, 1], np.uint32)
    a = oracle.sparse_prefill(q, 0, latent, None, 0, idx, lens, 0.06)
    b = oracle.sparse_prefill(q, 0, lat16, None, 0, idx, lens, 0.06)
    assert np.array_equal(a, b)
    L, H = 23, 2
    seqs = wl.make_seqs(rng, [L], [L], 8)
    lat = wl.to_bf16_bits(rng.standard_normal((seqs.phys_rows, 576)).astype(np.float32))
    qq = wl.to_bf16_bits(rng.standard_normal((L, H, 576)).astype(np.float32))
    rows = wl.logical_to_phys(seqs, 0, np.arange(L))
    ind = np.full((L, L), 0xFFFFFFFF, np.uint32)
    for t in range(L):
        ind[t, :t + 1] = rows[:t + 1]
    sc = 1 / math.sqrt(576)
    out = oracle.sparse_prefill(qq, 0, lat, None, 0, ind, np.arange(1, L + 1, dtype=np.uint32), sc)
    K = torch.from_numpy(lat[rows].view(np.int16)).view(torch.bfloat16).double()
    Q = torch.from_numpy(qq.view(np.int16)).view(torch.bfloat16).double().permute(1, 0, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(
        Q[None], K[None, None].expand(1, H, L, 576), K[None, None, :, :512].expand(1, H, L, 512),
        is_causal=True, scale=sc)[0].permute(1, 0, 2).numpy()
    assert np.allclose(out, ref, rtol=1e-11, atol=1e-13)

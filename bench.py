#!/usr/bin/env python3
"""Benchmark of the FP8 indexer -> top-k -> sparse MLA prefill path.

One step = one pass of the whole path over the end-to-end prefill chunk
(8 sequences x 8192 cached tokens, 2048 new tokens each at positions
6144..8191; indexer H_idx=64 FP8 -> causal top-2048 -> sparse MLA with
H=128, bf16 q, tensorwise-scaled e4m3 latent, bf16 output [16384,128,512]),
inputs resident in HBM.  Prints one JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the float64 CPU oracle on bounded samples of the
same workload (the path's reference arm).  Under torchrun with N > 1 every
rank runs its own replica of the chunk (weak scaling, no collective on the
data path); rank 0 prints.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse-MLA prefill TFLOP/s (% GB300 tensor peak); indexer+topk keys·tok/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            return d, "measured"
        except Exception:
            pass
    return dict(FALLBACK_PEAKS), "fallback"


def max_over_ranks(values, device):
    """Each timing's maximum over all ranks (the slowest replica sets the step
    time); values unchanged on one rank."""
    import torch
    if not torch.distributed.is_available() or not torch.distributed.is_initialized() or \
            torch.distributed.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(x) for x in t]


def weak_scaling_value(world, work_per_rank, ms_per_step):
    """Whole-job throughput when every rank processes the same work per step."""
    return world * work_per_rank / (ms_per_step * 1e-3)


def dtype_label(w):
    """The arithmetic the path runs in, per workload."""
    from serving_fp8_indexer_gb300 import workloads as wl
    if not w.H:
        return "e4m3 MMA (indexer q and k), f32 accumulate"
    if w.q_dtype == wl.Q_E4M3 and 0 < w.scale_block_size < 576:
        return "e4m3 MMA (e4m3 q; blockwise rows re-expressed as e4m3 hi+lo; P e4m3), f32 accumulate"
    if w.q_dtype == wl.Q_E4M3:
        return "e4m3 MMA (e4m3 q, e4m3 rows, P e4m3), f32 accumulate"
    return "e4m3 MMA (bf16 q and P as e4m3 hi+lo), f32 accumulate"


def profiled_traffic(kernel_src, variant, tokens, caps_path=None):
    """DRAM bytes per launch of `variant` from the committed ncu capture
    (profiles/dram_traffic.json: dram__bytes_read.sum + dram__bytes_write.sum
    of one launch at a size whose q and output exceed L2), scaled by the
    tokens a launch processes (q, output and indices all scale with them).
    None when there is no capture or the kernel source changed since."""
    try:
        src = open(os.path.join(ROOT, kernel_src), "rb").read()
        caps = json.load(open(caps_path or os.path.join(ROOT, "profiles", "dram_traffic.json")))
    except (OSError, ValueError):
        return None
    c = caps.get(variant)
    if not c or c.get("source_sha1") != hashlib.sha1(src).hexdigest():
        return None
    return (float(c["dram_bytes_read"]) + float(c["dram_bytes_write"])) * tokens / float(c["tokens"])


def peak_value(peaks, key):
    v = peaks.get(key)
    if isinstance(v, dict):
        v = v.get("value", v.get("median"))
    return float(v) if v is not None else FALLBACK_PEAKS[key]


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.lines = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", str(self.gpu_index)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (FileNotFoundError, OSError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------- workload
def sparse_flops(lens, H):
    return float(sum(int(x) for x in lens)) * H * 2.0 * (576 + 512)


def keys_tok(w):
    from serving_fp8_indexer_gb300 import workloads as wl
    return float((wl.token_positions(w.seqs) + 1).sum())


CASES = {
    # the benchmarked workload: the whole path on the end-to-end chunk
    "chunk": ("e2e_chunk", dict()),
    # the same shapes with one sequence of 1024 new tokens (inputs still
    # larger than L2), for ncu captures
    "chunk_small": ("e2e_chunk", dict(B=1, q_len=1024)),
    # two sequences of 2048 new tokens (4096 tokens: q 604 MB and the output
    # 537 MB exceed L2), for DRAM-traffic captures
    "chunk_4k": ("e2e_chunk", dict(B=2)),
    # the other workloads, stage by stage
    "tiny": ("tiny_prefill", dict()),
    "mtp_decode": ("mtp_decode_indexer", dict()),
    "dsv32": ("dsv32_prefill", dict()),
    "blockwise": ("blockwise_fp8_prefill", dict()),
    # two of its four sequences (3072 tokens), for ncu captures
    "blockwise_small": ("blockwise_fp8_prefill", dict(lens=(1024, 2048))),
    # the other entry points: split-K decode (8 x 2 tokens over 8192 keys),
    # dense short-prompt prefill, and the BF16-cache form of the T=4096 shape
    "decode": ("sparse_decode", dict()),
    "dense": ("dense_prefill", dict()),
    "dsv32_bf16cache": ("dsv32_prefill", dict(latent_bf16=True)),
}
# which attention entry point a case runs (default: smla_sparse_prefill)
CASE_ATTN = {"decode": "decode", "dense": "dense", "dsv32_bf16cache": "bf16cache"}


def make_workload(case="chunk"):
    from serving_fp8_indexer_gb300 import workloads as wl
    fn, kw = CASES[case]
    return getattr(wl, fn)(**kw)


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_sample(w, tokens):
    """The float64 oracle over `tokens` of the workload (whole path);
    returns (seconds, attention FLOPs, keys*tok of those tokens)."""
    import numpy as np
    import oracle
    s = w.seqs
    stride = int(s.kv_len.max() + 3) // 4 * 4
    t0 = time.perf_counter()
    sc = oracle.indexer_scores(w.q_idx, w.q_scale, w.k_pool, w.k_scale, s.cu_q, s.kv_len, s.page_table, s.page_size,
                               stride, tokens=tokens)
    idx, lens = oracle.topk(sc, w.topk, s.cu_q, s.kv_len, s.page_table, s.page_size, tokens=tokens)
    full_idx = np.zeros((int(tokens.max()) + 1, w.topk), np.uint32)
    full_len = np.zeros(int(tokens.max()) + 1, np.uint32)
    full_idx[tokens], full_len[tokens] = idx, lens
    oracle.sparse_prefill(w.q_attn, w.q_dtype, w.latent, w.scales, w.scale_block_size, full_idx, full_len,
                          w.softmax_scale, tokens=tokens)
    dt = time.perf_counter() - t0
    from serving_fp8_indexer_gb300 import workloads as wl
    pos = wl.token_positions(s)
    return dt, sparse_flops(lens, w.H), float((pos[tokens] + 1).sum())


def sample_tokens(w, n, seed=0):
    import numpy as np
    rng = np.random.default_rng(seed)
    return np.sort(rng.choice(w.seqs.T, size=min(n, w.seqs.T), replace=False))


def cpu_baseline(w, budget_s=12.0):
    n = 4
    dt, fl, _ = oracle_sample(w, sample_tokens(w, n, 1))
    per_tok = dt / n
    n2 = int(max(4, min(512, budget_s / max(per_tok, 1e-6))))
    toks = sample_tokens(w, n2, 2)
    dt, fl, _ = oracle_sample(w, toks)
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
            "sample": f"{len(toks)} random tokens of the chunk through the float64 oracle (indexer, top-k, attention), "
                      f"{dt:.1f} s"}


# ----------------------------------------------------------------------------- reference arm
def run_reference(args, rank, world):
    if rank != 0:
        return
    w = make_workload(args.case)
    steps, warm = args.steps, args.warmup
    per_step = 2
    for i in range(warm):
        oracle_sample(w, sample_tokens(w, per_step, 100 + i))
    times, flops = [], []
    for i in range(steps):
        dt, fl, _ = oracle_sample(w, sample_tokens(w, per_step, 1000 + i))
        times.append(dt)
        flops.append(fl)
    value = sum(flops) / sum(times) / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": steps, "warmup": warm, "ms_per_step": 1e3 * sum(times) / steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(w, world),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
                             "sample": f"{per_step} random tokens per step through the float64 oracle"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def config_dict(w, world):
    d = {"workload": w.name, "tokens": int(w.seqs.T), "sequences": int(w.seqs.B),
         "kv_len_max": int(w.seqs.kv_len.max()), "page_size": w.seqs.page_size, "parallelism": f"replicas x{world}"}
    if w.h_idx:
        d.update({"H_idx": w.h_idx, "topk": w.topk})
    if w.H:
        d.update({"H": w.H, "q": "bf16" if w.q_dtype == 0 else "e4m3",
                  "scale_block_size": w.scale_block_size, "v_depth": 512,
                  "indices": "from the indexer + top-k" if w.h_idx else f"sampled top-{w.topk}"})
    big = w.H and w.seqs.T * w.H * 576 * (2 if w.q_dtype == 0 else 1) > (129 << 20)
    d["l2"] = ("inputs larger than L2 (q, out); the latent pool is L2-resident by design" if big else
               "small workload: inputs fit in L2 (launch/latency-bound case)")
    return d


# ----------------------------------------------------------------------------- our arm
class Case:
    """One workload resident on the device, and one step of the path over it
    through the C ABI (indexer -> top-k -> attention, the stages it has)."""

    def __init__(self, name, dev, fused=False):
        import numpy as np
        import torch

        import serving_fp8_indexer_gb300 as smla
        from serving_fp8_indexer_gb300 import workloads as wl
        self.smla, self.torch = smla, torch
        self.name = name
        self.attn = CASE_ATTN.get(name, "sparse")
        self.w = w = make_workload(name)
        s = w.seqs
        self.T, self.H, self.k = s.T, w.H, w.topk
        self.has_idx, self.has_attn = w.h_idx > 0, w.H > 0
        # indexer + top-k through the fused entry point (rows on chip)
        self.fused = fused and self.has_idx
        self.ws = None  # split-K decode workspace
        self.stride = int(s.kv_len.max() + 3) // 4 * 4
        self.pos = wl.token_positions(s)
        self.kt = float((self.pos + 1).sum())
        self.dev = dev
        self.seqs = smla.Seqs.from_host(s, dev)
        self.t_in = {}
        if self.has_idx:
            self.t_in["q_idx"] = torch.from_numpy(w.q_idx).to(dev)
            self.t_in["q_scale"] = torch.from_numpy(w.q_scale).to(dev)
            self.k_pool = torch.from_numpy(w.k_pool).to(dev)
            self.k_scale = torch.from_numpy(w.k_scale).to(dev)
            self.scores = torch.empty((self.T, self.stride), device=dev)
            self.idx = torch.empty((self.T, self.k), dtype=torch.uint32, device=dev)
            self.lens = torch.empty((self.T,), dtype=torch.uint32, device=dev)
        else:
            self.idx = torch.from_numpy(w.indices).to(dev) if w.indices is not None else None
            self.lens = torch.from_numpy(w.topk_lengths).to(dev) if w.topk_lengths is not None else None
        if self.has_attn:
            self.latent = torch.from_numpy(w.latent).to(dev)
            if self.attn == "bf16cache":
                self.latent = self.latent.view(torch.bfloat16)
            if self.attn == "decode":
                n = smla.sparse_decode_workspace_size(self.T, self.H, w.indices.shape[1])
                self.ws = torch.empty(n, dtype=torch.uint8, device=dev) if n else None
            self.scales = None if w.scales is None else torch.from_numpy(w.scales).to(dev)
            if w.q_dtype == wl.Q_BF16:
                self.t_in["q_attn"] = torch.from_numpy(w.q_attn.view(np.int16)).view(torch.bfloat16).to(dev)
            else:
                self.t_in["q_attn"] = torch.from_numpy(w.q_attn).to(dev)
            self.out = torch.empty((self.T, self.H, 512), dtype=torch.bfloat16, device=dev)
        self.stream = torch.cuda.current_stream(dev)
        self.n_kernels = ((1 if self.fused else 2) if self.has_idx else 0) + (
            (2 if self.ws is not None else 1) if self.has_attn else 0)
        if self.attn == "dense":
            attn_len = self.pos + 1
        else:
            attn_len = np.minimum(self.pos + 1, self.k) if self.has_idx else (
                w.topk_lengths.astype(np.int64) if self.has_attn else np.zeros(0))
        self.flops = sparse_flops(attn_len, self.H) if self.has_attn else 0.0

    def step(self, ev=None, tin=None, o=None):
        """One pass of the path.  tin / o: the step's input tensors and result
        (attention output, or the top-k indices for indexer-only workloads);
        default the case's own.  ev: events recorded between the stages."""
        smla, w = self.smla, self.w
        tin = self.t_in if tin is None else tin
        o_idx = o if (o is not None and not self.has_attn) else self.idx
        o_out = o if (o is not None and self.has_attn) else (self.out if self.has_attn else None)
        if ev is not None:
            ev[0].record(self.stream)
        if self.fused:
            smla.indexer_topk(tin["q_idx"], tin["q_scale"], self.k_pool, self.k_scale, self.seqs, self.stride, self.k,
                              o_idx, self.lens)
            if ev is not None:
                ev[1].record(self.stream)
                ev[2].record(self.stream)
        elif self.has_idx:
            smla.indexer_scores(tin["q_idx"], tin["q_scale"], self.k_pool, self.k_scale, self.seqs, self.scores)
            if ev is not None:
                ev[1].record(self.stream)
            smla.topk(self.scores, self.seqs, self.k, o_idx, self.lens)
            if ev is not None:
                ev[2].record(self.stream)
        if self.has_attn:
            if self.attn == "dense":
                smla.dense_prefill(tin["q_attn"], self.latent, self.scales, w.scale_block_size, self.seqs,
                                   w.softmax_scale, o_out)
            elif self.attn == "decode":
                smla.sparse_decode(tin["q_attn"], self.latent, self.scales, w.scale_block_size, o_idx, self.lens,
                                   w.softmax_scale, o_out, self.ws)
            elif self.attn == "bf16cache":
                smla.sparse_prefill_bf16_cache(tin["q_attn"], self.latent, o_idx, self.lens, w.softmax_scale, o_out)
            else:
                smla.sparse_prefill(tin["q_attn"], self.latent, self.scales, w.scale_block_size, o_idx, self.lens,
                                    w.softmax_scale, o_out)
            if ev is not None:
                ev[3].record(self.stream)

    def time_steps(self, steps, warmup, graph=False, world=1, sampler=None):
        """Device time of `steps` steps after `warmup`; returns (total ms,
        per-stage mean ms)."""
        torch = self.torch
        for _ in range(warmup):
            self.step()
        torch.cuda.synchronize(self.dev)
        self.smla.check_device_errors()
        g = None
        if graph:
            # launch-bound workloads: replay one step as a CUDA graph
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self.step()
            g.replay()
            torch.cuda.synchronize(self.dev)
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
        if sampler is not None:
            sampler.start()
            time.sleep(0.3)
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(self.dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(self.stream)
        for i in range(steps):
            if g is not None:
                g.replay()
            else:
                self.step(evs[i])
        e1.record(self.stream)
        torch.cuda.synchronize(self.dev)
        if world > 1:
            torch.distributed.barrier()
        clocks = sampler.stop() if sampler is not None else None
        self.smla.check_device_errors()
        total_ms = e0.elapsed_time(e1)
        stage = {}
        if g is None:
            if self.fused:
                stage["indexer_topk"] = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
            elif self.has_idx:
                stage["indexer"] = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
                stage["topk"] = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
            if self.has_attn:
                a = 2 if self.has_idx else 0
                stage["sparse_mla"] = statistics.mean(e[a].elapsed_time(e[3]) for e in evs)
        return total_ms, stage, clocks

    def e2e(self, steps, world):
        """The same metric through the C ABI from pinned host buffers, host
        copies inside the timed region.  Serving-style pipeline: every step
        copies its inputs in and its result out on copy streams of their own,
        into two device buffer sets used in turn, so step i's copies overlap
        the compute of steps i - 1 and i + 1 (each step's copies stay inside
        the timed region)."""
        import numpy as np
        torch, w = self.torch, self.w
        from serving_fp8_indexer_gb300 import workloads as wl
        host = {name: (torch.from_numpy(w.q_attn.view(np.int16)).view(torch.bfloat16) if name == "q_attn" and
                       w.q_dtype == wl.Q_BF16 else
                       torch.from_numpy({"q_idx": w.q_idx, "q_scale": w.q_scale, "q_attn": w.q_attn}[name])).pin_memory()
                for name in self.t_in}
        res0 = self.out if self.has_attn else self.idx
        h_out = (torch.empty((self.T, self.H, 512), dtype=torch.bfloat16) if self.has_attn else
                 torch.empty((self.T, self.k), dtype=torch.int32)).pin_memory()
        sets = [(self.t_in, res0), ({name: torch.empty_like(x) for name, x in self.t_in.items()},
                                    torch.empty_like(res0))]
        dev, stream = self.dev, self.stream
        h2d, d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        in_ready = [torch.cuda.Event() for _ in range(2)]
        in_free = [torch.cuda.Event() for _ in range(2)]
        out_ready = [torch.cuda.Event() for _ in range(2)]
        out_free = [torch.cuda.Event() for _ in range(2)]
        for b in range(2):  # all buffers start free
            in_free[b].record(stream)
            out_free[b].record(stream)
        # the same K steps as the device-timed loop: the pipeline's fill (the
        # first step's input copy) and drain (the last step's output copy)
        # are inside the timed region once, as for a server loop of K steps
        n_e2e = max(4, steps)

        def e2e_step(i):
            b = i % 2
            tin, res = sets[b]
            with torch.cuda.stream(h2d):
                h2d.wait_event(in_free[b])
                for name, ht in host.items():
                    tin[name].copy_(ht, non_blocking=True)
                in_ready[b].record(h2d)
            stream.wait_event(in_ready[b])
            stream.wait_event(out_free[b])
            self.step(tin=tin, o=res)
            in_free[b].record(stream)
            out_ready[b].record(stream)
            with torch.cuda.stream(d2h):
                d2h.wait_event(out_ready[b])
                h_out.copy_(res if self.has_attn else res.view(torch.int32), non_blocking=True)
                out_free[b].record(d2h)

        for i in range(2):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        a = torch.cuda.Event(enable_timing=True)
        b_ev = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        h2d.wait_event(a)
        d2h.wait_event(a)
        for i in range(n_e2e):
            e2e_step(i)
        stream.wait_stream(d2h)  # the last result is back on the host
        b_ev.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = a.elapsed_time(b_ev) / n_e2e
        if world > 1:
            e2e_ms = max_over_ranks([e2e_ms], dev)[0]
        self.smla.check_device_errors()
        bi = sum(ht.numel() * ht.element_size() for ht in host.values())
        bo = h_out.numel() * h_out.element_size()
        ev = weak_scaling_value(world, self.flops if self.has_attn else self.kt, e2e_ms)
        return {"value": ev / 1e12 if self.has_attn else ev, "unit": "TFLOP/s" if self.has_attn else "keys·tok/s",
                "h2d_bytes_per_step": int(bi), "d2h_bytes_per_step": int(bo), "ms_per_step": e2e_ms}

    def free(self):
        for name in [n for n in vars(self) if isinstance(getattr(self, n), self.torch.Tensor)]:
            setattr(self, name, None)
        self.t_in = {}
        self.torch.cuda.empty_cache()


def attn_peaks(peaks, src, fp8_q, timed_s):
    """(peak TFLOP/s of the attention's logical dtype, label): bf16 for bf16 q,
    FP8 = 2 x the bf16 figure (the nominal ratio) for e4m3 q.  The burst bf16
    figure applies to a timed region under a second, the sustained one to a
    longer region."""
    key = "bf16_tflops" if timed_s < 1.0 else "bf16_tflops_sustained"
    bf16 = peak_value(peaks, key)
    kind = "burst" if key == "bf16_tflops" else "sustained"
    if fp8_q:
        return 2.0 * bf16, f"{src} fp8 dense = 2 x bf16 ({kind})"
    return bf16, f"{src} bf16 dense ({kind})"


# Issued tcgen05 MMA work per unit of the method's FLOPs, by path: bf16 q and
# the bf16-accuracy P each run as two e4m3 terms, and blockwise-scaled rows as
# two e4m3 terms (hi + lo), so the FP8 pipe executes twice the logical
# FLOPs on those paths (QK and PV alike); native e4m3 runs them once.
def issued_ratio(w):
    from serving_fp8_indexer_gb300 import workloads as wl
    if w.q_dtype == wl.Q_BF16:
        return 2.0
    if 0 < w.scale_block_size < 576:
        return 2.0
    return 1.0


def attn_variant(w):
    from serving_fp8_indexer_gb300 import workloads as wl
    q = "bf16 q" if w.q_dtype == wl.Q_BF16 else "e4m3 q"
    sc = {0: "unit scale"}.get(w.scale_block_size, "tensorwise scale" if w.scale_block_size >= 576 else
                               f"blockwise-{w.scale_block_size} scale")
    return f"prefill_kernel, {q}, {sc}, H={w.H}"


def run_ours(args, rank, world):
    import torch

    from serving_fp8_indexer_gb300 import build as smla_build
    smla_build.build()

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    # the step: indexer -> top-k -> attention (--fused: indexer + top-k as one
    # kernel with the score rows on chip)
    c = Case(args.case, dev, fused=args.fused)
    w = c.w
    sampler = ClockSampler(int(os.environ.get("LOCAL_RANK", 0)))
    total_ms, stage, clocks = c.time_steps(args.steps, args.warmup, graph=args.graph, world=world, sampler=sampler)
    if world > 1:
        keys = sorted(stage)
        red = max_over_ranks([total_ms] + [stage[x] for x in keys], dev)
        total_ms = red[0]
        for i, x in enumerate(keys):
            stage[x] = red[i + 1]
    ms_step = total_ms / args.steps
    e2e = None if args.no_e2e else c.e2e(args.steps, world)
    c_flops, n_kernels = c.flops, c.n_kernels
    # the other form of indexer + top-k on the same inputs
    other_form = {}
    if c.has_idx and not args.graph:
        c.fused = not c.fused
        _, ost, _ = c.time_steps(max(5, args.steps // 2), 2)
        other_form = ost
        c.fused = not c.fused

    # the other workloads, in the same launch configuration as the tests
    extra = {}
    if not args.no_extra and args.case == "chunk":
        c.free()
        del c
        for name, graph in (("dsv32", False), ("blockwise", False), ("dsv32_bf16cache", False), ("dense", False),
                            ("decode", True), ("mtp_decode", True), ("tiny", True)):
            reps = max(5, args.steps // 2) if not graph else 200
            # workloads with an indexer run both forms of indexer + top-k (the
            # fused kernel wins for two tokens a sequence at H_idx 64, the pair
            # for the tiny workload's 32-token tiles at H_idx 4); the faster
            # one is reported, the other beside it
            forms = {}
            for fused in ((True, False) if name in ("mtp_decode", "tiny") else (True,)):
                x = Case(name, dev, fused=fused)
                t, st, _ = x.time_steps(reps, args.warmup, graph=graph)
                forms[fused] = (x, t / reps, st)
                x.free()
            best = min(forms, key=lambda f: forms[f][1])
            extra[name] = forms[best] + ({f: forms[f][1] for f in forms},)
    if rank != 0:
        return
    peaks, src = load_peaks()
    hbm = peak_value(peaks, "hbm_gbs")
    fp8_peak_burst = 2.0 * peak_value(peaks, "bf16_tflops")
    fp8_q = w.q_dtype == 1
    stages = {}
    kt = c_kt(w)
    fused_ms = stage.get("indexer_topk", other_form.get("indexer_topk"))
    if fused_ms:
        tf_idx = 1e-12 * kt * w.h_idx * 256 / (fused_ms * 1e-3)
        stages["fused_indexer_topk"] = {"ms": fused_ms, "keys_tok_per_s": kt / (fused_ms * 1e-3),
                                        "indexer_TFLOP/s": tf_idx, "frac_fp8_peak": tf_idx / fp8_peak_burst,
                                        "entry": "smla_indexer_topk (score rows on chip)",
                                        "in_step": "indexer_topk" in stage}
    if "indexer" in stage or "indexer" in other_form:
        u = stage if "indexer" in stage else other_form
        idx_bytes = w.q_idx.nbytes + w.q_scale.nbytes + w.k_pool.nbytes + w.k_scale.nbytes + 4 * kt
        tf_idx = 1e-12 * kt * w.h_idx * 256 / (u["indexer"] * 1e-3)
        topk_bytes = 4 * kt + 4 * w.seqs.T * w.topk + 4 * w.seqs.T
        gbs = 1e-9 * topk_bytes / (u["topk"] * 1e-3)
        stages["indexer"] = {"ms": u["indexer"], "TFLOP/s": tf_idx, "frac_fp8_peak": tf_idx / fp8_peak_burst,
                             "GB/s_algorithmic": 1e-9 * idx_bytes / (u["indexer"] * 1e-3), "in_step": "indexer" in stage}
        stages["topk"] = {"ms": u["topk"], "GB/s_algorithmic": gbs, "frac_hbm": gbs / hbm, "in_step": "topk" in stage}
    flops = c_flops
    if "sparse_mla" in stage:
        tf = flops / (stage["sparse_mla"] * 1e-3) / 1e12
        peak, pname = attn_peaks(peaks, src, fp8_q, total_ms * 1e-3)
        fp8_attn_peak = peak if fp8_q else 2.0 * peak
        r = issued_ratio(w)
        stages["sparse_mla"] = {"ms": stage["sparse_mla"], "TFLOP/s": tf, "frac_peak": tf / peak,
                                "peak_dtype": "fp8" if fp8_q else "bf16"}
    if w.H:
        value, unit = weak_scaling_value(world, flops, ms_step) / 1e12, "TFLOP/s"
    else:
        value, unit = weak_scaling_value(world, kt, ms_step), "keys·tok/s"
    line = {
        "metric": METRIC,
        "value": value,
        "unit": unit,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": dtype_label(w),
        "data": "synthetic",
        "config": config_dict(w, world),
        "stages": stages,
        "gpu_launches": n_kernels * args.steps,
        "clocks": clocks,
    }
    line["config"]["step"] = ("smla_indexer_topk -> smla_sparse_prefill" if args.fused else
                              "smla_indexer_scores -> smla_topk -> smla_sparse_prefill")
    if args.graph:
        line["config"]["launch"] = "CUDA graph replay of one step"
    if w.h_idx:
        ms_it = stage.get("indexer_topk", stage.get("indexer", 0.0) + stage.get("topk", 0.0)) or ms_step
        line["indexer_topk"] = {"value": world * kt / (ms_it * 1e-3), "unit": "keys·tok/s"}
    if "sparse_mla" in stage:
        tf = stages["sparse_mla"]["TFLOP/s"]
        traffic = profiled_traffic("serving_fp8_indexer_gb300/csrc/prefill.cu", attn_variant(w), int(w.seqs.T))
        line["roofline"] = {"bound": "tensor", "kernel": "prefill_kernel (sparse MLA)", "achieved": tf,
                            "peak": peak, "unit": "TFLOP/s", "frac": tf / peak, "traffic": traffic,
                            "peak_source": pname,
                            # the MMAs actually issued run on the FP8 pipe: their FLOPs
                            # (r x the method's) against the FP8 peak
                            "issued": {"mma": "tcgen05 kind::f8f6f4 (e4m3)", "flops_per_logical_flop": r,
                                       "achieved": tf * r, "peak": fp8_attn_peak,
                                       "frac": tf * r / fp8_attn_peak}}
    elif "topk" in stage:
        line["roofline"] = {"bound": "hbm", "kernel": "topk_kernel", "achieved": stages["topk"]["GB/s_algorithmic"],
                            "peak": hbm, "unit": "GB/s", "frac": stages["topk"]["frac_hbm"], "traffic": None,
                            "peak_source": f"{src} HBM copy"}
    if extra:
        line["other_workloads"] = {}
        for name, (x, ms_rep, st, form_ms) in extra.items():
            xw = x.w
            d = {"workload": xw.name, "entry": {"sparse": "smla_sparse_prefill", "dense": "smla_dense_prefill",
                                                "decode": "smla_sparse_decode (split-K)",
                                                "bf16cache": "smla_sparse_prefill_bf16_cache"}[x.attn]
                 if xw.H else ("smla_indexer_topk" if x.fused else "smla_indexer_scores + smla_topk"),
                 "dtype": dtype_label(xw)}
            if x.has_idx:
                d["indexer_topk_form"] = "fused (smla_indexer_topk)" if x.fused else "pair (smla_indexer_scores + smla_topk)"
                if len(form_ms) > 1:
                    d["whole_path_ms_by_form"] = {("fused" if f else "pair"): v for f, v in form_ms.items()}
            if x.has_attn:
                ms = st.get("sparse_mla", ms_rep)
                xfp8 = xw.q_dtype == 1
                pk, pn = attn_peaks(peaks, src, xfp8, ms * 1e-3 * max(5, args.steps // 2))
                tf = x.flops / (ms * 1e-3) / 1e12
                d.update({"stage": "attention", "ms": ms, "TFLOP/s": tf, "frac_peak": tf / pk, "peak_source": pn})
                if x.attn != "bf16cache":
                    d["issued_frac_fp8"] = tf * issued_ratio(xw) / (pk if xfp8 else 2.0 * pk)
            if x.has_idx and not x.has_attn:
                d.update({"stage": "indexer + top-k", "ms": ms_rep, "keys_tok_per_s": x.kt / (ms_rep * 1e-3)})
            if x.has_idx and x.has_attn:
                d["whole_path_ms"] = ms_rep
            if name in ("decode", "mtp_decode", "tiny"):
                d["launch"] = "CUDA graph replay, 200 steps (launch-latency regime)"
            line["other_workloads"][name] = d
    if e2e is not None:
        line["e2e"] = e2e
    if world == 1 and not args.no_cpu_baseline and args.case == "chunk":
        line["cpu_baseline"] = cpu_baseline(w)
    print(json.dumps(line), flush=True)


def c_pos(w):
    from serving_fp8_indexer_gb300 import workloads as wl
    return wl.token_positions(w.seqs)


def c_kt(w):
    return float((c_pos(w) + 1).sum())


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--case", choices=sorted(CASES), default="chunk")
    ap.add_argument("--graph", action="store_true", help="replay each step as a CUDA graph")
    ap.add_argument("--no-extra", action="store_true", help="skip the other workloads")
    ap.add_argument("--fused", action="store_true", help="indexer + top-k as one kernel (score rows on chip)")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.gpus != world:
        sys.exit(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world}; launch N > 1 ranks with "
                 f"torch.distributed.run --nproc-per-node {args.gpus}")
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        torch.distributed.init_process_group("nccl")
    try:
        run_ours(args, rank, world)
    finally:
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()

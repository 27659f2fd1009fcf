"""The multi-replica timing of bench.py on CPU: two gloo ranks, each with
its own timings; the reported step time is the slowest rank's and the value
counts every rank's work (weak scaling, no data-path collective)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r's timings: total 10 + r ms, stage 5 - r ms
        red = bench.max_over_ranks([10.0 + rank, 5.0 - rank], "cpu")
        out[rank] = red
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == [11.0, 5.0] and res[1] == [11.0, 5.0]


def test_single_rank_is_identity_and_weak_scaling_value():
    assert bench.max_over_ranks([3.0, 4.5], "cpu") == [3.0, 4.5]
    # 2 replicas, each 9.346 TFLOP per step in 12 ms -> 2 x 779 TFLOP/s
    v = bench.weak_scaling_value(2, 9.346e12, 12.0) / 1e12
    assert v == pytest.approx(2 * 9.346 / 0.012)


def test_reference_arm_other_ranks_do_nothing():
    class A:
        pass
    # ranks other than 0 return at once without touching the oracle
    assert bench.run_reference(A(), 1, 2) is None


def test_profiled_traffic_scales_a_capture_of_the_current_source(tmp_path):
    # a capture of the current kernel source gives read + write bytes scaled
    # by tokens; a capture of another source (sha1 mismatch) gives None
    import hashlib
    import json
    src = "serving_fp8_indexer_gb300/csrc/prefill.cu"
    sha = hashlib.sha1(open(os.path.join(bench.ROOT, src), "rb").read()).hexdigest()
    cap = {"v": {"tokens": 4096, "dram_bytes_read": 1.0e9, "dram_bytes_write": 0.5e9, "source_sha1": sha},
           "old": {"tokens": 4096, "dram_bytes_read": 1.0e9, "dram_bytes_write": 0.5e9, "source_sha1": "0" * 40}}
    f = tmp_path / "caps.json"
    f.write_text(json.dumps(cap))
    assert bench.profiled_traffic(src, "v", 16384, str(f)) == pytest.approx(6.0e9)
    assert bench.profiled_traffic(src, "old", 16384, str(f)) is None
    assert bench.profiled_traffic(src, "missing", 16384, str(f)) is None


def test_gpus_flag_must_match_world_size():
    import subprocess
    import sys
    r = subprocess.run([sys.executable, os.path.join(bench.ROOT, "bench.py"), "--gpus", "2"], capture_output=True,
                       text=True, env={**os.environ, "WORLD_SIZE": "1"})
    assert r.returncode != 0 and "WORLD_SIZE" in r.stderr


def test_dtype_labels_follow_the_workload():
    from serving_fp8_indexer_gb300 import workloads as wl
    assert "bf16 q" in bench.dtype_label(bench.make_workload("tiny"))
    assert "blockwise" in bench.dtype_label(bench.make_workload("blockwise_small"))
    assert "indexer" in bench.dtype_label(bench.make_workload("mtp_decode"))
    assert wl.Q_E4M3 != wl.Q_BF16

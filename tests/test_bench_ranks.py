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


def test_profiled_traffic_reads_the_committed_capture(tmp_path):
    # the committed capture of the current kernel source parses to read + write
    # bytes scaled by tokens; another source (sha1 mismatch) gives None
    t = bench.profiled_traffic("serving_fp8_indexer_gb300/csrc/prefill.cu",
                               "profiles/prefill_kernel_chunk_small.md", 1024, 16384)
    assert t is not None and 3.0e9 < t < 5.0e9
    md = tmp_path / "p.md"
    md.write_text("sha1 0000\n| `dram__bytes_read.sum` / `dram__bytes_write.sum` | 1.0 MB / 2.0 MB |\n")
    assert bench.profiled_traffic("serving_fp8_indexer_gb300/csrc/prefill.cu", str(md), 1, 2) is None


def test_dtype_labels_follow_the_workload():
    from serving_fp8_indexer_gb300 import workloads as wl
    assert "bf16 q" in bench.dtype_label(bench.make_workload("tiny"))
    assert "blockwise" in bench.dtype_label(bench.make_workload("blockwise_small"))
    assert "indexer" in bench.dtype_label(bench.make_workload("mtp_decode"))
    assert wl.Q_E4M3 != wl.Q_BF16

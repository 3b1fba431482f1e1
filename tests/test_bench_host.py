"""Host-side logic of bench.py: the algorithmic work counts (closed forms for the
workloads) and the replica aggregation over ranks under torch.distributed (gloo,
world size 2, on CPU)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from relative_bias_hybrid_gb300 import inputs as gen


def test_sliding_window_pair_count_closed_form():
    w = gen.workload("swa")
    # sum_{i<8192} min(i+1, 4096) = 4096*4097/2 + 4096*4096
    assert bench.visible_pairs(w) == 4096 * 4097 // 2 + 4096 * 4096 == 25_167_872
    assert bench.biased_pairs(w) == 512 * 513 // 2 + (8192 - 512) * 512
    assert bench.attention_flops(w) == pytest.approx(8.247e11 + 1.664e10, rel=2e-3)


def test_full_layer_pair_count_closed_form():
    w = gen.workload("full")
    assert bench.visible_pairs(w) == 32768 * 32769 // 2 == 536_887_296


def test_decode_bytes_and_prologue_bytes():
    w = gen.workload("decode")
    # K+V of 32 sequences x 8 KV heads x 32768 keys x 128 x bf16 = 4 GiB, plus small terms
    assert bench.decode_bytes(w) == pytest.approx(4.314e9, rel=1e-3)
    s = gen.workload("swa")
    assert bench.prologue_bytes(s) == 40_964 * 8192 + 2 * 2 * 3 * 1024 * 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE="2")
    dist.init_process_group("gloo", rank=rank, world_size=2)
    ms, units = bench.aggregate_over_ranks(10.0 + rank * 5.0, 100.0 * (rank + 1), 2)
    q.put((rank, ms, units))
    dist.destroy_process_group()


def test_replica_aggregation_gloo_world_2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for _, ms, units in res:
        assert ms == 15.0          # max over ranks
        assert units == 300.0      # total over ranks

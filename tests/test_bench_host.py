"""Host-side checks of the benchmark: its byte accounting against the KV-size
formula the pages print, and the replica timing across ranks (world size 2,
gloo, CPU)."""
import math
import os

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from fp8_quantised_paged_gb300 import workloads as W


def test_llama_layer_accounting():
    w = W.make_workload(2, "full")
    acc = bench.accounting(w)
    # codes: K and V, 8 kv heads x 128 dims, 1 byte each; scales: 4 B per
    # (token, kv head) for K and V
    assert acc["bytes_per_token"] == 2 * 8 * 128 + 2 * 8 * 4 == 2112
    assert acc["kv_tokens"] == 12 * 16384
    assert acc["split"] == 196608 * 2112 + 12 * 64 * 128 * 2 + 12 * 1024 * 4 + 12 * 4
    # "Llama 3 70B FP8 deployment" (dpshk.com/news/5605006) sec. 2.2: KV bytes =
    # 2 x layers(80) x kv heads(8) x head_dim(128) x tokens x 2 bytes (bf16),
    # about 2.6 GB at 8K.  Our per-token code bytes are the FP8 half of it.
    codes_per_token_layer = 2 * w.n_kv_heads * w.head_dim
    bf16_8k = codes_per_token_layer * 2 * 80 * 8192
    assert bf16_8k == 2 * 80 * 8 * 128 * 8192 * 2
    assert abs(bf16_8k / 2 ** 30 - 2.6) < 0.1 * 2.6 or abs(bf16_8k / 1e9 - 2.6) < 0.1 * 2.6


def test_mla_and_static_accounting():
    w5 = W.make_workload(5, "full")
    assert bench.accounting(w5)["bytes_per_token"] == 576 + 9 * 4
    w4 = W.make_workload(4, "full")
    a4 = bench.accounting(w4)
    assert a4["bytes_per_token"] == 2 * 8 * 128
    assert a4["split"] >= a4["kv_tokens"] * 2048 + 2 * 8 * 128 * 4


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q.put((rank, bench.max_over_ranks(1.5 + rank, "cpu")))
    finally:
        dist.destroy_process_group()


def test_replica_time_is_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 1000)
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == {0: 2.5, 1: 2.5}


def test_single_process_time_passes_through():
    assert bench.max_over_ranks(3.25, "cpu") == 3.25

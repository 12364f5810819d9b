"""Host-side logic of the benchmark: algorithmic work counts and the max-over-ranks reduction
(world size 2 over gloo, on the CPU)."""

import os
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from workloads import random_small_batch  # noqa: E402


def test_workload_counts_by_brute_force():
    b = random_small_batch(3, page_size=4, num_q_heads=4, num_kv_heads=2, head_dim=16,
                           decode_lens=(5, 9, 12), extend=((3, 4), (0, 6)), share_decode_prefix=4)
    c = bench.workload_counts(b)
    # unique physical slots read by the decodes, by brute force
    seen = set()
    total = 0
    ind, idx = b.dec_kv_indptr.tolist(), b.dec_kv_indices.tolist()
    for r, L in enumerate(b.dec_kv_lens.tolist()):
        for j in range(L):
            seen.add(idx[ind[r] + j // 4] * 4 + j % 4)
            total += 1
    assert c["decode_kv_tokens_unique"] == len(seen)
    assert c["decode_kv_tokens_logical"] == total
    assert len(seen) < total  # the shared prefix is counted once
    # unmasked (query, key) pairs of the extends, by brute force
    pairs = 0
    qo = b.ext_qo_indptr.tolist()
    for r, P in enumerate(b.ext_prefix_lens.tolist()):
        for i in range(qo[r + 1] - qo[r]):
            pairs += P + i + 1
    assert c["extend_pairs"] == pairs
    assert c["extend_flops"] == 4 * 16 * 4 * pairs
    assert c["attn_tokens"] == 3 + qo[-1]


def _worker(rank, world, port, q):
    import torch.distributed as dist

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    out = bench.max_over_ranks([1.0 + rank, 10.0 - rank])
    q.put((rank, out))
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 1000)
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
    assert res[0] == [2.0, 10.0] and res[1] == [2.0, 10.0]


def test_max_over_ranks_without_group():
    assert bench.max_over_ranks([3.0, 4.0]) == [3.0, 4.0]

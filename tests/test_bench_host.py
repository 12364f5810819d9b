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


def test_extend_bytes_and_cascade_counts_by_brute_force():
    from paged_kv_attention_10_gb300.cascade import plan_shared_prefix

    b = random_small_batch(4, page_size=4, num_q_heads=4, num_kv_heads=2, head_dim=16,
                           decode_lens=(21, 30, 26, 7), extend=((8, 4), (0, 6)),
                           share_decode_prefix=16, share_extend_prefix=8)
    c = bench.workload_counts(b)
    row = 2 * 16 * 2  # one token's K (or V) row: Hkv x D x bf16
    # extend: each physical slot of the extend requests once (the shared prefix once), K and V,
    # plus q in, out and lse, plus the page lists
    seen = set()
    ind, idx = b.ext_kv_indptr.tolist(), b.ext_kv_indices.tolist()
    qo = b.ext_qo_indptr.tolist()
    for r, P in enumerate(b.ext_prefix_lens.tolist()):
        for j in range(P + qo[r + 1] - qo[r]):
            seen.add(idx[ind[r] + j // 4] * 4 + j % 4)
    meta = (len(ind) + len(idx) + 2 * len(qo) - 1) * 4
    assert c["extend_bytes"] == len(seen) * row * 2 + qo[-1] * 4 * (16 * 2 * 2 + 4) + meta
    # cascade: the shared-prefix parts' unmasked pairs, the own-pages decode's unique slots
    sharers = [i for i, r in enumerate(b.requests) if r.kind == "decode" and r.share_group == 0]
    assert sharers == [0, 1, 2]
    plan = plan_shared_prefix(b.dec_kv_indptr, b.dec_kv_indices, b.dec_kv_lens, [(0, 3)], 4,
                              num_kv_heads=2, group_size=2, num_sms=1, min_chunk_tokens=4)
    cc = bench.cascade_counts(b, plan)
    assert plan.shared_tokens == [16]
    assert cc["prefix_flops"] == 4 * 16 * 4 * (3 * 16)  # 3 queries x 16 shared positions, all heads
    own = set()
    sptr, sidx = plan.suffix_kv_indptr.tolist(), plan.suffix_kv_indices.tolist()
    for r, L in enumerate(plan.suffix_kv_lens.tolist()):
        for j in range(L):
            own.add(sidx[sptr[r] + j // 4] * 4 + j % 4)
    B = b.num_decode
    meta = (len(sptr) + len(sidx) + B) * 4
    assert cc["suffix_bytes"] == len(own) * row * 2 + B * 4 * (16 * 2 * 2 + 4) + meta
    S = plan.num_splits
    assert cc["merge_bytes"] == (S + 2) * B * 4 * (16 * 2 + 4)


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


def test_reference_arm_json_contract():
    """`bench.py --impl reference` (the oracle on the host cores) prints one JSON line with the
    contract's keys, for the workload asked for."""
    import json
    import subprocess

    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3", "--workload", "tiny"], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in line, k
    assert line["impl"] == "reference" and line["n_gpus"] == 1 and line["value"] > 0
    assert line["config"]["workload"].startswith("tiny")
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"], "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_decode_shared_tokens_match_the_page_lists():
    """The decode's L2 keep hint the benchmark passes: each decode request's count of leading
    positions whose physical pages another request of the step also lists (brute force over the
    page lists), on the mixed-step shape and a small batch."""
    from workloads import make_config

    for b in (make_config(5), random_small_batch(5, page_size=16, num_q_heads=8, num_kv_heads=2,
                                                 head_dim=64, decode_lens=(40, 700, 900, 90),
                                                 share_decode_prefix=32)):
        ind, idx = b.dec_kv_indptr.tolist(), b.dec_kv_indices.tolist()
        pages = [idx[ind[r]:ind[r + 1]] for r in range(b.num_decode)]
        owners = {}
        for r, pl in enumerate(pages):
            for p in pl:
                owners.setdefault(p, set()).add(r)
        hint = b.dec_shared_tokens.tolist()
        for r, pl in enumerate(pages):
            n = 0
            while n < len(pl) and len(owners[pl[n]]) > 1:
                n += 1
            assert hint[r] == n * b.page_size, (r, hint[r], n)
        assert sum(1 for h in hint if h > 0) >= 2

"""Shared-prefix (cascade) attention on the GPU against the fp64 oracle: the shared-prefix parts
element by element, the merge of bf16 partial states, and the whole cascade decode (parts, a
decode over each request's own pages, merge) against the plain decode of the oracle."""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_10_gb300.cascade import plan_shared_prefix
from workloads import random_small_batch
from workloads.paged import RequestSpec, build_paged_batch
from _gpu_helpers import assert_attention_close

pytestmark = pytest.mark.gpu


def _pool_batch(seed, ps, Hq, Hkv, lens, D=128):
    """Page lists of the given lengths over a NaN-filled pool (unused slots poison any stray read)."""
    b = random_small_batch(seed, page_size=ps, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                           decode_lens=lens, decode_new=0)
    return b


@pytest.mark.parametrize("ps,Hq,Hkv,D", [(16, 32, 8, 128), (8, 8, 8, 128), (64, 16, 2, 128), (32, 16, 16, 128),
                                         (16, 14, 2, 64), (16, 12, 2, 128), (1, 16, 8, 128), (24, 14, 2, 64)])
def test_shared_prefix_parts_match_oracle(lib, ps, Hq, Hkv, D):
    lens = (700, 64, 129, 1, 300, 2000)
    b = _pool_batch(90 + ps + Hq, ps, Hq, Hkv, lens, D)
    G = Hq // Hkv
    tpt = 128 // G
    g = torch.Generator().manual_seed(ps * 7 + Hq)
    Nq = 3 * tpt + 5
    q = torch.randn((Nq, Hq, D), generator=g).to(torch.bfloat16)
    # parts: (q_start, q_len, kv length used of page list p); list 3 is cut to 0 (an empty part)
    spec = [(0, Nq, 700), (5, 2 * tpt + 1, 64), (tpt - 3, 7, 129), (Nq - 1, 1, 0), (1, tpt, 300),
            (2, tpt + 9, 1999)]
    q_start = [s for s, _, _ in spec]
    q_len = [n for _, n, _ in spec]
    kv_lens = [L for _, _, L in spec]
    o_start, cur = [], 3
    for n in q_len:  # disjoint output rows, with gaps that must stay untouched
        o_start.append(cur)
        cur += n + 2
    n_out = cur
    i32 = lambda v: torch.tensor(v, dtype=torch.int32)
    kp, vp = b.k_pool, b.v_pool  # decode_new = 0: the pool as drawn
    o_ref, l_ref = oracle.shared_prefix_attention(q, kp, vp, i32(q_start), i32(q_len), i32(o_start),
                                                  b.dec_kv_indptr, b.dec_kv_indices, i32(kv_lens),
                                                  n_out, ps, b.sm_scale)
    o = torch.full((n_out, Hq, D), 7.0, dtype=torch.bfloat16, device="cuda")
    l = torch.full((n_out, Hq), 7.0, dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    d = lambda t: t.cuda()
    lib.shared_prefix_attention(d(q), d(kp), d(vp), d(i32(q_start)), d(i32(q_len)), d(i32(o_start)),
                                d(b.dec_kv_indptr), d(b.dec_kv_indices), d(i32(kv_lens)), max(q_len),
                                b.sm_scale, o, l, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    written = ~np.isnan(l_ref[:, 0])
    rows = np.nonzero(written)[0]
    empty = np.arange(o_start[3], o_start[3] + q_len[3])
    assert (o.cpu()[torch.tensor(empty)] == 0).all() and torch.isneginf(l.cpu()[torch.tensor(empty)]).all()
    full = np.setdiff1d(rows, empty)
    assert_attention_close(o, l, o_ref, l_ref, rows=full, what=f"shared prefix ps={ps} G={G}")
    untouched = torch.tensor(np.nonzero(~written)[0])
    assert (o.cpu()[untouched] == 7.0).all() and (l.cpu()[untouched] == 7.0).all()


def test_shared_prefix_row_out_of_range_is_reported(lib):
    b = _pool_batch(5, 16, 32, 8, (200, 300))
    q = torch.randn((40, 32, 128), generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    i32 = lambda v: torch.tensor(v, dtype=torch.int32).cuda()
    o = torch.zeros((80, 32, 128), dtype=torch.bfloat16, device="cuda")
    l = torch.zeros((80, 32), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    # part 0 reads rows 30..49 of a 40-row q: skipped and reported; part 1 is computed
    lib.shared_prefix_attention(q.cuda(), b.k_pool.cuda(), b.v_pool.cuda(), i32([30, 0]), i32([20, 10]),
                                i32([0, 50]), b.dec_kv_indptr.cuda(), b.dec_kv_indices.cuda(),
                                i32([200, 300]), 20, b.sm_scale, o, l, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & lib.DEVERR_ROW_OOB
    assert (o[:20].cpu() == 0).all()
    o_ref, l_ref = oracle.shared_prefix_attention(q, b.k_pool, b.v_pool, torch.tensor([0], dtype=torch.int32),
                                                  torch.tensor([10], dtype=torch.int32),
                                                  torch.tensor([50], dtype=torch.int32),
                                                  b.dec_kv_indptr[1:] - b.dec_kv_indptr[1],
                                                  b.dec_kv_indices[int(b.dec_kv_indptr[1]):],
                                                  torch.tensor([300], dtype=torch.int32), 80, 16, b.sm_scale)
    assert_attention_close(o, l, o_ref, l_ref, rows=np.arange(50, 60), what="part after a skipped one")


@pytest.mark.parametrize("S,N,H", [(2, 5, 8), (5, 33, 32)])
def test_merge_bf16_partials(lib, S, N, H):
    g = torch.Generator().manual_seed(S + N)
    o = (torch.randn((S, N, H, 128), generator=g) * 0.25).to(torch.bfloat16)
    l = torch.randn((S, N, H), generator=g) * 3
    l[0, 0, 0] = -float("inf")
    l[:, -1, -1] = -float("inf")
    out, lse = lib.merge_states(o.cuda(), l.cuda())
    o_ref, lse_ref = oracle.merge_states(o.double().numpy(), l.double().numpy())
    fin = np.isfinite(lse_ref)
    assert np.all(np.isneginf(lse.cpu().numpy()[~fin]))
    assert torch.all(out.float().cpu()[torch.tensor(~fin)] == 0)
    assert_attention_close(out.reshape(N * H, 128), lse.reshape(-1), o_ref.reshape(N * H, 128),
                           lse_ref.reshape(-1), rows=np.nonzero(fin.reshape(-1))[0], what="bf16 merge")


def _grouped_batch(seed, groups, loners, ps=16, Hq=32, Hkv=8):
    """Decode requests in contiguous share groups [(count, shared_tokens, (lo, hi))] followed by
    unshared requests with lengths in ``loners``."""
    gen = torch.Generator().manual_seed(seed)
    reqs, shared = [], {}
    for gid, (count, st, (lo, hi)) in enumerate(groups):
        shared[gid] = st
        for _ in range(count):
            L = int(torch.randint(max(lo, st + 1), hi + 1, (1,), generator=gen))
            reqs.append(RequestSpec("decode", L, 1, share_group=gid))
    for L in loners:
        reqs.append(RequestSpec("decode", L, 1))
    return build_paged_batch(gen, reqs, name=f"cascade-{seed}", page_size=ps, num_q_heads=Hq,
                             num_kv_heads=Hkv, head_dim=128, shared_tokens=shared)


@pytest.mark.parametrize("case", ["two-groups", "one-big-group"])
def test_cascade_decode_matches_oracle(lib, case):
    if case == "two-groups":
        b = _grouped_batch(11, [(5, 512, (513, 900)), (40, 1024, (1025, 1400))], (33, 700, 1))
        groups = [(0, 5), (5, 40)]
    else:
        b = _grouped_batch(12, [(150, 2048, (2049, 2300))], (17, 90))
        groups = [(0, 150)]
    kp, vp = oracle.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.slot_mapping, b.page_size)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    plan = plan_shared_prefix(b.dec_kv_indptr, b.dec_kv_indices, b.dec_kv_lens, groups, b.page_size,
                              num_kv_heads=b.num_kv_heads, group_size=b.num_q_heads // b.num_kv_heads,
                              num_sms=sms)
    assert len(plan.shared_tokens) == len(groups) and plan.num_splits >= 1
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = lib.cascade_decode(b.dec_q.cuda(), kp.cuda(), vp.cuda(), plan.to("cuda"), b.sm_scale,
                                  err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    B = b.num_decode
    check = sorted(set(range(0, B, max(1, B // 24))) | {B - 1, 4, 5})
    o_ref, l_ref = oracle.paged_decode(b.dec_q, kp, vp, b.dec_kv_indptr, b.dec_kv_indices, b.dec_kv_lens,
                                       b.page_size, b.sm_scale, requests=check)
    assert_attention_close(out, lse, o_ref, l_ref, rows=np.array(check), what=f"cascade {case}")


@pytest.mark.slow
def test_cascade_full_shared_prefix_workload(lib):
    """The shared-prefix workload at full size (256 decodes over a 4096-token shared prefix), planned
    as the benchmark plans it, on a sample of requests."""
    from workloads import make_shared_prefix_decode

    b = make_shared_prefix_decode()
    kp, vp = oracle.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.slot_mapping, b.page_size)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    plan = plan_shared_prefix(b.dec_kv_indptr, b.dec_kv_indices, b.dec_kv_lens, [(0, b.num_decode)],
                              b.page_size, num_kv_heads=b.num_kv_heads,
                              group_size=b.num_q_heads // b.num_kv_heads, num_sms=sms)
    assert plan.shared_tokens == [4096] and plan.num_splits > 1
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = lib.cascade_decode(b.dec_q.cuda(), kp.cuda(), vp.cuda(), plan.to("cuda"), b.sm_scale,
                                  err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rng = np.random.default_rng(1)
    sample = sorted(rng.choice(b.num_decode, 24, replace=False).tolist())
    o_ref, l_ref = oracle.paged_decode(b.dec_q, kp, vp, b.dec_kv_indptr, b.dec_kv_indices, b.dec_kv_lens,
                                       b.page_size, b.sm_scale, requests=sample)
    assert_attention_close(out, lse, o_ref, l_ref, rows=np.array(sample), what="cascade, full workload")

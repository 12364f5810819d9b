"""The shared-prefix (cascade) plan's integer bookkeeping, on the CPU: every (split, request)
state is written by exactly one part, a group's parts cover its shared pages in order, each
request's own pages follow them, and every request keeps at least one position of its own."""

import numpy as np
import pytest
import torch

from paged_kv_attention_10_gb300.cascade import plan_shared_prefix
from workloads import random_small_batch


def _batch(seed, lens, share, ps=4):
    return random_small_batch(seed, page_size=ps, num_q_heads=8, num_kv_heads=2, head_dim=8,
                              decode_lens=lens, decode_new=1, share_decode_prefix=share)


def _sharers(b):
    return [i for i, r in enumerate(b.requests) if r.share_group == 0]


def _check(b, plan, groups):
    ps, B, S = b.page_size, b.num_decode, plan.num_splits
    ind, ptr, lens = b.dec_kv_indices.tolist(), b.dec_kv_indptr.tolist(), b.dec_kv_lens.tolist()
    cover = np.zeros((S, B), dtype=int)
    qs, ql, os_ = plan.part_q_start.tolist(), plan.part_q_len.tolist(), plan.part_o_start.tolist()
    pptr, pind, plen = plan.part_kv_indptr.tolist(), plan.part_kv_indices.tolist(), plan.part_kv_lens.tolist()
    assert len(qs) == plan.num_parts and pptr[0] == 0 and len(pptr) == plan.num_parts + 1
    shared_of = {}
    for p in range(plan.num_parts):
        s, r0 = divmod(os_[p], B)
        assert r0 == qs[p] and 0 <= s < S
        cover[s, r0:r0 + ql[p]] += 1
        assert plen[p] == (pptr[p + 1] - pptr[p]) * ps
        shared_of.setdefault(r0, []).extend(pind[pptr[p]:pptr[p + 1]])
    assert (cover == 1).all()
    assert plan.max_part_rows == max(ql)
    sptr, sind, slen = plan.suffix_kv_indptr.tolist(), plan.suffix_kv_indices.tolist(), plan.suffix_kv_lens.tolist()
    for r in range(B):
        first = max(k for k in shared_of if k <= r)
        shared = shared_of[first]
        own = sind[sptr[r]:sptr[r + 1]]
        assert shared + own == ind[ptr[r]:ptr[r + 1]]  # shared pages, then the request's own
        assert slen[r] == lens[r] - len(shared) * ps and slen[r] >= 1


@pytest.mark.parametrize("num_sms", [1, 4, 152])
def test_plan_covers_every_state_once(num_sms):
    b = _batch(3, (5, 40, 44, 61, 37, 50, 9), share=32)
    s = _sharers(b)
    assert len(s) >= 3 and s == list(range(s[0], s[0] + len(s)))
    plan = plan_shared_prefix(b.dec_kv_indptr, b.dec_kv_indices, b.dec_kv_lens, [(s[0], len(s))],
                              b.page_size, num_kv_heads=2, group_size=4, num_sms=num_sms,
                              min_chunk_tokens=8)
    assert plan.shared_tokens == [32]
    _check(b, plan, [(s[0], len(s))])
    if num_sms == 152:
        assert plan.num_splits == 4  # 32 shared tokens in chunks of at least 8


def test_plan_keeps_one_own_position():
    # a sharer whose whole KV is the shared prefix plus one token keeps that token
    b = _batch(4, (33, 33, 60), share=32, ps=4)
    plan = plan_shared_prefix(b.dec_kv_indptr, b.dec_kv_indices, b.dec_kv_lens, [(0, 3)], b.page_size,
                              num_kv_heads=2, group_size=4, num_sms=152, min_chunk_tokens=8)
    assert plan.shared_tokens == [32]
    _check(b, plan, [(0, 3)])
    b = _batch(5, (32, 40, 60), share=28, ps=4)  # one member has exactly the shared pages
    plan = plan_shared_prefix(b.dec_kv_indptr, b.dec_kv_indices, b.dec_kv_lens, [(0, 3)], b.page_size,
                              num_kv_heads=2, group_size=4, num_sms=152, min_chunk_tokens=8)
    assert plan.shared_tokens == [28]  # (32 - 1) // 4 = 7 pages
    _check(b, plan, [(0, 3)])


def test_group_without_common_pages_is_unshared():
    b = _batch(6, (20, 30, 40), share=0)
    plan = plan_shared_prefix(b.dec_kv_indptr, b.dec_kv_indices, b.dec_kv_lens, [(0, 3)], b.page_size,
                              num_kv_heads=2, group_size=4, num_sms=152)
    assert plan.shared_tokens == [] and plan.num_splits == 1
    assert (plan.part_kv_lens == 0).all()
    assert torch.equal(plan.suffix_kv_indices, b.dec_kv_indices)
    assert torch.equal(plan.suffix_kv_lens, b.dec_kv_lens)


def test_bad_groups_rejected():
    b = _batch(7, (20, 30, 40), share=16)
    args = (b.dec_kv_indptr, b.dec_kv_indices, b.dec_kv_lens)
    with pytest.raises(ValueError):
        plan_shared_prefix(*args, [(1, 3)], b.page_size, num_kv_heads=2, group_size=4, num_sms=1)
    with pytest.raises(ValueError):
        plan_shared_prefix(*args, [(0, 2), (1, 2)], b.page_size, num_kv_heads=2, group_size=4, num_sms=1)

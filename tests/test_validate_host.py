"""The library's host-side metadata checks (no GPU): a generated batch passes, and each kind of
corrupted page table or slot mapping is rejected with the first offending request or token."""

import pytest
import torch

from workloads import random_small_batch


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_attention_10_gb300 import build

    build.build()
    import paged_kv_attention_10_gb300 as p

    p.load()
    return p


@pytest.fixture(scope="module")
def batch():
    return random_small_batch(5, page_size=16, num_q_heads=8, num_kv_heads=2, head_dim=64,
                              decode_lens=(1, 16, 17, 300, 40), decode_new=1,
                              extend=((0, 20), (33, 5)))


def _table(b):
    return b.dec_kv_indptr.clone(), b.dec_kv_indices.clone(), b.dec_kv_lens.clone()


def _bad(pkv, fn, *args, **kw):
    with pytest.raises(pkv.PagedKVError) as e:
        fn(*args, **kw)
    assert e.value.status == 1
    return e.value.bad


def test_generated_batches_pass(pkv, batch):
    b = batch
    pkv.validate_page_table(*_table(b), b.num_pages, b.page_size)
    ext_lens = (b.ext_prefix_lens + (b.ext_qo_indptr[1:] - b.ext_qo_indptr[:-1])).to(torch.int32)
    pkv.validate_page_table(b.ext_kv_indptr, b.ext_kv_indices, ext_lens, b.num_pages, b.page_size)
    pkv.validate_slots(b.slot_mapping, b.num_pages * b.page_size)
    pad = b.slot_mapping.clone()
    pad[1] = -1  # padding tokens are allowed
    pkv.validate_slots(pad, b.num_pages * b.page_size)


def test_page_table_corruptions(pkv, batch):
    b = batch
    n, ps = b.num_pages, b.page_size
    ptr, idx, lens = _table(b)
    bad_page = idx.clone()
    bad_page[int(ptr[3]) + 1] = n  # request 3's second page
    assert _bad(pkv, pkv.validate_page_table, ptr, bad_page, lens, n, ps) == 3
    neg = idx.clone()
    neg[int(ptr[2])] = -5
    assert _bad(pkv, pkv.validate_page_table, ptr, neg, lens, n, ps) == 2
    long = lens.clone()
    long[4] = (int(ptr[5]) - int(ptr[4])) * ps + 1  # one position past its pages
    assert _bad(pkv, pkv.validate_page_table, ptr, idx, long, n, ps) == 4
    zero = lens.clone()
    zero[1] = 0
    assert _bad(pkv, pkv.validate_page_table, ptr, idx, zero, n, ps) == 1
    pkv.validate_page_table(ptr, idx, zero, n, ps, min_len=0)  # allowed when asked
    down = ptr.clone()
    down[2] = down[3] + 1  # request 2 ends before it starts
    assert _bad(pkv, pkv.validate_page_table, down, idx, lens, n, ps) == 2
    shifted = ptr.clone()
    shifted[0] = 1
    assert _bad(pkv, pkv.validate_page_table, shifted, idx, lens, n, ps) == 0


def test_slot_corruptions(pkv, batch):
    b = batch
    slots = b.slot_mapping.clone()
    total = b.num_pages * b.page_size
    out = slots.clone()
    out[3] = total
    assert _bad(pkv, pkv.validate_slots, out, total) == 3
    dup = slots.clone()
    dup[5] = dup[2]  # token 5 writes token 2's slot
    dup[7] = dup[6]
    assert _bad(pkv, pkv.validate_slots, dup, total) == 5
    with pytest.raises(TypeError):
        pkv.validate_slots(slots.to(torch.int32), total)

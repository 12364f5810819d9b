"""KV append and page gather on the GPU: bit-exact against the oracle."""

import pytest
import torch

import oracle
from workloads import random_small_batch
from _gpu_helpers import DeviceBatch, bits_equal, config_with_append

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("idx", [1, 3, 5])
def test_append_bit_exact_on_workload(lib, idx):
    b, kp_ref, vp_ref = config_with_append(idx)
    d = DeviceBatch(b)
    lib.kv_append(d.k_pool, d.v_pool, d.k_new, d.v_new, d.slot_mapping)
    torch.cuda.synchronize()
    assert bits_equal(d.k_pool, kp_ref)
    assert bits_equal(d.v_pool, vp_ref)


@pytest.mark.parametrize("ps,hkv,D", [(1, 8, 128), (16, 2, 64), (5, 3, 64), (64, 1, 128)])
def test_append_padding_and_oob_slots(lib, ps, hkv, D):
    b = random_small_batch(31 + ps, page_size=ps, num_q_heads=hkv, num_kv_heads=hkv, head_dim=D,
                           decode_lens=(3, 40, 7), decode_new=3, extend=((5, 9),))
    slots = b.slot_mapping.clone()
    slots[0] = -1  # padding token
    d = DeviceBatch(b)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.kv_append(d.k_pool, d.v_pool, d.k_new, d.v_new, slots.cuda(), err_word=err)
    kp_ref, vp_ref = oracle.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, slots, ps)
    assert bits_equal(d.k_pool, kp_ref) and bits_equal(d.v_pool, vp_ref)
    assert int(err.item()) == 0
    # a slot past the pool is skipped and reported; the others are still written
    slots2 = b.slot_mapping.clone()
    slots2[1] = b.num_pages * ps + 7
    d2 = DeviceBatch(b)
    lib.kv_append(d2.k_pool, d2.v_pool, d2.k_new, d2.v_new, slots2.cuda(), err_word=err)
    slots_ok = slots2.clone()
    slots_ok[1] = -1
    kp_ref, vp_ref = oracle.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, slots_ok, ps)
    assert bits_equal(d2.k_pool, kp_ref) and bits_equal(d2.v_pool, vp_ref)
    assert int(err.item()) & lib.DEVERR_SLOT_OOB


def test_append_of_nothing(lib):
    b = random_small_batch(2, page_size=4, num_q_heads=2, num_kv_heads=2, head_dim=64, decode_lens=(4,))
    d = DeviceBatch(b)
    e = torch.zeros((0, 2, 64), dtype=torch.bfloat16, device="cuda")
    lib.kv_append(d.k_pool, d.v_pool, e, e, torch.zeros(0, dtype=torch.int64, device="cuda"))
    assert bits_equal(d.k_pool, b.k_pool)


@pytest.mark.parametrize("idx", [1, 2, 3])
def test_gather_bit_exact_on_workload(lib, idx):
    b, kp, vp = config_with_append(idx)
    kpd, vpd = kp.cuda(), vp.cuda()
    if b.num_decode:
        ind, idx_, lens = b.dec_kv_indptr, b.dec_kv_indices, b.dec_kv_lens
    else:
        ind, idx_ = b.ext_kv_indptr, b.ext_kv_indices
        lens = b.ext_prefix_lens + (b.ext_qo_indptr[1:] - b.ext_qo_indptr[:-1])
    total = int(lens.sum())
    k_out, v_out = lib.paged_gather(kpd, vpd, ind.cuda(), idx_.cuda(), lens.to(torch.int32).cuda(), total)
    k_ref = oracle.paged_gather(kp, ind, idx_, lens, b.page_size)
    v_ref = oracle.paged_gather(vp, ind, idx_, lens, b.page_size)
    assert bits_equal(k_out, k_ref) and bits_equal(v_out, v_ref)


def test_gather_reports_bad_page_index(lib):
    b = random_small_batch(3, page_size=4, num_q_heads=2, num_kv_heads=2, head_dim=64, decode_lens=(9, 5))
    kp, vp = oracle.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.slot_mapping, 4)
    ind = b.dec_kv_indices.clone()
    ind[0] = b.num_pages + 100  # outside the pool: must be skipped, not read
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.paged_gather(kp.cuda(), vp.cuda(), b.dec_kv_indptr.cuda(), ind.cuda(), b.dec_kv_lens.cuda(), 14,
                     err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & lib.DEVERR_PAGE_OOB

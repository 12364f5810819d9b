"""Paged decode on the GPU against the fp64 oracle (bf16 output, stated tolerances)."""

import math

import numpy as np
import pytest
import torch

import oracle
from workloads import random_small_batch
from _fixtures import golden_tensors, load_golden
from _gpu_helpers import DeviceBatch, assert_attention_close, config_with_append

pytestmark = pytest.mark.gpu

GOLD = load_golden()


def run_decode(lib, b, kp, vp, **kw):
    q = b.dec_q.cuda()
    return lib.paged_decode(q, kp.cuda() if not kp.is_cuda else kp, vp.cuda() if not vp.is_cuda else vp,
                            b.dec_kv_indptr.cuda(), b.dec_kv_indices.cuda(), b.dec_kv_lens.cuda(),
                            b.sm_scale, **kw)


@pytest.mark.parametrize("name", ["two_keys_ln3", "gqa_head_map"])
def test_golden_decode_on_gpu(lib, name):
    c = GOLD[name]
    t = golden_tensors(c)
    # head_dim of the worked examples is 2: embed them in head_dim 64 with zero padding, which
    # changes neither the scores nor the first two output columns
    D = 64

    def pad(x):
        y = torch.zeros(x.shape[:-1] + (D,), dtype=x.dtype)
        y[..., : x.shape[-1]] = x
        return y

    out, lse = lib.paged_decode(pad(t["q"]).cuda(), pad(t["k_pool"]).cuda(), pad(t["v_pool"]).cuda(),
                                t["kv_indptr"].cuda(), t["kv_indices"].cuda(), t["kv_lens"].cuda(),
                                c["sm_scale"])
    o = out.float().cpu().numpy()
    assert np.abs(o[..., :2] - np.array(c["expect_o"])).max() <= 1e-2
    assert np.all(o[..., 2:] == 0)
    assert np.abs(lse.cpu().numpy() - np.array(c["expect_lse"])).max() <= 1e-3


@pytest.mark.parametrize("idx", [1, 2])
def test_decode_full_workload(lib, idx):
    b, kp, vp = config_with_append(idx)
    # the product path: append on the GPU, then decode over the appended pool
    d = DeviceBatch(b)
    lib.kv_append(d.k_pool, d.v_pool, d.k_new, d.v_new, d.slot_mapping)
    out, lse = run_decode(lib, b, d.k_pool, d.v_pool)
    o_ref, lse_ref = oracle.paged_decode(b.dec_q, kp, vp, b.dec_kv_indptr, b.dec_kv_indices,
                                         b.dec_kv_lens, b.page_size, b.sm_scale)
    assert_attention_close(out, lse, o_ref, lse_ref, what=f"config {idx}")


@pytest.mark.slow
def test_decode_long_context_split(lib):
    """8 x 32768 tokens: every request is split across many CTAs and merged."""
    b, kp, vp = config_with_append(4)
    out, lse = run_decode(lib, b, kp, vp)
    o_ref, lse_ref = oracle.paged_decode(b.dec_q, kp, vp, b.dec_kv_indptr, b.dec_kv_indices,
                                         b.dec_kv_lens, b.page_size, b.sm_scale)
    assert_attention_close(out, lse, o_ref, lse_ref, what="config 4")


@pytest.mark.slow
@pytest.mark.parametrize("spare_sms", [0, 12, 16])
def test_decode_mixed_step_decodes(lib, spare_sms):
    """The 256 decodes of the mixed step (64 share a prefix), on a sample of requests; also on
    all but 12 SMs, as the benchmark's branched step runs it beside the extend (and 16)."""
    b, kp, vp = config_with_append(5)
    d = DeviceBatch(b)
    lib.kv_append(d.k_pool, d.v_pool, d.k_new, d.v_new, d.slot_mapping)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    out, lse = run_decode(lib, b, d.k_pool, d.v_pool, max_ctas=sms - spare_sms if spare_sms else 0)
    rng = np.random.default_rng(0)
    sample = sorted(rng.choice(b.num_decode, 64, replace=False).tolist())
    o_ref, lse_ref = oracle.paged_decode(b.dec_q, kp, vp, b.dec_kv_indptr, b.dec_kv_indices,
                                         b.dec_kv_lens, b.page_size, b.sm_scale, requests=sample)
    assert_attention_close(out, lse, o_ref, lse_ref, rows=sample, what="config 5 decodes")


CASES = [
    # (page_size, Hq, Hkv, D, lens)
    (16, 14, 2, 64, (1, 15, 16, 17, 33, 300)),
    (1, 16, 8, 128, (1, 2, 100, 640)),
    (2, 8, 8, 128, (1, 3, 4, 5, 77)),
    (64, 32, 8, 128, (63, 64, 65, 1000)),
    (16, 16, 1, 128, (5, 16, 200, 1500)),
    (16, 16, 16, 64, (31, 32, 2, 1)),
    (8, 28, 4, 128, (9, 129, 4000)),
    (16, 64, 4, 128, (17, 700)),
    (4, 6, 3, 64, (1, 2, 3, 50, 51)),
    (16, 40, 5, 128, (100, 2000, 16)),
]


@pytest.mark.parametrize("case", CASES, ids=[f"ps{c[0]}-q{c[1]}-kv{c[2]}-d{c[3]}" for c in CASES])
def test_decode_property_sweep(lib, case):
    ps, hq, hkv, D, lens = case
    b = random_small_batch(100 + ps + hq + D, page_size=ps, num_q_heads=hq, num_kv_heads=hkv,
                           head_dim=D, decode_lens=lens, decode_new=1)
    kp, vp = oracle.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.slot_mapping, ps)
    out, lse = run_decode(lib, b, kp, vp)
    o_ref, lse_ref = oracle.paged_decode(b.dec_q, kp, vp, b.dec_kv_indptr, b.dec_kv_indices,
                                         b.dec_kv_lens, ps, b.sm_scale)
    assert_attention_close(out, lse, o_ref, lse_ref, what=str(case))


def test_decode_shared_prefix_pages(lib):
    b = random_small_batch(7, page_size=16, num_q_heads=32, num_kv_heads=8, head_dim=128,
                           decode_lens=(600, 700, 1200, 90, 1500), share_decode_prefix=512)
    kp, vp = oracle.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.slot_mapping, 16)
    out, lse = run_decode(lib, b, kp, vp)
    o_ref, lse_ref = oracle.paged_decode(b.dec_q, kp, vp, b.dec_kv_indptr, b.dec_kv_indices,
                                         b.dec_kv_lens, 16, b.sm_scale)
    assert_attention_close(out, lse, o_ref, lse_ref, what="shared prefix")


def test_decode_is_deterministic(lib):
    b = random_small_batch(8, page_size=16, num_q_heads=32, num_kv_heads=8, head_dim=128,
                           decode_lens=(3000, 40, 9000, 1))
    kp, vp = oracle.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.slot_mapping, 16)
    kpd, vpd = kp.cuda(), vp.cuda()
    o1, l1 = run_decode(lib, b, kpd, vpd)
    o2, l2 = run_decode(lib, b, kpd, vpd)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(l1, l2)


def test_decode_zero_length_and_bad_page(lib):
    b = random_small_batch(9, page_size=16, num_q_heads=8, num_kv_heads=2, head_dim=64,
                           decode_lens=(20, 40, 60))
    kp, vp = oracle.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.slot_mapping, 16)
    lens = b.dec_kv_lens.clone()
    lens[1] = 0
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = lib.paged_decode(b.dec_q.cuda(), kp.cuda(), vp.cuda(), b.dec_kv_indptr.cuda(),
                                b.dec_kv_indices.cuda(), lens.cuda(), b.sm_scale, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & lib.DEVERR_LENGTH
    assert torch.all(out[1] == 0) and torch.all(torch.isneginf(lse[1]))
    o_ref, lse_ref = oracle.paged_decode(b.dec_q, kp, vp, b.dec_kv_indptr, b.dec_kv_indices, lens, 16,
                                         b.sm_scale, requests=[0, 2])
    assert_attention_close(out, lse, o_ref, lse_ref, rows=[0, 2], what="zero-length neighbours")
    # a page index outside the pool is skipped (never dereferenced) and reported
    ind = b.dec_kv_indices.clone()
    ind[0] = b.num_pages + 5
    err.zero_()
    lib.paged_decode(b.dec_q.cuda(), kp.cuda(), vp.cuda(), b.dec_kv_indptr.cuda(), ind.cuda(),
                     b.dec_kv_lens.cuda(), b.sm_scale, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & lib.DEVERR_PAGE_OOB


def test_decode_host_checks(lib):
    b = random_small_batch(10, page_size=16, num_q_heads=8, num_kv_heads=2, head_dim=64,
                           decode_lens=(20,))
    kp, vp = b.k_pool.cuda(), b.v_pool.cuda()
    args = (b.dec_kv_indptr.cuda(), b.dec_kv_indices.cuda(), b.dec_kv_lens.cuda(), b.sm_scale)
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(lib.PagedKVError) as e:
        lib.paged_decode(b.dec_q.cuda(), kp, vp, *args, workspace=small)
    assert e.value.status == 3  # workspace too small
    q_bad = torch.zeros((1, 7, 64), dtype=torch.bfloat16, device="cuda")  # 7 % 2 != 0
    with pytest.raises(lib.PagedKVError) as e:
        lib.paged_decode(q_bad, kp, vp, *args)
    assert e.value.status == 1
    kp96 = torch.zeros((4, 16, 2, 96), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(lib.PagedKVError) as e:
        lib.paged_decode(torch.zeros((1, 8, 96), dtype=torch.bfloat16, device="cuda"), kp96, kp96, *args)
    assert e.value.status == 2  # head_dim 96 not built


@pytest.mark.parametrize("max_ctas", [1, 5, 100, 100000])
def test_decode_on_fewer_sms(lib, max_ctas):
    # the persistent grid limited to max_ctas SMs (the rest left to other streams): a different
    # split of the token stream, the same attention within tolerance; a limit at or above the SM
    # count is the ordinary decode, bit for bit
    b = random_small_batch(12, page_size=16, num_q_heads=32, num_kv_heads=8, head_dim=128,
                           decode_lens=(5000, 1, 700, 12000, 33, 2500), share_decode_prefix=512)
    kp, vp = oracle.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.slot_mapping, 16)
    kpd, vpd = kp.cuda(), vp.cuda()
    out, lse = run_decode(lib, b, kpd, vpd, max_ctas=max_ctas)
    o_ref, lse_ref = oracle.paged_decode(b.dec_q, kp, vp, b.dec_kv_indptr, b.dec_kv_indices,
                                         b.dec_kv_lens, 16, b.sm_scale)
    assert_attention_close(out, lse, o_ref, lse_ref, what=f"decode on {max_ctas} SMs")
    if max_ctas >= torch.cuda.get_device_properties(0).multi_processor_count:
        o2, l2 = run_decode(lib, b, kpd, vpd)
        assert torch.equal(out.view(torch.int16), o2.view(torch.int16)) and torch.equal(lse, l2)


def test_decode_negative_sm_limit_rejected(lib):
    b = random_small_batch(13, page_size=16, num_q_heads=8, num_kv_heads=2, head_dim=64, decode_lens=(20,))
    with pytest.raises(lib.PagedKVError) as e:
        run_decode(lib, b, b.k_pool.cuda(), b.v_pool.cuda(), max_ctas=-1)
    assert e.value.status == 1


@pytest.mark.parametrize("page_size", [16, 1], ids=["tma-boxes", "row-copies"])
def test_decode_l2_keep_hint_changes_nothing(lib, page_size):
    """The L2 keep hint only steers the L2's evictions: with each request's shared prefix, with
    zeros, or with values outside [0, kv_lens] the decode is bit for bit the one without a hint,
    and within tolerance of the oracle."""
    b = random_small_batch(41, page_size=page_size, num_q_heads=32, num_kv_heads=8, head_dim=128,
                           decode_lens=(40, 700, 900, 1300, 650, 90), share_decode_prefix=512)
    kp, vp = oracle.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.slot_mapping, page_size)
    kpd, vpd = kp.cuda(), vp.cuda()
    out0, lse0 = run_decode(lib, b, kpd, vpd)
    o_ref, lse_ref = oracle.paged_decode(b.dec_q, kp, vp, b.dec_kv_indptr, b.dec_kv_indices,
                                         b.dec_kv_lens, page_size, b.sm_scale)
    assert_attention_close(out0, lse0, o_ref, lse_ref, what="decode without a hint")
    out40, lse40 = run_decode(lib, b, kpd, vpd, max_ctas=40)
    B = b.num_decode
    hints = [b.dec_shared_tokens, torch.zeros(B, dtype=torch.int32),
             torch.tensor([-5, 10**9, 0, 7, 2**31 - 1, -(2**31)][:B], dtype=torch.int32)]
    for hint in hints:
        for max_ctas, (o_plain, l_plain) in ((0, (out0, lse0)), (40, (out40, lse40))):
            err = torch.zeros(1, dtype=torch.int32, device="cuda")
            out, lse = run_decode(lib, b, kpd, vpd, l2_keep_tokens=hint.cuda(), max_ctas=max_ctas, err_word=err)
            torch.cuda.synchronize()
            assert int(err.item()) == 0
            assert torch.equal(out.view(torch.int16), o_plain.view(torch.int16)) and torch.equal(lse, l_plain)

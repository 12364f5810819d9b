"""Ragged extend (tcgen05) on the GPU against the fp64 oracle."""

import numpy as np
import pytest
import torch

import oracle
from workloads import random_small_batch
from _fixtures import golden_tensors, load_golden
from _gpu_helpers import DeviceBatch, assert_attention_close, config_with_append

pytestmark = pytest.mark.gpu


def run_extend(lib, b, kp, vp, max_extend_len=None, **kw):
    dev = "cuda"
    mel = b.max_extend_len if max_extend_len is None else max_extend_len
    return lib.paged_extend(b.ext_q.to(dev), kp.to(dev), vp.to(dev), b.ext_qo_indptr.to(dev),
                            b.ext_kv_indptr.to(dev), b.ext_kv_indices.to(dev),
                            b.ext_prefix_lens.to(dev), mel, b.sm_scale, **kw)


def oracle_extend(b, kp, vp, **kw):
    return oracle.paged_extend(b.ext_q, kp, vp, b.ext_qo_indptr, b.ext_kv_indptr, b.ext_kv_indices,
                               b.ext_prefix_lens, b.page_size, b.sm_scale, **kw)


def _repage(pool, indptr, indices, lens, ps, new_ps):
    """The same requests' rows laid out in a fresh NaN-filled pool of page size new_ps, pages in
    reverse order (a test-side re-layout: position j of request b -> page j // new_ps)."""
    B = len(lens)
    need = [-(-int(L) // new_ps) for L in lens]
    n = sum(need) + 1
    out = torch.full((n, new_ps) + tuple(pool.shape[2:]), float("nan"), dtype=pool.dtype)
    new_ind, new_ptr, nxt = [], [0], n - 1
    for b in range(B):
        pages = []
        for _ in range(need[b]):
            pages.append(nxt)
            nxt -= 1
        for j in range(int(lens[b])):
            src = pool[indices[indptr[b] + j // ps], j % ps]
            out[pages[j // new_ps], j % new_ps] = src
        new_ind += pages
        new_ptr.append(len(new_ind))
    return out, torch.tensor(new_ptr, dtype=torch.int32), torch.tensor(new_ind, dtype=torch.int32)


def test_golden_extend_on_gpu(lib):
    c = load_golden()["extend_prefix_offset_uniform"]
    t = golden_tensors(c)
    D = 128

    def pad(x):
        y = torch.zeros(x.shape[:-1] + (D,), dtype=x.dtype)
        y[..., : x.shape[-1]] = x
        return y

    lens = (t["prefix_lens"] + t["qo_indptr"][1:] - t["qo_indptr"][:-1]).tolist()
    ind, idx = t["kv_indptr"].tolist(), t["kv_indices"].tolist()
    kp, ptr, new_idx = _repage(pad(t["k_pool"]), ind, idx, lens, c["page_size"], 8)
    vp, _, _ = _repage(pad(t["v_pool"]), ind, idx, lens, c["page_size"], 8)
    out, lse = lib.paged_extend(pad(t["q"]).cuda(), kp.cuda(), vp.cuda(), t["qo_indptr"].cuda(),
                                ptr.cuda(), new_idx.cuda(), t["prefix_lens"].cuda(), 2, c["sm_scale"])
    o = out.float().cpu().numpy()
    assert np.abs(o[..., :2] - np.array(c["expect_o"])).max() <= 1e-2
    assert np.all(o[..., 2:] == 0)
    assert np.abs(lse.cpu().numpy() - np.array(c["expect_lse"])).max() <= 1e-3


def test_extend_radix_prefix_workload(lib):
    b, kp, vp = config_with_append(3)
    d = DeviceBatch(b)
    lib.kv_append(d.k_pool, d.v_pool, d.k_new, d.v_new, d.slot_mapping)
    out, lse = run_extend(lib, b, d.k_pool, d.v_pool)
    o_ref, lse_ref = oracle_extend(b, kp, vp)
    assert_attention_close(out, lse, o_ref, lse_ref, what="config 3")


@pytest.mark.slow
def test_extend_mixed_step_chunks(lib):
    b, kp, vp = config_with_append(5)
    d = DeviceBatch(b)
    lib.kv_append(d.k_pool, d.v_pool, d.k_new, d.v_new, d.slot_mapping)
    out, lse = run_extend(lib, b, d.k_pool, d.v_pool)
    o_ref, lse_ref = oracle_extend(b, kp, vp)
    assert_attention_close(out, lse, o_ref, lse_ref, what="config 5 extends")


CASES = [
    # (page_size, Hq, Hkv, [(prefix, extend), ...])
    (16, 32, 8, [(0, 1), (0, 5), (3, 40), (100, 33), (700, 129)]),
    (16, 8, 8, [(0, 128), (5, 200), (64, 64)]),
    (8, 16, 2, [(7, 31), (0, 64)]),
    (64, 32, 4, [(63, 65), (128, 1), (0, 300)]),
    (128, 16, 1, [(5, 130), (250, 10)]),
    (256, 16, 16, [(300, 100)]),
    (16, 32, 2, [(31, 17), (0, 9)]),
    (32, 16, 8, [(0, 3), (50, 0), (999, 77)]),          # group 2; a request with no new token
    (16, 32, 8, [(40, 0), (0, 1), (17, 0), (300, 64)]),  # empty extends between others
    (16, 32, 8, [((i * 37) % 300, (i * 11) % 40) for i in range(70)]),  # 70 requests, mixed lengths
]


@pytest.mark.parametrize("case", CASES, ids=[f"ps{c[0]}-q{c[1]}-kv{c[2]}" for c in CASES])
def test_extend_property_sweep(lib, case):
    ps, hq, hkv, ext = case
    b = random_small_batch(200 + ps + hq, page_size=ps, num_q_heads=hq, num_kv_heads=hkv, head_dim=128,
                           extend=ext)
    kp, vp = oracle.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.slot_mapping, ps)
    out, lse = run_extend(lib, b, kp, vp)
    o_ref, lse_ref = oracle_extend(b, kp, vp)
    assert_attention_close(out, lse, o_ref, lse_ref, what=str(case))


# any group size up to 16 (the Q tile then holds group x floor(128 / group) rows) and head_dim 64
GENERAL = [
    # (page_size, Hq, Hkv, head_dim, [(prefix, extend), ...])
    (16, 14, 2, 64, [(0, 37), (100, 70), (511, 1), (16, 18)]),  # Qwen2.5-0.5B attention: group 7
    (16, 6, 2, 128, [(0, 50), (77, 43), (3, 1)]),                # group 3: 126 rows
    (32, 20, 4, 128, [(64, 26), (0, 100)]),                      # group 5: 125 rows
    (8, 12, 2, 64, [(9, 22), (0, 21), (130, 5)]),                # group 6, page 8
    (16, 16, 16, 64, [(0, 129), (200, 64)]),                     # group 1, head_dim 64
    (64, 64, 4, 64, [(63, 17), (1, 8)]),                         # group 16, head_dim 64
    (16, 24, 2, 128, [(0, 30), (45, 11)]),                       # group 12: 120 rows
    # page sizes the TMA boxes do not take (below 8 rows, or not a power of two): row copies
    (1, 16, 8, 128, [(0, 40), (77, 13), (200, 64)]),             # page size 1 (Qwen3-0.6B shape)
    (2, 14, 2, 64, [(5, 33), (0, 7)]),
    (4, 32, 8, 128, [(63, 65), (128, 1), (0, 100)]),
    (24, 8, 8, 128, [(47, 30), (0, 24), (100, 3)]),              # page size 24
    (12, 6, 2, 64, [(11, 40), (36, 36)]),
]


@pytest.mark.parametrize("case", GENERAL, ids=[f"ps{c[0]}-q{c[1]}-kv{c[2]}-d{c[3]}" for c in GENERAL])
def test_extend_any_group_and_head_dim_64(lib, case):
    ps, hq, hkv, d, ext = case
    b = random_small_batch(300 + ps + hq + d, page_size=ps, num_q_heads=hq, num_kv_heads=hkv,
                           head_dim=d, extend=ext)
    kp, vp = oracle.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.slot_mapping, ps)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = run_extend(lib, b, kp, vp, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    o_ref, lse_ref = oracle_extend(b, kp, vp)
    assert_attention_close(out, lse, o_ref, lse_ref, what=f"extend {case[:4]}")


def test_extend_shared_prefix_pages(lib):
    b = random_small_batch(17, page_size=16, num_q_heads=32, num_kv_heads=8, head_dim=128,
                           extend=[(512, 100), (600, 37), (1000, 256), (40, 50)], share_extend_prefix=512)
    kp, vp = oracle.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.slot_mapping, 16)
    out, lse = run_extend(lib, b, kp, vp)
    o_ref, lse_ref = oracle_extend(b, kp, vp)
    assert_attention_close(out, lse, o_ref, lse_ref, what="shared prefix")


def test_extend_is_deterministic_and_matches_decode(lib):
    b = random_small_batch(18, page_size=16, num_q_heads=32, num_kv_heads=8, head_dim=128,
                           decode_lens=(77, 500, 1031), extend=[(300, 70)])
    kp, vp = oracle.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.slot_mapping, 16)
    kpd, vpd = kp.cuda(), vp.cuda()
    o1, l1 = run_extend(lib, b, kpd, vpd)
    o2, l2 = run_extend(lib, b, kpd, vpd)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(l1, l2)
    # decode requests viewed as one-token extends give the decode result (within tolerance)
    B = b.num_decode
    qo = torch.arange(B + 1, dtype=torch.int32).cuda()
    eo, el = lib.paged_extend(b.dec_q.cuda(), kpd, vpd, qo, b.dec_kv_indptr.cuda(), b.dec_kv_indices.cuda(),
                              (b.dec_kv_lens - 1).cuda(), 1, b.sm_scale)
    do, dl = lib.paged_decode(b.dec_q.cuda(), kpd, vpd, b.dec_kv_indptr.cuda(), b.dec_kv_indices.cuda(),
                              b.dec_kv_lens.cuda(), b.sm_scale)
    assert (eo.float() - do.float()).abs().max().item() <= 2e-2
    assert (el - dl).abs().max().item() <= 1e-3


def test_extend_bad_page_index_is_reported(lib):
    b = random_small_batch(19, page_size=16, num_q_heads=8, num_kv_heads=2, head_dim=128, extend=[(40, 30)])
    kp, vp = oracle.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.slot_mapping, 16)
    ind = b.ext_kv_indices.clone()
    ind[1] = b.num_pages + 3
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.paged_extend(b.ext_q.cuda(), kp.cuda(), vp.cuda(), b.ext_qo_indptr.cuda(), b.ext_kv_indptr.cuda(),
                     ind.cuda(), b.ext_prefix_lens.cuda(), b.max_extend_len, b.sm_scale, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & lib.DEVERR_PAGE_OOB


@pytest.mark.parametrize("pad", [0, 38], ids=["ranked-in-kernel", "order-kernel"])
def test_extend_rows_past_max_extend_len_are_reported(lib, pad):
    """A max_extend_len below a request's new-token count is a caller error the kernel reports:
    PKV_DEVERR_LENGTH, the rows the grid covers computed, the rows past it left untouched.  Two
    requests take the compact grid of a batch ranked in the kernel; 38 one-token requests more
    take the full grid and the order kernel."""
    b = random_small_batch(27, page_size=16, num_q_heads=8, num_kv_heads=2, head_dim=128,
                           extend=[(0, 300), (50, 70)] + [(5 + i, 1) for i in range(pad)])
    kp, vp = oracle.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.slot_mapping, 16)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full_like(b.ext_q, 7.0).cuda()
    too_small = 100  # group 4: the grid covers ceil(100 / 32) * 32 = 128 rows of each request
    lib.paged_extend(b.ext_q.cuda(), kp.cuda(), vp.cuda(), b.ext_qo_indptr.cuda(), b.ext_kv_indptr.cuda(),
                     b.ext_kv_indices.cuda(), b.ext_prefix_lens.cuda(), too_small, b.sm_scale, out=out,
                     err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == lib.DEVERR_LENGTH
    o_ref, _ = oracle_extend(b, kp, vp)
    covered = list(range(0, 128)) + list(range(300, 370))
    assert_attention_close(out, None, o_ref, None, rows=covered, what="covered rows")
    assert bool((out[128:300].float() == 7.0).all())
    # with a large enough bound the same call reports nothing
    err.zero_()
    run_extend(lib, b, kp, vp, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0


def test_extend_host_checks(lib):
    b = random_small_batch(20, page_size=16, num_q_heads=8, num_kv_heads=2, head_dim=96, extend=[(4, 4)])
    with pytest.raises(lib.PagedKVError) as e:
        run_extend(lib, b, b.k_pool, b.v_pool)
    assert e.value.status == 2  # head_dim 96 not built
    b = random_small_batch(22, page_size=16, num_q_heads=34, num_kv_heads=2, head_dim=128, extend=[(4, 4)])
    with pytest.raises(lib.PagedKVError) as e:
        run_extend(lib, b, b.k_pool, b.v_pool)
    assert e.value.status == 2  # group size 17
    # up to 32 requests are ranked inside the kernel (no workspace); more take the order kernel's
    b = random_small_batch(24, page_size=16, num_q_heads=8, num_kv_heads=2, head_dim=128,
                           extend=[(4, 4), (0, 9)])
    assert lib.extend_workspace_size(2, 8, 2, 128, b.max_extend_len) == 0
    b = random_small_batch(24, page_size=16, num_q_heads=8, num_kv_heads=2, head_dim=128,
                           extend=[(4, 4), (0, 9)] * 20)
    need = lib.extend_workspace_size(40, 8, 2, 128, b.max_extend_len)
    assert need > 0
    with pytest.raises(lib.PagedKVError) as e:
        run_extend(lib, b, b.k_pool, b.v_pool,
                   workspace=torch.zeros(need - 16, dtype=torch.uint8, device="cuda"))
    assert e.value.status == 3  # workspace too small for the request order


def test_extend_huge_max_extend_len_on_a_ranked_batch(lib):
    """A batch ranked in the kernel sizes its compact grid by the rows it has, not by
    max_extend_len: a loose bound costs nothing and the result is unchanged."""
    b = random_small_batch(25, page_size=16, num_q_heads=8, num_kv_heads=2, head_dim=128,
                           extend=[(3, 40), (90, 7)])
    kp, vp = oracle.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.slot_mapping, 16)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = run_extend(lib, b, kp, vp, err_word=err, max_extend_len=2_000_000_000)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    o_ref, lse_ref = oracle_extend(b, kp, vp)
    assert_attention_close(out, lse, o_ref, lse_ref, what="loose max_extend_len")


def test_extend_speculative_verify_shape(lib):
    """k drafted tokens + 1 verified in one extend over long contexts (sampled requests)."""
    from workloads import make_spec_verify

    b = make_spec_verify(num_requests=24, draft_tokens=5)
    kp, vp = oracle.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.slot_mapping, 16)
    out, lse = run_extend(lib, b, kp, vp)
    sample = list(range(0, 24, 3))
    o_ref, lse_ref = oracle_extend(b, kp, vp, requests=sample)
    qo = b.ext_qo_indptr.tolist()
    rows = [i for r in sample for i in range(qo[r], qo[r + 1])]
    assert_attention_close(out, lse, o_ref, lse_ref, rows=rows, what="spec verify")


@pytest.mark.slow
def test_extend_more_requests_than_the_plan_sorts(lib):
    # 4500 requests: above the 4096 the plan kernel sorts in shared memory, so they keep batch
    # order, and the item prefix is scanned in several chunks; a sample is checked
    ext = [((i * 13) % 90, 1 + (i * 7) % 3) for i in range(4500)]
    b = random_small_batch(77, page_size=16, num_q_heads=8, num_kv_heads=2, head_dim=128, extend=ext)
    kp, vp = oracle.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.slot_mapping, 16)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = run_extend(lib, b, kp, vp, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    sample = list(range(0, 4500, 97)) + [4095, 4096, 4499]
    o_ref, lse_ref = oracle_extend(b, kp, vp, requests=sample)
    qo = b.ext_qo_indptr.tolist()
    rows = np.concatenate([np.arange(qo[r], qo[r + 1]) for r in sample])
    assert_attention_close(out, lse, o_ref, lse_ref, rows=rows, what="4500 requests")


@pytest.mark.slow
def test_extend_small_model_prefill_workload(lib):
    """The small-model prefill workload at full size (Qwen2.5-0.5B attention: group 7, head_dim
    64), as the benchmark runs it: append, then extend, against the oracle."""
    from workloads import make_small_prefill

    b = make_small_prefill()
    kp, vp = oracle.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.slot_mapping, b.page_size)
    d = DeviceBatch(b)
    lib.kv_append(d.k_pool, d.v_pool, d.k_new, d.v_new, d.slot_mapping)
    out, lse = run_extend(lib, b, d.k_pool, d.v_pool)
    o_ref, lse_ref = oracle_extend(b, kp, vp)
    assert_attention_close(out, lse, o_ref, lse_ref, what="small-model prefill")

"""The kernels' failure path without a GPU fault: a wait that nothing completes gives up after its
bounded limit and reports PKV_DEVERR_TIMEOUT into the error word, and the context stays usable."""

import time

import numpy as np
import pytest
import torch

import oracle
from workloads import random_small_batch
from _gpu_helpers import assert_attention_close

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_reports(lib):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    lib.selftest_bounded_wait(err)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert int(err.item()) == lib.DEVERR_TIMEOUT
    assert 0.4 < waited < 10.0  # the 0.5 s limit of %globaltimer, then the kernel returns
    # the context is still usable: a decode right after gives the oracle's result
    b = random_small_batch(31, page_size=16, num_q_heads=8, num_kv_heads=2, head_dim=128,
                           decode_lens=(40, 300))
    kp, vp = oracle.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.slot_mapping, 16)
    out, lse = lib.paged_decode(b.dec_q.cuda(), kp.cuda(), vp.cuda(), b.dec_kv_indptr.cuda(),
                                b.dec_kv_indices.cuda(), b.dec_kv_lens.cuda(), b.sm_scale)
    o_ref, l_ref = oracle.paged_decode(b.dec_q, kp, vp, b.dec_kv_indptr, b.dec_kv_indices,
                                       b.dec_kv_lens, 16, b.sm_scale)
    assert_attention_close(out, lse, o_ref, l_ref, what="decode after a timed-out wait")

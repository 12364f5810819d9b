"""The hot path captured in a CUDA graph: append + decode (split + merge) + extend in one graph,
replayed on new inputs copied into the same device buffers (the fixed-buffer contract the
mini-sglang-from-Scratch handbook describes for CUDA Graph).  The library allocates nothing and
never synchronises inside a call, so the captured step must give the eager step's results."""

import pytest
import torch

import oracle
from workloads import random_small_batch
from _gpu_helpers import DeviceBatch, assert_attention_close, bits_equal

pytestmark = pytest.mark.gpu


def _batch(seed):
    return random_small_batch(seed, page_size=16, num_q_heads=32, num_kv_heads=8, head_dim=128,
                              decode_lens=(1, 300, 2100, 77, 4000), decode_new=1,
                              extend=((0, 70), (190, 33), (1024, 300)))


def test_captured_step_matches_eager_and_oracle(lib):
    b1, b2 = _batch(61), _batch(62)
    assert b1.k_pool.shape == b2.k_pool.shape and b1.dec_kv_indices.shape == b2.dec_kv_indices.shape
    d = DeviceBatch(b1)
    st = torch.cuda.Stream()
    dws = torch.empty(lib.decode_workspace_size(5, 32, 8, 128), dtype=torch.uint8, device="cuda")
    d_out = torch.empty_like(d.dec_q)
    d_lse = torch.empty(d.dec_q.shape[:2], dtype=torch.float32, device="cuda")
    e_out = torch.empty_like(d.ext_q)
    e_lse = torch.empty(d.ext_q.shape[:2], dtype=torch.float32, device="cuda")
    max_e = max(b1.max_extend_len, b2.max_extend_len)
    ews = torch.empty(max(256, lib.extend_workspace_size(b1.num_extend, 32, 8, 128, max_e)),
                      dtype=torch.uint8, device="cuda")

    def step():
        lib.kv_append(d.k_pool, d.v_pool, d.k_new, d.v_new, d.slot_mapping, stream=st)
        lib.paged_decode(d.dec_q, d.k_pool, d.v_pool, d.dec_kv_indptr, d.dec_kv_indices, d.dec_kv_lens,
                         b1.sm_scale, out=d_out, lse=d_lse, workspace=dws, stream=st)
        lib.paged_extend(d.ext_q, d.k_pool, d.v_pool, d.ext_qo_indptr, d.ext_kv_indptr, d.ext_kv_indices,
                         d.ext_prefix_lens, max_e, b1.sm_scale, out=e_out, lse=e_lse, workspace=ews,
                         stream=st)

    with torch.cuda.stream(st):
        step()  # warm-up: one-time attribute setup happens outside the capture
    st.synchronize()
    eager = [t.clone() for t in (d_out, d_lse, e_out, e_lse)]

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        step()

    def load(b):  # copy a step's inputs into the captured buffers
        for name in ("k_pool", "v_pool", "k_new", "v_new", "slot_mapping", "dec_q", "dec_kv_indptr",
                     "dec_kv_indices", "dec_kv_lens", "ext_q", "ext_qo_indptr", "ext_kv_indptr",
                     "ext_kv_indices", "ext_prefix_lens"):
            getattr(d, name).copy_(getattr(b, name))

    # replay on the first step's inputs: identical to eager (deterministic kernels)
    load(b1)
    g.replay()
    torch.cuda.synchronize()
    for x, y in zip((d_out, d_lse, e_out, e_lse), eager):
        assert bits_equal(x, y) if x.dtype == torch.bfloat16 else torch.equal(x, y)
    # replay on different inputs of the same shapes: matches the oracle
    load(b2)
    g.replay()
    torch.cuda.synchronize()
    kp, vp = oracle.kv_append(b2.k_pool, b2.v_pool, b2.k_new, b2.v_new, b2.slot_mapping, 16)
    assert bits_equal(d.k_pool, kp) and bits_equal(d.v_pool, vp)
    o_ref, l_ref = oracle.paged_decode(b2.dec_q, kp, vp, b2.dec_kv_indptr, b2.dec_kv_indices,
                                       b2.dec_kv_lens, 16, b2.sm_scale)
    assert_attention_close(d_out, d_lse, o_ref, l_ref, what="graph decode")
    o_ref, l_ref = oracle.paged_extend(b2.ext_q, kp, vp, b2.ext_qo_indptr, b2.ext_kv_indptr,
                                       b2.ext_kv_indices, b2.ext_prefix_lens, 16, b2.sm_scale)
    assert_attention_close(e_out, e_lse, o_ref, l_ref, what="graph extend")


def test_two_branch_step_matches_serial_and_oracle(lib):
    # The step as two graph branches that share no data (the decodes' new tokens, then decode and
    # its merge, beside the extend tokens, then extend), as the benchmark captures it: the same
    # bits as the serial step, and the pool and outputs the oracle gives.
    b = _batch(63)
    nd = sum(r.new_tokens for r in b.requests if r.kind == "decode")
    assert all(r.kind == "decode" for r in b.requests[: b.num_decode])
    st, st2 = torch.cuda.Stream(), torch.cuda.Stream()
    dws = torch.empty(lib.decode_workspace_size(b.num_decode, 32, 8, 128), dtype=torch.uint8,
                      device="cuda")
    ews = torch.empty(max(256, lib.extend_workspace_size(b.num_extend, 32, 8, 128, b.max_extend_len)),
                      dtype=torch.uint8, device="cuda")
    fork, join = torch.cuda.Event(), torch.cuda.Event()
    # the decode leaves 12 SMs to the extend beside it, as the benchmark's branched step does
    ctas = torch.cuda.get_device_properties(0).multi_processor_count - 12

    def run(branches):
        d = DeviceBatch(b)
        d_out = torch.empty_like(d.dec_q)
        d_lse = torch.empty(d.dec_q.shape[:2], dtype=torch.float32, device="cuda")
        e_out = torch.empty_like(d.ext_q)
        e_lse = torch.empty(d.ext_q.shape[:2], dtype=torch.float32, device="cuda")

        def step():
            s_ext = st2 if branches else st
            if branches:
                fork.record(st)
                st2.wait_event(fork)
            lib.kv_append(d.k_pool, d.v_pool, d.k_new[:nd], d.v_new[:nd], d.slot_mapping[:nd], stream=st)
            lib.paged_decode(d.dec_q, d.k_pool, d.v_pool, d.dec_kv_indptr, d.dec_kv_indices,
                             d.dec_kv_lens, b.sm_scale, out=d_out, lse=d_lse, workspace=dws, stream=st,
                             max_ctas=ctas)
            lib.kv_append(d.k_pool, d.v_pool, d.k_new[nd:], d.v_new[nd:], d.slot_mapping[nd:],
                          stream=s_ext)
            lib.paged_extend(d.ext_q, d.k_pool, d.v_pool, d.ext_qo_indptr, d.ext_kv_indptr,
                             d.ext_kv_indices, d.ext_prefix_lens, b.max_extend_len, b.sm_scale,
                             out=e_out, lse=e_lse, workspace=ews, stream=s_ext)
            if branches:
                join.record(st2)
                st.wait_event(join)

        if branches:
            with torch.cuda.stream(st):
                step()  # warm-up outside the capture
            st.synchronize()
            d = DeviceBatch(b)  # fresh pool: the capture below must start from the same state
            d_out.zero_(), d_lse.zero_(), e_out.zero_(), e_lse.zero_()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=st):
                step()
            g.replay()
        else:
            with torch.cuda.stream(st):
                step()
        torch.cuda.synchronize()
        return d, (d_out, d_lse, e_out, e_lse)

    d_ser, serial = run(False)
    d_br, branched = run(True)
    for x, y in zip(branched, serial):
        assert bits_equal(x, y) if x.dtype == torch.bfloat16 else torch.equal(x, y)
    kp, vp = oracle.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.slot_mapping, 16)
    assert bits_equal(d_br.k_pool, kp) and bits_equal(d_br.v_pool, vp)
    o_ref, l_ref = oracle.paged_decode(b.dec_q, kp, vp, b.dec_kv_indptr, b.dec_kv_indices,
                                       b.dec_kv_lens, 16, b.sm_scale)
    assert_attention_close(branched[0], branched[1], o_ref, l_ref, what="two-branch decode")
    o_ref, l_ref = oracle.paged_extend(b.ext_q, kp, vp, b.ext_qo_indptr, b.ext_kv_indptr,
                                       b.ext_kv_indices, b.ext_prefix_lens, 16, b.sm_scale)
    assert_attention_close(branched[2], branched[3], o_ref, l_ref, what="two-branch extend")

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

    def step():
        lib.kv_append(d.k_pool, d.v_pool, d.k_new, d.v_new, d.slot_mapping, stream=st)
        lib.paged_decode(d.dec_q, d.k_pool, d.v_pool, d.dec_kv_indptr, d.dec_kv_indices, d.dec_kv_lens,
                         b1.sm_scale, out=d_out, lse=d_lse, workspace=dws, stream=st)
        lib.paged_extend(d.ext_q, d.k_pool, d.v_pool, d.ext_qo_indptr, d.ext_kv_indptr, d.ext_kv_indices,
                         d.ext_prefix_lens, max_e, b1.sm_scale, out=e_out, lse=e_lse, stream=st)

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

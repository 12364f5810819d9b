"""Pins for the oracle's shared-prefix (cascade) level, each resting on something other than the
function itself:

- brute force: the pure-Python dense attention over contiguous K/V, every position visible;
- the cascade identity: the state over the shared pages merged with a decode over each request's
  own pages equals the decode over the whole page list (the decode is pinned by brute force);
- closed forms: q = 0 gives the mean of the part's V rows and lse = ln(kv_len); an empty part
  gives o = 0 and lse = -inf;
- a planted mistake (a causal mask over the shared positions) is caught.
"""

import math

import numpy as np
import pytest
import torch

import oracle
import oracle.attention as oa
from workloads import random_small_batch
from _fixtures import contiguous_case
from test_oracle_pins import brute_attention, kv_head_list, _worst


def _parts_case(seed, lens, Hq, Hkv, D, ps):
    """Parts over contiguous K/V scattered into pages; queries read and written at unrelated
    rows (two parts read the same query rows, output rows in a different order)."""
    contig, paged = contiguous_case(seed, lens=lens, Hq=Hq, Hkv=Hkv, D=D, page_size=ps)
    rng = np.random.default_rng(seed + 7)
    Nq = 9
    q = torch.tensor(rng.standard_normal((Nq, Hq, D)), dtype=torch.float32).to(torch.bfloat16)
    P = len(lens)
    q_len = [int(x) for x in rng.integers(1, 4, size=P)]
    q_start = [int(rng.integers(0, Nq - n + 1)) for n in q_len]
    q_start[-1] = q_start[0]  # two parts on the same query rows
    q_len[-1] = q_len[0]
    o_start, cur = [0] * P, 0
    for p in reversed(range(P)):  # outputs laid out in reverse part order
        o_start[p] = cur
        cur += q_len[p]
    num_out = cur + 2  # two rows nobody writes
    as_i32 = lambda v: torch.tensor(v, dtype=torch.int32)
    args = dict(q_start=as_i32(q_start), q_len=as_i32(q_len), o_start=as_i32(o_start))
    return contig, paged, q, args, num_out


@pytest.mark.parametrize("ps", [1, 4, 16])
@pytest.mark.parametrize("Hq,Hkv", [(2, 2), (6, 2), (4, 1)])
def test_shared_prefix_matches_bruteforce(ps, Hq, Hkv):
    D = 8
    lens = [5, 17, 1, 33]
    contig, paged, q, args, num_out = _parts_case(40 + ps + Hq, lens, Hq, Hkv, D, ps)
    scale = 1.0 / math.sqrt(D)
    o, lse = oracle.shared_prefix_attention(q, paged["k_pool"], paged["v_pool"], args["q_start"],
                                            args["q_len"], args["o_start"], paged["kv_indptr"],
                                            paged["kv_indices"], paged["kv_lens"], num_out, ps, scale)
    qf = q.float().numpy().astype(np.float64)
    kvh = kv_head_list(Hq, Hkv)
    err = 0.0
    written = np.zeros(num_out, dtype=bool)
    for p, L in enumerate(lens):
        for i in range(int(args["q_len"][p])):
            r_in, r_out = int(args["q_start"][p]) + i, int(args["o_start"][p]) + i
            written[r_out] = True
            for h in range(Hq):
                g = kvh[h]
                bo, bl = brute_attention(qf[r_in, h].tolist(), contig["K"][p][:, g].tolist(),
                                         contig["V"][p][:, g].tolist(), L, scale)
                err = _worst(err, np.abs(np.array(bo) - o[r_out, h]), abs(bl - lse[r_out, h]))
    assert err < 1e-12
    assert np.isnan(o[~written]).all() and np.isnan(lse[~written]).all()


def _cascade_pieces(b, cut_pages):
    """Shared pages of the decode sharers (share group 0) split at ``cut_pages``; each sharer's own
    pages after them.  Returns the part arrays, the suffix page lists and the sharer list."""
    ps = b.page_size
    shared = b.shared_pages[0].to(torch.int32)
    sharers = [i for i, r in enumerate(b.requests) if r.kind == "decode" and r.share_group == 0]
    assert sharers == list(range(sharers[0], sharers[0] + len(sharers)))  # contiguous rows
    cuts = [0] + list(cut_pages) + [shared.numel()]
    indptr, indices, lens = [0], [], []
    for a, c in zip(cuts[:-1], cuts[1:]):
        indices += shared[a:c].tolist()
        indptr.append(len(indices))
        lens.append((c - a) * ps)
    S = len(lens)
    B = b.num_decode
    parts = dict(q_start=torch.full((S,), sharers[0], dtype=torch.int32),
                 q_len=torch.full((S,), len(sharers), dtype=torch.int32),
                 o_start=torch.tensor([s * B + sharers[0] for s in range(S)], dtype=torch.int32),
                 kv_indptr=torch.tensor(indptr, dtype=torch.int32),
                 kv_indices=torch.tensor(indices, dtype=torch.int32),
                 kv_lens=torch.tensor(lens, dtype=torch.int32))
    sp = shared.numel()
    s_indptr, s_indices, s_lens = [0], [], []
    for r in range(B):
        lo, hi = int(b.dec_kv_indptr[r]), int(b.dec_kv_indptr[r + 1])
        skip = sp if r in sharers else 0
        s_indices += b.dec_kv_indices[lo + skip:hi].tolist()
        s_indptr.append(len(s_indices))
        s_lens.append(int(b.dec_kv_lens[r]) - skip * ps)
    suffix = dict(kv_indptr=torch.tensor(s_indptr, dtype=torch.int32),
                  kv_indices=torch.tensor(s_indices, dtype=torch.int32),
                  kv_lens=torch.tensor(s_lens, dtype=torch.int32))
    return parts, suffix, sharers


@pytest.mark.parametrize("cut_pages", [(), (1,), (2, 3)])
def test_cascade_identity_equals_decode(cut_pages):
    b = random_small_batch(71, page_size=4, num_q_heads=4, num_kv_heads=2, head_dim=8,
                           decode_lens=(3, 30, 25, 40, 7), decode_new=1, share_decode_prefix=16)
    kp, vp = oracle.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.slot_mapping, b.page_size)
    parts, suffix, sharers = _cascade_pieces(b, cut_pages)
    assert len(sharers) == 3
    B, S = b.num_decode, len(cut_pages) + 1
    o_p, l_p = oracle.shared_prefix_attention(b.dec_q, kp, vp, parts["q_start"], parts["q_len"],
                                              parts["o_start"], parts["kv_indptr"], parts["kv_indices"],
                                              parts["kv_lens"], S * B, b.page_size, b.sm_scale)
    o_s, l_s = oracle.paged_decode(b.dec_q, kp, vp, suffix["kv_indptr"], suffix["kv_indices"],
                                   suffix["kv_lens"], b.page_size, b.sm_scale)
    o_p = o_p.reshape(S, B, *o_p.shape[1:])
    l_p = l_p.reshape(S, B, -1)
    # rows that share nothing have empty shared splits
    for r in range(B):
        if r not in sharers:
            o_p[:, r], l_p[:, r] = 0.0, -np.inf
    o, lse = oracle.merge_states(np.concatenate([o_p, o_s[None]]), np.concatenate([l_p, l_s[None]]))
    o_ref, l_ref = oracle.paged_decode(b.dec_q, kp, vp, b.dec_kv_indptr, b.dec_kv_indices,
                                       b.dec_kv_lens, b.page_size, b.sm_scale)
    assert np.abs(o - o_ref).max() < 1e-12 and np.abs(lse - l_ref).max() < 1e-12


def test_shared_prefix_closed_forms():
    D, ps = 8, 4
    lens = [6, 0, 9]
    contig, paged, _, args, num_out = _parts_case(5, lens, 2, 1, D, ps)
    q = torch.zeros((9, 2, D), dtype=torch.bfloat16)
    o, lse = oracle.shared_prefix_attention(q, paged["k_pool"], paged["v_pool"], args["q_start"],
                                            args["q_len"], args["o_start"], paged["kv_indptr"],
                                            paged["kv_indices"], paged["kv_lens"], num_out, ps, 0.3)
    for p, L in enumerate(lens):
        rows = slice(int(args["o_start"][p]), int(args["o_start"][p]) + int(args["q_len"][p]))
        if L == 0:
            assert (o[rows] == 0).all() and np.isneginf(lse[rows]).all()
        else:
            mean_v = contig["V"][p][:, 0].mean(axis=0)
            assert np.abs(o[rows] - mean_v).max() < 1e-12
            assert np.abs(lse[rows] - math.log(L)).max() < 1e-12


def test_pin_catches_causal_mask_over_shared_part(monkeypatch):
    real = oa.attend_rows

    def causal_rows(q, K, V, visible, scale, return_probs=False):  # planted: row i sees i+1 keys
        vis = np.minimum(np.asarray(visible), np.arange(1, len(np.asarray(visible)) + 1))
        return real(q, K, V, vis, scale, return_probs)

    monkeypatch.setattr(oa, "attend_rows", causal_rows)
    with pytest.raises(AssertionError):
        test_shared_prefix_matches_bruteforce(4, 6, 2)

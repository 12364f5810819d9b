"""Pins for the CPU oracle: each check rests on something other than the oracle itself.

- brute force: a pure-Python triple loop over contiguous (never paged) K/V;
- hand-derived worked examples (tests/golden/worked_examples.json);
- closed forms (q = 0, constant V, length 1) and a library routine
  (torch scaled_dot_product_attention in fp64 with an explicit mask);
- invariants (page relabelling, softmax rows summing to 1, split/merge = unsplit,
  decode = extend with one query);
- a brute-force byte check of the KV append, and of the RoPE append (pure-Python rotation per
  token at its own position, bf16 rounding with exact rationals, V bit copies, padding skipped).
The mutation tests at the end plant plausible mistakes in the oracle (on the
CPU) and check that a pin catches each one.
"""

import math
import struct
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import oracle.attention as oa
from workloads import random_small_batch
from _fixtures import contiguous_case, golden_tensors, load_golden


# ---------------------------------------------------------------------------
# brute force over contiguous K/V (pure Python, math.exp, no numpy)
# ---------------------------------------------------------------------------
def brute_attention(q_vec, K_rows, V_rows, n_visible, scale):
    scores = []
    for j in range(n_visible):
        s = 0.0
        for d in range(len(q_vec)):
            s += q_vec[d] * K_rows[j][d]
        scores.append(s * scale)
    m = max(scores)
    w = [math.exp(s - m) for s in scores]
    tot = sum(w)
    out = [0.0] * len(V_rows[0])
    for j in range(n_visible):
        for d in range(len(out)):
            out[d] += w[j] * V_rows[j][d]
    return [x / tot for x in out], m + math.log(tot)


def _worst(err, *vals):
    """Running maximum that treats NaN as an infinite error (Python's max() would drop it)."""
    for v in vals:
        v = float(np.max(v))
        err = math.inf if math.isnan(v) else max(err, v)
    return err


def kv_head_list(Hq, Hkv):
    # repeat each kv head once per member of its group, in order
    G = Hq // Hkv
    heads = []
    for g in range(Hkv):
        heads += [g] * G
    return heads


def _pin_decode_bruteforce(seed, lens, Hq, Hkv, D, ps):
    contig, paged = contiguous_case(seed, lens=lens, Hq=Hq, Hkv=Hkv, D=D, page_size=ps)
    rng = np.random.default_rng(seed + 1)
    q = torch.tensor(rng.standard_normal((len(lens), Hq, D)), dtype=torch.float32).to(torch.bfloat16)
    scale = 1.0 / math.sqrt(D)
    o, lse = oracle.paged_decode(q, paged["k_pool"], paged["v_pool"], paged["kv_indptr"],
                                 paged["kv_indices"], paged["kv_lens"], ps, scale)
    qf = q.float().numpy().astype(np.float64)
    kvh = kv_head_list(Hq, Hkv)
    err = 0.0
    for b, L in enumerate(lens):
        for h in range(Hq):
            g = kvh[h]
            Krows = contig["K"][b][:, g].tolist()
            Vrows = contig["V"][b][:, g].tolist()
            bo, bl = brute_attention(qf[b, h].tolist(), Krows, Vrows, L, scale)
            err = _worst(err, np.abs(np.array(bo) - o[b, h]), abs(bl - lse[b, h]))
    return err


def _pin_extend_bruteforce(seed, prefixes, exts, Hq, Hkv, D, ps):
    lens = [p + e for p, e in zip(prefixes, exts)]
    contig, paged = contiguous_case(seed, lens=lens, Hq=Hq, Hkv=Hkv, D=D, page_size=ps)
    rng = np.random.default_rng(seed + 2)
    N = sum(exts)
    q = torch.tensor(rng.standard_normal((N, Hq, D)), dtype=torch.float32).to(torch.bfloat16)
    qo = torch.tensor(np.concatenate([[0], np.cumsum(exts)]), dtype=torch.int32)
    pref = torch.tensor(prefixes, dtype=torch.int32)
    scale = 1.0 / math.sqrt(D)
    o, lse = oracle.paged_extend(q, paged["k_pool"], paged["v_pool"], qo, paged["kv_indptr"],
                                 paged["kv_indices"], pref, ps, scale)
    qf = q.float().numpy().astype(np.float64)
    kvh = kv_head_list(Hq, Hkv)
    err = 0.0
    row = 0
    for b, (P, E) in enumerate(zip(prefixes, exts)):
        for i in range(E):
            for h in range(Hq):
                g = kvh[h]
                Krows = contig["K"][b][:, g].tolist()
                Vrows = contig["V"][b][:, g].tolist()
                # query i of the extend is at absolute position P + i and sees 0..P+i
                bo, bl = brute_attention(qf[row, h].tolist(), Krows, Vrows, P + i + 1, scale)
                err = _worst(err, np.abs(np.array(bo) - o[row, h]), abs(bl - lse[row, h]))
            row += 1
    return err


@pytest.mark.parametrize("ps", [1, 3, 16])
@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (6, 2), (7, 1)])
def test_decode_matches_bruteforce(ps, Hq, Hkv):
    assert _pin_decode_bruteforce(11 + ps + Hq, [1, 5, 17, 33], Hq, Hkv, 8, ps) < 1e-12


@pytest.mark.parametrize("ps", [1, 4, 16])
@pytest.mark.parametrize("Hq,Hkv", [(2, 2), (4, 2), (3, 1)])
def test_extend_matches_bruteforce(ps, Hq, Hkv):
    assert _pin_extend_bruteforce(5 + ps * Hq, [0, 3, 16, 21], [5, 1, 7, 4], Hq, Hkv, 8, ps) < 1e-12


# ---------------------------------------------------------------------------
# hand-derived worked examples
# ---------------------------------------------------------------------------
GOLD = load_golden()


@pytest.mark.parametrize("name", [k for k, v in GOLD.items() if v["kind"] == "decode"])
def test_golden_decode(name):
    c = GOLD[name]
    t = golden_tensors(c)
    o, lse = oracle.paged_decode(t["q"], t["k_pool"], t["v_pool"], t["kv_indptr"], t["kv_indices"],
                                 t["kv_lens"], c["page_size"], c["sm_scale"])
    np.testing.assert_allclose(o, np.array(c["expect_o"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, np.array(c["expect_lse"]), rtol=0, atol=1e-12)


@pytest.mark.parametrize("name", [k for k, v in GOLD.items() if v["kind"] == "extend"])
def test_golden_extend(name):
    c = GOLD[name]
    t = golden_tensors(c)
    o, lse = oracle.paged_extend(t["q"], t["k_pool"], t["v_pool"], t["qo_indptr"], t["kv_indptr"],
                                 t["kv_indices"], t["prefix_lens"], c["page_size"], c["sm_scale"])
    np.testing.assert_allclose(o, np.array(c["expect_o"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, np.array(c["expect_lse"]), rtol=0, atol=1e-12)


def test_golden_merge():
    c = GOLD["merge_two_splits"]
    o, lse = oracle.merge_states(np.array(c["o_parts"]), np.array(c["lse_parts"]))
    np.testing.assert_allclose(o, np.array(c["expect_o"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, np.array(c["expect_lse"]), rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# closed forms and a library routine
# ---------------------------------------------------------------------------
def _small(seed=3, **kw):
    args = dict(page_size=4, num_q_heads=6, num_kv_heads=2, head_dim=16,
                decode_lens=(1, 4, 9, 30), extend=((0, 5), (6, 3), (13, 8)))
    args.update(kw)
    return random_small_batch(seed, **args)


def _after_append(b):
    return oracle.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.slot_mapping, b.page_size)


def test_q_zero_gives_mean_of_visible_v():
    b = _small()
    kp, vp = _after_append(b)
    q0 = torch.zeros_like(b.dec_q)
    o, lse = oracle.paged_decode(q0, kp, vp, b.dec_kv_indptr, b.dec_kv_indices, b.dec_kv_lens,
                                 b.page_size, b.sm_scale)
    G = b.num_q_heads // b.num_kv_heads
    for r in range(b.num_decode):
        L = int(b.dec_kv_lens[r])
        V = oa.as_f64(oracle.request_kv(vp, b.dec_kv_indptr, b.dec_kv_indices, r, L, b.page_size))
        for h in range(b.num_q_heads):
            np.testing.assert_allclose(o[r, h], V[:, h // G].mean(0), atol=1e-13, rtol=0)
            assert abs(lse[r, h] - math.log(L)) < 1e-13


def test_constant_v_rows_give_that_row():
    b = _small(seed=4)
    kp, vp = _after_append(b)
    vp = torch.ones_like(vp) * 0.375  # exactly representable in bf16
    o, _ = oracle.paged_extend(b.ext_q, kp, vp, b.ext_qo_indptr, b.ext_kv_indptr, b.ext_kv_indices,
                               b.ext_prefix_lens, b.page_size, b.sm_scale)
    assert np.abs(o - 0.375).max() < 1e-14


def test_length_one_returns_v_exactly():
    b = random_small_batch(5, page_size=2, num_q_heads=4, num_kv_heads=2, head_dim=8,
                           decode_lens=(1, 1, 1), decode_new=1)
    kp, vp = _after_append(b)
    o, lse = oracle.paged_decode(b.dec_q, kp, vp, b.dec_kv_indptr, b.dec_kv_indices, b.dec_kv_lens,
                                 b.page_size, b.sm_scale)
    q = oa.as_f64(b.dec_q)
    for r in range(3):
        V = oa.as_f64(oracle.request_kv(vp, b.dec_kv_indptr, b.dec_kv_indices, r, 1, b.page_size))[0]
        K = oa.as_f64(oracle.request_kv(kp, b.dec_kv_indptr, b.dec_kv_indices, r, 1, b.page_size))[0]
        for h in range(4):
            assert np.array_equal(o[r, h], V[h // 2])
            assert abs(lse[r, h] - b.sm_scale * float(q[r, h] @ K[h // 2])) < 1e-14


def _sdpa_reference(q, K, V, P, scale):
    """torch's fused attention (fp64, CPU) with an explicit boolean mask for a prefix offset."""
    E, L = q.shape[0], K.shape[0]
    mask = torch.zeros(E, L, dtype=torch.bool)
    for i in range(E):
        mask[i, : P + i + 1] = True
    out = torch.nn.functional.scaled_dot_product_attention(
        torch.tensor(q)[None, None], torch.tensor(K)[None, None], torch.tensor(V)[None, None],
        attn_mask=mask[None, None], scale=scale)
    return out[0, 0].numpy()


def test_extend_matches_sdpa_with_prefix_mask():
    b = _small(seed=6, extend=((0, 9), (7, 5), (16, 12)))
    kp, vp = _after_append(b)
    o, _ = oracle.paged_extend(b.ext_q, kp, vp, b.ext_qo_indptr, b.ext_kv_indptr, b.ext_kv_indices,
                               b.ext_prefix_lens, b.page_size, b.sm_scale)
    q = oa.as_f64(b.ext_q)
    G = b.num_q_heads // b.num_kv_heads
    qo = b.ext_qo_indptr.tolist()
    for r in range(b.num_extend):
        P = int(b.ext_prefix_lens[r])
        E = qo[r + 1] - qo[r]
        K = oa.as_f64(oracle.request_kv(kp, b.ext_kv_indptr, b.ext_kv_indices, r, P + E, b.page_size))
        V = oa.as_f64(oracle.request_kv(vp, b.ext_kv_indptr, b.ext_kv_indices, r, P + E, b.page_size))
        for h in range(b.num_q_heads):
            ref = _sdpa_reference(q[qo[r]:qo[r + 1], h], K[:, h // G], V[:, h // G], P, b.sm_scale)
            np.testing.assert_allclose(o[qo[r]:qo[r + 1], h], ref, atol=1e-12, rtol=0)


def test_extend_without_prefix_is_textbook_causal():
    b = _small(seed=7, extend=((0, 11), (0, 4)))
    kp, vp = _after_append(b)
    o, _ = oracle.paged_extend(b.ext_q, kp, vp, b.ext_qo_indptr, b.ext_kv_indptr, b.ext_kv_indices,
                               b.ext_prefix_lens, b.page_size, b.sm_scale)
    q = oa.as_f64(b.ext_q)
    G = b.num_q_heads // b.num_kv_heads
    qo = b.ext_qo_indptr.tolist()
    for r in range(b.num_extend):
        E = qo[r + 1] - qo[r]
        K = oa.as_f64(oracle.request_kv(kp, b.ext_kv_indptr, b.ext_kv_indices, r, E, b.page_size))
        V = oa.as_f64(oracle.request_kv(vp, b.ext_kv_indptr, b.ext_kv_indices, r, E, b.page_size))
        for h in range(b.num_q_heads):
            ref = torch.nn.functional.scaled_dot_product_attention(
                torch.tensor(q[qo[r]:qo[r + 1], h])[None, None], torch.tensor(K[:, h // G])[None, None],
                torch.tensor(V[:, h // G])[None, None], is_causal=True, scale=b.sm_scale)[0, 0].numpy()
            np.testing.assert_allclose(o[qo[r]:qo[r + 1], h], ref, atol=1e-12, rtol=0)


# ---------------------------------------------------------------------------
# invariants
# ---------------------------------------------------------------------------
def test_page_relabelling_is_bit_invariant():
    b = _small(seed=8)
    kp, vp = _after_append(b)
    rng = np.random.default_rng(0)
    perm = torch.tensor(rng.permutation(b.num_pages))
    kp2 = torch.empty_like(kp)
    vp2 = torch.empty_like(vp)
    kp2[perm] = kp
    vp2[perm] = vp
    ind2 = perm[b.dec_kv_indices.long()].to(torch.int32)
    o1, l1 = oracle.paged_decode(b.dec_q, kp, vp, b.dec_kv_indptr, b.dec_kv_indices, b.dec_kv_lens,
                                 b.page_size, b.sm_scale)
    o2, l2 = oracle.paged_decode(b.dec_q, kp2, vp2, b.dec_kv_indptr, ind2, b.dec_kv_lens,
                                 b.page_size, b.sm_scale)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    e_ind2 = perm[b.ext_kv_indices.long()].to(torch.int32)
    o1, l1 = oracle.paged_extend(b.ext_q, kp, vp, b.ext_qo_indptr, b.ext_kv_indptr, b.ext_kv_indices,
                                 b.ext_prefix_lens, b.page_size, b.sm_scale)
    o2, l2 = oracle.paged_extend(b.ext_q, kp2, vp2, b.ext_qo_indptr, b.ext_kv_indptr, e_ind2,
                                 b.ext_prefix_lens, b.page_size, b.sm_scale)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_softmax_rows_sum_to_one_and_respect_mask():
    b = _small(seed=9)
    kp, vp = _after_append(b)
    _, _, probs = oracle.paged_extend(b.ext_q, kp, vp, b.ext_qo_indptr, b.ext_kv_indptr,
                                      b.ext_kv_indices, b.ext_prefix_lens, b.page_size, b.sm_scale,
                                      return_probs=True)
    for (r, h), p in probs.items():
        assert np.abs(p.sum(1) - 1).max() < 1e-12
        P = int(b.ext_prefix_lens[r])
        for i in range(p.shape[0]):
            assert np.all(p[i, P + i + 1:] == 0)
            assert np.all(p[i, : P + i + 1] > 0)
    _, _, probs = oracle.paged_decode(b.dec_q, kp, vp, b.dec_kv_indptr, b.dec_kv_indices,
                                      b.dec_kv_lens, b.page_size, b.sm_scale, return_probs=True)
    for p in probs.values():
        assert abs(p.sum() - 1) < 1e-12


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_split_merge_equals_unsplit(seed):
    b = _small(seed=10 + seed, decode_lens=(1, 7, 40, 64))
    kp, vp = _after_append(b)
    rng = np.random.default_rng(seed)
    bounds = []
    for L in b.dec_kv_lens.tolist():
        S = int(rng.integers(1, 6))
        cuts = sorted(rng.integers(0, L + 1, size=S - 1).tolist())
        bounds.append([0] + cuts + [L])  # repeated cut points make empty splits
    o, lse = oracle.paged_decode(b.dec_q, kp, vp, b.dec_kv_indptr, b.dec_kv_indices, b.dec_kv_lens,
                                 b.page_size, b.sm_scale)
    o2, lse2, _ = oracle.decode_split_reference(b.dec_q, kp, vp, b.dec_kv_indptr, b.dec_kv_indices,
                                                b.dec_kv_lens, b.page_size, b.sm_scale, bounds)
    assert np.abs(o - o2).max() < 1e-12
    assert np.abs(lse - lse2).max() < 1e-12


def test_merge_of_all_empty_splits():
    o, lse = oracle.merge_states(np.zeros((3, 2, 4)), np.full((3, 2), -np.inf))
    assert np.all(o == 0) and np.all(np.isneginf(lse))


def test_decode_equals_extend_with_one_query():
    b = _small(seed=12, decode_lens=(3, 17, 32), extend=())
    kp, vp = _after_append(b)
    o, lse = oracle.paged_decode(b.dec_q, kp, vp, b.dec_kv_indptr, b.dec_kv_indices, b.dec_kv_lens,
                                 b.page_size, b.sm_scale)
    B = b.num_decode
    qo = torch.arange(B + 1, dtype=torch.int32)
    pref = b.dec_kv_lens - 1
    o2, lse2 = oracle.paged_extend(b.dec_q, kp, vp, qo, b.dec_kv_indptr, b.dec_kv_indices, pref,
                                   b.page_size, b.sm_scale)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)


# ---------------------------------------------------------------------------
# KV append, page gather
# ---------------------------------------------------------------------------
def test_kv_append_bruteforce_bytes():
    b = _small(seed=13)
    slots = b.slot_mapping.clone()
    slots[1] = -1  # padding token: skipped
    kp, vp = oracle.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, slots, b.page_size)
    before_k = b.k_pool.view(torch.int16).reshape(-1, b.num_kv_heads * b.head_dim)
    after_k = kp.view(torch.int16).reshape(-1, b.num_kv_heads * b.head_dim)
    after_v = vp.view(torch.int16).reshape(-1, b.num_kv_heads * b.head_dim)
    new_k = b.k_new.view(torch.int16).reshape(len(slots), -1)
    new_v = b.v_new.view(torch.int16).reshape(len(slots), -1)
    written = {}
    for t, s in enumerate(slots.tolist()):
        if s >= 0:
            written[s] = t
    for s in range(after_k.shape[0]):
        if s in written:
            assert torch.equal(after_k[s], new_k[written[s]])
            assert torch.equal(after_v[s], new_v[written[s]])
        else:
            assert torch.equal(after_k[s], before_k[s])  # NaN rows compare by their bits


def test_gather_bruteforce():
    contig, paged = contiguous_case(21, lens=[3, 1, 9], Hq=2, Hkv=2, D=4, page_size=4)
    g = oracle.paged_gather(paged["k_pool"], paged["kv_indptr"], paged["kv_indices"],
                            paged["kv_lens"], 4)
    ref = np.concatenate(contig["K"], 0)
    assert np.array_equal(g.float().numpy().astype(np.float64), ref)


def test_generator_slots_agree_with_page_lists():
    b = _small(seed=14, share_decode_prefix=4)
    kp, vp = _after_append(b)
    # every position a request can see holds a finite value after the append
    for r in range(b.num_decode):
        L = int(b.dec_kv_lens[r])
        assert torch.isfinite(oracle.request_kv(kp, b.dec_kv_indptr, b.dec_kv_indices, r, L,
                                                b.page_size).float()).all()
    for r in range(b.num_extend):
        L = int(b.ext_prefix_lens[r]) + int(b.ext_qo_indptr[r + 1] - b.ext_qo_indptr[r])
        assert torch.isfinite(oracle.request_kv(vp, b.ext_kv_indptr, b.ext_kv_indices, r, L,
                                                b.page_size).float()).all()
    # the appended slots were NaN before the append
    assert torch.isnan(b.k_pool.view(-1, b.num_kv_heads, b.head_dim)[b.slot_mapping].float()).all()


# ---------------------------------------------------------------------------
# mutation tests: plausible oracle mistakes must be caught by a pin above
# ---------------------------------------------------------------------------
def test_pin_catches_wrong_gqa_map(monkeypatch):
    monkeypatch.setattr(oa, "_kv_head_of", lambda h, Hq, Hkv: h % Hkv)
    assert _pin_decode_bruteforce(3, [5, 9], 4, 2, 8, 4) > 1e-3


def test_pin_catches_top_left_causal(monkeypatch):
    orig = oa.attend_rows

    def top_left(q, K, V, visible, scale, return_probs=False):
        vis = np.asarray(visible)
        vis = vis - vis.min() + 1 if vis.size else vis  # forgets the prefix offset
        return orig(q, K, V, vis, scale, return_probs)

    monkeypatch.setattr(oa, "attend_rows", top_left)
    assert _pin_extend_bruteforce(4, [6], [5], 2, 1, 8, 4) > 1e-3


def test_pin_catches_off_by_one_page_row(monkeypatch):
    orig = oa._positions_to_page_rows

    def shifted(kv_indptr, kv_indices, b, kv_len, page_size):
        pages, rows = orig(kv_indptr, kv_indices, b, kv_len, page_size)
        return pages, (rows + 1) % page_size

    monkeypatch.setattr(oa, "_positions_to_page_rows", shifted)
    with np.errstate(invalid="ignore"):
        err = _pin_decode_bruteforce(5, [6, 12], 2, 2, 8, 4)
    assert err > 1e-3  # an unused (NaN) row was read, or the values moved


def test_pin_catches_missing_scale(monkeypatch):
    orig = oa.attend_rows
    monkeypatch.setattr(oa, "attend_rows", lambda q, K, V, vis, scale, rp=False: orig(q, K, V, vis, 1.0, rp))
    assert _pin_decode_bruteforce(6, [7], 2, 2, 16, 4) > 1e-3


# ---------------------------------------------------------------------------
# RoPE (half-split pairing)
# ---------------------------------------------------------------------------
def test_golden_rope():
    c = GOLD["rope_quarter_turns"]
    out = oracle.rope(np.array(c["x"], dtype=np.float64), c["positions"], c["theta"])
    np.testing.assert_allclose(out, np.array(c["expect"]), rtol=0, atol=1e-15)


def _rope_bruteforce(x, pos, theta):
    """Explicit 2x2 rotation of each (i, i + D/2) pair, pure Python."""
    D = len(x)
    y = list(x)
    for i in range(D // 2):
        a = pos * theta ** (-2.0 * i / D)
        c, s = math.cos(a), math.sin(a)
        y[i] = c * x[i] - s * x[i + D // 2]
        y[i + D // 2] = s * x[i] + c * x[i + D // 2]
    return y


def test_rope_matches_explicit_rotation():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((5, 3, 16))
    pos = [0, 1, 17, 4095, 32767]
    out = oracle.rope(x, pos, 1e6)
    for t in range(5):
        for h in range(3):
            ref = _rope_bruteforce(x[t, h].tolist(), pos[t], 1e6)
            assert np.abs(np.array(ref) - out[t, h]).max() < 1e-12


def test_rope_invariants():
    rng = np.random.default_rng(1)
    D = 128
    q = rng.standard_normal((1, 1, D))
    k = rng.standard_normal((1, 1, D))
    # position 0 is the identity; each pair keeps its norm
    assert np.array_equal(oracle.rope(q, [0], 1e4), q)
    r = oracle.rope(q, [777], 1e4)[0, 0]
    assert np.allclose(r[: D // 2] ** 2 + r[D // 2:] ** 2, q[0, 0, : D // 2] ** 2 + q[0, 0, D // 2:] ** 2, atol=1e-12)
    # scores depend only on the relative position
    for m, n in ((10, 3), (5000, 4993), (2, 9)):
        a = oracle.rope(q, [m], 1e4)[0, 0] @ oracle.rope(k, [n], 1e4)[0, 0]
        b = oracle.rope(q, [m - n], 1e4)[0, 0] @ k[0, 0]
        assert abs(a - b) < 1e-9


def test_pin_catches_interleaved_rope(monkeypatch):
    """The adjacent-pair (interleaved) convention is a different rotation: the golden case sees it."""
    def interleaved(x, positions, theta):
        x = np.asarray(x, dtype=np.float64)
        D = x.shape[-1]
        ang = oa.rope_angles(positions, D, theta)[:, None, :]
        c, s = np.cos(ang), np.sin(ang)
        ev, od = x[..., 0::2], x[..., 1::2]
        y = np.empty_like(x)
        y[..., 0::2] = ev * c - od * s
        y[..., 1::2] = od * c + ev * s
        return y

    monkeypatch.setattr(oa, "rope", interleaved)
    c = GOLD["rope_quarter_turns"]
    out = oa.rope(np.array(c["x"], dtype=np.float64), c["positions"], c["theta"])
    assert np.abs(out - np.array(c["expect"])).max() > 0.1


# ---------------------------------------------------------------------------
# RoPE fused with the KV append: K rotated at its own position and rounded once to bf16, V copied,
# padding skipped, nothing else touched
# ---------------------------------------------------------------------------
def _bf16_rne_bruteforce(x):
    """The bf16 value nearest to x (ties to the even significand), found with exact rationals:
    the two bf16 neighbours are consecutive multiples of the spacing at |x|, and the nearer one
    wins.  Independent of the oracle's frexp/round formulation."""
    if x == 0.0 or math.isnan(x) or math.isinf(x):
        return x
    _, e = math.frexp(abs(x))              # 2**(e-1) <= |x| < 2**e
    ulp = Fraction(2) ** (max(e, -125) - 8)  # 8 significant bits; fixed spacing below 2**-126
    fx = Fraction(x)
    lo = (fx / ulp).__floor__()
    below, above = fx - lo * ulp, (lo + 1) * ulp - fx
    n = lo if below < above or (below == above and lo % 2 == 0) else lo + 1
    y = float(n * ulp)
    return math.copysign(math.inf, x) if abs(y) >= 2.0 ** 128 else y


def _bits_of_bf16(v):
    """bf16 bit pattern of a value that is exactly a bf16 value (the top half of its fp32 bits)."""
    b = struct.unpack("<I", struct.pack("<f", v))[0]
    assert b & 0xFFFF == 0
    b >>= 16
    return b - 0x10000 if b >= 0x8000 else b  # as int16, like torch's int16 view


def _pin_rope_append(seed=41, theta=1.0e4):
    """Check oracle.rope_kv_append against a byte-level brute force; returns the failures."""
    b = _small(seed=seed)
    T, Hkv, D, ps = b.num_new_tokens, b.num_kv_heads, b.head_dim, b.page_size
    gen = torch.Generator().manual_seed(seed)
    positions = torch.randint(0, 20000, (T,), generator=gen, dtype=torch.int32)
    slots = b.slot_mapping.clone()
    slots[2] = -1  # padding token
    kp, vp, k_rot = oa.rope_kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, slots, positions, ps, theta)
    fails = []
    width = Hkv * D
    before_k = b.k_pool.view(torch.int16).reshape(-1, width)
    before_v = b.v_pool.view(torch.int16).reshape(-1, width)
    after_k = kp.view(torch.int16).reshape(-1, width)
    after_v = vp.view(torch.int16).reshape(-1, width)
    new_v = b.v_new.view(torch.int16).reshape(T, width)
    kx = b.k_new.float().double().numpy()
    written = {}
    for t, s in enumerate(slots.tolist()):
        if s >= 0:
            written[s] = t
    for s in range(after_k.shape[0]):
        t = written.get(s)
        if t is None:  # padding or untouched slot: every byte as before (NaN rows by their bits)
            if not (torch.equal(after_k[s], before_k[s]) and torch.equal(after_v[s], before_v[s])):
                fails.append(f"slot {s} changed without a token")
            continue
        if not torch.equal(after_v[s], new_v[t]):
            fails.append(f"V of token {t} is not a bit copy")
        p = int(positions[t])
        for h in range(Hkv):
            rot = _rope_bruteforce(kx[t, h].tolist(), p, theta)
            if np.abs(np.array(rot) - k_rot[t, h]).max() > 1e-12:
                fails.append(f"rotation of token {t} head {h}")
            want = [_bits_of_bf16(_bf16_rne_bruteforce(v)) for v in rot]
            got = after_k[s, h * D:(h + 1) * D].tolist()
            if got != want:
                fails.append(f"K bits of token {t} head {h}")
    return fails


def test_rope_append_bruteforce_bytes():
    assert _pin_rope_append() == []


def test_bf16_rounding_ties_and_edges():
    """Round-to-nearest-even cases fixed by the bf16 format itself (8 significant bits)."""
    r = oracle.bf16_round_nearest_even
    cases = {
        1.0 + 2.0 ** -8: 1.0,                           # halfway, even neighbour below
        1.0 + 3 * 2.0 ** -8: 1.0 + 2.0 ** -6,           # halfway, even neighbour above
        1.0 + 2.0 ** -8 + 2.0 ** -40: 1.0 + 2.0 ** -7,  # just above halfway (a cast via fp32 gives 1.0)
        -(1.0 + 2.0 ** -8 + 2.0 ** -40): -(1.0 + 2.0 ** -7),
        2.0 ** -133: 2.0 ** -133,                       # smallest subnormal
        3 * 2.0 ** -135: 2.0 ** -133,                   # 0.75 of it rounds up
        (2.0 - 2.0 ** -7) * 2.0 ** 127: (2.0 - 2.0 ** -7) * 2.0 ** 127,  # largest finite
        (2.0 - 2.0 ** -8) * 2.0 ** 127: math.inf,       # halfway to 2**128: overflows
        0.0: 0.0,
    }
    got = r(np.array(list(cases)))
    assert got.tolist() == list(cases.values())
    rng = np.random.default_rng(3)
    x = rng.standard_normal(2000) * np.exp(rng.uniform(-30, 30, 2000))
    assert r(x).tolist() == [_bf16_rne_bruteforce(v) for v in x.tolist()]


def test_pin_catches_rotated_v(monkeypatch):
    orig = oa.rope_kv_append

    def rotates_v(k_pool, v_pool, k_new, v_new, slot_mapping, positions, page_size, theta):
        v_rot = oa.bf16_round_nearest_even(oa.rope(oa.as_f64(v_new), oa._as_int(positions), theta))
        v_b = torch.tensor(v_rot).float().to(torch.bfloat16)
        return orig(k_pool, v_pool, k_new, v_b, slot_mapping, positions, page_size, theta)

    monkeypatch.setattr(oa, "rope_kv_append", rotates_v)
    assert any("V of token" in f for f in _pin_rope_append())


def test_pin_catches_token_index_as_position(monkeypatch):
    orig = oa.rope_kv_append

    def by_index(k_pool, v_pool, k_new, v_new, slot_mapping, positions, page_size, theta):
        return orig(k_pool, v_pool, k_new, v_new, slot_mapping, np.arange(len(positions)), page_size, theta)

    monkeypatch.setattr(oa, "rope_kv_append", by_index)
    assert any("rotation of token" in f for f in _pin_rope_append())


def test_pin_catches_truncation(monkeypatch):
    def truncate(x):
        x = np.asarray(x, dtype=np.float64)
        m, e = np.frexp(x)
        step = np.maximum(e, -125) - 8
        return np.ldexp(np.trunc(np.ldexp(x, -step)), step)

    monkeypatch.setattr(oa, "bf16_round_nearest_even", truncate)
    fails = _pin_rope_append()
    assert fails and all("K bits" in f for f in fails)


def test_pin_catches_padding_written(monkeypatch):
    orig = oa.kv_append

    def no_skip(k_pool, v_pool, k_new, v_new, slot_mapping, page_size):
        s = oa._as_int(slot_mapping).copy()
        free = next(x for x in range(k_pool.shape[0] * page_size) if x not in set(s.tolist()))
        s[s < 0] = free  # a padding token written into a slot no token owns
        return orig(k_pool, v_pool, k_new, v_new, s, page_size)

    monkeypatch.setattr(oa, "kv_append", no_skip)
    assert any("changed without a token" in f or "V of token" in f for f in _pin_rope_append())

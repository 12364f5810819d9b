"""fp64 reference for paged KV append, page gather, decode, extend and LSE merge.

Test infrastructure only (see the package docstring).  The functions follow
the behaviour the Mini-SGLang README ("Reference Attention Backends", torch
backend) gives its plain-PyTorch attention backend: gather each request's K/V
from the paged pool, map query heads onto KV heads the way
``repeat_interleave`` does, and apply causal attention offset by the cached
prefix.  Page layout and slot convention follow the nanoSGLang README
("Architecture": block-based KV cache in FlashInfer NHD layout) and the
mini-sglang-from-Scratch handbook ("What you will be able to do": paged KV
pool, page table and token pool).  Split-KV partials and their merge restate
the log-sum-exp identity of flash-decoding; no page prints it, so it is the
plainest reading that keeps the split result equal to the unsplit one.

Precision: inputs are bf16 and are widened exactly to fp64; every product,
sum, exponential and logarithm below is fp64; outputs are returned unrounded.
"""

from __future__ import annotations

import numpy as np

try:  # torch is only used to read bf16 tensors from the input generator
    import torch
except Exception:  # pragma: no cover - numpy-only use
    torch = None


def as_f64(x) -> np.ndarray:
    """Exact widening of a bf16/fp32 tensor or array to fp64."""
    if torch is not None and isinstance(x, torch.Tensor):
        x = x.detach().cpu()
        if x.dtype in (torch.bfloat16, torch.float16):
            x = x.to(torch.float32)  # exact: every bf16/fp16 value is an fp32 value
        return x.numpy().astype(np.float64)
    return np.asarray(x, dtype=np.float64)


def _as_int(x) -> np.ndarray:
    if torch is not None and isinstance(x, torch.Tensor):
        return x.detach().cpu().numpy().astype(np.int64)
    return np.asarray(x, dtype=np.int64)


# ---------------------------------------------------------------------------
# KV-cache write (the handbook's "KV-cache writes"; nanoSGLang's zero-copy KV)
# ---------------------------------------------------------------------------
def kv_append(k_pool, v_pool, k_new, v_new, slot_mapping, page_size):
    """Write token t's K/V row into flat pool slot ``slot_mapping[t]``.

    The pool ``[num_pages, page_size, Hkv, D]`` is addressed as rows
    ``slot = page * page_size + row``.  A negative slot marks a padding token
    and writes nothing.  Returns new pools; the copy is bit-exact (the dtype of
    the pools is kept, no arithmetic happens).
    """
    slots = _as_int(slot_mapping)
    kp = k_pool.clone() if torch is not None and isinstance(k_pool, torch.Tensor) else np.array(k_pool, copy=True)
    vp = v_pool.clone() if torch is not None and isinstance(v_pool, torch.Tensor) else np.array(v_pool, copy=True)
    num_pages = kp.shape[0]
    for t, s in enumerate(slots.tolist()):
        if s < 0:
            continue
        page, row = divmod(s, page_size)
        if page >= num_pages:
            raise IndexError(f"slot {s} lies outside a pool of {num_pages} pages")
        kp[page, row] = k_new[t]
        vp[page, row] = v_new[t]
    return kp, vp


# ---------------------------------------------------------------------------
# Page gather: position j of request b lives in page kv_indices[indptr[b] + j // ps], row j % ps
# ---------------------------------------------------------------------------
def _positions_to_page_rows(kv_indptr, kv_indices, b, kv_len, page_size):
    indptr = _as_int(kv_indptr)
    indices = _as_int(kv_indices)
    j = np.arange(kv_len, dtype=np.int64)
    page_slot = indptr[b] + j // page_size
    if kv_len and page_slot[-1] >= indptr[b + 1]:
        raise IndexError(f"request {b}: kv_len {kv_len} exceeds its {indptr[b+1]-indptr[b]} pages")
    pages = indices[page_slot]
    rows = j % page_size
    return pages, rows


def request_kv(pool, kv_indptr, kv_indices, b, kv_len, page_size):
    """Request b's K (or V) rows ``[kv_len, Hkv, D]`` gathered from the pool, in position order.

    Keeps the pool's dtype (a bit-exact copy).
    """
    pages, rows = _positions_to_page_rows(kv_indptr, kv_indices, b, kv_len, page_size)
    if torch is not None and isinstance(pool, torch.Tensor):
        return pool[torch.as_tensor(pages), torch.as_tensor(rows)]
    return np.asarray(pool)[pages, rows]


def paged_gather(pool, kv_indptr, kv_indices, kv_lens, page_size):
    """All requests' rows concatenated: ``[sum(kv_lens), Hkv, D]``, bit-exact."""
    lens = _as_int(kv_lens)
    parts = [request_kv(pool, kv_indptr, kv_indices, b, int(L), page_size) for b, L in enumerate(lens)]
    if torch is not None and isinstance(pool, torch.Tensor):
        if not parts:
            return pool.new_zeros((0,) + tuple(pool.shape[2:]))
        return torch.cat(parts, 0)
    if not parts:
        return np.zeros((0,) + np.asarray(pool).shape[2:], dtype=np.asarray(pool).dtype)
    return np.concatenate(parts, 0)


# ---------------------------------------------------------------------------
# Softmax attention of query rows over a KV sequence, with a per-row visible length
# ---------------------------------------------------------------------------
def attend_rows(q, K, V, visible, scale, return_probs=False):
    """Attention of query rows over KV positions ``[0, visible[i])``.

    q ``[n, D]``, K, V ``[L, D]`` (fp64), ``visible`` ``[n]`` ints.  Row i:
    ``s_j = scale * q_i . k_j`` for visible j, ``m = max_j s_j``,
    ``p_j = exp(s_j - m)``, ``l = sum_j p_j``, ``lse = m + ln l``,
    ``o = sum_j p_j v_j / l``.  A row with nothing visible gets ``o = 0`` and
    ``lse = -inf`` (the empty-split convention).
    """
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    visible = np.asarray(visible, dtype=np.int64)
    n, D = q.shape
    L = K.shape[0]
    s = (q @ K.T) * scale  # [n, L]
    j = np.arange(L)[None, :]
    mask = j < visible[:, None]
    s = np.where(mask, s, -np.inf)
    o = np.zeros((n, V.shape[1]), dtype=np.float64)
    lse = np.full(n, -np.inf, dtype=np.float64)
    probs = np.zeros((n, L), dtype=np.float64)
    has = visible > 0
    if has.any():
        sh = s[has]
        m = sh.max(axis=1, keepdims=True)
        p = np.exp(sh - m)
        l = p.sum(axis=1, keepdims=True)
        o[has] = (p @ V) / l
        lse[has] = m[:, 0] + np.log(l[:, 0])
        probs[has] = p / l
    if return_probs:
        return o, lse, probs
    return o, lse


def attend_range(q, K, V, j0, j1, scale):
    """Partial state of query rows over KV positions ``[j0, j1)`` only: ``(o_s, lse_s)``.

    o_s is normalised by the split's own sum; an empty range gives
    ``o_s = 0`` and ``lse_s = -inf``.
    """
    q = np.asarray(q, dtype=np.float64)
    if j1 <= j0:
        return np.zeros((q.shape[0], np.asarray(V).shape[1])), np.full(q.shape[0], -np.inf)
    Ks = np.asarray(K, dtype=np.float64)[j0:j1]
    Vs = np.asarray(V, dtype=np.float64)[j0:j1]
    return attend_rows(q, Ks, Vs, np.full(q.shape[0], j1 - j0), scale)


def merge_states(o_parts, lse_parts):
    """Merge split partials: ``lse = ln sum_s exp(lse_s)``, ``o = sum_s exp(lse_s - lse) o_s``.

    o_parts ``[S, ..., D]``, lse_parts ``[S, ...]``.  Splits with
    ``lse_s = -inf`` contribute nothing; if every split is empty the result is
    ``o = 0``, ``lse = -inf``.
    """
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    m = lse_parts.max(axis=0)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    w = np.exp(lse_parts - m_safe[None])  # exp(-inf) = 0 for empty splits
    tot = w.sum(axis=0)
    with np.errstate(divide="ignore", invalid="ignore"):
        lse = np.where(finite, m_safe + np.log(tot), -np.inf)
        o = np.where(finite[..., None], (w[..., None] * o_parts).sum(axis=0) / np.where(finite, tot, 1.0)[..., None], 0.0)
    return o, lse


# ---------------------------------------------------------------------------
# Decode and extend over the paged pool
# ---------------------------------------------------------------------------
def _kv_head_of(h, num_q_heads, num_kv_heads):
    # repeat_interleave of the KV heads by the group size: q heads
    # [g*G, (g+1)*G) all read kv head g.
    G = num_q_heads // num_kv_heads
    return h // G


def paged_decode(q, k_pool, v_pool, kv_indptr, kv_indices, kv_lens, page_size, sm_scale,
                 return_probs=False, requests=None):
    """One query per request (its last position), attending over all ``kv_lens[b]`` positions.

    q ``[B, Hq, D]`` -> o ``[B, Hq, D]`` fp64, lse ``[B, Hq]`` fp64 (natural log).
    ``requests`` optionally restricts the work to a subset of request ids
    (rows not computed are left NaN).
    """
    qf = as_f64(q)
    B, Hq, D = qf.shape
    Hkv = k_pool.shape[2]
    lens = _as_int(kv_lens)
    o = np.full((B, Hq, D), np.nan)
    lse = np.full((B, Hq), np.nan)
    probs = {}
    for b in (range(B) if requests is None else requests):
        L = int(lens[b])
        Kb = as_f64(request_kv(k_pool, kv_indptr, kv_indices, b, L, page_size))  # [L, Hkv, D]
        Vb = as_f64(request_kv(v_pool, kv_indptr, kv_indices, b, L, page_size))
        for h in range(Hq):
            g = _kv_head_of(h, Hq, Hkv)
            res = attend_rows(qf[b, h][None], Kb[:, g], Vb[:, g], [L], sm_scale, return_probs)
            o[b, h], lse[b, h] = res[0][0], res[1][0]
            if return_probs:
                probs[(b, h)] = res[2][0]
    if return_probs:
        return o, lse, probs
    return o, lse


def paged_extend(q, k_pool, v_pool, qo_indptr, kv_indptr, kv_indices, prefix_lens, page_size,
                 sm_scale, return_probs=False, requests=None, heads=None):
    """Ragged extend: request b's queries are rows ``qo_indptr[b]..qo_indptr[b+1]`` of q.

    Query i (0-based within the request) sits at absolute position
    ``prefix_lens[b] + i`` and sees KV positions ``j <= prefix_lens[b] + i``
    (causal, aligned to the end of the cached prefix).  The request's KV length
    is ``prefix_lens[b] + E_b`` and all of it is read through the pool (the new
    tokens are appended before attention).  ``requests``/``heads`` optionally
    restrict the work (rows not computed are left NaN).
    """
    qf = as_f64(q)
    N, Hq, D = qf.shape
    Hkv = k_pool.shape[2]
    qo = _as_int(qo_indptr)
    pref = _as_int(prefix_lens)
    B = len(pref)
    o = np.full((N, Hq, D), np.nan)
    lse = np.full((N, Hq), np.nan)
    probs = {}
    for b in (range(B) if requests is None else requests):
        P = int(pref[b])
        E = int(qo[b + 1] - qo[b])
        L = P + E
        Kb = as_f64(request_kv(k_pool, kv_indptr, kv_indices, b, L, page_size))
        Vb = as_f64(request_kv(v_pool, kv_indptr, kv_indices, b, L, page_size))
        visible = P + np.arange(E) + 1
        for h in (range(Hq) if heads is None else heads):
            g = _kv_head_of(h, Hq, Hkv)
            res = attend_rows(qf[qo[b]:qo[b + 1], h], Kb[:, g], Vb[:, g], visible, sm_scale, return_probs)
            o[qo[b]:qo[b + 1], h] = res[0]
            lse[qo[b]:qo[b + 1], h] = res[1]
            if return_probs:
                probs[(b, h)] = res[2]
    if return_probs:
        return o, lse, probs
    return o, lse


def shared_prefix_attention(q, k_pool, v_pool, q_start, q_len, o_start, kv_indptr, kv_indices,
                            kv_lens, num_out_rows, page_size, sm_scale):
    """Attention of several requests' queries over KV pages they share (a cascade level).

    Radix-cache prefix sharing (mini-sglang README, "KVcache Management") lets requests point at
    the same physical pages for a common prefix.  Over those positions every sharer's query sees
    every position (the prefix lies before all of its queries), so the part's state is plain
    unmasked attention; merged with the state over the request's own pages (``merge_states``)
    it gives the request's full attention.

    Part p: query rows ``q_start[p] .. q_start[p] + q_len[p] - 1`` of q ``[Nq, Hq, D]``
    attend to the ``kv_lens[p]`` positions of page list p (``kv_indptr``/``kv_indices``, as for
    the decode), query head h reading KV head ``h // (Hq / Hkv)``.  Output row ``o_start[p] + i``
    gets the normalised output and the natural-log LSE of query row ``q_start[p] + i``.  A part
    with no positions gives ``o = 0``, ``lse = -inf``.  Returns ``(o [num_out_rows, Hq, D],
    lse [num_out_rows, Hq])`` in fp64; rows that no part writes are NaN.
    """
    qf = as_f64(q)
    _, Hq, D = qf.shape
    Hkv = k_pool.shape[2]
    qs, ql, os_ = _as_int(q_start), _as_int(q_len), _as_int(o_start)
    lens = _as_int(kv_lens)
    o = np.full((num_out_rows, Hq, D), np.nan)
    lse = np.full((num_out_rows, Hq), np.nan)
    for p in range(len(lens)):
        L = int(lens[p])
        n = int(ql[p])
        Kp = as_f64(request_kv(k_pool, kv_indptr, kv_indices, p, L, page_size))
        Vp = as_f64(request_kv(v_pool, kv_indptr, kv_indices, p, L, page_size))
        rows_in = slice(int(qs[p]), int(qs[p]) + n)
        rows_out = slice(int(os_[p]), int(os_[p]) + n)
        for h in range(Hq):
            g = _kv_head_of(h, Hq, Hkv)
            res = attend_rows(qf[rows_in, h], Kp[:, g], Vp[:, g], np.full(n, L), sm_scale)
            o[rows_out, h] = res[0]
            lse[rows_out, h] = res[1]
    return o, lse


def decode_split_reference(q, k_pool, v_pool, kv_indptr, kv_indices, kv_lens, page_size, sm_scale, bounds):
    """Decode computed as split partials over ``bounds`` and merged.

    ``bounds[b]`` is a non-decreasing list of cut points ``0 = c_0 <= ... <= c_S = kv_lens[b]``;
    split s covers positions ``[c_s, c_{s+1})`` (possibly empty).  Returns
    (o, lse, partials) where partials[b] = (o_parts [S, Hq, D], lse_parts [S, Hq]).
    """
    qf = as_f64(q)
    B, Hq, D = qf.shape
    Hkv = k_pool.shape[2]
    lens = _as_int(kv_lens)
    o = np.zeros((B, Hq, D))
    lse = np.zeros((B, Hq))
    partials = []
    for b in range(B):
        L = int(lens[b])
        cuts = list(bounds[b])
        assert cuts[0] == 0 and cuts[-1] == L
        Kb = as_f64(request_kv(k_pool, kv_indptr, kv_indices, b, L, page_size))
        Vb = as_f64(request_kv(v_pool, kv_indptr, kv_indices, b, L, page_size))
        S = len(cuts) - 1
        op = np.zeros((S, Hq, D))
        lp = np.zeros((S, Hq))
        for h in range(Hq):
            g = _kv_head_of(h, Hq, Hkv)
            for s in range(S):
                a, c = attend_range(qf[b, h][None], Kb[:, g], Vb[:, g], cuts[s], cuts[s + 1], sm_scale)
                op[s, h], lp[s, h] = a[0], c[0]
        mo, ml = merge_states(op, lp)
        o[b], lse[b] = mo, ml
        partials.append((op, lp))
    return o, lse, partials


# ---------------------------------------------------------------------------
# Rotary position embedding, half-split pairing (the rotate_half convention of HF Llama/Qwen
# checkpoints, nanoSGLang README "Notable Fixes"), applied to K before it is written into the
# pool and to Q before attention.
# ---------------------------------------------------------------------------
def rope_angles(positions, head_dim, theta):
    """Angle of pair i at position p: p * theta**(-2i/D), fp64 ``[T, D/2]``."""
    pos = np.asarray(positions, dtype=np.float64)
    i = np.arange(head_dim // 2, dtype=np.float64)
    inv_freq = theta ** (-2.0 * i / head_dim)
    return pos[:, None] * inv_freq[None, :]


def rope(x, positions, theta):
    """Rotate x ``[T, H, D]`` (fp64) by the position of each token: for i < D/2,
    x'[i] = x[i] cos a_i - x[i + D/2] sin a_i and x'[i + D/2] = x[i + D/2] cos a_i + x[i] sin a_i."""
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    ang = rope_angles(positions, D, theta)[:, None, :]  # [T, 1, D/2]
    c, s = np.cos(ang), np.sin(ang)
    lo, hi = x[..., : D // 2], x[..., D // 2:]
    return np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1)


def bf16_round_nearest_even(x):
    """Round fp64 values once to the nearest bf16 value, ties to the even significand.

    bf16 keeps 8 significant bits and fp32's exponent range: with x = m * 2**e (0.5 <= |m| < 1)
    the neighbours are multiples of 2**(e - 8), or of 2**-133 below the smallest normal 2**-126.
    ``np.round`` rounds halves to even.  Values past the largest finite bf16 become +-inf (the
    result is returned in fp64, every element exactly a bf16 value).  Rounding straight from fp64
    avoids the second rounding a cast through fp32 would add.
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    step = np.maximum(e, -125) - 8  # exponent of the bf16 spacing at x
    with np.errstate(over="ignore"):
        y = np.ldexp(np.round(np.ldexp(x, -step)), step)
        y = np.where(np.abs(y) >= 2.0 ** 128, np.copysign(np.inf, x), y)
    return np.where(np.isfinite(x), y, x)


def rope_kv_append(k_pool, v_pool, k_new, v_new, slot_mapping, positions, page_size, theta):
    """KV write with RoPE applied to K: pool.k[slot[t]] = bf16(rope(k_new[t], pos[t])), rounded
    once to nearest even from the fp64 rotation; pool.v[slot[t]] = v_new[t] bit-exact.  Negative
    slots write nothing.  Returns (k_pool, v_pool, k_rot_f64) where k_rot_f64 is the unrounded
    rotation."""
    k_rot = rope(as_f64(k_new), _as_int(positions), theta)
    k_r = bf16_round_nearest_even(k_rot)
    # exact: every value of k_r is a bf16 value, so the casts through fp32 do not round
    k_bf16 = torch.tensor(k_r).to(torch.float32).to(torch.bfloat16) if torch is not None else k_r
    kp, vp = kv_append(k_pool, v_pool, k_bf16, v_new, slot_mapping, page_size)
    return kp, vp, k_rot

"""Host plan for shared-prefix (cascade) decoding.

When a decode batch holds groups of requests whose page lists start with the same physical pages
(radix-cache prefix sharing, mini-sglang README "KVcache Management"), the attention over the
shared pages can be computed once per group, for all of the group's queries together, on tensor
cores (``shared_prefix_attention``), and merged with a decode over each request's own pages
(``merge_states`` of bf16 partials).  This module turns a batch's page lists and its groups into
the integer arrays those calls take.  It is metadata only: no attention arithmetic happens here.

Layout of the partial states: split ``s < num_splits`` of row r is the shared-prefix chunk s of
r's group (an empty state, lse = -inf, for rows outside every group and chunks a group does not
have); split ``num_splits`` is the decode over r's own pages.  Both go to one bf16 buffer
``[num_splits + 1, B, Hq, D]`` and one fp32 buffer ``[num_splits + 1, B, Hq]``.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, fields

import numpy as np
import torch

_TILE_ROWS = 128  # query rows (token, group head) per tile of the shared-prefix kernel


@dataclass
class CascadePlan:
    num_requests: int
    num_splits: int       # shared-prefix splits; the own-pages decode is split num_splits
    num_parts: int
    max_part_rows: int
    shared_tokens: list   # per group: the shared positions used (a whole number of pages)
    # shared-prefix parts, int32 [num_parts] (kv_indptr [num_parts + 1])
    part_q_start: torch.Tensor
    part_q_len: torch.Tensor
    part_o_start: torch.Tensor
    part_kv_indptr: torch.Tensor
    part_kv_indices: torch.Tensor
    part_kv_lens: torch.Tensor
    # each request's own pages, int32 (kv_indptr [B + 1], kv_lens [B])
    suffix_kv_indptr: torch.Tensor
    suffix_kv_indices: torch.Tensor
    suffix_kv_lens: torch.Tensor

    def to(self, device) -> "CascadePlan":
        vals = {}
        for f in fields(self):
            v = getattr(self, f.name)
            vals[f.name] = v.to(device) if isinstance(v, torch.Tensor) else v
        return CascadePlan(**vals)


def _common_pages(lists):
    """Length of the longest common leading run of page ids over the given lists."""
    n = min(len(x) for x in lists)
    first = lists[0][:n]
    for x in lists[1:]:
        diff = np.nonzero(x[:n] != first)[0]
        if diff.size:
            n = int(diff[0])
            first = first[:n]
    return n


def plan_shared_prefix(kv_indptr, kv_indices, kv_lens, groups, page_size: int, *, num_kv_heads: int,
                       group_size: int, num_sms: int, ctas_per_sm: int = 2,
                       min_chunk_tokens: int = 512) -> CascadePlan:
    """Plan a cascade decode.

    ``kv_indptr``/``kv_indices``/``kv_lens``: the decode batch's page lists (CPU int tensors or
    arrays).  ``groups``: ``(first_request, num_requests)`` pairs of consecutive requests that
    share leading pages; the shared length is the longest common run of page ids, cut so that
    every member keeps at least one position of its own.  A group that shares nothing is treated
    as unshared.  The shared pages are split into the same number of chunks for every group,
    chosen so that one wave of CTAs (``num_sms * ctas_per_sm``) covers all groups' chunks and no
    chunk is shorter than ``min_chunk_tokens``.
    """
    indptr = np.asarray(kv_indptr, dtype=np.int64)
    indices = np.asarray(kv_indices, dtype=np.int64)
    lens = np.asarray(kv_lens, dtype=np.int64)
    B = lens.size
    ps = int(page_size)
    if indptr.size != B + 1 or ps <= 0 or not 1 <= group_size <= 16:
        raise ValueError("bad page lists, page size or group size")
    tpt = _TILE_ROWS // group_size  # tokens per Q tile (group x tpt <= 128 rows)
    owner = np.full(B, -1, dtype=np.int64)
    kept = []  # (first, count, shared pages)
    for first, count in groups:
        first, count = int(first), int(count)
        if count < 1 or first < 0 or first + count > B:
            raise ValueError(f"group ({first}, {count}) outside the batch of {B}")
        if (owner[first:first + count] >= 0).any():
            raise ValueError("groups overlap")
        lists = [indices[indptr[r]:indptr[r + 1]] for r in range(first, first + count)]
        sp = _common_pages(lists)
        sp = min(sp, int(((lens[first:first + count] - 1) // ps).min()))  # keep one own position
        if sp <= 0:
            continue
        owner[first:first + count] = len(kept)
        kept.append((first, count, sp))

    # splits: as many as one wave of CTAs holds, each chunk at least min_chunk_tokens long
    ctas_per_split = num_kv_heads * sum(math.ceil(c / tpt) for _, c, _ in kept)
    max_sp = max((sp for _, _, sp in kept), default=0)
    S = 1
    if kept:
        S = max(1, (num_sms * ctas_per_sm) // max(1, ctas_per_split))
        S = max(1, min(S, (max_sp * ps) // max(1, min_chunk_tokens)))

    q_start, q_len, o_start, p_indptr, p_indices, p_lens = [], [], [], [0], [], []

    def add_part(r0, n, s, pages):
        q_start.append(r0)
        q_len.append(n)
        o_start.append(s * B + r0)
        p_indices.extend(pages)
        p_indptr.append(len(p_indices))
        p_lens.append(len(pages) * ps)

    r = 0
    while r < B:
        g = owner[r]
        if g >= 0:
            first, count, sp = kept[g]
            shared = indices[indptr[first]:indptr[first] + sp].tolist()
            c = math.ceil(sp / S)
            for s in range(S):
                add_part(first, count, s, shared[s * c:min((s + 1) * c, sp)])
            r = first + count
        else:
            r1 = r
            while r1 < B and owner[r1] < 0:
                r1 += 1
            for s in range(S):  # rows that share nothing: empty states
                add_part(r, r1 - r, s, [])
            r = r1

    s_indptr, s_indices, s_lens = [0], [], []
    for r in range(B):
        skip = kept[owner[r]][2] if owner[r] >= 0 else 0
        s_indices.extend(indices[indptr[r] + skip:indptr[r + 1]].tolist())
        s_indptr.append(len(s_indices))
        s_lens.append(int(lens[r]) - skip * ps)

    i32 = lambda v: torch.tensor(v, dtype=torch.int32)
    return CascadePlan(
        num_requests=B, num_splits=S, num_parts=len(q_len), max_part_rows=max(q_len, default=0),
        shared_tokens=[sp * ps for _, _, sp in kept],
        part_q_start=i32(q_start), part_q_len=i32(q_len), part_o_start=i32(o_start),
        part_kv_indptr=i32(p_indptr), part_kv_indices=i32(p_indices), part_kv_lens=i32(p_lens),
        suffix_kv_indptr=i32(s_indptr), suffix_kv_indices=i32(s_indices), suffix_kv_lens=i32(s_lens),
    )

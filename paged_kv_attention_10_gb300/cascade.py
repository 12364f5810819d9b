"""Host plan for shared-prefix (cascade) decoding.

When a decode batch holds groups of requests whose page lists start with the same physical pages
(radix-cache prefix sharing, mini-sglang README "KVcache Management"), the attention over the
shared pages can be computed once per group, for all of the group's queries together, on tensor
cores (``shared_prefix_attention``), and merged with a decode over each request's own pages
(``merge_states`` of bf16 partials).  This module turns a batch's page lists and its groups into
the integer arrays those calls take, through the library's host planner
(``pkv_plan_shared_prefix``).  It is metadata only: no attention arithmetic happens here.

Layout of the partial states: split ``s < num_splits`` of row r is the shared-prefix chunk s of
r's group (an empty state, lse = -inf, for rows outside every group and chunks a group does not
have); split ``num_splits`` is the decode over r's own pages.  Both go to one bf16 buffer
``[num_splits + 1, B, Hq, D]`` and one fp32 buffer ``[num_splits + 1, B, Hq]``.
"""

from __future__ import annotations

import ctypes
from dataclasses import dataclass, fields

import numpy as np
import torch


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


def _host_i32(x, name):
    t = torch.as_tensor(np.asarray(x), dtype=torch.int32) if not isinstance(x, torch.Tensor) else x
    t = t.detach().to("cpu", torch.int32).contiguous()
    if t.dim() != 1:
        raise ValueError(f"{name} must be one-dimensional")
    return t


def plan_shared_prefix(kv_indptr, kv_indices, kv_lens, groups, page_size: int, *, num_kv_heads: int,
                       group_size: int, num_sms: int, ctas_per_sm: int = 2,
                       min_chunk_tokens: int = 512) -> CascadePlan:
    """Plan a cascade decode with the library's host planner (``pkv_plan_shared_prefix``).

    ``kv_indptr``/``kv_indices``/``kv_lens``: the decode batch's page lists (CPU int tensors or
    arrays).  ``groups``: ``(first_request, num_requests)`` pairs of consecutive requests that
    share leading pages; the shared length is the longest common run of page ids, cut so that
    every member keeps at least one position of its own.  A group that shares nothing is treated
    as unshared.  The shared pages are split into the same number of chunks for every group,
    chosen so that one wave of CTAs (``num_sms * ctas_per_sm``) covers all groups' chunks and no
    chunk is shorter than ``min_chunk_tokens``.  Argument marshalling only: the planning runs in
    the C library.
    """
    from . import CascadeSizes, PagedKVError, load

    lib = load()
    indptr = _host_i32(kv_indptr, "kv_indptr")
    indices = _host_i32(kv_indices, "kv_indices")
    lens = _host_i32(kv_lens, "kv_lens")
    B = lens.numel()
    if indptr.numel() != B + 1:
        raise ValueError("kv_indptr must have batch_size + 1 entries")
    gf = torch.tensor([int(g[0]) for g in groups], dtype=torch.int32)
    gc = torch.tensor([int(g[1]) for g in groups], dtype=torch.int32)
    ng = gf.numel()
    p = lambda t: ctypes.c_void_p(t.data_ptr()) if t.numel() else None
    shared = torch.zeros(max(ng, 1), dtype=torch.int32)
    sizes = CascadeSizes()
    common = (p(indptr), p(indices), p(lens), B, p(gf), p(gc), ng, int(page_size), int(num_kv_heads),
              int(group_size), int(num_sms), int(ctas_per_sm), int(min_chunk_tokens), ctypes.byref(sizes))
    st = lib.pkv_plan_shared_prefix(*common, None, *([None] * 9), 0, 0)  # size query
    if st == 1:
        raise ValueError("bad page lists, page size, group size or groups")
    if st != 0:
        raise PagedKVError("pkv_plan_shared_prefix", st)
    n_parts = sizes.num_parts
    cap = max(int(indptr[-1]), 1)
    arr = lambda n: torch.zeros(max(n, 1), dtype=torch.int32)
    q_start, q_len, o_start, p_lens = arr(n_parts), arr(n_parts), arr(n_parts), arr(n_parts)
    p_indptr, p_indices = arr(n_parts + 1), arr(cap)
    s_indptr, s_indices, s_lens = arr(B + 1), arr(cap), arr(B)
    st = lib.pkv_plan_shared_prefix(*common, p(shared), p(q_start), p(q_len), p(o_start), p(p_indptr),
                                    p(p_indices), p(p_lens), p(s_indptr), p(s_indices), p(s_lens),
                                    n_parts, cap)
    if st != 0:
        raise PagedKVError("pkv_plan_shared_prefix", st)
    return CascadePlan(
        num_requests=B, num_splits=sizes.num_splits, num_parts=n_parts, max_part_rows=sizes.max_part_rows,
        shared_tokens=[int(t) for t in shared[:ng].tolist() if t > 0],
        part_q_start=q_start[:n_parts], part_q_len=q_len[:n_parts], part_o_start=o_start[:n_parts],
        part_kv_indptr=p_indptr[:n_parts + 1], part_kv_indices=p_indices[:sizes.num_part_indices],
        part_kv_lens=p_lens[:n_parts], suffix_kv_indptr=s_indptr,
        suffix_kv_indices=s_indices[:sizes.num_suffix_indices], suffix_kv_lens=s_lens,
    )

"""Seeded synthetic batches for attention over a paged KV pool.

A batch is what a serving engine's scheduler hands to one attention layer in
one step: a K pool and a V pool of fixed-size pages (layout
``[num_pages, page_size, num_kv_heads, head_dim]``, the NHD page layout of the
nanoSGLang README, "Architecture"/"Features"), the new tokens' K/V with the
slot each one is written to, and per-request page lists in CSR form
(``kv_indptr`` / ``kv_indices``) for the decode requests and for the extend
(chunked-prefill) requests.

Everything here is drawn, nothing is computed: lengths and page permutations
come from one ``torch.Generator`` seeded per workload, values are N(0, 1)
rounded to bf16.  Pool slots that hold no token (free pages, the tail of a
request's last page, and the slots the step's append is about to fill) are set
to NaN, so any read of a slot the attention must not see poisons the result.

A slot is the flat row index of the pool viewed as ``[num_pages * page_size,
num_kv_heads, head_dim]``; a scheduler that owns page ``p`` hands out slots
``p * page_size + r`` for ``r < page_size``.  This is the input convention of
the library, stated here because the generator must produce slots that agree
with the page lists it draws.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np
import torch

CONFIG_NAMES = {
    1: "tiny paged decode + append: B=4, KV lens {37,100,256,511}+1, 14q/2kv heads, D=64, page 16",
    2: "batched decode, page size 1: B=32, KV len U[100,640], 16q/8kv heads, D=128, 200k-slot pool",
    3: "ragged extend with radix prefixes: 16 requests, 32q/8kv heads, D=128, page 16, prefix U[0,1024] (8 share 512), extend U[128,512]",
    4: "long-context split-KV decode: B=8, KV len 32768, 32q/8kv heads, D=128, page 16",
    5: "mixed continuous-batching step: 256 decodes (KV U[512,4096], 64 share a 2048-token prefix) + 4x512 chunked-prefill extends, 32q/8kv heads, D=128, page 16, append 2304 tokens",
}

SEED_BASE = 20260


@dataclass
class RequestSpec:
    """One request of a step.

    ``kv_len`` is the KV length *after* this step's append; the request's last
    ``new_tokens`` positions are the ones appended this step.  A decode request
    issues one query (its last position); an extend request issues one query
    per new token.  Requests with the same ``share_group`` (>= 0) share the
    physical pages of their first ``shared_tokens`` positions.
    """

    kind: str
    kv_len: int
    new_tokens: int
    share_group: int = -1


@dataclass
class PagedBatch:
    name: str
    page_size: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    num_pages: int
    sm_scale: float
    requests: List[RequestSpec]
    # pool state before the step's append (bf16, CPU)
    k_pool: torch.Tensor
    v_pool: torch.Tensor
    # the append
    k_new: torch.Tensor
    v_new: torch.Tensor
    slot_mapping: torch.Tensor  # int64 [T]
    # decode requests
    dec_q: torch.Tensor  # bf16 [Bd, Hq, D]
    dec_kv_indptr: torch.Tensor  # int32 [Bd+1]
    dec_kv_indices: torch.Tensor  # int32 [nnz]
    dec_kv_lens: torch.Tensor  # int32 [Bd]
    # extend requests
    ext_q: torch.Tensor  # bf16 [N, Hq, D]
    ext_qo_indptr: torch.Tensor  # int32 [Be+1]
    ext_kv_indptr: torch.Tensor  # int32 [Be+1]
    ext_kv_indices: torch.Tensor  # int32 [nnz]
    ext_prefix_lens: torch.Tensor  # int32 [Be]
    shared_pages: dict = field(default_factory=dict)

    @property
    def dec_shared_tokens(self) -> torch.Tensor:
        """int32 [Bd]: how many leading positions each decode request shares with other requests
        of the step (its share group's pages; 0 outside every group) -- what a radix cache knows
        of each request's shared prefix."""
        return torch.tensor([int(self.shared_pages[r.share_group].numel()) * self.page_size
                             if r.share_group >= 0 else 0
                             for r in self.requests if r.kind == "decode"], dtype=torch.int32)

    @property
    def num_decode(self) -> int:
        return int(self.dec_kv_lens.numel())

    @property
    def num_extend(self) -> int:
        return int(self.ext_prefix_lens.numel())

    @property
    def num_new_tokens(self) -> int:
        return int(self.slot_mapping.numel())

    @property
    def max_extend_len(self) -> int:
        if self.num_extend == 0:
            return 0
        d = self.ext_qo_indptr[1:] - self.ext_qo_indptr[:-1]
        return int(d.max())

    @property
    def max_decode_len(self) -> int:
        return int(self.dec_kv_lens.max()) if self.num_decode else 0


def _randn_bf16(gen: torch.Generator, shape) -> torch.Tensor:
    return torch.randn(shape, generator=gen, dtype=torch.float32).to(torch.bfloat16)


def build_paged_batch(
    gen: torch.Generator,
    requests: List[RequestSpec],
    *,
    name: str,
    page_size: int,
    num_q_heads: int,
    num_kv_heads: int,
    head_dim: int,
    num_pages: Optional[int] = None,
    shared_tokens: Optional[dict] = None,
    pool_slack: float = 1.25,
    unused_fill: float = float("nan"),
    sm_scale: Optional[float] = None,
) -> PagedBatch:
    """Draw a step over a paged pool for the given requests.

    ``shared_tokens`` maps a share group id to the number of leading positions
    (a multiple of ``page_size``) whose pages the group's requests share.
    """
    ps = page_size
    shared_tokens = dict(shared_tokens or {})
    for gid, s in shared_tokens.items():
        assert s % ps == 0, "a shared prefix covers whole pages"
    # page counts
    shared_page_count = {g: s // ps for g, s in shared_tokens.items()}
    priv_counts = []
    for r in requests:
        n = math.ceil(r.kv_len / ps)
        if r.share_group >= 0:
            s = shared_tokens[r.share_group]
            assert r.kv_len - r.new_tokens >= s, "a shared prefix must already be cached"
            n -= shared_page_count[r.share_group]
        priv_counts.append(n)
    used = sum(priv_counts) + sum(shared_page_count.values())
    if num_pages is None:
        num_pages = max(1, math.ceil(pool_slack * used))
    assert used <= num_pages, f"pool of {num_pages} pages cannot hold {used}"

    perm = torch.randperm(num_pages, generator=gen).to(torch.int64)
    cursor = 0
    group_pages = {}
    for g in sorted(shared_page_count):
        c = shared_page_count[g]
        group_pages[g] = perm[cursor:cursor + c]
        cursor += c
    page_lists = []
    for r, n in zip(requests, priv_counts):
        own = perm[cursor:cursor + n]
        cursor += n
        if r.share_group >= 0:
            page_lists.append(torch.cat([group_pages[r.share_group], own]))
        else:
            page_lists.append(own)

    def slots_of(pages: torch.Tensor, positions: torch.Tensor) -> torch.Tensor:
        return pages[positions // ps] * ps + positions % ps

    # slots already holding cached tokens (each physical slot once)
    cached = []
    for g, pages in group_pages.items():
        pos = torch.arange(shared_tokens[g], dtype=torch.int64)
        cached.append(slots_of(pages, pos))
    for r, pages in zip(requests, page_lists):
        start = shared_tokens[r.share_group] if r.share_group >= 0 else 0
        pos = torch.arange(start, r.kv_len - r.new_tokens, dtype=torch.int64)
        cached.append(slots_of(pages, pos))
    cached_slots = torch.cat(cached) if cached else torch.zeros(0, dtype=torch.int64)

    Hkv, D = num_kv_heads, head_dim
    k_pool = torch.full((num_pages, ps, Hkv, D), unused_fill, dtype=torch.bfloat16)
    v_pool = torch.full((num_pages, ps, Hkv, D), unused_fill, dtype=torch.bfloat16)
    nc = int(cached_slots.numel())
    k_pool.view(-1, Hkv, D)[cached_slots] = _randn_bf16(gen, (nc, Hkv, D))
    v_pool.view(-1, Hkv, D)[cached_slots] = _randn_bf16(gen, (nc, Hkv, D))

    # the step's new tokens, request by request
    new_slots = []
    for r, pages in zip(requests, page_lists):
        pos = torch.arange(r.kv_len - r.new_tokens, r.kv_len, dtype=torch.int64)
        new_slots.append(slots_of(pages, pos))
    slot_mapping = torch.cat(new_slots) if new_slots else torch.zeros(0, dtype=torch.int64)
    T = int(slot_mapping.numel())
    k_new = _randn_bf16(gen, (T, Hkv, D))
    v_new = _randn_bf16(gen, (T, Hkv, D))

    dec = [(r, p) for r, p in zip(requests, page_lists) if r.kind == "decode"]
    ext = [(r, p) for r, p in zip(requests, page_lists) if r.kind == "extend"]

    def csr(items):
        counts = [int(p.numel()) for _, p in items]
        indptr = torch.zeros(len(items) + 1, dtype=torch.int32)
        if counts:
            indptr[1:] = torch.tensor(np.cumsum(counts), dtype=torch.int32)
            indices = torch.cat([p for _, p in items]).to(torch.int32)
        else:
            indices = torch.zeros(0, dtype=torch.int32)
        return indptr, indices

    dec_indptr, dec_indices = csr(dec)
    dec_lens = torch.tensor([r.kv_len for r, _ in dec], dtype=torch.int32)
    ext_indptr, ext_indices = csr(ext)
    ext_prefix = torch.tensor([r.kv_len - r.new_tokens for r, _ in ext], dtype=torch.int32)
    qo = torch.zeros(len(ext) + 1, dtype=torch.int32)
    if ext:
        qo[1:] = torch.tensor(np.cumsum([r.new_tokens for r, _ in ext]), dtype=torch.int32)
    Hq = num_q_heads
    dec_q = _randn_bf16(gen, (len(dec), Hq, D))
    ext_q = _randn_bf16(gen, (int(qo[-1]), Hq, D))

    return PagedBatch(
        name=name, page_size=ps, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
        num_pages=num_pages,
        sm_scale=float(sm_scale if sm_scale is not None else 1.0 / math.sqrt(D)),
        requests=list(requests), k_pool=k_pool, v_pool=v_pool,
        k_new=k_new, v_new=v_new, slot_mapping=slot_mapping,
        dec_q=dec_q, dec_kv_indptr=dec_indptr, dec_kv_indices=dec_indices, dec_kv_lens=dec_lens,
        ext_q=ext_q, ext_qo_indptr=qo, ext_kv_indptr=ext_indptr, ext_kv_indices=ext_indices,
        ext_prefix_lens=ext_prefix,
        shared_pages={g: p.clone() for g, p in group_pages.items()},
    )


def _ri(gen: torch.Generator, lo: int, hi_inclusive: int, n: int) -> List[int]:
    return torch.randint(lo, hi_inclusive + 1, (n,), generator=gen).tolist()


def make_config(idx: int) -> PagedBatch:
    """The five synthetic workloads (shapes of Qwen2.5-0.5B / Qwen3-0.6B / Qwen3-8B attention)."""
    gen = torch.Generator().manual_seed(SEED_BASE + idx)
    name = CONFIG_NAMES[idx]
    if idx == 1:
        # lens are the cached lengths before the append; each request appends one token
        reqs = [RequestSpec("decode", L + 1, 1) for L in (37, 100, 256, 511)]
        return build_paged_batch(gen, reqs, name=name, page_size=16, num_q_heads=14,
                                  num_kv_heads=2, head_dim=64, num_pages=256)
    if idx == 2:
        lens = _ri(gen, 100, 640, 32)
        reqs = [RequestSpec("decode", L, 0) for L in lens]
        return build_paged_batch(gen, reqs, name=name, page_size=1, num_q_heads=16,
                                 num_kv_heads=8, head_dim=128, num_pages=200_000)
    if idx == 3:
        order = torch.randperm(16, generator=gen).tolist()
        sharer = set(order[:8])
        reqs = []
        for i in range(16):
            E = _ri(gen, 128, 512, 1)[0]
            if i in sharer:
                P = _ri(gen, 512, 1024, 1)[0]
                reqs.append(RequestSpec("extend", P + E, E, share_group=0))
            else:
                P = _ri(gen, 0, 1024, 1)[0]
                reqs.append(RequestSpec("extend", P + E, E))
        return build_paged_batch(gen, reqs, name=name, page_size=16, num_q_heads=32,
                                 num_kv_heads=8, head_dim=128, shared_tokens={0: 512})
    if idx == 4:
        reqs = [RequestSpec("decode", 32768, 0) for _ in range(8)]
        return build_paged_batch(gen, reqs, name=name, page_size=16, num_q_heads=32,
                                 num_kv_heads=8, head_dim=128, num_pages=32768)
    if idx == 5:
        order = torch.randperm(256, generator=gen).tolist()
        sharer = set(order[:64])
        reqs = []
        for i in range(256):
            if i in sharer:
                reqs.append(RequestSpec("decode", _ri(gen, 2049, 4096, 1)[0], 1, share_group=0))
            else:
                reqs.append(RequestSpec("decode", _ri(gen, 512, 4096, 1)[0], 1))
        for P in (0, 512, 1024, 1536):
            reqs.append(RequestSpec("extend", P + 512, 512))
        return build_paged_batch(gen, reqs, name=name, page_size=16, num_q_heads=32,
                                 num_kv_heads=8, head_dim=128, shared_tokens={0: 2048})
    raise ValueError(f"no workload {idx}")


def make_spec_verify(num_requests: int = 64, draft_tokens: int = 5, seed: int = SEED_BASE + 6) -> PagedBatch:
    """Target-model verification of speculative drafts: each request checks ``draft_tokens``
    drafted tokens plus the bonus position in one extend of draft_tokens + 1 new tokens over its
    cached context (Mini-SGLang README, "Speculative Decoding": k drafts verified in one parallel
    prefill).  Context lengths U[512, 4096], Qwen3-8B attention shape, page 16."""
    gen = torch.Generator().manual_seed(seed)
    E = draft_tokens + 1
    reqs = [RequestSpec("extend", _ri(gen, 512, 4096, 1)[0] + E, E) for _ in range(num_requests)]
    return build_paged_batch(gen, reqs, name=f"speculative verify: {num_requests} requests x {E} tokens "
                             "over contexts U[512,4096], 32q/8kv heads, D=128, page 16",
                             page_size=16, num_q_heads=32, num_kv_heads=8, head_dim=128)


def make_small_prefill(num_requests: int = 32, seed: int = SEED_BASE + 8) -> PagedBatch:
    """The prefill of the nanoSGLang benchmark's prompts for its model: 32 requests with prompts of
    U[100, 512] tokens and no cached prefix, Qwen2.5-0.5B attention (14 query heads over 2 KV
    heads, so GQA groups of 7, head_dim 64), page 16 (nanoSGLang README, "Performance")."""
    gen = torch.Generator().manual_seed(seed)
    reqs = [RequestSpec("extend", E, E) for E in _ri(gen, 100, 512, num_requests)]
    return build_paged_batch(gen, reqs, name=f"small-model prefill: {num_requests} prompts of U[100,512] "
                             "tokens, Qwen2.5-0.5B attention 14q/2kv heads (group 7), D=64, page 16",
                             page_size=16, num_q_heads=14, num_kv_heads=2, head_dim=64)


def make_shared_prefix_decode(num_requests: int = 256, shared_tokens: int = 4096,
                              seed: int = SEED_BASE + 7) -> PagedBatch:
    """A decode batch whose requests all continue one long shared prompt: every request shares the
    pages of its first ``shared_tokens`` positions (a radix-cache hit on a common system prompt
    or parallel samples of one prompt: mini-sglang README, "KVcache Management") and owns
    U[64, 1024] further positions, the last one appended this step.  Qwen3-8B attention shape,
    page 16.  The requests are consecutive, so the shared-prefix (cascade) decode can take them
    as one group."""
    gen = torch.Generator().manual_seed(seed)
    reqs = [RequestSpec("decode", shared_tokens + own, 1, share_group=0)
            for own in _ri(gen, 64, 1024, num_requests)]
    return build_paged_batch(gen, reqs, name=f"shared-prefix decode: {num_requests} requests sharing a "
                             f"{shared_tokens}-token prefix, own KV U[64,1024], 32q/8kv heads, D=128, "
                             "page 16", page_size=16, num_q_heads=32, num_kv_heads=8, head_dim=128,
                             shared_tokens={0: shared_tokens})


def random_small_batch(
    seed: int,
    *,
    page_size: int,
    num_q_heads: int,
    num_kv_heads: int,
    head_dim: int,
    decode_lens=(),
    decode_new: int = 1,
    extend=(),
    share_decode_prefix: int = 0,
    share_extend_prefix: int = 0,
    pool_slack: float = 1.5,
    sm_scale: Optional[float] = None,
    unused_fill: float = float("nan"),
) -> PagedBatch:
    """A small batch for property and parity tests.

    ``decode_lens`` are KV lengths after the append (``decode_new`` tokens each,
    clamped to the length); ``extend`` is a sequence of ``(prefix, extend_len)``.
    ``share_*_prefix`` > 0 makes the requests of that kind whose cached part is
    long enough share their first that-many positions' pages.
    """
    gen = torch.Generator().manual_seed(seed)
    reqs: List[RequestSpec] = []
    shared = {}
    if share_decode_prefix:
        shared[0] = share_decode_prefix
    if share_extend_prefix:
        shared[1] = share_extend_prefix
    for L in decode_lens:
        new = min(decode_new, L)
        g = 0 if (share_decode_prefix and L - new >= share_decode_prefix) else -1
        reqs.append(RequestSpec("decode", L, new, share_group=g))
    for P, E in extend:
        g = 1 if (share_extend_prefix and P >= share_extend_prefix) else -1
        reqs.append(RequestSpec("extend", P + E, E, share_group=g))
    # drop share groups nobody joined
    used_groups = {r.share_group for r in reqs if r.share_group >= 0}
    shared = {g: s for g, s in shared.items() if g in used_groups}
    return build_paged_batch(gen, reqs, name=f"small-{seed}", page_size=page_size,
                             num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                             head_dim=head_dim, shared_tokens=shared, pool_slack=pool_slack,
                             sm_scale=sm_scale, unused_fill=unused_fill)

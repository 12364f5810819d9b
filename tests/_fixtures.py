"""Small helpers shared by the tests (loading golden cases, building contiguous-KV cases)."""

import json
import math
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _num(x):
    if isinstance(x, str):
        try:
            return float(x)  # "nan", "-inf"
        except ValueError:
            return x
    if isinstance(x, list):
        return [_num(v) for v in x]
    return x


def load_golden(name="worked_examples.json"):
    with open(os.path.join(GOLDEN, name)) as f:
        raw = json.load(f)
    out = {}
    for k, v in raw.items():
        if k.startswith("_"):
            continue
        out[k] = {kk: _num(vv) for kk, vv in v.items()}
    return out


def golden_tensors(case):
    """Torch tensors (bf16 data, int32 metadata) for a golden case."""
    t = {}
    for key in ("k_pool", "v_pool", "q"):
        if key in case:
            t[key] = torch.tensor(case[key], dtype=torch.float32).to(torch.bfloat16)
    for key in ("kv_indptr", "kv_indices", "kv_lens", "qo_indptr", "prefix_lens"):
        if key in case:
            t[key] = torch.tensor(case[key], dtype=torch.int32)
    return t


def contiguous_case(seed, *, lens, prefixes=None, Hq, Hkv, D, page_size, spare_pages=3):
    """Per-request contiguous K/V (the naive contiguous cache) plus the same data scattered into a
    page pool by the test's own loop.  Returns (contig, paged) where contig has per-request fp64
    arrays K[b], V[b] of shape [L_b, Hkv, D] and paged has bf16 pools and CSR page lists."""
    rng = np.random.default_rng(seed)
    B = len(lens)
    Kc, Vc = [], []
    for L in lens:
        k = torch.tensor(rng.standard_normal((L, Hkv, D)), dtype=torch.float32).to(torch.bfloat16)
        v = torch.tensor(rng.standard_normal((L, Hkv, D)), dtype=torch.float32).to(torch.bfloat16)
        Kc.append(k)
        Vc.append(v)
    need = [math.ceil(L / page_size) for L in lens]
    num_pages = sum(need) + spare_pages
    order = rng.permutation(num_pages)
    k_pool = torch.full((num_pages, page_size, Hkv, D), float("nan"), dtype=torch.bfloat16)
    v_pool = torch.full((num_pages, page_size, Hkv, D), float("nan"), dtype=torch.bfloat16)
    indptr = [0]
    indices = []
    cur = 0
    for b, L in enumerate(lens):
        pages = order[cur:cur + need[b]].tolist()
        cur += need[b]
        indices += pages
        indptr.append(len(indices))
        for j in range(L):
            pg, r = pages[j // page_size], j % page_size
            k_pool[pg, r] = Kc[b][j]
            v_pool[pg, r] = Vc[b][j]
    paged = dict(
        k_pool=k_pool, v_pool=v_pool,
        kv_indptr=torch.tensor(indptr, dtype=torch.int32),
        kv_indices=torch.tensor(indices, dtype=torch.int32),
        kv_lens=torch.tensor(lens, dtype=torch.int32),
        page_size=page_size,
    )
    contig = dict(K=[k.float().numpy().astype(np.float64) for k in Kc],
                  V=[v.float().numpy().astype(np.float64) for v in Vc])
    return contig, paged

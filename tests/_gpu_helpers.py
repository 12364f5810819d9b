"""Helpers for the GPU parity tests: moving a generated batch to the device and comparing with the
fp64 oracle under the stated tolerances."""

import numpy as np
import torch

# Tolerances for bf16 attention outputs against the fp64 oracle (absolute).
O_MAX_ABS = 1e-2
O_MEAN_ABS = 1e-3
LSE_ABS = 1e-3


class DeviceBatch:
    def __init__(self, b, device="cuda"):
        self.b = b
        d = device
        self.k_pool = b.k_pool.to(d)
        self.v_pool = b.v_pool.to(d)
        self.k_new = b.k_new.to(d)
        self.v_new = b.v_new.to(d)
        self.slot_mapping = b.slot_mapping.to(d)
        self.dec_q = b.dec_q.to(d)
        self.dec_kv_indptr = b.dec_kv_indptr.to(d)
        self.dec_kv_indices = b.dec_kv_indices.to(d)
        self.dec_kv_lens = b.dec_kv_lens.to(d)
        self.ext_q = b.ext_q.to(d)
        self.ext_qo_indptr = b.ext_qo_indptr.to(d)
        self.ext_kv_indptr = b.ext_kv_indptr.to(d)
        self.ext_kv_indices = b.ext_kv_indices.to(d)
        self.ext_prefix_lens = b.ext_prefix_lens.to(d)


def bits_equal(a: torch.Tensor, b: torch.Tensor) -> bool:
    """Bitwise equality of bf16 tensors (NaNs compare by their bits)."""
    return torch.equal(a.contiguous().view(torch.int16).cpu(), b.contiguous().view(torch.int16).cpu())


def attention_errors(out, lse, o_ref, lse_ref, rows=None):
    """(max_abs, mean_abs, lse_max_abs, floor) over the given leading-index rows of o_ref.

    floor = mean |bf16(o_ref) - o_ref|, the error of the best possible bf16 answer."""
    o = out.float().cpu().numpy().astype(np.float64)
    if rows is not None:
        o, o_ref = o[rows], o_ref[rows]
    d = np.abs(o - o_ref)
    floor = np.abs(torch.tensor(o_ref).to(torch.bfloat16).double().numpy() - o_ref).mean()
    lerr = 0.0
    if lse is not None:
        l = lse.cpu().numpy().astype(np.float64)
        lr = lse_ref
        if rows is not None:
            l, lr = l[rows], lr[rows]
        lerr = float(np.abs(l - lr).max()) if l.size else 0.0
        if np.isnan(lerr):
            lerr = np.inf
    mx = float(d.max()) if d.size else 0.0
    mean = float(d.mean()) if d.size else 0.0
    if np.isnan(mx) or np.isnan(mean):
        mx = mean = np.inf
    return mx, mean, lerr, float(floor)


def assert_attention_close(out, lse, o_ref, lse_ref, rows=None, what=""):
    mx, mean, lerr, floor = attention_errors(out, lse, o_ref, lse_ref, rows)
    msg = f"{what}: max_abs={mx:.3g} mean_abs={mean:.3g} lse_abs={lerr:.3g} (bf16 floor {floor:.3g})"
    assert mx <= O_MAX_ABS, msg
    assert mean <= O_MEAN_ABS, msg
    assert lerr <= LSE_ABS, msg
    return mx, mean, lerr, floor


_CFG = {}


def config_with_append(idx):
    """(batch, k_pool_after, v_pool_after) for a named workload; the appended pools come from the
    oracle.  Cached per process (the big workloads take seconds to draw)."""
    if idx not in _CFG:
        import oracle
        from workloads import make_config

        b = make_config(idx)
        kp, vp = oracle.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.slot_mapping, b.page_size)
        if idx in (4, 5) or any(k in (4, 5) for k in _CFG):
            _CFG.clear()  # keep at most one large workload in host memory
        _CFG[idx] = (b, kp, vp)
    return _CFG[idx]

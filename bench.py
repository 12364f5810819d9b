"""Throughput of one attention step over a paged KV pool on GB300.

A step is one pass of the whole hot path over the mixed continuous-batching workload:
KV append of all 2304 new tokens through the slot mapping, paged decode of 256 requests
(64 of them sharing a 2048-token prefix on the same pages; long requests split and merged by
log-sum-exp), and ragged extend of 4 chunked-prefill chunks of 512 tokens over cached prefixes.
Shapes are Qwen3-8B attention (32 query heads, 8 KV heads, head_dim 128), page size 16, bf16.

Prints one JSON line.  ``--impl reference`` times the fp64 CPU oracle on the same workload
instead (a bounded sample per step).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time
import types

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode KV GB/s (% HBM peak); extend TFLOP/s (% bf16 peak); attn tokens/s"


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def _dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(values, device=None):
    """Element-wise maximum of per-rank timings (identity without a process group)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


# ---------------------------------------------------------------------------------------------
# algorithmic work of the workload (from the generated lengths)
# ---------------------------------------------------------------------------------------------
def _packed(named, device, pin=False):
    """One byte buffer holding each (name, tensor) at a 256-byte-aligned offset, filled with the
    tensors' values: returns (buffer, {name: view of the buffer})."""
    import torch

    offs, total = [], 0
    for _, t in named:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    buf = torch.empty(max(total, 256), dtype=torch.uint8, device=device)
    if pin:
        buf = buf.pin_memory()
    views = {}
    for (name, t), off in zip(named, offs):
        nb = t.numel() * t.element_size()
        v = buf[off:off + nb].view(t.dtype).view(t.shape)
        v.copy_(t)
        views[name] = v
    return buf, views


def workload_counts(b):
    import numpy as np

    Hkv, D, Hq = b.num_kv_heads, b.head_dim, b.num_q_heads
    row = Hkv * D * 2  # bytes of one token's K (or V) row
    ps = b.page_size
    # decode: each physical KV slot read counted once (shared prefix pages once), K and V
    indptr = b.dec_kv_indptr.numpy()
    indices = b.dec_kv_indices.numpy().astype(np.int64)
    lens = b.dec_kv_lens.numpy().astype(np.int64)
    slots = []
    for r in range(len(lens)):
        pos = np.arange(lens[r])
        slots.append(indices[indptr[r] + pos // ps] * ps + pos % ps)
    uniq = np.unique(np.concatenate(slots)).size if len(slots) else 0
    logical = int(lens.sum())
    qo_bytes = len(lens) * Hq * D * 2 * 2 + len(lens) * Hq * 4  # q in, out + lse
    meta = (indptr.size + indices.size + lens.size) * 4
    dec_bytes = uniq * row * 2 + qo_bytes + meta
    dec_bytes_logical = logical * row * 2 + qo_bytes + meta
    # extend: unmasked (query, key) pairs, 2 matmuls of 2*D flops each per pair and head
    qo = b.ext_qo_indptr.numpy().astype(np.int64)
    pref = b.ext_prefix_lens.numpy().astype(np.int64)
    pairs = 0
    for r in range(len(pref)):
        E = qo[r + 1] - qo[r]
        pairs += E * pref[r] + E * (E + 1) // 2
    ext_flops = 4 * D * Hq * pairs
    # extend bytes: each physical KV slot of the extend requests once (prefix and new rows), K and
    # V; the queries in, outputs and LSE out; the page lists
    eptr = b.ext_kv_indptr.numpy()
    eind = b.ext_kv_indices.numpy().astype(np.int64)
    eslots = []
    for r in range(len(pref)):
        pos = np.arange(pref[r] + qo[r + 1] - qo[r])
        eslots.append(eind[eptr[r] + pos // ps] * ps + pos % ps)
    euniq = np.unique(np.concatenate(eslots)).size if len(eslots) else 0
    ext_bytes = (euniq * row * 2 + int(qo[-1]) * Hq * (D * 2 * 2 + 4)
                 + (eptr.size + eind.size + pref.size + qo.size) * 4)
    T = b.num_new_tokens
    app_bytes = T * row * 2 * 2 + T * 8  # read new K/V, write K/V rows, slots
    tokens = len(lens) + int(qo[-1])
    return {"decode_bytes": int(dec_bytes), "decode_bytes_logical": int(dec_bytes_logical),
            "decode_kv_tokens_unique": int(uniq), "decode_kv_tokens_logical": logical,
            "extend_flops": int(ext_flops), "extend_pairs": int(pairs), "extend_bytes": int(ext_bytes),
            "append_bytes": int(app_bytes),
            "attn_tokens": int(tokens)}


def cascade_counts(b, plan):
    """Algorithmic work of the cascade's pieces: the shared-prefix parts' unmasked (query, key)
    flops, the own-pages decode's bytes (each physical slot once, plus q in, partial out) and the
    merge's bytes (every partial state read, the output written)."""
    import numpy as np

    Hkv, D, Hq, ps = b.num_kv_heads, b.head_dim, b.num_q_heads, b.page_size
    row = Hkv * D * 2
    ql = plan.part_q_len.numpy().astype(np.int64)
    kl = plan.part_kv_lens.numpy().astype(np.int64)
    prefix_flops = int(4 * D * Hq * (ql * kl).sum())
    ind = plan.suffix_kv_indices.numpy().astype(np.int64)
    ptr = plan.suffix_kv_indptr.numpy()
    lens = plan.suffix_kv_lens.numpy().astype(np.int64)
    slots = [ind[ptr[r] + np.arange(lens[r]) // ps] * ps + np.arange(lens[r]) % ps for r in range(len(lens))]
    uniq = np.unique(np.concatenate(slots)).size if slots else 0
    B = len(lens)
    suffix_bytes = uniq * row * 2 + B * Hq * (D * 2 * 2 + 4) + (ptr.size + ind.size + lens.size) * 4
    merge_bytes = (plan.num_splits + 1) * B * Hq * (D * 2 + 4) + B * Hq * (D * 2 + 4)
    return {"prefix_flops": prefix_flops, "suffix_bytes": int(suffix_bytes), "merge_bytes": int(merge_bytes)}


# ---------------------------------------------------------------------------------------------
# clocks sampled by nvidia-smi during the timed region
# ---------------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[1]), float(parts[2]), parts[5:9], parts[4]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return None
        sm = [r[0] for r in rows]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[2]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(r[1] for r in rows),
                "samples": len(rows), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------------------------
def _kernel_hash():
    h = hashlib.sha256()
    for f in ("decode.cu", "common.cuh"):
        with open(os.path.join(ROOT, "paged_kv_attention_10_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _traffic_record():
    """DRAM bytes per decode launch from the committed ncu summary of the mixed step, if that
    capture was taken on the current decode source (its hash is recorded beside the figure)."""
    p = os.path.join(ROOT, "profiles", "paged_decode_mixed_step_dram.md")
    if not os.path.exists(p):
        return None
    fields = {}
    with open(p) as f:
        for line in f:
            if line.startswith("- ") and ": " in line:
                k, v = line[2:].split(": ", 1)
                fields[k.strip("` ")] = v.strip().strip("`")
    if fields.get("source_hash") != _kernel_hash():
        return None
    try:
        return int(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def run_ours(args, ws, rank, local):
    import numpy as np
    import torch
    import torch.distributed as dist

    import paged_kv_attention_10_gb300 as pkv
    from workloads import make_config

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pkv.load()
    b = load_workload(args.workload)
    counts = workload_counts(b)
    st = torch.cuda.Stream(device=dev)

    # device-resident state: the pool (the KV cache).  A step's inputs and outputs each live in one
    # buffer (256-byte-aligned views), so the end-to-end run moves them with one copy each way.
    kp, vp = b.k_pool.to(dev), b.v_pool.to(dev)
    inputs = [("kn", b.k_new), ("vn", b.v_new), ("sm", b.slot_mapping), ("d_ind", b.dec_kv_indptr),
              ("d_idx", b.dec_kv_indices), ("d_len", b.dec_kv_lens), ("e_qo", b.ext_qo_indptr),
              ("e_ind", b.ext_kv_indptr), ("e_idx", b.ext_kv_indices), ("e_pre", b.ext_prefix_lens)]
    # each decode request's shared prefix length, the decode's L2 keep hint (a radix cache knows
    # it: the length of the match other requests of the step share)
    use_keep = not args.no_l2_keep and not args.cascade and b.num_decode > 0
    if use_keep:
        inputs += [("d_keep", b.dec_shared_tokens)]
    table = None
    if args.rope:
        # the step's queries are the new tokens' (decodes first, then extend tokens, the slot
        # order): one buffer the fused RoPE-append rotates in place, with decode/extend views
        pos = []
        for r in b.requests:
            pos += list(range(r.kv_len - r.new_tokens, r.kv_len))
        inputs += [("q_all", torch.cat([b.dec_q, b.ext_q])),
                   ("positions", torch.tensor(pos, dtype=torch.int32))]
        table = pkv.rope_cos_sin_table(max(pos) + 1, b.head_dim, 1.0e6, device=dev)
    else:
        inputs += [("dq", b.dec_q), ("eq", b.ext_q)]
    plan = None
    if args.cascade:
        from paged_kv_attention_10_gb300.cascade import plan_shared_prefix

        # each share group must be a run of consecutive decode requests
        groups = {}
        for i, r in enumerate(b.requests[: b.num_decode]):
            if r.share_group >= 0:
                groups.setdefault(r.share_group, []).append(i)
        for g, rows in groups.items():
            if rows != list(range(rows[0], rows[0] + len(rows))):
                raise SystemExit(f"--cascade: share group {g} is not a run of consecutive requests")
        plan = plan_shared_prefix(b.dec_kv_indptr, b.dec_kv_indices, b.dec_kv_lens,
                                  [(rows[0], len(rows)) for rows in groups.values()], b.page_size,
                                  num_kv_heads=b.num_kv_heads, group_size=b.num_q_heads // b.num_kv_heads,
                                  num_sms=torch.cuda.get_device_properties(dev).multi_processor_count)
        # the step's metadata is the plan's: the parts, and each request's own pages
        inputs = [x for x in inputs if x[0] not in ("d_ind", "d_idx", "d_len")]
        inputs += [("d_ind", plan.suffix_kv_indptr), ("d_idx", plan.suffix_kv_indices),
                   ("d_len", plan.suffix_kv_lens), ("p_qs", plan.part_q_start), ("p_ql", plan.part_q_len),
                   ("p_os", plan.part_o_start), ("p_ind", plan.part_kv_indptr),
                   ("p_idx", plan.part_kv_indices), ("p_len", plan.part_kv_lens)]
        S = plan.num_splits
        o_parts = torch.empty((S + 1, b.num_decode, b.num_q_heads, b.head_dim), dtype=torch.bfloat16,
                              device=dev)
        lse_parts = torch.empty((S + 1, b.num_decode, b.num_q_heads), dtype=torch.float32, device=dev)
        pws = torch.empty(max(256, pkv.shared_prefix_workspace_size(plan.num_parts, b.num_q_heads,
                                                                    b.num_kv_heads, b.head_dim,
                                                                    plan.max_part_rows, dev)),
                          dtype=torch.uint8, device=dev)
    ws_bytes = pkv.decode_workspace_size(b.num_decode, b.num_q_heads, b.num_kv_heads, b.head_dim, dev)
    dws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    ext_ws = pkv.extend_workspace_size(b.num_extend, b.num_q_heads, b.num_kv_heads, b.head_dim,
                                       b.max_extend_len, dev) if b.num_extend else 0
    ews = torch.empty(max(256, ext_ws), dtype=torch.uint8, device=dev)
    max_e = b.max_extend_len

    def make_bufs():
        """One set of the step's device inputs and outputs (views of two packed buffers)."""
        f = types.SimpleNamespace()
        f.in_buf, din = _packed(inputs, dev)
        for n in ("kn", "vn", "sm", "d_ind", "d_idx", "d_len", "e_qo", "e_ind", "e_idx", "e_pre"):
            setattr(f, n, din[n])
        f.d_keep = din["d_keep"] if use_keep else None
        if plan is not None:
            for n in ("p_qs", "p_ql", "p_os", "p_ind", "p_idx", "p_len"):
                setattr(f, n, din[n])
        if args.rope:
            f.q_all, f.positions = din["q_all"], din["positions"]
            f.dq, f.eq = f.q_all[: b.num_decode], f.q_all[b.num_decode:]
        else:
            f.q_all = f.positions = None
            f.dq, f.eq = din["dq"], din["eq"]
        outputs = [("d_out", torch.empty(f.dq.shape, dtype=f.dq.dtype)),
                   ("d_lse", torch.empty((b.num_decode, b.num_q_heads), dtype=torch.float32)),
                   ("e_out", torch.empty(f.eq.shape, dtype=f.eq.dtype)),
                   ("e_lse", torch.empty((f.eq.shape[0], b.num_q_heads), dtype=torch.float32))]
        f.out_buf, dout = _packed(outputs, dev)
        f.d_out, f.d_lse, f.e_out, f.e_lse = dout["d_out"], dout["d_lse"], dout["e_out"], dout["e_lse"]
        return f

    bufs = make_bufs()

    do_app = args.op in ("all", "append")
    do_dec = args.op in ("all", "decode") and b.num_decode > 0
    do_ext = args.op in ("all", "extend") and b.num_extend > 0

    def append_range(f, lo, hi, stream):
        if hi <= lo:
            return
        if args.rope:
            pkv.rope_kv_append(kp, vp, f.kn[lo:hi], f.vn[lo:hi], f.sm[lo:hi], f.positions[lo:hi],
                               table, q=f.q_all[lo:hi], stream=stream)
        else:
            pkv.kv_append(kp, vp, f.kn[lo:hi], f.vn[lo:hi], f.sm[lo:hi], stream=stream)

    def decode(f, stream, sub=None):
        if plan is None:
            pkv.paged_decode(f.dq, kp, vp, f.d_ind, f.d_idx, f.d_len, b.sm_scale, out=f.d_out,
                             lse=f.d_lse, workspace=dws, stream=stream, max_ctas=decode_ctas,
                             l2_keep_tokens=f.d_keep)
            return
        # shared pages once per group (splits 0..S-1), each request's own pages (split S), merge
        # (the scratch partial states are shared by both buffer sets: steps run in stream order)
        H, D = b.num_q_heads, b.head_dim
        pkv.shared_prefix_attention(f.dq, kp, vp, f.p_qs, f.p_ql, f.p_os, f.p_ind, f.p_idx, f.p_len,
                                    plan.max_part_rows, b.sm_scale, o_parts.view(-1, H, D),
                                    lse_parts.view(-1, H), workspace=pws, stream=stream)
        if sub is not None:
            sub[0].record(stream)
        pkv.paged_decode(f.dq, kp, vp, f.d_ind, f.d_idx, f.d_len, b.sm_scale, out=o_parts[S],
                         lse=lse_parts[S], workspace=dws, stream=stream, max_ctas=decode_ctas)
        if sub is not None:
            sub[1].record(stream)
        pkv.merge_states(o_parts, lse_parts, out=f.d_out, lse=f.d_lse, stream=stream)

    def extend(f, stream):
        pkv.paged_extend(f.eq, kp, vp, f.e_qo, f.e_ind, f.e_idx, f.e_pre, max_e, b.sm_scale,
                         out=f.e_out, lse=f.e_lse, workspace=ews, stream=stream)

    def step(f=bufs, ev=None):
        if ev is not None:
            ev[0].record(st)
        if do_app:
            append_range(f, 0, f.kn.shape[0], st)
        if ev is not None:
            ev[1].record(st)
        if do_dec:
            decode(f, st, sub=ev[4:6] if ev is not None and len(ev) > 4 else None)
        if ev is not None:
            ev[2].record(st)
        if do_ext:
            extend(f, st)
        if ev is not None:
            ev[3].record(st)

    # The same step as two branches that share no data: the decodes' new tokens then decode (and
    # its split merge), beside the extend chunks' new tokens then extend.  New tokens are laid out
    # request by request with the decodes first, so each branch appends a contiguous range.  The
    # extend's append then runs during the decode, and extend CTAs take SMs as decode CTAs finish.
    nd_new = sum(r.new_tokens for r in b.requests if r.kind == "decode")
    decodes_first = all(r.kind == "decode" for r in b.requests[: b.num_decode])
    overlap = (do_app and do_dec and do_ext and decodes_first and not args.serial_step
               and (not args.rope or nd_new == b.num_decode))
    st2 = torch.cuda.Stream(device=dev)
    fork_ev, join_ev = torch.cuda.Event(), torch.cuda.Event()
    # SMs the decode runs on: in the branched step a few stay free for the extend beside it (the
    # decode is HBM-bound, the extend tensor-bound); otherwise all of them
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    if args.decode_sms >= 0:
        decode_ctas = args.decode_sms
    else:
        decode_ctas = sms - EXTEND_SPARE_SMS if overlap and not args.eager else 0

    def step_branches(f=bufs):
        # the extend branch forks once the decodes' tokens are appended, so the decode's
        # persistent CTAs are dispatched before the extend branch's kernels can take their SMs
        append_range(f, 0, nd_new, st)
        fork_ev.record(st)
        st2.wait_event(fork_ev)
        decode(f, st)
        append_range(f, nd_new, f.kn.shape[0], st2)
        extend(f, st2)
        join_ev.record(st2)
        st.wait_event(join_ev)

    whole_step = step_branches if overlap else step

    def barrier():
        if ws > 1:
            dist.barrier()

    with torch.cuda.stream(st):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize(dev)

    # ---- device-resident timed region ----------------------------------------------------
    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4 if plan is None else 6)] for _ in range(K)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    barrier()
    torch.cuda.synchronize(dev)
    clocks.start()
    time.sleep(0.3)  # let the sampler take its first reading
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev) if args.flush_l2 else None
    with torch.cuda.stream(st):
        start.record(st)
        for k in range(K):
            if flush is not None:
                flush.zero_()
            step(ev=evs[k])
        stop.record(st)
    torch.cuda.synchronize(dev)
    barrier()
    clk = clocks.stop()
    elapsed_ms = start.elapsed_time(stop)
    if flush is not None:  # exclude the flushes: the step is the span of its own operations
        elapsed_ms = sum(e[0].elapsed_time(e[3]) for e in evs)
    eager_ms = elapsed_ms

    if not args.eager:
        # the same step captured once as a CUDA graph (the library allocates nothing and never
        # synchronises inside a call) and replayed; per-kernel figures stay from the eager loop
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            whole_step()
        with torch.cuda.stream(st):
            for _ in range(args.warmup):
                g.replay()
        torch.cuda.synchronize(dev)
        barrier()
        gs, ge = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        gclocks = ClockSampler(local)
        gclocks.start()
        time.sleep(0.3)
        with torch.cuda.stream(st):
            gs.record(st)
            for _ in range(K):
                g.replay()
            ge.record(st)
        torch.cuda.synchronize(dev)
        barrier()
        clk = gclocks.stop() or clk
        elapsed_ms = gs.elapsed_time(ge)
    t_app = [e[0].elapsed_time(e[1]) for e in evs]
    t_dec = [e[1].elapsed_time(e[2]) for e in evs]
    t_ext = [e[2].elapsed_time(e[3]) for e in evs]

    # ---- end to end through the public API with host buffers -----------------------------
    # Every step copies its inputs from pinned host memory (one buffer, laid out as on the
    # device), runs, and copies all its outputs back.  Two device buffer sets let the copies of
    # one step overlap the computation of its neighbours: the inputs of step k+1 go in and the
    # outputs of step k-1 come out while step k computes, on their own copy streams.
    host_in_buf, _ = _packed(inputs, "cpu", pin=True)
    host_out_buf = torch.empty(bufs.out_buf.numel(), dtype=torch.uint8).pin_memory()
    h2d = host_in_buf.numel()
    d2h = host_out_buf.numel()
    sets = [bufs, make_bufs()]
    # Each buffer set's step is captured once as a CUDA graph (as a serving engine replays its
    # captured step), so the per-step cost is one graph launch instead of a launch per call; the
    # host copies stay outside the graphs on their own streams.
    set_graphs = [None, None]
    if not args.eager:
        set_graphs[0] = g
        g1 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g1, stream=st):
            whole_step(sets[1])
        set_graphs[1] = g1
    cs_in, cs_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_step(k):
        i = k % 2
        f = sets[i]
        if k >= 2:
            cs_in.wait_event(ev_comp[i])  # step k-2 has finished reading set i's inputs
        with torch.cuda.stream(cs_in):
            f.in_buf.copy_(host_in_buf, non_blocking=True)
        ev_in[i].record(cs_in)
        st.wait_event(ev_in[i])
        if k >= 2:
            st.wait_event(ev_out[i])  # step k-2's outputs (set i) are back on the host
        if set_graphs[i] is not None:
            set_graphs[i].replay()
        else:
            whole_step(f)
        ev_comp[i].record(st)
        cs_out.wait_event(ev_comp[i])
        with torch.cuda.stream(cs_out):
            host_out_buf.copy_(f.out_buf, non_blocking=True)
        ev_out[i].record(cs_out)

    K2 = max(1, min(K, 200)) if not args.no_e2e else 1
    with torch.cuda.stream(st):
        for k in range(max(2, args.warmup)):
            e2e_step(k)
    torch.cuda.synchronize(dev)
    barrier()
    s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(st):
        s2.record(st)
        cs_in.wait_event(s2)
        for k in range(K2):
            e2e_step(k)
        st.wait_event(ev_out[(K2 - 1) % 2])  # the last step's outputs are on the host
        e2.record(st)
    torch.cuda.synchronize(dev)
    barrier()
    e2e_ms = s2.elapsed_time(e2)

    # ---- max over ranks --------------------------------------------------------------------
    elapsed_ms, e2e_ms = max_over_ranks([elapsed_ms, e2e_ms], dev)

    peaks = _peaks()
    ms_step = elapsed_ms / K
    tokens = counts["attn_tokens"]
    value = tokens * K * ws / (elapsed_ms / 1e3)
    dec_ms = statistics.mean(t_dec) if do_dec else None
    ext_ms = statistics.mean(t_ext) if do_ext else None
    app_ms = statistics.mean(t_app) if (do_app and b.num_new_tokens) else None
    kernels = {}
    # decode and its split merge; with the cascade also the part order, the shared-prefix kernel and
    # the final merge
    dec_launches = 2 if plan is None else 4 + int(
        pkv.shared_prefix_workspace_size(plan.num_parts, b.num_q_heads, b.num_kv_heads, b.head_dim,
                                         plan.max_part_rows, dev) > 0)
    if dec_ms:
        dec_gbs = counts["decode_bytes"] / (dec_ms / 1e3) / 1e9
        kernels["decode"] = {"ms": round(dec_ms, 4), "gbs": round(dec_gbs, 1),
                             "frac_hbm": round(dec_gbs / peaks["hbm_gbs"], 4),
                             "gbs_logical": round(counts["decode_bytes_logical"] / (dec_ms / 1e3) / 1e9, 1)}
    if dec_ms and plan is not None:
        # the cascade's pieces: the whole path above counts every unique KV byte once
        cc = cascade_counts(b, plan)
        t_pre = statistics.mean(e[1].elapsed_time(e[4]) for e in evs)
        t_suf = statistics.mean(e[4].elapsed_time(e[5]) for e in evs)
        t_mrg = statistics.mean(e[5].elapsed_time(e[2]) for e in evs)
        pre_tf = cc["prefix_flops"] / (t_pre / 1e3) / 1e12
        suf_gbs = cc["suffix_bytes"] / (t_suf / 1e3) / 1e9
        kernels["decode"]["path"] = "cascade: shared-prefix parts + own-pages decode + merge"
        kernels["shared_prefix"] = {"ms": round(t_pre, 4), "tflops": round(pre_tf, 1),
                                    "frac_bf16": round(pre_tf / peaks["bf16_tflops"], 4),
                                    "peak_tflops": peaks["bf16_tflops"], "peak_kind": "burst",
                                    "flops": cc["prefix_flops"]}
        kernels["own_pages_decode"] = {"ms": round(t_suf, 4), "gbs": round(suf_gbs, 1),
                                       "frac_hbm": round(suf_gbs / peaks["hbm_gbs"], 4),
                                       "bytes": cc["suffix_bytes"]}
        kernels["merge"] = {"ms": round(t_mrg, 4),
                            "gbs": round(cc["merge_bytes"] / (t_mrg / 1e3) / 1e9, 1)}
    # per-kernel times come from CUDA events around each call of an eager pass: a kernel timed on
    # its own for tens of microseconds, so the burst tensor peak is its denominator
    ext_peak = peaks["bf16_tflops"]
    if ext_ms:
        ext_tflops = counts["extend_flops"] / (ext_ms / 1e3) / 1e12
        ext_gbs = counts["extend_bytes"] / (ext_ms / 1e3) / 1e9
        kernels["extend"] = {"ms": round(ext_ms, 4), "tflops": round(ext_tflops, 1),
                             "frac_bf16": round(ext_tflops / ext_peak, 4), "peak_tflops": ext_peak,
                             "peak_kind": "burst",
                             "flops": counts["extend_flops"], "gbs": round(ext_gbs, 1),
                             "frac_hbm": round(ext_gbs / peaks["hbm_gbs"], 4),
                             "bytes": counts["extend_bytes"]}
    if app_ms:
        kernels["kv_append"] = {"ms": round(app_ms, 4),
                                "gbs": round(counts["append_bytes"] / (app_ms / 1e3) / 1e9, 1)}
    traffic = _traffic_record() if args.workload == "mixed" else None
    if dec_ms and plan is not None and kernels["own_pages_decode"]["ms"] >= kernels["shared_prefix"]["ms"]:
        k = kernels["own_pages_decode"]
        roofline = {"kernel": "paged_decode over each request's own pages (decode + split merge)",
                    "bound": "hbm", "achieved": k["gbs"], "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": k["frac_hbm"], "traffic": None, "algorithmic_bytes": k["bytes"],
                    "peak_source": "of measured (MEASURED_PEAKS.json hbm_gbs)" if peaks["source"] == "measured" else "of fallback"}
    elif dec_ms and plan is not None:
        k = kernels["shared_prefix"]
        roofline = {"kernel": "shared-prefix attention (paged_extend_kernel, unmasked parts)",
                    "bound": "tensor", "achieved": k["tflops"], "peak": k["peak_tflops"],
                    "unit": "TFLOP/s", "frac": k["frac_bf16"], "traffic": None,
                    "algorithmic_flops": k["flops"],
                    "peak_source": "of measured (MEASURED_PEAKS.json bf16_tflops, burst)" if peaks["source"] == "measured" else "of fallback"}
    elif dec_ms:
        roofline = {"kernel": "paged_decode (decode + split merge)", "bound": "hbm",
                    "achieved": kernels["decode"]["gbs"], "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": kernels["decode"]["frac_hbm"], "traffic": traffic,
                    "algorithmic_bytes": counts["decode_bytes"],
                    "peak_source": "of measured (MEASURED_PEAKS.json hbm_gbs)" if peaks["source"] == "measured" else "of fallback"}
    elif not ext_ms:
        # only the append was timed: a copy, bounded by HBM bandwidth
        k = kernels["kv_append"]
        roofline = {"kernel": "kv_append", "bound": "hbm", "achieved": k["gbs"], "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": round(k["gbs"] / peaks["hbm_gbs"], 4), "traffic": None,
                    "algorithmic_bytes": counts["append_bytes"],
                    "peak_source": "of measured (MEASURED_PEAKS.json hbm_gbs)" if peaks["source"] == "measured" else "of fallback"}
    elif counts["extend_flops"] * peaks["hbm_gbs"] >= counts["extend_bytes"] * ext_peak * 1e3:
        # arithmetic intensity at or above the ridge point: bounded by the tensor cores
        roofline = {"kernel": "paged_extend", "bound": "tensor", "achieved": kernels["extend"]["tflops"],
                    "peak": ext_peak, "unit": "TFLOP/s", "frac": kernels["extend"]["frac_bf16"],
                    "traffic": None, "algorithmic_flops": counts["extend_flops"],
                    "peak_source": "of measured (MEASURED_PEAKS.json bf16_tflops, burst)" if peaks["source"] == "measured" else "of fallback"}
    else:
        # few queries per KV row (speculative verify): bounded by reading the KV pages
        roofline = {"kernel": "paged_extend", "bound": "hbm", "achieved": kernels["extend"]["gbs"],
                    "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": kernels["extend"]["frac_hbm"],
                    "traffic": None, "algorithmic_bytes": counts["extend_bytes"],
                    "peak_source": "of measured (MEASURED_PEAKS.json hbm_gbs)" if peaks["source"] == "measured" else "of fallback"}
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "tokens/s",
        "n_gpus": ws,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 q/k/v, seeded lengths and page permutation)",
        "config": {
            "workload": workload_label(args.workload, b),
            "decode_requests": b.num_decode, "extend_requests": b.num_extend,
            "new_tokens": b.num_new_tokens, "page_size": b.page_size, "num_pages": b.num_pages,
            "l2": ("L2 flushed (256 MB written) before every step" if args.flush_l2 else
                   "inputs larger than L2: each step reads ~%.1f GB of KV" % (counts["decode_bytes_logical"] / 1e9)),
            "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
            "append": "fused RoPE (theta 1e6) + KV append, queries rotated in place" if args.rope else "KV append",
            "decode_path": ("plain paged decode" if plan is None else
                            f"shared-prefix cascade: {plan.num_parts} parts in {plan.num_splits} splits of "
                            f"the shared pages ({plan.shared_tokens} tokens) on tensor cores, a decode over "
                            "each request's own pages, bf16 partial-state merge"),
            "decode_sms": decode_ctas or sms,
            "decode_l2_keep": ("each request's shared prefix evict-last in L2, the rest evict-first"
                               if use_keep else "none"),
            "launch": ("eager launches" if args.eager else "CUDA graph of the whole step")
            + ("; two branches: (append of the decodes' tokens, decode, merge) beside (append of the "
               "extend tokens, extend)" if overlap else "; one stream")
            + " (per-kernel times from an eager pass on one stream)",
        "e2e_copies": "each step's inputs (one pinned buffer) in and outputs out on two copy streams, "
                      "overlapping the neighbouring steps' computation (two device buffer sets)",
        },
        "ms_per_step_eager": round(eager_ms / K, 4),
        "roofline": roofline,
        "kernels": kernels,
        "e2e": {"value": round(tokens * K2 * ws / (e2e_ms / 1e3), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "step": "captured graph per buffer set" if set_graphs[0] is not None else "eager calls"},
        # kernels of the timed step: the append (two, one per branch, when the step is branched),
        # decode and its split merge, the extend's request ordering and the extend
        "gpu_launches": ((2 if overlap and not args.eager else int(bool(app_ms))) + dec_launches * int(do_dec)
                         + (1 + int(ext_ws > 0)) * int(do_ext)) * K,
        "clocks": clk,
    }
    return line


# ---------------------------------------------------------------------------------------------
# CPU oracle (reported baseline and reference arm)
# ---------------------------------------------------------------------------------------------
def _oracle_sample_runner(b, kp, vp):
    """A bounded slice of the workload for the oracle: callable(k) -> attention tokens done.

    Slice k is decode request k (all heads) and up to 8 consecutive query rows of extend chunk k,
    for whichever of the two the workload has."""
    import torch as _t

    import oracle

    B = b.num_decode
    qo = b.ext_qo_indptr.tolist()
    rows_per_call = 8

    def run(k):
        done = 0
        if B:
            oracle.paged_decode(b.dec_q, kp, vp, b.dec_kv_indptr, b.dec_kv_indices, b.dec_kv_lens,
                                b.page_size, b.sm_scale, requests=[k % B])
            done += 1
        if b.num_extend:
            e = k % b.num_extend
            E = qo[e + 1] - qo[e]
            i0 = (k * rows_per_call) % E
            n = min(rows_per_call, E - i0)
            q_rows = b.ext_q[qo[e] + i0: qo[e] + i0 + n]
            lo, hi = int(b.ext_kv_indptr[e]), int(b.ext_kv_indptr[e + 1])
            oracle.paged_extend(q_rows, kp, vp, _t.tensor([0, n], dtype=_t.int32),
                                _t.tensor([0, hi - lo], dtype=_t.int32), b.ext_kv_indices[lo:hi],
                                (b.ext_prefix_lens[e:e + 1] + i0).to(_t.int32), b.page_size, b.sm_scale)
            done += n
        return done

    return run


def cpu_baseline(b, seconds=12.0, threads=0):
    import torch as _t

    import oracle

    cores = threads if threads > 0 else len(os.sched_getaffinity(0))
    _t.set_num_threads(cores)
    kp, vp = oracle.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.slot_mapping, b.page_size)
    run = _oracle_sample_runner(b, kp, vp)
    t0 = time.perf_counter()
    toks, k = 0, 0
    while time.perf_counter() - t0 < seconds:
        toks += run(k)
        k += 1
    el = time.perf_counter() - t0
    return {"value": round(toks / el, 2), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{k} slices of the workload, each 1 decode request (all heads) and/or up to 8 "
                      f"extend query rows of one request; {toks} attention tokens in {el:.1f} s; fp64 NumPy, "
                      f"BLAS and torch limited to {cores} threads"}


def workload_label(name, b):
    """The workload as the JSON line's config names it (the same for both arms)."""
    if name != "mixed":
        return b.name
    return ("mixed continuous-batching step: kv_append 2304 tokens + paged decode of 256 requests (KV "
            "U[512,4096], 64 share a 2048-token prefix) + ragged extend of 4x512 chunked-prefill tokens "
            "(prefixes 0/512/1024/1536); Qwen3-8B attention 32q/8kv heads, head_dim 128, page 16")


def run_reference(args, ws, rank):
    if rank != 0:
        return None
    import oracle

    import torch as _t

    cores = args.cpu_threads if args.cpu_threads > 0 else len(os.sched_getaffinity(0))
    _t.set_num_threads(cores)
    b = load_workload(args.workload)
    kp, vp = oracle.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.slot_mapping, b.page_size)
    run = _oracle_sample_runner(b, kp, vp)
    for k in range(args.warmup):
        run(k)
    budget = 150.0
    t0 = time.perf_counter()
    toks, done = 0, 0
    for k in range(args.steps):
        toks += run(k)
        done += 1
        if time.perf_counter() - t0 > budget:
            break
    el = time.perf_counter() - t0
    val = toks / el
    return {"impl": "reference", "metric": METRIC, "value": round(val, 2), "unit": "tokens/s",
            "n_gpus": ws, "steps": args.steps, "steps_completed": done, "warmup": args.warmup,
            "ms_per_step": round(el / done * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_label(args.workload, b) + " (a bounded oracle sample per step)"},
            "cpu_baseline": {"value": round(val, 2), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": "per step: 1 decode request (all heads) and/or up to 8 extend query "
                                       "rows of one request of this workload"},
            "e2e": {"value": round(val, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# SMs the branched step's decode leaves to the extend beside it (swept on the mixed step: 12 of
# 152 gave the shortest step once the decode kept its shared prefix in L2; 16 before)
EXTEND_SPARE_SMS = 12

WORKLOADS = {"mixed": 5, "tiny": 1, "batched-decode": 2, "radix-extend": 3, "long-decode": 4}


def load_workload(name):
    """The mixed step (default), the other four workloads, or a few-hundred-MB profiler case."""
    if name in WORKLOADS:
        from workloads import make_config

        return make_config(WORKLOADS[name])
    if name == "spec-verify":
        from workloads import make_spec_verify

        return make_spec_verify()
    if name == "shared-prefix-decode":
        from workloads import make_shared_prefix_decode

        return make_shared_prefix_decode()
    if name == "small-prefill":
        from workloads import make_small_prefill

        return make_small_prefill()
    if name == "profile":
        from workloads import random_small_batch

        return random_small_batch(7001, page_size=16, num_q_heads=32, num_kv_heads=8, head_dim=128,
                                  decode_lens=(4096,) * 16, decode_new=1,
                                  extend=((1024, 512), (1536, 512)), pool_slack=1.1)
    raise ValueError(name)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="mixed",
                    choices=sorted(WORKLOADS) + ["spec-verify", "shared-prefix-decode", "small-prefill",
                                                 "profile"])
    ap.add_argument("--cascade", action="store_true",
                    help="decode through the shared-prefix (cascade) plan: the shared pages once per "
                         "group on tensor cores, each request's own pages, and a merge")
    ap.add_argument("--flush-l2", action="store_true",
                    help="zero a 256 MB buffer before every timed step (for workloads that fit in L2); "
                         "the step time is then the sum of the per-operation event times")
    ap.add_argument("--op", default="all", choices=["all", "decode", "extend", "append"],
                    help="time only one operation of the step (default: the whole step)")
    ap.add_argument("--no-e2e", action="store_true",
                    help="skip the end-to-end run (host buffers, copies inside the timed region)")
    ap.add_argument("--rope", action="store_true",
                    help="fuse the rotary embedding of the new K and of all queries into the append")
    ap.add_argument("--eager", action="store_true",
                    help="time eager launches instead of the step captured as one CUDA graph")
    ap.add_argument("--decode-sms", type=int, default=-1,
                    help="SMs the decode may use (0 = all; default: all but 16 when the step's extend "
                         "runs beside the decode in its own graph branch, else all)")
    ap.add_argument("--no-l2-keep", action="store_true",
                    help="decode without the L2 keep hint for the requests' shared prefixes")
    ap.add_argument("--serial-step", action="store_true",
                    help="run the step's operations one after another on one stream (no branches)")
    ap.add_argument("--gpus", type=int, default=1,
                    help="GPUs of this node; N > 1 runs under torchrun, one replica per rank")
    ap.add_argument("--steps", type=int, default=3000, help="timed steps")
    ap.add_argument("--warmup", type=int, default=10, help="untimed warm-up steps (at least 3)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"],
                    help="reference: time the fp64 CPU oracle on the host cores instead")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="seconds of CPU-oracle work for the cpu_baseline figure")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the cpu_baseline figure")
    ap.add_argument("--cpu-threads", type=int, default=0,
                    help="threads the CPU oracle may use (default: every affinity core)")
    args = ap.parse_args()
    if args.cpu_threads > 0:  # before NumPy or torch start their thread pools
        for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[var] = str(args.cpu_threads)
    if args.warmup < 3:
        args.warmup = 3
    ws, rank, local = _dist_env()
    if args.impl == "reference":
        line = run_reference(args, ws, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if ws > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    line = run_ours(args, ws, rank, local)
    if rank == 0:
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(load_workload(args.workload), args.cpu_seconds,
                                                args.cpu_threads)
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()

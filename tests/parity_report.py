"""Parity report: every workload run through the library as the benchmark runs it, compared with
the fp64 oracle, one markdown row per operation (max-abs and mean-abs error of O, max LSE error,
and the bf16 floor mean|bf16(oracle) - oracle|, the error of the best possible bf16 answer).

Test infrastructure (it calls the oracle): ``python tests/parity_report.py`` on a GPU machine.
Large workloads are checked on a sample of requests, named in the row.
"""

import os
import sys

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

import oracle  # noqa: E402
import paged_kv_attention_10_gb300 as pkv  # noqa: E402
from paged_kv_attention_10_gb300.cascade import plan_shared_prefix  # noqa: E402
from workloads import (make_config, make_shared_prefix_decode, make_small_prefill,  # noqa: E402
                       make_spec_verify)
from _gpu_helpers import DeviceBatch, attention_errors  # noqa: E402


def _row(name, what, out, lse, o_ref, l_ref, rows=None):
    mx, mean, lerr, floor = attention_errors(out, lse, o_ref, l_ref, rows)
    ok = mx <= 1e-2 and mean <= 1e-3 and lerr <= 1e-3
    print(f"| {name} | {what} | {mx:.2e} | {mean:.2e} | {lerr:.2e} | {floor:.2e} | {'yes' if ok else 'NO'} |")
    return ok


def _appended(b):
    d = DeviceBatch(b)
    pkv.kv_append(d.k_pool, d.v_pool, d.k_new, d.v_new, d.slot_mapping)
    kp, vp = oracle.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.slot_mapping, b.page_size)
    torch.cuda.synchronize()
    same = torch.equal(d.k_pool.cpu().view(torch.int16), kp.view(torch.int16)) and \
        torch.equal(d.v_pool.cpu().view(torch.int16), vp.view(torch.int16))
    return d, kp, vp, same


def main():
    torch.cuda.set_device(0)
    pkv.load()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rng = np.random.default_rng(0)
    print("| workload | operation (rows checked) | O max-abs | O mean-abs | LSE max-abs | bf16 floor | within 1e-2 / 1e-3 / 1e-3 |")
    print("|---|---|---|---|---|---|---|")
    ok = True
    names = {1: "tiny decode + append", 2: "batched decode, page 1", 3: "radix extend",
             4: "long-context decode 8 x 32K", 5: "mixed step"}
    for idx in (1, 2, 3, 4, 5):
        b = make_config(idx)
        d, kp, vp, same = _appended(b)
        if b.num_new_tokens:
            print(f"| {names[idx]} | kv_append ({b.num_new_tokens} tokens) | bit-exact: {'yes' if same else 'NO'} | | | | {'yes' if same else 'NO'} |")
            ok &= same
        if b.num_decode:
            ctas = sms - 12 if idx == 5 else 0  # the branched step's decode leaves 12 SMs to the extend
            out, lse = pkv.paged_decode(d.dec_q, d.k_pool, d.v_pool, d.dec_kv_indptr, d.dec_kv_indices,
                                        d.dec_kv_lens, b.sm_scale, max_ctas=ctas)
            sample = None
            if b.num_decode > 64:
                sample = sorted(rng.choice(b.num_decode, 64, replace=False).tolist())
            o_ref, l_ref = oracle.paged_decode(b.dec_q, kp, vp, b.dec_kv_indptr, b.dec_kv_indices,
                                               b.dec_kv_lens, b.page_size, b.sm_scale, requests=sample)
            what = f"decode ({'all ' + str(b.num_decode) if sample is None else '64 of ' + str(b.num_decode)} requests)"
            ok &= _row(names[idx], what, out, lse, o_ref, l_ref, None if sample is None else np.array(sample))
        if b.num_extend:
            out, lse = pkv.paged_extend(d.ext_q, d.k_pool, d.v_pool, d.ext_qo_indptr, d.ext_kv_indptr,
                                        d.ext_kv_indices, d.ext_prefix_lens, b.max_extend_len, b.sm_scale)
            o_ref, l_ref = oracle.paged_extend(b.ext_q, kp, vp, b.ext_qo_indptr, b.ext_kv_indptr,
                                               b.ext_kv_indices, b.ext_prefix_lens, b.page_size, b.sm_scale)
            ok &= _row(names[idx], f"extend (all {int(b.ext_qo_indptr[-1])} query rows)", out, lse, o_ref, l_ref)
        del d
        torch.cuda.empty_cache()

    for name, b in (("speculative verify", make_spec_verify()), ("small-model prefill", make_small_prefill())):
        d, kp, vp, same = _appended(b)
        out, lse = pkv.paged_extend(d.ext_q, d.k_pool, d.v_pool, d.ext_qo_indptr, d.ext_kv_indptr,
                                    d.ext_kv_indices, d.ext_prefix_lens, b.max_extend_len, b.sm_scale)
        o_ref, l_ref = oracle.paged_extend(b.ext_q, kp, vp, b.ext_qo_indptr, b.ext_kv_indptr,
                                           b.ext_kv_indices, b.ext_prefix_lens, b.page_size, b.sm_scale)
        ok &= _row(name, f"extend (all {int(b.ext_qo_indptr[-1])} query rows)", out, lse, o_ref, l_ref)
        ok &= same

    b = make_shared_prefix_decode()
    d, kp, vp, same = _appended(b)
    plan = plan_shared_prefix(b.dec_kv_indptr, b.dec_kv_indices, b.dec_kv_lens, [(0, b.num_decode)], b.page_size,
                              num_kv_heads=b.num_kv_heads, group_size=b.num_q_heads // b.num_kv_heads,
                              num_sms=sms)
    out, lse = pkv.cascade_decode(d.dec_q, d.k_pool, d.v_pool, plan.to("cuda"), b.sm_scale)
    sample = sorted(rng.choice(b.num_decode, 32, replace=False).tolist())
    o_ref, l_ref = oracle.paged_decode(b.dec_q, kp, vp, b.dec_kv_indptr, b.dec_kv_indices, b.dec_kv_lens,
                                       b.page_size, b.sm_scale, requests=sample)
    ok &= _row("shared-prefix decode", f"cascade decode (32 of {b.num_decode} requests)", out, lse, o_ref, l_ref,
               np.array(sample))
    print()
    print("all within tolerance" if ok else "SOME OUTSIDE TOLERANCE")
    return 0 if ok else 1


if __name__ == "__main__":
    sys.exit(main())

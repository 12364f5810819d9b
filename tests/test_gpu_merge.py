"""merge_states on the GPU against the oracle's log-sum-exp merge."""

import numpy as np
import pytest
import torch

import oracle
from _fixtures import load_golden
from _gpu_helpers import assert_attention_close

pytestmark = pytest.mark.gpu


def test_golden_merge_on_gpu(lib):
    c = load_golden()["merge_two_splits"]
    o = torch.zeros((3, 1, 1, 4), dtype=torch.float32)
    o[..., :2] = torch.tensor(c["o_parts"], dtype=torch.float32)[:, :, None, :]
    l = torch.tensor(c["lse_parts"], dtype=torch.float32)[:, :, None]
    out, lse = lib.merge_states(o.cuda(), l.cuda())
    assert np.abs(out[0, 0, :2].float().cpu().numpy() - np.array(c["expect_o"][0])).max() <= 1e-2
    assert abs(float(lse[0, 0]) - c["expect_lse"][0]) <= 1e-3


@pytest.mark.parametrize("S,N,H,D", [(1, 3, 4, 64), (4, 17, 8, 128), (16, 8, 32, 128), (5, 2, 3, 256),
                                     (40, 3, 2, 64), (70, 2, 4, 132)])
def test_merge_random(lib, S, N, H, D):
    g = torch.Generator().manual_seed(S * 1000 + N)
    # partial outputs of attention are averages of V rows: magnitudes well below 1
    o = torch.randn((S, N, H, D), generator=g) * 0.25
    l = torch.randn((S, N, H), generator=g) * 3
    # some empty splits, and one row whose splits are all empty
    l[0, 0, 0] = -float("inf")
    if S > 1:
        l[:, -1, -1] = -float("inf")
    o_dev = o.clone()
    o_dev[0, 0, 0] = float("nan")  # an empty split contributes nothing, whatever its o holds
    out, lse = lib.merge_states(o_dev.cuda(), l.cuda())
    o_ref, lse_ref = oracle.merge_states(o.double().numpy(), l.double().numpy())
    fin = np.isfinite(lse_ref)
    assert np.all(np.isneginf(lse.cpu().numpy()[~fin]))
    assert torch.all(out.float().cpu()[torch.tensor(~fin)] == 0)
    assert_attention_close(out.reshape(N * H, D), lse.reshape(-1), o_ref.reshape(N * H, D),
                           lse_ref.reshape(-1), rows=np.nonzero(fin.reshape(-1))[0], what="merge")

"""The backward run with a bounded workspace: below the full size the dK/dV
and dQ kernels take the (sample, head) pairs in consecutive groups that
reuse one region of dS tiles. Every output must be byte-identical to the
single-group run (a pair's arithmetic never depends on its group), for a
ragged last group and for one pair per group."""

import pytest

import invariant_mmdit_joint_gb300 as pkg
from invariant_mmdit_joint_gb300 import workloads as W
from tests import _helpers as Hh

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


def _run(w, batch, dev, budget=None):
    import torch
    ja = pkg.JointAttention(w.B, w.T_txt, w.grid_h, w.grid_w, w.H, device=dev, ws_budget_bytes=budget)
    res = Hh.run_gpu(ja, batch, dev)
    pkg.rlk_joint_attn_check_status()
    torch.cuda.synchronize()
    return ja, res


CASES = [
    # 1328^2 on 3 heads: 12 pairs; room for 5 -> groups of 5, 5, 2
    (Hh.workload("img1328_h3", 4, 3, 256, 83, 83, (40, 40, 256, 129), scale=3.0), 5),
    # odd tiles, one pair per group
    (Hh.workload("ragged", 3, 2, 200, 13, 21, (0, 130, 200)), 1),
]


@pytest.mark.parametrize("w,pairs", CASES, ids=[c[0].name for c in CASES])
def test_bounded_workspace_gives_the_same_bytes(dev, w, pairs):
    batch = W.make_batch(w, seed=8)
    ja_full, full = _run(w, batch, dev)
    least = pkg.rlk_joint_attn_bwd_workspace_min_bytes(ja_full.shape)
    one_pair = (pkg.rlk_joint_attn_bwd_workspace_bytes(ja_full.shape) - least) // (w.B * w.H - 1)
    ja, part = _run(w, batch, dev, budget=least + (pairs - 1) * one_pair)
    assert ja.workspace.numel() < ja_full.workspace.numel()
    for key in ("out", "lse", "dq", "dk", "dv", "dgp", "dg"):
        assert Hh.bits_equal(part[key], full[key]), key


def test_budget_below_the_minimum_is_refused(dev):
    w = W.TINY
    shape = pkg.Shape.make(w.B, w.T_txt, w.grid_h, w.grid_w, w.H)
    with pytest.raises(pkg.RlkError):
        pkg.JointAttention(w.B, w.T_txt, w.grid_h, w.grid_w, w.H, device=dev,
                           ws_budget_bytes=pkg.rlk_joint_attn_bwd_workspace_min_bytes(shape) - 1)

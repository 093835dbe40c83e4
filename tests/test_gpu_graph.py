"""The forward and backward captured into one CUDA graph: replays give the
same bytes as eager calls, including after new inputs are copied into the
captured tensors (the calls read host arguments and encode their tensor
maps at capture time; only device memory changes between replays)."""

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


CASES = [W.TINY, Hh.workload("ragged", 3, 2, 200, 9, 13, (0, 200, 77))]


def _inputs(w, seed, dev):
    import torch
    batch = W.make_batch(w, seed)
    q, k, v, do = (Hh.to_dev(batch[n], dev) for n in ("q", "k", "v", "do"))
    gains = torch.from_numpy(batch["gains"]).to(dev)
    return (q, k, v, do, gains), [int(x) for x in batch["valid_len"]]


def _step(ja, tensors, vl, outs):
    q, k, v, do, gains = tensors
    out, lse, dq, dk, dv, dgp, dg = outs
    ja.forward(q, k, v, gains, vl, out=out, lse=lse)
    ja.backward(q, k, v, gains, vl, out, do, lse, dq=dq, dk=dk, dv=dv, dg_partial=dgp, dg=dg)


def _alloc(w, tensors, dev):
    import torch
    q = tensors[0]
    return (torch.empty_like(q), torch.empty((w.B, w.H, q.shape[1]), dtype=torch.float32, device=dev),
            torch.empty_like(q), torch.empty_like(q), torch.empty_like(q),
            torch.empty((w.B, w.H, 4, 128), dtype=torch.float32, device=dev),
            torch.empty((4, 128), dtype=torch.float32, device=dev))


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_graph_replay_matches_eager(w, dev):
    import torch
    a, vl = _inputs(w, 11, dev)
    b, _ = _inputs(w, 12, dev)  # same valid lengths (fixed per workload), other values
    ja = pkg.JointAttention(w.B, w.T_txt, w.grid_h, w.grid_w, w.H, device=dev)
    # eager results on both input sets
    ref = []
    for t in (a, b):
        o = _alloc(w, t, dev)
        _step(ja, t, vl, o)
        torch.cuda.synchronize()
        ref.append([x.clone() for x in o])
    # capture on inputs that start as a, on a side stream as torch requires
    cap_in = [x.clone() for x in a]
    cap_out = _alloc(w, cap_in, dev)
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            _step(ja, cap_in, vl, cap_out)
    torch.cuda.current_stream().wait_stream(s)
    for which, src in ((0, a), (1, b), (0, a)):
        for dst, x in zip(cap_in, src):
            dst.copy_(x)
        g.replay()
        torch.cuda.synchronize()
        pkg.rlk_joint_attn_check_status()
        for name, got, want in zip(("out", "lse", "dq", "dk", "dv", "dg_partial", "dg"), cap_out, ref[which]):
            assert Hh.bits_equal(got, want), (w.name, which, name)

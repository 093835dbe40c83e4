"""The operator trace on real calls: each C ABI call leaves one record with
the kernels it enqueued, the backend that ran them and no fallback (the
RFC's qwenimage_operator_trace row and the WS1 kernel list's rule 7)."""

import pytest

import invariant_mmdit_joint_gb300 as pkg
from invariant_mmdit_joint_gb300 import workloads as W
from tests import _helpers as Hh

pytestmark = pytest.mark.gpu

FWD = ["rope_table_kernel", "prologue_kernel", "attn_fwd_tc_kernel"]
BWD = ["bwd_pre_kernel", "attn_bwd_dkdv_tc_kernel", "attn_bwd_dq_tc_kernel", "norm_rope_bwd_k_kernel",
       "dg_fold_kernels"]


@pytest.fixture(scope="module")
def dev():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


def test_each_call_records_its_kernels(dev):
    import torch
    w = W.TINY
    batch = W.make_batch(w, 3)
    q, k, v, do = (Hh.to_dev(batch[n], dev) for n in ("q", "k", "v", "do"))
    gains = torch.from_numpy(batch["gains"]).to(dev)
    vl = [int(x) for x in batch["valid_len"]]
    ja = pkg.JointAttention(w.B, w.T_txt, w.grid_h, w.grid_w, w.H, device=dev)
    shape = pkg.Shape.make(w.B, w.T_txt, w.grid_h, w.grid_w, w.H)
    with pkg.op_trace() as t:
        out, lse = ja.forward(q, k, v, gains, vl)
        ja.backward(q, k, v, gains, vl, out, do, lse)
        ja.forward_unfused(q, k, v, gains, vl)
        out2 = torch.empty_like(q)
        pkg.rlk_joint_attn_fwd_noalloc(shape, q, k, v, gains[0], gains[1], gains[2], gains[3], vl, out2, None)
        torch.cuda.synchronize()
    pkg.rlk_joint_attn_check_status()
    got = [(r["entry_point"], r["kernels"]) for r in t.records]
    assert got == [
        ("rlk_joint_attn_fwd", FWD),
        ("rlk_joint_attn_bwd", BWD),
        ("rlk_qk_norm_rope", FWD[:2]),
        ("rlk_joint_attn_qk_gemm", ["qk_gemm_kernel"]),
        ("rlk_joint_attn_softmax", ["softmax_kernel"]),
        ("rlk_joint_attn_av_gemm", ["av_gemm_kernel"]),
        # the allocation-free forward is one record: the regular forward it
        # runs inside adds its kernels there
        ("rlk_joint_attn_fwd_noalloc", FWD),
    ]
    for r in t.records:
        assert r["status"] == 0 and r["actual_backend"] == "sm_103a tcgen05" and r["fallback"] == 0
        assert (r["B"], r["H"], r["T_txt"], r["grid_h"], r["grid_w"]) == (w.B, w.H, w.T_txt, w.grid_h, w.grid_w)
    assert [r["seq"] for r in t.records] == list(range(1, 8))

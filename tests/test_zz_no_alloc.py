"""The allocation-free forward (rlk_joint_attn_fwd_noalloc) against the
regular forward (rlk_joint_attn_fwd), through the C ABI.

Callers that cannot allocate device memory on the call path (plugin hosts
without a workspace, serving processes whose pool owns the device) use the
allocation-free entry point; its context lives in a fixed device array in the
library. This file is collected last so that a failure here never hides the
other tests. It must pass alone in a fresh process and after the others.
"""

import ctypes

import numpy as np
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


def _inputs(w, seed, dev):
    import torch
    batch = W.make_batch(w, seed, with_dout=False)
    q, k, v = (Hh.to_dev(batch[n], dev) for n in ("q", "k", "v"))
    gains = torch.from_numpy(batch["gains"]).to(dev)
    return q, k, v, gains, [int(x) for x in batch["valid_len"]]


def _noalloc(w, q, k, v, gains, vl, dev):
    import torch
    shape = pkg.Shape.make(w.B, w.T_txt, w.grid_h, w.grid_w, w.H)
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, shape.S), dtype=torch.float32, device=dev)
    pkg.rlk_joint_attn_fwd_noalloc(shape, q, k, v, gains[0], gains[1], gains[2], gains[3], vl, out, lse)
    return out, lse


def _compare(w, a_out, a_lse, b_out, b_lse):
    Hh.assert_forward_close(Hh.f64(a_out), Hh.f64(a_lse), Hh.f64(b_out), Hh.f64(b_lse), w.name, scale=w.scale)
    # the same kernels run on the same inputs: the bytes agree as well
    assert Hh.bits_equal(a_out, b_out) and Hh.bits_equal(a_lse, b_lse)


def test_noalloc_forward_matches_regular_forward_twice_in_a_row(dev):
    import torch
    small = Hh.workload("small", 2, 4, 64, 16, 16, (50, 7))
    one_image = Hh.workload("cfg1024_one_sample", 1, 24, 256, 64, 64, (87,))
    for w, seed in ((small, 11), (one_image, 12)):
        ja = pkg.JointAttention(w.B, w.T_txt, w.grid_h, w.grid_w, w.H, device=dev)
        x1 = _inputs(w, seed, dev)
        x2 = _inputs(w, seed + 100, dev)
        n1 = _noalloc(w, *x1, dev)
        n2 = _noalloc(w, *x2, dev)   # second call in a row reuses the shared scratch
        torch.cuda.synchronize()
        pkg.rlk_joint_attn_check_status()
        r1 = ja.forward(*x1)
        r2 = ja.forward(*x2)
        torch.cuda.synchronize()
        _compare(w, n1[0], n1[1], r1[0], r1[1])
        _compare(w, n2[0], n2[1], r2[0], r2[1])


def test_noalloc_rejects_shapes_beyond_its_scratch(dev):
    import torch
    w = W.CFG1024  # two samples need about 109 MB of context
    shape = pkg.Shape.make(w.B, w.T_txt, w.grid_h, w.grid_w, w.H)
    assert pkg.rlk_joint_attn_ctx_bytes(shape) > (64 << 20)
    buf = torch.zeros(16, dtype=torch.bfloat16, device=dev)
    p = buf.data_ptr()
    vl = (ctypes.c_int32 * 2)(87, 193)
    rc = pkg.lib().rlk_joint_attn_fwd_noalloc(ctypes.byref(shape), p, p, p, p, p, p, p, vl, p, p, None)
    assert rc == 4  # RLK_ERR_WORKSPACE, nothing launched
    assert np.all(buf.cpu().float().numpy() == 0)

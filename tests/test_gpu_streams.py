"""Separate text and image buffers (no concatenation copy) against the
concatenated calls: every output byte must agree, forward and backward."""

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


CASES = [
    W.TINY,
    Hh.workload("ragged", 3, 2, 200, 13, 21, (0, 130, 200)),
    Hh.workload("no_text", 2, 3, 0, 5, 7, (0, 0)),
    W.CFG1024,
]


def _split(t, T):
    """Two separately allocated stream tensors (None for an empty text stream)."""
    txt = t[:, :T].clone() if T > 0 else None
    return txt, t[:, T:].clone()


def _join(pair):
    import torch
    return pair[1] if pair[0] is None else torch.cat(pair, dim=1)


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_separate_streams_give_the_concatenated_bytes(w, dev):
    import torch
    batch = W.make_batch(w, 41)
    q, k, v, do = (Hh.to_dev(batch[n], dev) for n in ("q", "k", "v", "do"))
    gains = torch.from_numpy(batch["gains"]).to(dev)
    vl = [int(x) for x in batch["valid_len"]]
    ja = pkg.JointAttention(w.B, w.T_txt, w.grid_h, w.grid_w, w.H, device=dev)
    ref = Hh.run_gpu(ja, batch, dev)
    ref = {key: val.clone() for key, val in ref.items()}
    T = w.T_txt
    qs, ks, vs, dos = (_split(t, T) for t in (q, k, v, do))
    out, lse = ja.forward_streams(qs, ks, vs, gains, vl)
    dq, dk, dv, dgp, dg = ja.backward_streams(qs, ks, vs, gains, vl, out, dos, lse)
    torch.cuda.synchronize()
    pkg.rlk_joint_attn_check_status()
    got = {"out": _join(out), "lse": lse, "dq": _join(dq), "dk": _join(dk), "dv": _join(dv), "dgp": dgp, "dg": dg}
    for key, val in got.items():
        assert Hh.bits_equal(val.contiguous(), ref[key].contiguous()), (w.name, key)

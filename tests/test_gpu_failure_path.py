"""The failure path of the bounded device waits, exercised without a fault:
a probe warp waits on an mbarrier that nothing completes, gives up after a
short limit and records the failure in the status word the host reads; the
context stays usable and the next calls run normally."""

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


def test_timed_out_wait_is_reported_and_the_context_stays_usable(dev):
    import torch
    w = W.TINY
    batch = W.make_batch(w, 7)
    q, k, v, do = (Hh.to_dev(batch[n], dev) for n in ("q", "k", "v", "do"))
    gains = torch.from_numpy(batch["gains"]).to(dev)
    vl = [int(x) for x in batch["valid_len"]]
    ja = pkg.JointAttention(w.B, w.T_txt, w.grid_h, w.grid_w, w.H, device=dev)
    out_ref, lse_ref = ja.forward(q, k, v, gains, vl)
    torch.cuda.synchronize()
    pkg.rlk_joint_attn_check_status()  # clean before the probe

    pkg.rlk_selftest_wait_timeout(50)
    torch.cuda.synchronize()
    with pytest.raises(pkg.RlkError) as e:
        pkg.rlk_joint_attn_check_status()
    assert e.value.code == 6  # RLK_ERR_DEVICE_TIMEOUT
    pkg.rlk_joint_attn_check_status()  # reading cleared it

    # the context is intact: the same call gives the same bytes
    out, lse = ja.forward(q, k, v, gains, vl)
    ja.backward(q, k, v, gains, vl, out, do, lse)
    torch.cuda.synchronize()
    pkg.rlk_joint_attn_check_status()
    assert Hh.bits_equal(out, out_ref) and Hh.bits_equal(lse, lse_ref)


def test_limit_out_of_range_fails_closed(dev):
    for bad in (0, -1, 2001):
        with pytest.raises(pkg.RlkError) as e:
            pkg.rlk_selftest_wait_timeout(bad)
        assert e.value.code == 1

"""GPU parity: the CUDA path through the C ABI against the CPU oracle, on the
same seeded inputs, at the declared tolerances. Small geometries are compared
element by element over every output; the full-size workloads are compared on
a head subset (all outputs of heads 0 and H-1) plus sampled forward rows."""

import numpy as np
import pytest

from invariant_mmdit_joint_gb300 import workloads as W
from oracle import joint_attn as O
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


def _ja(w, dev):
    import invariant_mmdit_joint_gb300 as pkg
    return pkg.JointAttention(w.B, w.T_txt, w.grid_h, w.grid_w, w.H, device=dev)


def _full_compare(w, batch, res, heads=None, where="", pure=True):
    """Compare every output of the given heads (all heads by default)."""
    all_heads = heads is None or len(heads) == w.H
    heads = list(range(w.H)) if heads is None else list(heads)
    sub = {n: batch[n][:, :, heads] for n in ("q", "k", "v", "do") if n in batch}
    sub["gains"] = batch["gains"]
    Q, K, V, dO, g = Hh.oracle_inputs(sub)
    vl = batch["valid_len"]
    ro, rl = O.joint_attn_forward(Q, K, V, g, w.T_txt, w.grid_h, w.grid_w, vl, store_bf16=True)
    out = Hh.f64(res["out"][:, :, heads])
    lse = Hh.f64(res["lse"][:, heads])
    Hh.assert_forward_close(out, lse, ro, rl, where, scale=w.scale)
    if pure:
        po, pl = O.joint_attn_forward(Q, K, V, g, w.T_txt, w.grid_h, w.grid_w, vl)
        Hh.assert_forward_close_exact(out, lse, (ro, rl), (po, pl), where + " (exact f64)", scale=w.scale)
    if "dq" not in res:
        return
    rdq, rdk, rdv, rdgp, rdg = O.joint_attn_backward(Q, K, V, g, dO, w.T_txt, w.grid_h, w.grid_w, vl,
                                                     store_bf16=True)
    got = {n: Hh.f64(res[n][:, :, heads]) for n in ("dq", "dk", "dv")}
    for name, b in (("dq", rdq), ("dk", rdk), ("dv", rdv)):
        for bb in range(w.B):
            for j, h in enumerate(heads):
                Hh.assert_grad_close(name, got[name][bb, :, j], b[bb, :, j], f"{where} b={bb} h={h}")
    gp = Hh.f64(res["dgp"][:, heads])
    for bb in range(w.B):
        for j, h in enumerate(heads):
            for slot in range(4):
                if np.linalg.norm(rdgp[bb, j, slot]) > 0:
                    Hh.assert_grad_close("dg_partial", gp[bb, j, slot], rdgp[bb, j, slot],
                                         f"{where} b={bb} h={h} slot={slot}")
    if all_heads:
        Hh.assert_grad_close("dg", Hh.f64(res["dg"]), rdg, where)
    # masked keys get exactly zero gradient
    for bb in range(w.B):
        L = int(vl[bb])
        assert np.all(got["dk"][bb, L:w.T_txt] == 0)
        assert np.all(got["dv"][bb, L:w.T_txt] == 0)


def test_tiny_forward_backward_matches_oracle(dev):
    w = W.TINY
    batch = W.make_batch(w, seed=0)
    res = Hh.run_gpu(_ja(w, dev), batch, dev)
    _full_compare(w, batch, res, where="tiny")


def test_prologue_matches_oracle_storage_rounding(dev):
    """The stored q and k are the oracle's exact values rounded to bf16: equal
    except where the FP32 arithmetic lands on the other side of a rounding
    midpoint (then one bf16 ulp off, and rare); the exact values are within
    one ulp plus the FP32 error of the rotation."""
    w = Hh.workload("pro", 2, 3, 40, 7, 9, (13, 40))
    batch = W.make_batch(w, seed=3, with_dout=False)
    ja = _ja(w, dev)
    Hh.run_gpu(ja, batch, dev, with_bwd=False)
    qh, kh, rq, rk = (Hh.f64(t) for t in ja.ctx_views())
    Q, K, V, _, g = Hh.oracle_inputs(batch)
    rqh, rkh, rrq, rrk = O.prologue(Q, K, g, w.T_txt, w.grid_h, w.grid_w)
    for got, ref in ((qh, rqh), (kh, rkh)):
        stored = O.round_bf16(ref)
        ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(stored), 2.0 ** -60))) - 7)
        diff = np.abs(got - stored)
        # FP32 error of the rotation, relative to the pair's norm (matters
        # where the two terms of a rotated coordinate cancel)
        pair = np.repeat(np.hypot(ref[..., 0::2], ref[..., 1::2]), 2, axis=-1)
        assert np.all(diff <= ulp + 1e-6 * pair)
        assert np.count_nonzero(diff) <= 2e-3 * diff.size, np.count_nonzero(diff)
        assert np.all(np.abs(got - ref) <= ulp + 1e-6 * pair)
    assert np.max(np.abs(rq - rrq) / rrq) <= 1e-6
    assert np.max(np.abs(rk - rrk) / rrk) <= 1e-6


EDGE = [
    # no text at all
    Hh.workload("no_text", 2, 3, 0, 5, 7, (0, 0)),
    # ragged: text tile partially filled; L = 0 and L = T_txt in one batch
    Hh.workload("ragged", 3, 1, 200, 9, 13, (0, 200, 77)),
    # text just over one 128 tile, odd grid
    Hh.workload("tile_edge", 1, 2, 130, 11, 12, (129,)),
    # a single image token
    Hh.workload("one_pixel", 1, 1, 5, 1, 1, (5,)),
    # exact tiles, L = 1
    Hh.workload("exact", 2, 2, 64, 16, 16, (64, 1)),
    # inputs scaled by 3
    Hh.workload("scaled", 1, 2, 24, 10, 10, (9,), scale=3.0),
    # the valid text length ending at and around every edge the kernels
    # split a 128-key tile at (the softmax threads' 64-key halves, their
    # 32-key P chunks, the 16-key k-steps), in two text tiles
    Hh.workload("mask_edges", 16, 2, 256, 8, 9,
                (0, 1, 15, 16, 31, 32, 33, 63, 64, 65, 95, 96, 97, 127, 128, 129)),
]


@pytest.mark.parametrize("w", EDGE, ids=[w.name for w in EDGE])
def test_edge_geometries_match_oracle(dev, w):
    batch = W.make_batch(w, seed=1)
    res = Hh.run_gpu(_ja(w, dev), batch, dev)
    _full_compare(w, batch, res, where=w.name)


@pytest.mark.parametrize("name", ["cfg1024", "img1664x928", "img1328"])
def test_full_size_workloads_match_oracle_on_head_subset(dev, name):
    w = W.WORKLOADS[name]
    batch = W.make_batch(w, seed=0)
    res = Hh.run_gpu(_ja(w, dev), batch, dev)
    _full_compare(w, batch, res, heads=[0, w.H - 1], where=name, pure=False)
    # sampled forward rows of other heads, computed one row at a time
    rng = np.random.default_rng(5)
    for b in range(w.B):
        h = int(rng.integers(1, w.H - 1))
        rows = sorted(set(rng.integers(0, w.S, 12).tolist()) | {0, w.T_txt - 1, w.T_txt, w.S - 1})
        sub = {n: batch[n][b:b + 1, :, h:h + 1] for n in ("q", "k", "v")}
        sub["gains"] = batch["gains"]
        Q, K, V, _, g = Hh.oracle_inputs(sub)
        L = batch["valid_len"][b]
        ro, rl = O.forward_rows(Q, K, V, g, w.T_txt, w.grid_h, w.grid_w, L, 0, 0, rows, store_bf16=True)
        out = Hh.f64(res["out"][b, rows, h])
        lse = Hh.f64(res["lse"][b, h, rows])
        Hh.assert_forward_close(out, lse, ro, rl, f"{name} rows b={b} h={h}", scale=w.scale)
        po, pl = O.forward_rows(Q, K, V, g, w.T_txt, w.grid_h, w.grid_w, L, 0, 0, rows)
        Hh.assert_forward_close_exact(out, lse, (ro, rl), (po, pl), f"{name} rows b={b} h={h} (exact f64)",
                                      scale=w.scale)


def test_masked_keys_have_no_effect_on_gpu(dev):
    w = Hh.workload("mask", 1, 2, 96, 8, 8, (37,))
    batch = W.make_batch(w, seed=2)
    ja = _ja(w, dev)
    a = Hh.run_gpu(ja, batch, dev)
    a = {k: v.clone() for k, v in a.items()}
    rng = np.random.default_rng(4)
    b2 = dict(batch)
    for n in ("k", "v"):
        x = batch[n].copy()
        x[:, 37:96] = W.f32_to_bf16_bits(rng.standard_normal(x[:, 37:96].shape).astype(np.float32) * 4)
        b2[n] = x
    b = Hh.run_gpu(ja, b2, dev)
    for key in ("out", "lse", "dq", "dgp", "dg"):
        assert Hh.bits_equal(a[key], b[key]), key
    for key in ("dk", "dv"):
        assert Hh.bits_equal(a[key][:, :37], b[key][:, :37]), key
        assert Hh.bits_equal(a[key][:, 96:], b[key][:, 96:]), key


def test_lse_request_and_repeat_runs_do_not_change_bytes(dev):
    import torch
    w = Hh.workload("rep", 2, 4, 64, 12, 12, (50, 7))
    batch = W.make_batch(w, seed=4)
    ja = _ja(w, dev)
    a = {k: v.clone() for k, v in Hh.run_gpu(ja, batch, dev).items()}
    b = Hh.run_gpu(ja, batch, dev)
    for key in a:
        assert Hh.bits_equal(a[key], b[key]), key
    q, k, v = (Hh.to_dev(batch[n], dev) for n in ("q", "k", "v"))
    gains = torch.from_numpy(batch["gains"]).to(dev)
    out, lse = ja.forward(q, k, v, gains, list(batch["valid_len"]), want_lse=False)
    torch.cuda.synchronize()
    assert lse is None and Hh.bits_equal(out, a["out"])

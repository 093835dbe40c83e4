"""Bit-exact batch invariance on the GPU (RFC #386 Numerical requirements:
a logical row's bytes must not change with batch size, batch position,
prompt padding, launch geometry or tiling; "WS1 Single-GPU Kernel List" rule
6 calls it the core acceptance test).

The sweep follows the 1024^2 shape: 8 rows with random valid text lengths in
U{1..256}; each row alone, then in batches of 2, 3, 5 and 8 built from the
row list in forward, reversed and shuffled order, and the single-row runs
repeated 3 times. O, lse, dQ, dK, dV and the per-(sample, head) gain
gradients must be byte-identical everywhere. Comparisons run on the device.
"""

import numpy as np
import pytest

from invariant_mmdit_joint_gb300 import workloads as W
from tests import _helpers as Hh

pytestmark = pytest.mark.gpu

SWEEP = dict(H=24, T_txt=256, grid_h=64, grid_w=64)


@pytest.fixture(scope="module")
def dev():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


def _run(dev, rows_data, gains, lens, geom):
    """Run one batch built by stacking per-row device tensors."""
    import torch

    import invariant_mmdit_joint_gb300 as pkg
    B = len(rows_data)
    ja = pkg.JointAttention(B, geom["T_txt"], geom["grid_h"], geom["grid_w"], geom["H"], device=dev)
    q, k, v, do = (torch.stack([r[n] for r in rows_data]) for n in ("q", "k", "v", "do"))
    out, lse = ja.forward(q, k, v, gains, lens)
    dq, dk, dv, dgp, dg = ja.backward(q, k, v, gains, lens, out, do, lse)
    torch.cuda.synchronize()
    pkg.rlk_joint_attn_check_status()
    return [{"out": out[i], "lse": lse[i], "dq": dq[i], "dk": dk[i], "dv": dv[i], "dgp": dgp[i]}
            for i in range(B)]


def _same(a, b):
    return all(Hh.bits_equal(a[k], b[k]) for k in a)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_batch_invariance_sweep(dev, seed):
    import torch
    S = SWEEP["T_txt"] + SWEEP["grid_h"] * SWEEP["grid_w"]
    lens = [int(x) for x in W.sweep_lengths(seed, 8, SWEEP["T_txt"])]
    rows = []
    for r in range(8):
        d = W.make_row(S, SWEEP["H"], seed, r)
        rows.append({n: Hh.to_dev(d[n], dev) for n in ("q", "k", "v", "do")})
    gains = torch.from_numpy(W.gains(seed)).to(dev)
    alone = [_run(dev, [rows[r]], gains, [lens[r]], SWEEP)[0] for r in range(8)]
    for _ in range(2):  # three runs in all
        again = [_run(dev, [rows[r]], gains, [lens[r]], SWEEP)[0] for r in range(8)]
        for r in range(8):
            assert _same(again[r], alone[r]), ("repeat", r)
    rng = np.random.default_rng([seed, 99])
    orders = {"forward": list(range(8)), "reversed": list(range(7, -1, -1)),
              "shuffled": [int(x) for x in rng.permutation(8)]}
    for oname, order in orders.items():
        for bs in (2, 3, 5, 8):
            for start in range(0, 8, bs):
                chunk = order[start:start + bs]
                res = _run(dev, [rows[r] for r in chunk], gains, [lens[r] for r in chunk], SWEEP)
                for pos, r in enumerate(chunk):
                    assert _same(res[pos], alone[r]), (oname, bs, pos, r)


def test_padding_invariance_with_zero_dout_on_padded_rows(dev):
    """A row's valid outputs and gradients are byte-identical whatever the
    padded text length, when dO is zero on the padded text rows (padded
    query rows then feed nothing back)."""
    import torch
    H, gh, gw, L = 4, 32, 32, 87
    T_img = gh * gw
    base = W.make_row(512 + T_img, H, 7, 0)
    gains = torch.from_numpy(W.gains(7)).to(dev)
    results = {}
    for T in (128, 256, 512):
        S = T + T_img
        row = {}
        rng = np.random.default_rng(T)
        for n in ("q", "k", "v", "do"):
            x = np.empty((S, H, 128), np.uint16)
            x[:L] = base[n][:L]
            x[T:] = base[n][512:]
            pad = W.f32_to_bf16_bits(rng.standard_normal((T - L, H, 128)).astype(np.float32))
            x[L:T] = 0 if n == "do" else pad
            row[n] = Hh.to_dev(x, dev)
        results[T] = (_run(dev, [row], gains, [L], dict(H=H, T_txt=T, grid_h=gh, grid_w=gw))[0], T)
    ref, T0 = results[128]
    for T, (res, _) in results.items():
        for key in ("out", "dq", "dk", "dv"):
            a, b = ref[key], res[key]
            assert Hh.bits_equal(a[:L], b[:L]), (T, key, "text")
            assert Hh.bits_equal(a[T0:], b[T:]), (T, key, "image")
        assert Hh.bits_equal(ref["lse"][:, :L], res["lse"][:, :L]), (T, "lse text")
        assert Hh.bits_equal(ref["lse"][:, T0:], res["lse"][:, T:]), (T, "lse image")
        assert Hh.bits_equal(ref["dgp"], res["dgp"]), (T, "dg_partial")


def test_head_composition_invariance(dev):
    """A head computed among 24 heads equals the same head computed alone."""
    import torch
    w = Hh.workload("heads", 1, 24, 96, 16, 16, (50,))
    batch = W.make_batch(w, seed=8)
    gains = torch.from_numpy(batch["gains"]).to(dev)
    full = {n: Hh.to_dev(batch[n][0], dev) for n in ("q", "k", "v", "do")}
    geom = dict(H=24, T_txt=96, grid_h=16, grid_w=16)
    res = _run(dev, [full], gains, [50], geom)[0]
    for h in (0, 5, 23):
        one = {n: full[n][:, h:h + 1].contiguous() for n in full}
        r1 = _run(dev, [one], gains, [50], dict(geom, H=1))[0]
        for key in ("out", "dq", "dk", "dv"):
            assert Hh.bits_equal(r1[key][:, 0], res[key][:, h]), (h, key)
        assert Hh.bits_equal(r1["lse"][0], res["lse"][h]) and Hh.bits_equal(r1["dgp"][0], res["dgp"][h])


@pytest.mark.parametrize("geom", [
    dict(name="cfg1024_h5", B=2, H=5, T_txt=256, gh=64, gw=64, vl=(87, 193)),
    dict(name="odd_tiles", B=3, H=2, T_txt=200, gh=13, gw=21, vl=(0, 130, 200)),
], ids=lambda g: g["name"])
def test_query_tile_schedule_never_changes_bytes(dev, geom):
    """Every pair of query tiles as one CTA, every tile alone, and the default
    mix give the same output bytes: a tile's arithmetic does not depend on
    the tile it shares a CTA with, whatever the SM count."""
    import torch

    import invariant_mmdit_joint_gb300 as pkg
    w = Hh.workload(geom["name"], geom["B"], geom["H"], geom["T_txt"], geom["gh"], geom["gw"], geom["vl"])
    batch = W.make_batch(w, seed=6, with_dout=False)
    q, k, v = (Hh.to_dev(batch[n], dev) for n in ("q", "k", "v"))
    gains = torch.from_numpy(batch["gains"]).to(dev)
    vl = [int(x) for x in batch["valid_len"]]
    ja = pkg.JointAttention(w.B, w.T_txt, w.grid_h, w.grid_w, w.H, device=dev)
    res = {}
    prev = pkg.rlk_fwd_tile_schedule("auto")
    try:
        for policy in ("auto", "pairs", "single"):
            pkg.rlk_fwd_tile_schedule(policy)
            out, lse = ja.forward(q, k, v, gains, vl)
            torch.cuda.synchronize()
            res[policy] = (out.clone(), lse.clone())
    finally:
        pkg.rlk_fwd_tile_schedule(prev)
    pkg.rlk_joint_attn_check_status()
    for policy in ("pairs", "single"):
        assert Hh.bits_equal(res[policy][0], res["auto"][0]), policy
        assert Hh.bits_equal(res[policy][1], res["auto"][1]), policy

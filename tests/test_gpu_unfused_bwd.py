"""The standalone backward of the attention operators (the backward calls of
joint_attn_softmax, joint_attn_av_gemm, joint_attn_qk_gemm and of
qk_rmsnorm + multi_axis_rope) against the fused backward and the oracle,
through the C ABI.

The RFC's WS1 table marks every attention row "fwd + bwd" and asks the fused
kernels to equal the operators' composition byte for byte: chained after a
forward, the backward calls must give the fused backward's dQ, dK, dV and
gain-gradient bytes exactly. Their intermediates are checked against the
oracle's definitions: P against the softmax of the storage-rounded oracle,
dP against dO V^T, dS against P (dP - Delta) and dq^, dk^ against the
oracle's attention backward.
"""

import numpy as np
import pytest

import invariant_mmdit_joint_gb300 as pkg
from invariant_mmdit_joint_gb300 import workloads as W
from tests import _helpers as Hh

pytestmark = pytest.mark.gpu

LOG2E = 1.4426950408889634


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
    batch = W.make_batch(w, seed)
    q, k, v, do = (Hh.to_dev(batch[n], dev) for n in ("q", "k", "v", "do"))
    return batch, q, k, v, do, torch.from_numpy(batch["gains"]).to(dev), [int(x) for x in batch["valid_len"]]


def _run_both(w, seed, dev):
    """The fused forward + backward, then the standalone forward and
    backward on the same inputs (same object: the context is rewritten with
    the same bytes)."""
    import torch
    batch, q, k, v, do, gains, vl = _inputs(w, seed, dev)
    ja = pkg.JointAttention(w.B, w.T_txt, w.grid_h, w.grid_w, w.H, device=dev)
    out, lse = ja.forward(q, k, v, gains, vl)
    fused = ja.backward(q, k, v, gains, vl, out, do, lse)
    fused = [t.clone() for t in fused]
    u = ja.forward_unfused(q, k, v, gains, vl)
    ub = ja.backward_unfused(q, k, v, gains, vl, u["out"], do, u["lse"], u["scores"])
    torch.cuda.synchronize()
    pkg.rlk_joint_attn_check_status()
    qh, kh, _, _ = ja.ctx_views()
    u["qh"], u["kh"] = Hh.f64(qh), Hh.f64(kh)
    return batch, u, ub, fused


SMALL = [
    W.TINY,
    # two text tiles (the second partly padded), a ragged 13 x 21 image,
    # a sample with no valid text key and one whose last text tile holds 2
    Hh.workload("ragged", 3, 2, 200, 13, 21, (0, 130, 200)),
    # the valid text length at and around the tile's half, chunk and k-step edges
    Hh.workload("mask_edges", 14, 1, 256, 8, 9, (1, 15, 16, 31, 32, 33, 63, 64, 65, 95, 96, 97, 127, 129)),
]


@pytest.mark.parametrize("w", SMALL + [Hh.workload("cfg1024_h4", 1, 4, 256, 64, 64, (87,))], ids=lambda w: w.name)
def test_backward_composition_is_byte_equal_to_the_fused_backward(w, dev):
    _, _, ub, fused = _run_both(w, 41, dev)
    for name, f in zip(("dq", "dk", "dv", "dgp", "dg"), fused):
        assert Hh.bits_equal(ub[name], f), (w.name, name)


def test_backward_composition_is_byte_equal_at_full_size(dev):
    _, _, ub, fused = _run_both(W.CFG1024, 0, dev)
    for name, f in zip(("dq", "dk", "dv", "dgp", "dg"), fused):
        assert Hh.bits_equal(ub[name], f), name


def _key_cols(w, L):
    """Columns of the visited key blocks and, for each, whether that key is
    valid (masked keys and columns past a text segment are not)."""
    ntq_txt = -(-w.T_txt // 128)
    cols, keys = [], []
    for t in range(-(-L // 128)):
        for c in range(128):
            cols.append(128 * t + c)
            keys.append(128 * t + c if 128 * t + c < L else -1)
    n_img = -(-(w.grid_h * w.grid_w) // 128)
    for i in range(n_img):
        for c in range(128):
            key = w.T_txt + 128 * i + c
            cols.append(128 * (ntq_txt + i) + c)
            keys.append(key if key < w.S else -1)
    return np.array(cols), np.array(keys)


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_backward_intermediates_match_the_oracle(w, dev):
    """Each intermediate against the oracle's definition applied to the
    operators' own inputs: the stored q^, k^ of the context (the prologue's
    bf16 values, which may sit one bf16 ulp from the oracle's rounding of its
    exact values), the bf16 inputs and the GPU's own O and lse."""
    from oracle import joint_attn as O
    batch, u, ub, _ = _run_both(w, 42, dev)
    _, _, V, dO, _ = Hh.oracle_inputs(batch)
    ja_q, ja_k = u["qh"], u["kh"]
    out = Hh.f64(u["out"])
    stats = Hh.f64(ub["stats"])
    p = Hh.f64(ub["p"])
    dp = Hh.f64(ub["dp"])
    ds = Hh.f64(ub["ds"])
    dqh = Hh.f64(ub["dqh"])
    dkh = Hh.f64(ub["dkh"])
    lse = Hh.f64(u["lse"])
    ntq_txt = -(-w.T_txt // 128)
    for b in range(w.B):
        L = int(batch["valid_len"][b])
        cols, keys = _key_cols(w, L)
        valid = keys >= 0
        kv = O.key_valid(w.T_txt, w.S, L)
        for h in range(w.H):
            qh, kh = ja_q[b, h], ja_k[b, h]
            _, ref_lse, ref_p = O.attention_forward(qh, kh, V[b, :, h], kv)
            ref_dqh, ref_dkh, _ = O.attention_backward(qh, kh, V[b, :, h], ref_p, dO[b, :, h])
            # stats: lse * log2(e) of every row in its tile-padded slot (+inf past a
            # segment), Delta = rowsum(dO * O) of the GPU's own O
            slots = np.array([n if n < w.T_txt else 128 * ntq_txt + n - w.T_txt for n in range(w.S)])
            l2 = stats[0, b, h, slots]
            assert np.all(np.abs(l2 - lse[b, h] * LOG2E) <= 4e-7 * np.abs(l2) + 1e-30)
            pad = np.setdiff1d(np.arange(stats.shape[-1]), slots)
            assert np.all(np.isinf(stats[0, b, h, pad])) and np.all(stats[1, b, h, pad] == 0)
            delta = np.sum(dO[b, :, h] * out[b, :, h], axis=1)
            assert np.all(np.abs(stats[1, b, h, slots] - delta) <= 1e-5 * np.sum(np.abs(dO[b, :, h] * out[b, :, h]),
                                                                                axis=1) + 1e-12)
            # P: the softmax, one bf16 rounding (2^-8 relative) plus its fp32
            # exponent's error, that of an fp32 score of 128 products against
            # the row's lse (below 2^-11 relative); masked keys exactly 0
            pg = p[b, h][:, cols]
            pr = ref_p[:, np.where(valid, keys, 0)]
            assert np.all(pg[:, ~valid] == 0)
            assert np.all(np.abs(pg[:, valid] - pr[:, valid]) <= (2 ** -8 + 2 ** -11) * pr[:, valid] + 1e-7), \
                (w.name, b, h, float(np.max(np.abs(pg[:, valid] - pr[:, valid]) / np.maximum(pr[:, valid], 1e-30))))
            # the lse the forward gave is that softmax's (fp32)
            assert np.max(np.abs(lse[b, h] - ref_lse) / np.abs(ref_lse)) <= 1e-5
            # dP = dO V^T: exact bf16 products, fp32 accumulation of 128 of them
            dpr = dO[b, :, h] @ V[b, :, h].T
            terms = np.abs(dO[b, :, h]) @ np.abs(V[b, :, h]).T
            dpg = dp[b, h][:, cols[valid]]
            assert np.all(np.abs(dpg - dpr[:, keys[valid]]) <= 2 ** -16 * terms[:, keys[valid]] + 1e-30)
            # dS = P (dP - Delta): within the bf16 roundings of P and dS (relative L2)
            dsr = ref_p * (dpr - np.sum(ref_p * dpr, axis=1, keepdims=True))
            Hh.assert_grad_close("dS", ds[b, h][:, cols[valid]], dsr[:, keys[valid]], f"{w.name} b={b} h={h}")
            # dq^, dk^ against the oracle's attention backward; masked keys 0
            Hh.assert_grad_close("dq^", dqh[b, h], ref_dqh, f"{w.name} b={b} h={h}")
            if np.linalg.norm(ref_dkh[kv]) > 0:
                Hh.assert_grad_close("dk^", dkh[b, h][kv], ref_dkh[kv], f"{w.name} b={b} h={h}")
            assert np.all(dkh[b, h][~kv] == 0)


def test_backward_calls_are_traced(dev):
    import torch
    w = W.TINY
    batch, q, k, v, do, gains, vl = _inputs(w, 43, dev)
    ja = pkg.JointAttention(w.B, w.T_txt, w.grid_h, w.grid_w, w.H, device=dev)
    u = ja.forward_unfused(q, k, v, gains, vl)
    with pkg.op_trace() as t:
        ja.backward_unfused(q, k, v, gains, vl, u["out"], do, u["lse"], u["scores"])
        torch.cuda.synchronize()
    assert [(r["entry_point"], r["kernels"]) for r in t.records] == [
        ("rlk_joint_attn_bwd_stats", ["bwd_pre_kernel"]),
        ("rlk_joint_attn_softmax_bwd", ["softmax_bwd_kernel"]),
        ("rlk_joint_attn_av_gemm_bwd", ["qk_gemm_kernel<dp>", "acc_gemm_kernel<key>"]),
        ("rlk_joint_attn_softmax_bwd", ["softmax_bwd_kernel"]),
        ("rlk_joint_attn_qk_gemm_bwd", ["acc_gemm_kernel<key>", "acc_gemm_kernel<query>"]),
        ("rlk_qk_norm_rope_bwd", ["norm_rope_bwd_q_kernel", "norm_rope_bwd_k_kernel", "dg_fold_kernels"]),
    ]

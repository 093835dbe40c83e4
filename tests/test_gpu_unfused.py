"""The standalone attention operators (joint_attn_qk_gemm, joint_attn_softmax,
joint_attn_av_gemm, after qk_rmsnorm + multi_axis_rope) against the fused
forward and the oracle, through the C ABI.

The RFC's WS1 table asks joint_attention_fused to be a byte-equal fusion of
the three operators, and the WS1 Single-GPU Kernel List says the fusion must
match their composition byte for byte: the chained operators must give the
fused forward's out and lse bytes exactly. Their intermediates are checked
against the oracle's definitions: the raw scores against q^ . k^, and the
probabilities rebuilt from P, the rescale factors and the row sums against
the oracle's softmax.
"""

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
    return batch, q, k, v, torch.from_numpy(batch["gains"]).to(dev), [int(x) for x in batch["valid_len"]]


def _n_tiles(w):
    return -(-w.T_txt // 128) + -(-(w.grid_h * w.grid_w) // 128)


def _key_blocks(w, L):
    """(column block, first key, end of valid keys, end of the tile's
    segment) of each key tile in the fixed visiting order: text tiles
    holding a valid key, then image tiles."""
    ntq_txt = -(-w.T_txt // 128)
    S = w.T_txt + w.grid_h * w.grid_w
    out = [(t, 128 * t, L, w.T_txt) for t in range(-(-L // 128))]
    out += [(ntq_txt + i, w.T_txt + 128 * i, S, S) for i in range(-(-(w.grid_h * w.grid_w) // 128))]
    return out


SMALL = [
    W.TINY,
    # two text tiles (the second partly padded), a ragged 13 x 21 image,
    # a sample with no valid text key and one whose last text tile holds 2
    Hh.workload("ragged", 3, 2, 200, 13, 21, (0, 130, 200)),
    # the valid text length at and around the tile's half, chunk and k-step edges
    Hh.workload("mask_edges", 14, 1, 256, 8, 9, (1, 15, 16, 31, 32, 33, 63, 64, 65, 95, 96, 97, 127, 129)),
]


@pytest.mark.parametrize("w", SMALL + [Hh.workload("cfg1024_h4", 1, 4, 256, 64, 64, (87,))], ids=lambda w: w.name)
def test_composition_is_byte_equal_to_the_fused_forward(w, dev):
    import torch
    _, q, k, v, gains, vl = _inputs(w, 21, dev)
    ja = pkg.JointAttention(w.B, w.T_txt, w.grid_h, w.grid_w, w.H, device=dev)
    out_f, lse_f = ja.forward(q, k, v, gains, vl)
    u = ja.forward_unfused(q, k, v, gains, vl)
    torch.cuda.synchronize()
    pkg.rlk_joint_attn_check_status()
    assert Hh.bits_equal(u["out"], out_f), w.name
    assert Hh.bits_equal(u["lse"], lse_f), w.name


def test_composition_is_byte_equal_at_full_size(dev):
    import torch
    w = W.CFG1024
    _, q, k, v, gains, vl = _inputs(w, 0, dev)
    ja = pkg.JointAttention(w.B, w.T_txt, w.grid_h, w.grid_w, w.H, device=dev)
    out_f, lse_f = ja.forward(q, k, v, gains, vl)
    u = ja.forward_unfused(q, k, v, gains, vl)
    torch.cuda.synchronize()
    pkg.rlk_joint_attn_check_status()
    assert Hh.bits_equal(u["out"], out_f)
    assert Hh.bits_equal(u["lse"], lse_f)


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_intermediates_match_the_oracle(w, dev):
    import torch
    from oracle import joint_attn as O
    batch, q, k, v, gains, vl = _inputs(w, 22, dev)
    ja = pkg.JointAttention(w.B, w.T_txt, w.grid_h, w.grid_w, w.H, device=dev)
    u = ja.forward_unfused(q, k, v, gains, vl)
    torch.cuda.synchronize()
    scores = u["scores"].cpu().numpy().astype(np.float64)
    p = u["p"].float().cpu().numpy().astype(np.float64)
    alpha = u["alpha"].cpu().numpy().astype(np.float64)
    l = u["l"].cpu().numpy().astype(np.float64)
    lse = u["lse"].cpu().numpy().astype(np.float64)
    Q, K, V, _, g64 = Hh.oracle_inputs(batch)
    S = w.T_txt + w.grid_h * w.grid_w
    # the operator's own inputs: the bf16 q^, k^ the prologue left in ctx
    qh_in, kh_in, _, _ = (Hh.f64(t) for t in ja.ctx_views())
    for b in range(w.B):
        for h in range(w.H):
            f = O._pair_forward(Q[b, :, h], K[b, :, h], V[b, :, h], g64, w.T_txt, w.grid_h, w.grid_w,
                                vl[b], O.EPS, O.THETA, O.AXES, store_bf16=True)
            qh, kh, p_ref = f["qh"], f["kh"], f["p"]
            blocks = _key_blocks(w, vl[b])
            # normalised probabilities rebuilt from the operator outputs:
            # p_ij = P_ij(t) * prod over later tiles t' of alpha_i(t') / l_i
            later = np.ones((S,))
            p_gpu = np.zeros((S, S))
            for blk, k0, kend, seg_end in reversed(blocks):
                n = min(128, seg_end - k0)  # the tile's keys inside its segment
                cols = slice(blk * 128, blk * 128 + n)
                valid = np.arange(k0, k0 + n) < kend
                got = scores[b, h, :, cols][:, valid]
                # (a) the operator's arithmetic on its own inputs: products
                # of bf16 values are exact in fp32 and the 128-term fp32 sum
                # errs by well under 2^-16 of the sum of |terms|
                qi, ki = qh_in[b, h], kh_in[b, h, k0:k0 + n][valid]
                tight = 2.0 ** -16 * (np.abs(qi) @ np.abs(ki).T) + 1e-30
                assert np.all(np.abs(got - qi @ ki.T) <= tight), (w.name, b, h, blk, "scores vs own inputs")
                # (b) against the oracle's q^ . k^: the prologue rounds q^ and
                # k^ to bf16 from fp32, the oracle from exact values, so an
                # element at a rounding tie may differ by one bf16 ulp (2^-8)
                sum_abs = np.abs(qh) @ np.abs(kh[k0:k0 + n][valid]).T
                ref = qh @ kh[k0:k0 + n][valid].T
                assert np.all(np.abs(got - ref) <= (2.0 ** -8 + 2.0 ** -16) * sum_abs + 1e-30), \
                    (w.name, b, h, blk, "scores vs oracle")
                # masked keys inside a visited tile: -inf scores, P exactly zero
                full_cols = slice(blk * 128, (blk + 1) * 128)
                masked = np.arange(k0, k0 + 128) >= kend
                assert np.all(scores[b, h, :, full_cols][:, masked] == -np.inf), (w.name, b, h, blk)
                assert np.all(p[b, h, :, full_cols][:, masked] == 0.0), (w.name, b, h, blk)
                p_gpu[:, k0:k0 + n] = p[b, h, :, cols] * later[:, None] / l[b, h][:, None]
                later = later * alpha[b, h, :, blk]
            # P is rounded to bf16 (2^-9 relative), exp2 errs by 2 ulp, and
            # the bf16 rounding of q^, k^ may move a score (see above)
            err = np.abs(p_gpu - p_ref)
            assert np.all(err <= 8e-3 * p_ref + 1e-7), (w.name, b, h, np.max(err / (p_ref + 1e-7)))
            assert np.max(np.abs(lse[b, h] - f["lse"]) / np.abs(f["lse"])) <= Hh.LSE_REL


def test_intermediates_are_batch_invariant(dev):
    """Each sample's scores, P, alpha and l bytes are the same computed alone
    and inside a batch, in any batch position."""
    import torch
    w = Hh.workload("ragged", 3, 2, 200, 13, 21, (0, 130, 200))
    batch, q, k, v, gains, vl = _inputs(w, 23, dev)
    ja = pkg.JointAttention(w.B, w.T_txt, w.grid_h, w.grid_w, w.H, device=dev)
    full = ja.forward_unfused(q, k, v, gains, vl)
    one = pkg.JointAttention(1, w.T_txt, w.grid_h, w.grid_w, w.H, device=dev)
    nt = _n_tiles(w)
    for b in range(w.B):
        u = one.forward_unfused(q[b:b + 1].contiguous(), k[b:b + 1].contiguous(), v[b:b + 1].contiguous(),
                                gains, [vl[b]])
        torch.cuda.synchronize()
        # compare the written blocks only: the visited key tiles' columns
        blocks = [blk for blk, _, _, _ in _key_blocks(w, vl[b])]
        for name, width in (("scores", 128), ("p", 128), ("alpha", 1)):
            for blk in blocks:
                a = full[name][b, :, :, blk * width:(blk + 1) * width]
                c = u[name][0, :, :, blk * width:(blk + 1) * width]
                assert Hh.bits_equal(a.contiguous(), c.contiguous()), (name, b, blk)
        assert Hh.bits_equal(full["l"][b].contiguous(), u["l"][0].contiguous())
        assert Hh.bits_equal(full["out"][b].contiguous(), u["out"][0].contiguous())
    assert nt == 2 + 3

"""The per-stream QKV projection (the WS1 row qkv_bias_gemm) on the tensor
cores, with qk_rmsnorm + multi_axis_rope fused into its epilogue: the plain
projections against the oracle, the fused context against the prologue run
on the stored projections (byte for byte), and the attention from that
context against the separate-stream forward (byte for byte)."""

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


CASES = [
    W.TINY,
    # odd H: 3C = 1152 columns, the last 256-column tile holds one head
    Hh.workload("odd_heads", 2, 3, 40, 9, 7, (40, 13)),
    # rows that do not fill the last 128-row tile of either stream
    Hh.workload("ragged", 3, 2, 200, 13, 21, (0, 130, 200)),
    Hh.workload("no_text", 2, 2, 0, 5, 7, (0, 0)),
]


def _inputs(w, seed, dev):
    import torch
    d = W.make_qkv_inputs(w, seed)

    def t(name):
        if d[name].size == 0:
            return None
        return Hh.to_dev(d[name], dev)
    x, wt, b = ((t(p + "_txt"), t(p + "_img")) for p in ("x", "w", "b"))
    gains = torch.from_numpy(W.gains(seed)).to(dev)
    return d, x, wt, b, gains


def _empty_pair(w, dev):
    import torch
    mk = (lambda T: None if T == 0 else
          torch.empty((w.B, T, w.H, 128), dtype=torch.bfloat16, device=dev))
    return mk(w.T_txt), mk(w.T_img)


def _cat(pair):
    import torch
    return pair[1] if pair[0] is None else torch.cat(pair, dim=1).contiguous()


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_plain_projection_matches_oracle(w, dev):
    import torch
    from oracle import joint_attn as O
    d, x, wt, b, _ = _inputs(w, 51, dev)
    shape = pkg.Shape.make(w.B, w.T_txt, w.grid_h, w.grid_w, w.H)
    q, k, v = (_empty_pair(w, dev) for _ in range(3))
    pkg.rlk_qkv_bias_gemm(shape, x, wt, b, None, None, q, k, v)
    torch.cuda.synchronize()
    pkg.rlk_joint_attn_check_status()
    for si, s in enumerate(("txt", "img")):
        if d["x_" + s].size == 0:
            continue
        X, Wm, bias = (O.widen_bf16(d[p + "_" + s]) for p in ("x", "w", "b"))
        exact = O.qkv_projection(X, Wm, bias)
        sum_abs = O.qkv_projection(np.abs(X), np.abs(Wm), np.abs(bias))
        for name, got, ref, sa in zip("qkv", (q[si], k[si], v[si]), exact, sum_abs):
            g = Hh.f64(got)
            # one bf16 rounding of an fp32 sum: within a bf16 ulp, plus the
            # fp32 accumulation error (far below 2^-16 of the sum of |terms|)
            assert np.all(np.abs(g - ref) <= 2.0 ** -8 * np.abs(ref) + 2.0 ** -16 * sa), (w.name, s, name)
            # and almost always the correctly rounded value itself
            assert np.mean(g == O.round_bf16(ref)) > 0.99, (w.name, s, name)


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_fused_epilogue_equals_the_prologue_on_the_stored_projections(w, dev):
    import torch
    d, x, wt, b, gains = _inputs(w, 52, dev)
    shape = pkg.Shape.make(w.B, w.T_txt, w.grid_h, w.grid_w, w.H)
    # unfused: store Q, K, V, then qk_rmsnorm + multi_axis_rope
    q, k, v = (_empty_pair(w, dev) for _ in range(3))
    pkg.rlk_qkv_bias_gemm(shape, x, wt, b, None, None, q, k, v)
    ja_a = pkg.JointAttention(w.B, w.T_txt, w.grid_h, w.grid_w, w.H, device=dev)
    pkg.rlk_qk_norm_rope(shape, _cat(q), _cat(k), gains[0], gains[1], gains[2], gains[3], ja_a.ctx)
    # fused, also storing Q and K (as a backward would want), and fused alone
    ja_b = pkg.JointAttention(w.B, w.T_txt, w.grid_h, w.grid_w, w.H, device=dev)
    q2, k2, v2 = (_empty_pair(w, dev) for _ in range(3))
    pkg.rlk_qkv_bias_gemm(shape, x, wt, b, gains, ja_b.ctx, q2, k2, v2)
    ja_c = pkg.JointAttention(w.B, w.T_txt, w.grid_h, w.grid_w, w.H, device=dev)
    v3 = _empty_pair(w, dev)
    pkg.rlk_qkv_bias_gemm(shape, x, wt, b, gains, ja_c.ctx, (None, None), (None, None), v3)
    torch.cuda.synchronize()
    pkg.rlk_joint_attn_check_status()
    ref = ja_a.ctx_views()
    for other in (ja_b, ja_c):
        for name, got, want in zip(("qh", "kh", "rq", "rk"), other.ctx_views(), ref):
            assert Hh.bits_equal(got, want), (w.name, name)
    for a_pair, b_pair in ((q, q2), (k, k2), (v, v2), (v, v3)):
        for a_t, b_t in zip(a_pair, b_pair):
            if a_t is not None:
                assert Hh.bits_equal(a_t, b_t), w.name


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_attention_from_the_projection_context(w, dev):
    import torch
    d, x, wt, b, gains = _inputs(w, 53, dev)
    vl = list(w.valid_len)
    shape = pkg.Shape.make(w.B, w.T_txt, w.grid_h, w.grid_w, w.H)
    q, k, v = (_empty_pair(w, dev) for _ in range(3))
    pkg.rlk_qkv_bias_gemm(shape, x, wt, b, None, None, q, k, v)
    ja = pkg.JointAttention(w.B, w.T_txt, w.grid_h, w.grid_w, w.H, device=dev)
    out_ref, lse_ref = ja.forward_streams(q, k, v, gains, vl)
    torch.cuda.synchronize()
    ja2 = pkg.JointAttention(w.B, w.T_txt, w.grid_h, w.grid_w, w.H, device=dev)
    v2 = _empty_pair(w, dev)
    pkg.rlk_qkv_bias_gemm(shape, x, wt, b, gains, ja2.ctx, (None, None), (None, None), v2)
    out = _empty_pair(w, dev)
    lse = torch.empty_like(lse_ref)
    pkg.rlk_joint_attn_fwd_ctx(shape, ja2.ctx, v2, vl, out, lse)
    torch.cuda.synchronize()
    pkg.rlk_joint_attn_check_status()
    assert Hh.bits_equal(_cat(out), _cat(out_ref)) and Hh.bits_equal(lse, lse_ref), w.name


def test_full_size_projection_on_sampled_rows(dev):
    import torch
    from oracle import joint_attn as O
    w = W.CFG1024
    d, x, wt, b, gains = _inputs(w, 54, dev)
    shape = pkg.Shape.make(w.B, w.T_txt, w.grid_h, w.grid_w, w.H)
    q, k, v = (_empty_pair(w, dev) for _ in range(3))
    pkg.rlk_qkv_bias_gemm(shape, x, wt, b, None, None, q, k, v)
    ja = pkg.JointAttention(w.B, w.T_txt, w.grid_h, w.grid_w, w.H, device=dev)
    pkg.rlk_qk_norm_rope(shape, _cat(q), _cat(k), gains[0], gains[1], gains[2], gains[3], ja.ctx)
    ja2 = pkg.JointAttention(w.B, w.T_txt, w.grid_h, w.grid_w, w.H, device=dev)
    pkg.rlk_qkv_bias_gemm(shape, x, wt, b, gains, ja2.ctx, (None, None), (None, None), _empty_pair(w, dev))
    torch.cuda.synchronize()
    pkg.rlk_joint_attn_check_status()
    for name, got, want in zip(("qh", "kh", "rq", "rk"), ja2.ctx_views(), ja.ctx_views()):
        assert Hh.bits_equal(got, want), name
    rng = np.random.default_rng(3)
    for si, s in enumerate(("txt", "img")):
        T = w.T_txt if si == 0 else w.T_img
        rows = sorted(set(rng.integers(0, w.B * T, 12).tolist()) | {0, w.B * T - 1})
        X = O.widen_bf16(d["x_" + s]).reshape(w.B * T, -1)[rows][None]
        Wm, bias = O.widen_bf16(d["w_" + s]), O.widen_bf16(d["b_" + s])
        exact = O.qkv_projection(X, Wm, bias)
        sum_abs = O.qkv_projection(np.abs(X), np.abs(Wm), np.abs(bias))
        for got_pair, ref, sa in zip((q, k, v), exact, sum_abs):
            g = Hh.f64(got_pair[si].reshape(w.B * T, w.H, 128)[rows])
            assert np.all(np.abs(g - ref[0]) <= 2.0 ** -8 * np.abs(ref[0]) + 2.0 ** -16 * sa[0]), s


@pytest.mark.parametrize("w", CASES + [W.CFG1024], ids=lambda w: w.name)
def test_output_projection_matches_oracle(w, dev):
    """attn_out_bias_gemm on separate stream buffers (seeded inputs: the
    activations x stand in for the attention output, the first C rows of the
    QKV weights and biases for the projection's)."""
    import torch
    from oracle import joint_attn as O
    d, x, wt, b, _ = _inputs(w, 55, dev)
    C = w.H * 128
    shape = pkg.Shape.make(w.B, w.T_txt, w.grid_h, w.grid_w, w.H)
    o = tuple(None if t is None else t.view(w.B, -1, w.H, 128) for t in x)
    wo = tuple(t[:C].contiguous() for t in wt)
    bo = tuple(t[:C].contiguous() for t in b)
    y = tuple(None if t is None else torch.empty_like(t) for t in x)
    pkg.rlk_attn_out_bias_gemm(shape, o, wo, bo, y)
    torch.cuda.synchronize()
    pkg.rlk_joint_attn_check_status()
    rng = np.random.default_rng(6)
    for si, s in enumerate(("txt", "img")):
        if y[si] is None:
            continue
        T = w.T_txt if si == 0 else w.T_img
        rows = np.arange(w.B * T)
        if rows.size > 64:  # full size: sampled rows
            rows = np.array(sorted(set(rng.integers(0, rows.size, 24).tolist()) | {0, rows.size - 1}))
        X = O.widen_bf16(d["x_" + s]).reshape(w.B * T, w.H, 128)[rows][None]
        Wm = O.widen_bf16(d["w_" + s])[:C]
        bias = O.widen_bf16(d["b_" + s])[:C]
        ref = O.attn_out_projection(X, Wm, bias)[0]
        sa = O.attn_out_projection(np.abs(X), np.abs(Wm), np.abs(bias))[0]
        g = Hh.f64(y[si].reshape(w.B * T, C)[torch.from_numpy(rows).to(dev)])
        assert np.all(np.abs(g - ref) <= 2.0 ** -8 * np.abs(ref) + 2.0 ** -16 * sa), (w.name, s)
        assert np.mean(g == O.round_bf16(ref)) > 0.99, (w.name, s)

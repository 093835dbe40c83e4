"""Pins of the CPU oracle to what the pages and the mathematics fix.

Each check ties the oracle to something other than itself: finite
differences, closed forms, invariants, an independent formulation through a
library routine (scipy's softmax / logsumexp, complex multiplication), and
hand-worked position values. ``test_planted_mistakes_are_caught`` plants a
plausible mistake in a copy of an oracle function and shows that a pin fails.
"""

import json
import os

import numpy as np
import pytest
import scipy.special

from oracle import joint_attn as O
from invariant_mmdit_joint_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _tiny(seed=0):
    w = W.TINY
    d = W.make_batch(w, seed)
    Q, K, V, dO = (O.widen_bf16(d[k]) for k in ("q", "k", "v", "do"))
    return w, Q, K, V, dO, d["gains"].astype(np.float64), d["valid_len"]


def _micro(seed=5, T=4, L=3, gh=2, gw=3, B=1, H=1, D=128):
    rng = np.random.default_rng(seed)
    S = T + gh * gw
    Q, K, V, dO = (rng.standard_normal((B, S, H, D)) for _ in range(4))
    g = rng.uniform(0.5, 1.5, (4, D))
    return (T, gh, gw, np.array([L] * B)), Q, K, V, dO, g


def _loss(Q, K, V, g, dO, geom):
    T, gh, gw, vl = geom
    o, _ = O.joint_attn_forward(Q, K, V, g, T, gh, gw, vl)
    return float(np.sum(o * dO))


# ------------------------------------------------------------ gradients
def directional_fd_error(geom, Q, K, V, dO, g, backward=O.joint_attn_backward,
                         n_dir=3, h=1e-6, seed=11):
    """max relative gap between <grad, d> and the central difference along d."""
    T, gh, gw, vl = geom
    dQ, dK, dV, _, dg = backward(Q, K, V, g, dO, T, gh, gw, vl)
    rng = np.random.default_rng(seed)
    worst = 0.0
    for _ in range(n_dir):
        for name, grad in (("Q", dQ), ("K", dK), ("V", dV), ("g", dg)):
            args = dict(Q=Q, K=K, V=V, g=g)
            d = rng.standard_normal(args[name].shape)
            plus = dict(args)
            minus = dict(args)
            plus[name] = args[name] + h * d
            minus[name] = args[name] - h * d
            fd = (_loss(dO=dO, geom=geom, **plus) - _loss(dO=dO, geom=geom, **minus)) / (2 * h)
            an = float(np.sum(grad * d))
            worst = max(worst, abs(fd - an) / max(abs(an), 1e-3))
    return worst


def test_gradients_match_directional_finite_differences():
    w, Q, K, V, dO, g, vl = _tiny()
    err = directional_fd_error((w.T_txt, w.grid_h, w.grid_w, vl), Q, K, V, dO, g)
    assert err < 1e-6, err


def test_gradients_match_elementwise_finite_differences():
    geom, Q, K, V, dO, g = _micro()
    T, gh, gw, vl = geom
    dQ, dK, dV, dgp, dg = O.joint_attn_backward(Q, K, V, g, dO, T, gh, gw, vl)
    h = 1e-6
    rng = np.random.default_rng(3)
    for name, grad in (("Q", dQ), ("K", dK), ("V", dV), ("g", dg)):
        base = dict(Q=Q, K=K, V=V, g=g)[name]
        flat = list(zip(*np.unravel_index(rng.choice(base.size, 120, replace=False), base.shape)))
        for idx in flat:
            args = dict(Q=Q, K=K, V=V, g=g)
            p = base.copy()
            p[idx] += h
            m = base.copy()
            m[idx] -= h
            args[name] = p
            lp = _loss(dO=dO, geom=geom, **args)
            args[name] = m
            lm = _loss(dO=dO, geom=geom, **args)
            fd = (lp - lm) / (2 * h)
            assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(grad[idx])), (name, idx, fd, grad[idx])
    # the four gain slots are the per-stream sums of the per-(b, h) partials
    assert np.allclose(dgp.sum(axis=(0, 1)), dg, rtol=0, atol=1e-12)


# ------------------------------------------------------------ softmax / mask
def test_softmax_rows_sum_to_one_and_masked_keys_get_zero():
    w, Q, K, V, dO, g, vl = _tiny()
    f = O._pair_forward(Q[0, :, 0], K[0, :, 0], V[0, :, 0], g, w.T_txt,
                        w.grid_h, w.grid_w, int(vl[0]), O.EPS, O.THETA, O.AXES)
    p = f["p"]
    assert np.max(np.abs(p.sum(axis=1) - 1.0)) <= 1e-14
    L = int(vl[0])
    assert np.all(p[:, L:w.T_txt] == 0.0)
    # valid keys: the first L text keys and every image key have p > 0
    assert np.all(p[:, :L] > 0) and np.all(p[:, w.T_txt:] > 0)
    assert int(np.count_nonzero(p[0])) == w.T_img + L


def test_constant_v_returns_v():
    w, Q, K, V, dO, g, vl = _tiny()
    Vc = np.full_like(V, 0.0)
    Vc[..., :] = np.linspace(-2.0, 3.0, V.shape[-1])
    o, _ = O.joint_attn_forward(Q, K, Vc, g, w.T_txt, w.grid_h, w.grid_w, vl)
    assert np.max(np.abs(o - Vc)) <= 1e-13


def test_masked_keys_have_no_effect():
    w, Q, K, V, dO, g, vl = _tiny()
    L = int(vl[0])
    rng = np.random.default_rng(9)
    K2, V2 = K.copy(), V.copy()
    K2[:, L:w.T_txt] = rng.standard_normal(K2[:, L:w.T_txt].shape) * 5
    V2[:, L:w.T_txt] = rng.standard_normal(V2[:, L:w.T_txt].shape) * 5
    a = O.joint_attn_forward(Q, K, V, g, w.T_txt, w.grid_h, w.grid_w, vl)
    b = O.joint_attn_forward(Q, K2, V2, g, w.T_txt, w.grid_h, w.grid_w, vl)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    ga = O.joint_attn_backward(Q, K, V, g, dO, w.T_txt, w.grid_h, w.grid_w, vl)
    gb = O.joint_attn_backward(Q, K2, V2, g, dO, w.T_txt, w.grid_h, w.grid_w, vl)
    assert np.array_equal(ga[0], gb[0])
    valid = O.key_valid(w.T_txt, w.S, L)
    assert np.array_equal(ga[1][:, valid], gb[1][:, valid])
    assert np.array_equal(ga[2][:, valid], gb[2][:, valid])
    # masked keys get exactly zero gradient
    assert np.all(ga[1][:, ~valid] == 0) and np.all(ga[2][:, ~valid] == 0)


def test_zero_query_gives_uniform_attention_closed_form():
    w, Q, K, V, dO, g, vl = _tiny()
    Q0 = np.zeros_like(Q)
    o, lse = O.joint_attn_forward(Q0, K, V, g, w.T_txt, w.grid_h, w.grid_w, vl)
    L = int(vl[0])
    n_valid = w.T_img + L
    for h in range(w.H):
        mean_v = (V[0, :L, h].sum(axis=0) + V[0, w.T_txt:, h].sum(axis=0)) / n_valid
        assert np.max(np.abs(o[0, :, h] - mean_v[None, :])) <= 1e-13
        assert np.max(np.abs(lse[0, h] - np.log(n_valid))) <= 1e-13


def core_vs_scipy_error(attention_forward=O.attention_forward, seed=4):
    """Attention core against scipy.special.softmax / logsumexp of the
    textbook softmax(q k^T / sqrt(d)) V with a -inf key mask."""
    rng = np.random.default_rng(seed)
    S, D = 37, 128
    qh, kh, v = (rng.standard_normal((S, D)) for _ in range(3))
    valid = np.ones(S, bool)
    valid[[3, 4, 5, 20]] = False
    o, lse, _ = attention_forward(qh, kh, v, valid)
    logits = qh @ kh.T / np.sqrt(D)
    logits[:, ~valid] = -np.inf
    ref_o = scipy.special.softmax(logits, axis=1) @ v
    ref_lse = scipy.special.logsumexp(logits, axis=1)
    return max(np.max(np.abs(o - ref_o)), np.max(np.abs(lse - ref_lse)))


def test_attention_core_matches_scipy_softmax():
    assert core_vs_scipy_error() <= 1e-12


# ------------------------------------------------------------ RoPE
def golden_positions_error(rope_positions=O.rope_positions):
    with open(os.path.join(GOLDEN, "rope_positions.json")) as f:
        cases = json.load(f)["cases"]
    bad = 0
    for c in cases:
        pos = rope_positions(c["T_txt"], *c["grid"])
        for n, p in c["tokens"].items():
            bad += int(list(pos[int(n)]) != p)
    return bad


def test_rope_positions_match_hand_worked_values():
    assert golden_positions_error() == 0


def rope_vs_complex_error(rope_rotate=O.rope_rotate, seed=2):
    """RoPE as multiplication of (y[2j] + i y[2j+1]) by exp(i * angle)."""
    rng = np.random.default_rng(seed)
    y = rng.standard_normal((50, 128))
    ang = O.rope_angles(O.rope_positions(10, 5, 8))
    z = (y[:, 0::2] + 1j * y[:, 1::2]) * np.exp(1j * ang)
    ref = np.empty_like(y)
    ref[:, 0::2], ref[:, 1::2] = z.real, z.imag
    return np.max(np.abs(rope_rotate(y, ang) - ref))


def test_rope_equals_complex_multiplication():
    assert rope_vs_complex_error() <= 1e-13


def test_rope_axis_split_and_first_pair_frequency():
    pos = O.rope_positions(16, 8, 8)
    ang = O.rope_angles(pos)
    y = np.random.default_rng(1).standard_normal((pos.shape[0], 128))
    out = O.rope_rotate(y, ang)
    # image tokens have frame index 0: the 16 frame dims are left unchanged
    assert np.array_equal(out[16:, :16], y[16:, :16])
    # grid row 4 is the centre (index 0) of the height axis: dims 16..71 unchanged
    row4 = [16 + 4 * 8 + c for c in range(8)]
    assert np.array_equal(out[row4, 16:72], y[row4, 16:72])
    # the first pair of each axis turns by exactly its position (frequency 1)
    e = np.zeros((pos.shape[0], 128))
    for start in (0, 16, 72):
        e[:] = 0
        e[:, start] = 1.0
        r = O.rope_rotate(e, ang)
        axis = {0: 0, 16: 1, 72: 2}[start]
        assert np.allclose(r[:, start], np.cos(pos[:, axis]), atol=1e-15)
        assert np.allclose(r[:, start + 1], np.sin(pos[:, axis]), atol=1e-15)
    # the last pair of the 56-wide axes turns by pos * 10000 ** (-54/56)
    e[:] = 0
    e[:, 16 + 54] = 1.0
    r = O.rope_rotate(e, ang)
    f = 10.0 ** (-4.0 * 54.0 / 56.0)
    assert np.allclose(r[:, 16 + 55], np.sin(pos[:, 1] * f), atol=1e-15)


def test_rope_preserves_pair_norms_and_inverse_undoes_it():
    rng = np.random.default_rng(0)
    y = rng.standard_normal((80, 128))
    ang = O.rope_angles(O.rope_positions(16, 8, 8))
    r = O.rope_rotate(y, ang)
    n0 = y[:, 0::2] ** 2 + y[:, 1::2] ** 2
    n1 = r[:, 0::2] ** 2 + r[:, 1::2] ** 2
    assert np.max(np.abs(n0 - n1)) <= 1e-12
    assert np.max(np.abs(O.rope_rotate_back(r, ang) - y)) <= 1e-13


def text_diagonal_relative_error(rope_positions=O.rope_positions):
    """Text scores depend only on t_q - t_k: shift all text positions (a change
    of the offset o by a bigger grid) and compare all text-text scores."""
    rng = np.random.default_rng(7)
    q = rng.standard_normal((12, 128))
    k = rng.standard_normal((12, 128))
    p1 = rope_positions(12, 8, 8)[:12]
    p2 = rope_positions(12, 40, 30)[:12]
    a1, a2 = O.rope_angles(p1), O.rope_angles(p2)
    s1 = O.rope_rotate(q, a1) @ O.rope_rotate(k, a1).T
    s2 = O.rope_rotate(q, a2) @ O.rope_rotate(k, a2).T
    # and within one layout: the score of (t, t + d) is the same for every t
    # when the same q and k vectors are placed there
    qq = np.repeat(q[:1], 12, axis=0)
    kk = np.repeat(k[:1], 12, axis=0)
    s3 = O.rope_rotate(qq, a1) @ O.rope_rotate(kk, a1).T
    diag_gap = max(np.ptp(np.diagonal(s3, offset=d)) for d in range(-11, 12))
    return max(np.max(np.abs(s1 - s2)), diag_gap)


def test_rope_text_diagonal_is_relative():
    assert text_diagonal_relative_error() <= 1e-11


def test_rope_image_shift_is_relative():
    rng = np.random.default_rng(8)
    q = rng.standard_normal((1, 128))
    k = rng.standard_normal((1, 128))

    def score(pq, pk):
        aq = O.rope_angles(np.array([pq]))
        ak = O.rope_angles(np.array([pk]))
        return float((O.rope_rotate(q, aq) @ O.rope_rotate(k, ak).T)[0, 0])

    base = score((0, 3, -2), (0, -1, 5))
    assert abs(score((0, 10, -2), (0, 6, 5)) - base) <= 1e-11
    assert abs(score((0, 3, 20), (0, -1, 27)) - base) <= 1e-11


# ------------------------------------------------------------ RMSNorm
def rmsnorm_unit_gain_error(rmsnorm=O.rmsnorm):
    """With g = 1: mean(y^2) = ms / (ms + eps); checked at ms ~ eps too."""
    rng = np.random.default_rng(3)
    worst = 0.0
    for scale in (1.0, 1e-3, 3e-4):
        x = rng.standard_normal((20, 128)) * scale
        y, _ = rmsnorm(x, np.ones_like(x), O.EPS)
        ms = np.mean(x * x, axis=1)
        worst = max(worst, np.max(np.abs(np.mean(y * y, axis=1) - ms / (ms + O.EPS))))
    return worst


def test_rmsnorm_unit_gain_mean_square():
    assert rmsnorm_unit_gain_error() <= 1e-13


def test_rmsnorm_scale_invariance_and_stream_gains():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((30, 128))
    g = rng.uniform(0.5, 1.5, (30, 128))
    y1, _ = O.rmsnorm(x, g)
    y2, _ = O.rmsnorm(37.0 * x, g)
    # equal up to the eps term: y2 / y1 = sqrt(ms + eps) / sqrt(ms + eps / 37^2)
    ms = np.mean(x * x, axis=1, keepdims=True)
    ratio = np.sqrt(ms + O.EPS) / np.sqrt(ms + O.EPS / 37.0 ** 2)
    assert np.max(np.abs(y2 - y1 * ratio)) <= 1e-13
    assert 0 < np.max(np.abs(y1 - y2)) <= 1e-5
    gains = np.stack([np.full(128, v) for v in (1.0, 2.0, 3.0, 4.0)])
    gq = O.token_gains(gains, 5, 30, "q")
    gk = O.token_gains(gains, 5, 30, "k")
    assert np.all(gq[:5] == 1.0) and np.all(gq[5:] == 3.0)
    assert np.all(gk[:5] == 2.0) and np.all(gk[5:] == 4.0)


# ------------------------------------------------------------ generator
def test_generator_bf16_rounding_matches_torch_and_rows_stack():
    torch = pytest.importorskip("torch")
    x = np.random.default_rng(0).standard_normal(100000).astype(np.float32)
    x[:4] = [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8, 3.0e38]  # ties and a big value
    ours = W.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    a = W.make_batch(W.TINY, 0)
    w2 = W.Workload("t2", B=3, H=2, T_txt=16, grid_h=8, grid_w=8, valid_len=(11, 3, 16))
    b = W.make_batch(w2, 0, rows=[5, 0, 2])
    assert np.array_equal(a["q"][0], b["q"][1]) and np.array_equal(a["do"][0], b["do"][1])
    assert W.credited_flops(W.CFG1024)["fwd"] == pytest.approx(453.06e9, rel=1e-5)
    assert W.credited_flops(W.CFG1024)["fwd_bwd"] == pytest.approx(1585.71e9, rel=1e-5)


# ------------------------------------------------------------ planted mistakes
def test_planted_mistakes_are_caught():
    """A copy of an oracle function with one plausible mistake fails a pin."""
    # RoPE: wrong sign of the sine term
    def rot_sign(y, ang):
        c, s = np.cos(ang), np.sin(ang)
        out = np.empty_like(y)
        out[:, 0::2] = y[:, 0::2] * c + y[:, 1::2] * s
        out[:, 1::2] = -y[:, 0::2] * s + y[:, 1::2] * c
        return out
    assert rope_vs_complex_error(rot_sign) > 1e-3

    # RoPE: floor instead of ceil when centring a side
    def pos_floor(T, gh, gw):
        p = O.rope_positions(T, gh, gw)
        p[T:, 1] += (gh + 1) // 2 - gh // 2
        p[T:, 2] += (gw + 1) // 2 - gw // 2
        return p
    assert golden_positions_error(pos_floor) > 0

    # RoPE: text offset missing
    def pos_no_offset(T, gh, gw):
        p = O.rope_positions(T, gh, gw)
        p[:T] -= max(gh // 2, gw // 2)
        return p
    assert golden_positions_error(pos_no_offset) > 0

    # RMSNorm: eps dropped
    def rms_no_eps(x, g, eps=O.EPS):
        r = 1.0 / np.sqrt(np.mean(x * x, axis=1))
        return x * r[:, None] * g, r
    assert rmsnorm_unit_gain_error(rms_no_eps) > 1e-3

    # attention: scale 1/d instead of 1/sqrt(d)
    def fwd_bad_scale(qh, kh, v, valid):
        return O.attention_forward(qh / np.sqrt(qh.shape[1]), kh, v, valid)
    assert core_vs_scipy_error(fwd_bad_scale) > 1e-3

    # backward: dS transposed in the dK product
    def bwd_transposed(qh, kh, v, p, do):
        D = qh.shape[1]
        dv = p.T @ do
        dp = do @ v.T
        ds = p * (dp - np.sum(p * dp, axis=1, keepdims=True))
        return (ds @ kh) / np.sqrt(D), (ds @ qh) / np.sqrt(D), dv

    def backward_mut(*a, **k):
        saved = O.attention_backward
        O.attention_backward = bwd_transposed
        try:
            return O.joint_attn_backward(*a, **k)
        finally:
            O.attention_backward = saved

    geom, Q, K, V, dO, g = _micro(T=3, L=2, gh=2, gw=2)
    assert directional_fd_error(geom, Q, K, V, dO, g, backward=backward_mut, n_dir=1) > 1e-3
    # and the unmodified oracle passes the same pin on the same case
    assert directional_fd_error(geom, Q, K, V, dO, g, n_dir=1) < 1e-6


def test_row_sample_equals_full_pair_when_all_rows_selected():
    w, Q, K, V, dO, g, vl = _tiny()
    o, lse = O.joint_attn_forward(Q, K, V, g, w.T_txt, w.grid_h, w.grid_w, vl)
    dQ, dK, dV, _, _ = O.joint_attn_backward(Q, K, V, g, dO, w.T_txt, w.grid_h, w.grid_w, vl)
    r = O.pair_rows_forward_backward(Q, K, V, g, dO, w.T_txt, w.grid_h, w.grid_w, vl[0], 0, 1, np.arange(w.S))
    for a, ref in zip(r, (o[0, :, 1], lse[0, 1], dQ[0, :, 1], dK[0, :, 1], dV[0, :, 1])):
        assert np.max(np.abs(a - ref)) <= 1e-12
    # a row subset gives exactly the selected rows of the forward
    rows = [0, 5, 40, 79]
    r2 = O.pair_rows_forward_backward(Q, K, V, g, dO, w.T_txt, w.grid_h, w.grid_w, vl[0], 0, 1, rows)
    assert np.max(np.abs(r2[0] - o[0, rows, 1])) <= 1e-12


def test_round_bf16_is_round_to_nearest_even():
    torch = pytest.importorskip("torch")
    x = np.random.default_rng(6).standard_normal(200000).astype(np.float32) * 7
    # exact ties between two bf16 neighbours, both parities, and a carry
    ties = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 255.5 / 128, 1.5 + 2 ** -8], np.float32)
    x = np.concatenate([x, ties])
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    got = O.round_bf16(x.astype(np.float64))
    assert np.array_equal(got, ref)
    assert O.round_bf16(np.array([1 + 2 ** -8]))[0] == 1.0          # tie to even (down)
    assert O.round_bf16(np.array([1 + 3 * 2 ** -8]))[0] == 1 + 2 ** -6  # tie to even (up)
    assert O.round_bf16(np.array([255.5 / 128]))[0] == 2.0           # carry into the exponent


def test_storage_rounding_only_rounds_q_and_k():
    """With store_bf16 the forward equals the exact attention of the rounded
    normed/rotated q and k; without it nothing is rounded."""
    w, Q, K, V, dO, g, vl = _tiny()
    qh, kh, _, _ = O.prologue(Q, K, g, w.T_txt, w.grid_h, w.grid_w)
    o, lse = O.joint_attn_forward(Q, K, V, g, w.T_txt, w.grid_h, w.grid_w, vl, store_bf16=True)
    valid = O.key_valid(w.T_txt, w.S, int(vl[0]))
    for h in range(w.H):
        ro, rl, _ = O.attention_forward(O.round_bf16(qh[0, h]), O.round_bf16(kh[0, h]), V[0, :, h], valid)
        assert np.max(np.abs(o[0, :, h] - ro)) <= 1e-13 and np.max(np.abs(lse[0, h] - rl)) <= 1e-13
    o2, lse2 = O.joint_attn_forward(Q, K, V, g, w.T_txt, w.grid_h, w.grid_w, vl)
    assert 0 < np.max(np.abs(lse2 - lse)) < 1e-2


# ---------------------------------------------------------------- qkv_bias_gemm
def _brute_qkv(X, W, b):
    """Every output feature as a plain Python sum, for tiny sizes."""
    B, T, C = X.shape
    out = np.zeros((B, T, 3 * C))
    for bb in range(B):
        for t in range(T):
            for o in range(3 * C):
                acc = 0.0
                for c in range(C):
                    acc += float(X[bb, t, c]) * float(W[o, c])
                out[bb, t, o] = acc + float(b[o])
    return out


def test_qkv_projection_matches_brute_force():
    rng = np.random.default_rng(7)
    B, T, C = 2, 3, 128
    X = rng.standard_normal((B, T, C))
    W = rng.standard_normal((3 * C, C))
    b = rng.standard_normal(3 * C)
    Q, K, V = O.qkv_projection(X, W, b)
    Y = _brute_qkv(X, W, b)
    for i, part in enumerate((Q, K, V)):
        assert part.shape == (B, T, 1, 128)
        assert np.allclose(part.reshape(B, T, C), Y[..., i * C:(i + 1) * C], rtol=0, atol=1e-11)


def test_qkv_projection_exact_on_integers_and_identity_blocks():
    rng = np.random.default_rng(8)
    B, T, H = 1, 5, 2
    C = H * 128
    X = rng.integers(-4, 5, (B, T, C)).astype(np.float64)
    b = rng.integers(-3, 4, 3 * C).astype(np.float64)
    # W = [I; 2I; -I]: Q = X + b_q, K = 2X + b_k, V = -X + b_v, head-major
    I = np.eye(C)
    Q, K, V = O.qkv_projection(X, np.concatenate([I, 2 * I, -I]), b)
    assert np.array_equal(Q.reshape(B, T, C), X + b[:C])
    assert np.array_equal(K.reshape(B, T, C), 2 * X + b[C:2 * C])
    assert np.array_equal(V.reshape(B, T, C), -X + b[2 * C:])
    # feature h * 128 + d is head h, dim d
    assert np.array_equal(Q[0, :, 1, 5], X[0, :, 128 + 5] + b[128 + 5])
    # integer operands: the general product is exact in float64
    W = rng.integers(-3, 4, (3 * C, C)).astype(np.float64)
    Q, K, V = O.qkv_projection(X, W, b)
    Y = np.einsum("btc,oc->bto", X.astype(np.int64), W.astype(np.int64)) + b.astype(np.int64)
    assert np.array_equal(V.reshape(B, T, C), Y[..., 2 * C:].astype(np.float64))


def test_attn_out_projection_matches_brute_force_and_identity():
    rng = np.random.default_rng(9)
    B, T, H = 2, 3, 1
    C = H * 128
    O_s = rng.standard_normal((B, T, H, 128))
    W = rng.standard_normal((C, C))
    b = rng.standard_normal(C)
    Y = O.attn_out_projection(O_s, W, b)
    for bb in range(B):
        for t in range(T):
            for o in (0, 17, C - 1):
                ref = sum(float(O_s[bb, t, 0, c]) * float(W[o, c]) for c in range(C)) + float(b[o])
                assert abs(Y[bb, t, o] - ref) <= 1e-11
    # W = permutation: output feature o reads input feature perm[o]
    perm = rng.permutation(C)
    P = np.eye(C)[perm]
    Y = O.attn_out_projection(O_s, P, np.zeros(C))
    assert np.array_equal(Y, O_s.reshape(B, T, C)[..., perm])


# ---------------------------------------------------------------- widening, row path, gain attribution
def bf16_by_definition(bits: int) -> float:
    """A bfloat16 bit pattern decoded from the format's definition: sign bit
    15, an 8-bit biased exponent (bias 127) in bits 14..7 and 7 fraction bits;
    exponent 0 is subnormal (0.f x 2^-126), exponent 255 is inf / NaN."""
    import math
    s = -1.0 if bits & 0x8000 else 1.0
    e = (bits >> 7) & 0xFF
    f = bits & 0x7F
    if e == 0xFF:
        return s * math.inf if f == 0 else math.nan
    if e == 0:
        return s * math.ldexp(f, -126 - 7)
    return s * math.ldexp(128 + f, e - 127 - 7)


def widen_mismatches(widen_bf16=O.widen_bf16) -> int:
    """Bit patterns (of all 65,536) that ``widen_bf16`` decodes differently
    from the definition; NaNs must stay NaN. The count, so a plant shows."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):  # signalling-NaN patterns warn when widened
        got = widen_bf16(bits)
    bad = 0
    for b in range(1 << 16):
        ref = bf16_by_definition(b)
        g = float(got[b])
        if np.isnan(ref):
            bad += int(not np.isnan(g))
        elif g != ref or np.signbit(g) != np.signbit(ref):
            bad += 1
    return bad


def test_widen_bf16_is_exact_over_every_bit_pattern():
    assert widen_mismatches() == 0
    torch = pytest.importorskip("torch")
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    with np.errstate(invalid="ignore"):
        got = O.widen_bf16(bits)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


RAGGED_ROWS = dict(B=2, H=2, T_txt=20, grid_h=3, grid_w=5, valid_len=(7, 20))


def forward_rows_error(forward_rows=O.forward_rows) -> float:
    """``forward_rows`` (one query row at a time, used for the full-size spot
    checks) against the selected rows of ``joint_attn_forward``, with and
    without the bf16 storage rounding, on the tiny case and a ragged one."""
    worst = 0.0
    w2 = W.Workload("ragged_rows", **RAGGED_ROWS)
    for w, seed in ((W.TINY, 0), (w2, 3)):
        d = W.make_batch(w, seed)
        Q, K, V = (O.widen_bf16(d[n]) for n in ("q", "k", "v"))
        g, vl = d["gains"].astype(np.float64), d["valid_len"]
        for store in (False, True):
            o, lse = O.joint_attn_forward(Q, K, V, g, w.T_txt, w.grid_h, w.grid_w, vl, store_bf16=store)
            for b in range(w.B):
                for h in range(w.H):
                    rows = list(range(w.S)) if w is W.TINY else [0, 1, w.T_txt - 1, w.T_txt, w.S - 1, 9]
                    ro, rl = forward_rows(Q, K, V, g, w.T_txt, w.grid_h, w.grid_w, vl[b], b, h, rows,
                                          store_bf16=store)
                    worst = max(worst, np.max(np.abs(ro - o[b, rows, h])), np.max(np.abs(rl - lse[b, h, rows])))
    return worst


def test_forward_rows_equals_the_full_forward():
    assert forward_rows_error() <= 1e-12


def dg_attribution_error(backward=O.joint_attn_backward, h=1e-6) -> float:
    """Each per-(sample, head) gain-gradient slot against a central difference
    of sum(O[b, :, h] * dO[b, :, h]) -- dO zeroed outside that (sample, head)
    -- in the gain of that slot, along a random direction and elementwise at
    a few dims. B = 2 and H = 2 with different valid lengths, so a partial
    credited to the wrong sample, head or slot fails."""
    rng = np.random.default_rng(21)
    T, gh, gw, vl = 3, 2, 3, np.array([2, 1])
    B, H, D = 2, 2, 128
    S = T + gh * gw
    Q, K, V, dO = (rng.standard_normal((B, S, H, D)) for _ in range(4))
    g = rng.uniform(0.5, 1.5, (4, D))
    _, _, _, dgp, _ = backward(Q, K, V, g, dO, T, gh, gw, vl)
    worst = 0.0
    for b in range(B):
        for hh in range(H):
            dOm = np.zeros_like(dO)
            dOm[b, :, hh] = dO[b, :, hh]

            def loss(gg):
                o, _ = O.joint_attn_forward(Q, K, V, gg, T, gh, gw, vl)
                return float(np.sum(o * dOm))
            for slot in range(4):
                d = rng.standard_normal(D)
                gp, gm = g.copy(), g.copy()
                gp[slot] += h * d
                gm[slot] -= h * d
                fd = (loss(gp) - loss(gm)) / (2 * h)
                an = float(np.dot(dgp[b, hh, slot], d))
                worst = max(worst, abs(fd - an) / max(abs(an), 1e-3))
                for j in rng.choice(D, 3, replace=False):
                    gp, gm = g.copy(), g.copy()
                    gp[slot, j] += h
                    gm[slot, j] -= h
                    fd = (loss(gp) - loss(gm)) / (2 * h)
                    worst = max(worst, abs(fd - dgp[b, hh, slot, j]) / max(1.0, abs(dgp[b, hh, slot, j])))
    return worst


def test_gain_gradient_partials_are_attributed_to_their_sample_head_and_slot():
    assert dg_attribution_error() <= 1e-6


def test_planted_mistakes_in_the_helpers_are_caught():
    """Widening, the row path and the per-(sample, head) gain partials each
    fail their pin with one plausible mistake planted."""
    # widening: a shift by 15 instead of 16
    def widen_shift(bits):
        u = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(15)
        with np.errstate(invalid="ignore"):
            return u.view(np.float32).astype(np.float64)
    assert widen_mismatches(widen_shift) > 1000

    # widening: the sign bit dropped
    def widen_unsigned(bits):
        with np.errstate(invalid="ignore"):
            return np.abs(O.widen_bf16(bits))
    assert widen_mismatches(widen_unsigned) > 1000

    # row path: every selected row rotated by the first token's angles
    def rows_first_angle(Q, K, V, g, T_txt, grid_h, grid_w, L, b, h, rows, store_bf16=False, **kw):
        S = Q.shape[1]
        ang = O.rope_angles(O.rope_positions(T_txt, grid_h, grid_w))
        gq, gk = O.token_gains(g, T_txt, S, "q"), O.token_gains(g, T_txt, S, "k")
        kh = O.rope_rotate(O.rmsnorm(K[b, :, h], gk)[0], ang)
        kh = O.round_bf16(kh) if store_bf16 else kh
        outs, lses = [], []
        for i in rows:
            qh = O.rope_rotate(O.rmsnorm(Q[b, i:i + 1, h], gq[i:i + 1])[0], ang[0:1])
            qh = O.round_bf16(qh) if store_bf16 else qh
            o, lse, _ = O.attention_forward(qh, kh, V[b, :, h], O.key_valid(T_txt, S, int(L)))
            outs.append(o[0])
            lses.append(lse[0])
        return np.array(outs), np.array(lses)
    assert forward_rows_error(rows_first_angle) > 1e-3

    # gain partials: the image Q and K slots swapped, and the (b, h) slots
    # transposed; both keep dgp.sum(axis=(0, 1)) equal to the true dg sum
    # of the swapped slots, so only the attribution pin sees them
    def bwd_slots_swapped(*a, **k):
        dQ, dK, dV, dgp, dg = O.joint_attn_backward(*a, **k)
        dgp = dgp[:, :, [0, 1, 3, 2]]
        return dQ, dK, dV, dgp, dgp.sum(axis=(0, 1))
    assert dg_attribution_error(bwd_slots_swapped) > 1e-3

    def bwd_bh_transposed(*a, **k):
        dQ, dK, dV, dgp, dg = O.joint_attn_backward(*a, **k)
        return dQ, dK, dV, dgp.transpose(1, 0, 2, 3).copy(), dg
    assert dg_attribution_error(bwd_bh_transposed) > 1e-3

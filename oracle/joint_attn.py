"""CPU oracle for the Qwen-Image joint attention path, forward and backward.

TEST INFRASTRUCTURE ONLY. Nothing in the product path may import, call or run
this module: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
legs of ``bench.py`` do. It shares no code, table or helper with the CUDA path.

Everything is computed in float64 from exactly widened bfloat16 inputs, with
no intermediate rounding, one (sample, head) pair at a time. Matrix products
use numpy's ``@`` as a library primitive; nothing is blocked, fused or
reordered beyond the plain definitions below.

Sources (the pages are GitHub threads of the RL-Kernel project):
  [RFC]  "[RFC][Qwen-Image][CUDA/ROCm] WS1/WS2 kernel roadmap, ablation matrix
         and integration plan #386" -- Model contract table (rows Streams,
         Text input, Q/K preprocessing, RoPE), Numerical requirements, WS1
         table (qk_rmsnorm, multi_axis_rope, joint_attn_qk_gemm,
         joint_attn_softmax, joint_attn_av_gemm, joint_attention_fused).
  [KL]   "[RFC] [Qwen-Image] WS1 Single-GPU Kernel List" (the older revision
         of #386) -- Kernel table (head_dim 128, axis split [16, 56, 56], text
         on the grid diagonal, QK^T / sqrt(d), online softmax, A . V, fwd+bwd).

Readings taken where the pages leave a step open (each is tested in
tests/test_oracle_pins.py against what the pages fix; the last three are not
fixed by the pages at all and are "parity unpinned" against the real model):
  * four gain vectors of shape [128], one per (stream, Q|K), shared by heads;
  * RoPE rotates interleaved pairs (2j, 2j+1) inside each axis block by
    pos_axis * theta ** (-2j / d_axis);                      [parity unpinned]
  * a side of N tokens is centred as i - ceil(N/2); text token t sits at
    o + t on all three axes with o = max(floor(gh/2), floor(gw/2)); the image
    frame index is 0;                                      [parity unpinned]
  * angles are formed in float64.                          [parity unpinned]
  * the key mask is a prefix valid length per sample over the text segment;
    padded query rows are computed like any other row.
  * storage rounding (``store_bf16=True``): qk_rmsnorm and multi_axis_rope
    are their own WS1 rows whose outputs are stored as bf16 ([RFC] Numerical
    requirements: cast to bf16 at the declared kernel output boundary), and
    the pages' CPU references round explicitly at storage. With the flag set
    the normed, rotated q and k are rounded to bf16 before the attention; the
    backward passes gradients through that rounding unchanged. With the flag
    clear (the default) everything stays exact float64.
"""

from __future__ import annotations

import numpy as np

D_HEAD = 128
AXES = (16, 56, 56)
THETA = 10000.0
EPS = 1e-6
# Gain slots, in the order the gains are passed.
Q_TXT, K_TXT, Q_IMG, K_IMG = 0, 1, 2, 3


def widen_bf16(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> exact float64 values."""
    u = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 value, ties to even,
    exactly (bfloat16 keeps 8 significant bits)."""
    m, e = np.frexp(x)
    return np.ldexp(np.rint(m * 256.0) / 256.0, e)


# ---------------------------------------------------------------- positions
def rope_positions(T_txt: int, grid_h: int, grid_w: int) -> np.ndarray:
    """Integer (frame, row, col) position of every token, [T_txt + gh*gw, 3].

    [RFC] Model contract, RoPE row: three axes, centred spatial indices, text
    offset max(H/2, W/2); [KL] multi_axis_rope: text on the grid diagonal.
    Image token n = T_txt + r * grid_w + c (row-major over the grid) has
    position (0, r - ceil(gh/2), c - ceil(gw/2)); text token t has
    (o + t, o + t, o + t) with o = max(gh // 2, gw // 2).
    """
    o = max(grid_h // 2, grid_w // 2)
    S = T_txt + grid_h * grid_w
    pos = np.zeros((S, 3), dtype=np.int64)
    for t in range(T_txt):
        pos[t, :] = o + t
    centre_h = (grid_h + 1) // 2
    centre_w = (grid_w + 1) // 2
    for r in range(grid_h):
        for c in range(grid_w):
            n = T_txt + r * grid_w + c
            pos[n, 0] = 0
            pos[n, 1] = r - centre_h
            pos[n, 2] = c - centre_w
    return pos


def rope_angles(pos: np.ndarray, axes=AXES, theta: float = THETA) -> np.ndarray:
    """Rotation angle of each of the D/2 pairs of each token, float64 [S, D/2].

    [RFC] RoPE row / [KL] multi_axis_rope: axis a owns a block of axes[a] dims;
    pair j of that block turns by pos_a * theta ** (-2j / axes[a]).
    """
    blocks = []
    for a, d_a in enumerate(axes):
        j = np.arange(d_a // 2, dtype=np.float64)
        freq = theta ** (-2.0 * j / d_a)
        blocks.append(pos[:, a].astype(np.float64)[:, None] * freq[None, :])
    return np.concatenate(blocks, axis=1)


def rope_rotate(y: np.ndarray, ang: np.ndarray) -> np.ndarray:
    """Rotate each pair (y[2j], y[2j+1]) of each row by ang[:, j]."""
    c, s = np.cos(ang), np.sin(ang)
    a, b = y[:, 0::2], y[:, 1::2]
    out = np.empty_like(y)
    out[:, 0::2] = a * c - b * s
    out[:, 1::2] = a * s + b * c
    return out


def rope_rotate_back(u: np.ndarray, ang: np.ndarray) -> np.ndarray:
    """The transpose (= inverse) of ``rope_rotate``: turn each pair by -ang."""
    return rope_rotate(u, -ang)


# ---------------------------------------------------------------- RMSNorm
def token_gains(g: np.ndarray, T_txt: int, S: int, which: str) -> np.ndarray:
    """Per-token gain rows [S, D]: the text gain before T_txt, image after."""
    txt, img = (Q_TXT, Q_IMG) if which == "q" else (K_TXT, K_IMG)
    rows = np.empty((S, g.shape[1]), dtype=np.float64)
    rows[:T_txt] = g[txt]
    rows[T_txt:] = g[img]
    return rows


def rmsnorm(x: np.ndarray, g_rows: np.ndarray, eps: float = EPS):
    """[RFC] Q/K preprocessing: y = x / sqrt(mean(x^2) + eps) * g, per row.

    Returns (y, r) with r = 1 / sqrt(mean(x^2) + eps) per row.
    """
    r = 1.0 / np.sqrt(np.mean(x * x, axis=1) + eps)
    return x * r[:, None] * g_rows, r


def rmsnorm_backward(x, r, g_rows, dy):
    """VJP of ``rmsnorm``: returns (dx, per-row gain gradient dy * x * r).

    With xh = x * r and w = dy * g:  dx = r * (w - xh * sum(w * xh) / D).
    """
    xh = x * r[:, None]
    w = dy * g_rows
    D = x.shape[1]
    dx = r[:, None] * (w - xh * (np.sum(w * xh, axis=1, keepdims=True) / D))
    return dx, dy * xh


# ---------------------------------------------------------------- attention
def key_valid(T_txt: int, S: int, L: int) -> np.ndarray:
    """[RFC] Text input row: padded prompts need a key mask. Key j is valid
    iff it is an image token (j >= T_txt) or one of the first L text tokens."""
    valid = np.ones(S, dtype=bool)
    valid[L:T_txt] = False
    return valid


def attention_forward(qh, kh, v, valid):
    """Joint non-causal attention of one (sample, head).

    [KL] joint_attn_qk_gemm (QK^T / sqrt(d)), joint_attn_softmax (masked
    softmax over the key sequence), joint_attn_av_gemm (A . V). The softmax is
    the plain two-pass definition; an online softmax reaches the same value.
    Returns O [S, D], lse [S] (natural log) and P [S, S].
    """
    D = qh.shape[1]
    s = (qh @ kh.T) / np.sqrt(D)
    s[:, ~valid] = -np.inf
    m = np.max(s, axis=1, keepdims=True)
    e = np.exp(s - m)
    l = np.sum(e, axis=1, keepdims=True)
    p = e / l
    return p @ v, m[:, 0] + np.log(l[:, 0]), p


def attention_backward(qh, kh, v, p, do):
    """VJP of ``attention_forward`` with respect to qh, kh and v.

    dV = P^T dO;  dP = dO V^T;  Delta_i = sum_j P_ij dP_ij;
    dS = P * (dP - Delta);  dqh = dS kh / sqrt(D);  dkh = dS^T qh / sqrt(D).
    """
    D = qh.shape[1]
    dv = p.T @ do
    dp = do @ v.T
    delta = np.sum(p * dp, axis=1, keepdims=True)
    ds = p * (dp - delta)
    return (ds @ kh) / np.sqrt(D), (ds.T @ qh) / np.sqrt(D), dv


# ---------------------------------------------------------------- full path
def _pair_forward(Qbh, Kbh, Vbh, g, T_txt, grid_h, grid_w, L, eps, theta, axes, store_bf16=False):
    S = Qbh.shape[0]
    ang = rope_angles(rope_positions(T_txt, grid_h, grid_w), axes, theta)
    gq = token_gains(g, T_txt, S, "q")
    gk = token_gains(g, T_txt, S, "k")
    yq, rq = rmsnorm(Qbh, gq, eps)
    yk, rk = rmsnorm(Kbh, gk, eps)
    qh = rope_rotate(yq, ang)
    kh = rope_rotate(yk, ang)
    if store_bf16:
        qh, kh = round_bf16(qh), round_bf16(kh)
    valid = key_valid(T_txt, S, L)
    o, lse, p = attention_forward(qh, kh, Vbh, valid)
    return dict(o=o, lse=lse, p=p, qh=qh, kh=kh, rq=rq, rk=rk, ang=ang,
                gq=gq, gk=gk, valid=valid)


def joint_attn_forward(Q, K, V, g, T_txt, grid_h, grid_w, valid_len,
                       eps=EPS, theta=THETA, axes=AXES, heads=None, store_bf16=False):
    """Forward of the whole path on float64 [B, S, H, D] inputs.

    g: float64 [4, D] gains (q_txt, k_txt, q_img, k_img); valid_len: [B].
    Returns O [B, S, H, D] and lse [B, H, S]; with ``heads`` given, only those
    heads are computed (the rest stay NaN).
    """
    B, S, H, D = Q.shape
    heads = range(H) if heads is None else heads
    O = np.full((B, S, H, D), np.nan)
    lse = np.full((B, H, S), np.nan)
    for b in range(B):
        for h in heads:
            f = _pair_forward(Q[b, :, h], K[b, :, h], V[b, :, h], g, T_txt,
                              grid_h, grid_w, int(valid_len[b]), eps, theta, axes, store_bf16)
            O[b, :, h] = f["o"]
            lse[b, h] = f["lse"]
    return O, lse


def joint_attn_backward(Q, K, V, g, dO, T_txt, grid_h, grid_w, valid_len,
                        eps=EPS, theta=THETA, axes=AXES, heads=None, store_bf16=False):
    """Backward of the whole path: gradients of sum(O * dO).

    Returns dQ, dK, dV [B, S, H, D], the per-(sample, head) gain-gradient
    partials dg_partial [B, H, 4, D] (slots q_txt, k_txt, q_img, k_img, each
    summed over that stream's tokens) and dg [4, D] = their sum over b and h.
    [RFC] Work items: every differentiable WS1 operator needs a backward too.
    """
    B, S, H, D = Q.shape
    heads = list(range(H)) if heads is None else list(heads)
    dQ = np.full((B, S, H, D), np.nan)
    dK = np.full_like(dQ, np.nan)
    dV = np.full_like(dQ, np.nan)
    dgp = np.full((B, H, 4, D), np.nan)
    for b in range(B):
        for h in heads:
            x_q, x_k = Q[b, :, h], K[b, :, h]
            f = _pair_forward(x_q, x_k, V[b, :, h], g, T_txt, grid_h, grid_w,
                              int(valid_len[b]), eps, theta, axes, store_bf16)
            dqh, dkh, dv = attention_backward(f["qh"], f["kh"], V[b, :, h],
                                              f["p"], dO[b, :, h])
            dyq = rope_rotate_back(dqh, f["ang"])
            dyk = rope_rotate_back(dkh, f["ang"])
            dxq, gq_rows = rmsnorm_backward(x_q, f["rq"], f["gq"], dyq)
            dxk, gk_rows = rmsnorm_backward(x_k, f["rk"], f["gk"], dyk)
            dQ[b, :, h], dK[b, :, h], dV[b, :, h] = dxq, dxk, dv
            dgp[b, h, Q_TXT] = gq_rows[:T_txt].sum(axis=0)
            dgp[b, h, K_TXT] = gk_rows[:T_txt].sum(axis=0)
            dgp[b, h, Q_IMG] = gq_rows[T_txt:].sum(axis=0)
            dgp[b, h, K_IMG] = gk_rows[T_txt:].sum(axis=0)
    dg = dgp[:, heads].sum(axis=(0, 1))
    return dQ, dK, dV, dgp, dg


def qkv_projection(X, W, b):
    """[RFC] WS1 row qkv_bias_gemm (each stream's Q, K and V projections in
    one GEMM with a bias; [KL] 3072 -> 3 x 3072, one weight set per stream) for one stream, in
    float64: Y = X W^T + b.

    X [B, T, C] with C = H * 128; W [3C, C], rows are output features in the
    nn.Linear layout: the Q features first (feature h * 128 + d is head h,
    dim d), then K, then V; b [3C]. Returns Q, K, V as [B, T, H, 128].
    """
    B, T, C = X.shape
    H = C // D_HEAD
    Y = X @ W.T + b
    parts = (Y[..., :C], Y[..., C:2 * C], Y[..., 2 * C:])
    return tuple(p.reshape(B, T, H, D_HEAD) for p in parts)


def attn_out_projection(O_s, W, b):
    """[RFC] WS1 row attn_out_bias_gemm (the attention output's projection,
    one per stream; [KL] 3072 -> 3072 with a bias) for one stream, in float64:
    Y = O W^T + b with O [B, T, H, 128] read as [B, T, C], W [C, C] (output
    feature rows), b [C]. Returns Y [B, T, C]."""
    B, T, H, D = O_s.shape
    return O_s.reshape(B, T, H * D) @ W.T + b


def prologue(Q, K, g, T_txt, grid_h, grid_w, eps=EPS, theta=THETA, axes=AXES):
    """qk_rmsnorm followed by multi_axis_rope on [B, S, H, D] inputs.

    Returns qh, kh in float64 [B, H, S, D] and the row factors rq, rk [B, H, S].
    """
    B, S, H, D = Q.shape
    ang = rope_angles(rope_positions(T_txt, grid_h, grid_w), axes, theta)
    gq = token_gains(g, T_txt, S, "q")
    gk = token_gains(g, T_txt, S, "k")
    qh = np.empty((B, H, S, D))
    kh = np.empty((B, H, S, D))
    rq = np.empty((B, H, S))
    rk = np.empty((B, H, S))
    for b in range(B):
        for h in range(H):
            yq, rq[b, h] = rmsnorm(Q[b, :, h], gq, eps)
            yk, rk[b, h] = rmsnorm(K[b, :, h], gk, eps)
            qh[b, h] = rope_rotate(yq, ang)
            kh[b, h] = rope_rotate(yk, ang)
    return qh, kh, rq, rk


def forward_rows(Q, K, V, g, T_txt, grid_h, grid_w, L, b, h, rows,
                 eps=EPS, theta=THETA, axes=AXES, store_bf16=False):
    """O and lse of selected query rows of one (sample, head), computed one
    row at a time against all keys (for spot checks at full size)."""
    S = Q.shape[1]
    ang = rope_angles(rope_positions(T_txt, grid_h, grid_w), axes, theta)
    gk = token_gains(g, T_txt, S, "k")
    gq = token_gains(g, T_txt, S, "q")
    yk, _ = rmsnorm(K[b, :, h], gk, eps)
    kh = rope_rotate(yk, ang)
    if store_bf16:
        kh = round_bf16(kh)
    valid = key_valid(T_txt, S, int(L))
    outs, lses = [], []
    for i in rows:
        yq, _ = rmsnorm(Q[b, i:i + 1, h], gq[i:i + 1], eps)
        qh = rope_rotate(yq, ang[i:i + 1])
        if store_bf16:
            qh = round_bf16(qh)
        o, lse, _ = attention_forward(qh, kh, V[b, :, h], valid)
        outs.append(o[0])
        lses.append(lse[0])
    return np.array(outs), np.array(lses)


def pair_rows_forward_backward(Q, K, V, g, dO, T_txt, grid_h, grid_w, L, b, h, rows,
                               eps=EPS, theta=THETA, axes=AXES):
    """Forward and backward of one (sample, head) restricted to the query rows
    ``rows``: their O and lse, the gradient of sum(O[rows] * dO[rows]) with
    respect to Q[rows], and that loss's gradient with respect to all of K and
    V. With every row selected this is the full per-(sample, head) result.
    (Used to time bounded samples of the oracle.)"""
    S = Q.shape[1]
    rows = np.asarray(rows)
    ang = rope_angles(rope_positions(T_txt, grid_h, grid_w), axes, theta)
    gq = token_gains(g, T_txt, S, "q")
    gk = token_gains(g, T_txt, S, "k")
    x_q, x_k = Q[b, rows, h], K[b, :, h]
    yq, rq = rmsnorm(x_q, gq[rows], eps)
    yk, rk = rmsnorm(x_k, gk, eps)
    qh = rope_rotate(yq, ang[rows])
    kh = rope_rotate(yk, ang)
    o, lse, p = attention_forward(qh, kh, V[b, :, h], key_valid(T_txt, S, int(L)))
    dqh, dkh, dv = attention_backward(qh, kh, V[b, :, h], p, dO[b, rows, h])
    dxq, _ = rmsnorm_backward(x_q, rq, gq[rows], rope_rotate_back(dqh, ang[rows]))
    dxk, _ = rmsnorm_backward(x_k, rk, gk, rope_rotate_back(dkh, ang))
    return o, lse, dxq, dxk, dv

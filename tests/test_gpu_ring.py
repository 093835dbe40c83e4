"""The forward run as key shards handing the online-softmax state on in the
fixed global block order (the RFC's WS2 row sp_attention_ring, emulated on
one GPU): every split of the key blocks into consecutive shards must give
the fused forward's out and lse bytes (topology invariance), and each split's
out and lse are also compared with the CPU oracle at the declared bounds, so
the hand-off itself (the rescale at a shard's first block, a shard with no
valid key passing its state through, the last shard's O / l) is checked
against the mathematics, not only against the fused kernel."""

import random

import pytest

from oracle import joint_attn as O

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


def _splits(n_blocks, n_txt, seed):
    """Shard boundaries: one shard, every block its own shard, the
    text/image boundary, and a few seeded random splits."""
    out = [[], list(range(1, n_blocks))]
    if 0 < n_txt < n_blocks:
        out.append([n_txt])
        out.append([1] if n_txt > 1 else [n_txt, n_txt + 1])
    rng = random.Random(seed)
    for _ in range(3):
        k = rng.randint(1, min(6, n_blocks - 1))
        out.append(sorted(rng.sample(range(1, n_blocks), k)))
    # boundaries strictly inside (0, n_blocks): every shard non-empty
    out = [sorted(set(b for b in bounds if 0 < b < n_blocks)) for bounds in out]
    return [list(x) for x in dict.fromkeys(tuple(b) for b in out)]


CASES = [
    W.TINY,
    # two text blocks; L = 0 gives a first shard with no valid key; L = 130
    # puts 2 valid keys in the second text block; a ragged image tail
    Hh.workload("ragged", 3, 2, 200, 13, 21, (0, 130, 200)),
    Hh.workload("cfg1024_h3", 2, 3, 256, 64, 64, (87, 193), scale=3.0),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_every_shard_split_gives_the_fused_bytes(w, dev):
    import torch
    batch = W.make_batch(w, 31, with_dout=False)
    q, k, v = (Hh.to_dev(batch[n], dev) for n in ("q", "k", "v"))
    gains = torch.from_numpy(batch["gains"]).to(dev)
    vl = [int(x) for x in batch["valid_len"]]
    ja = pkg.JointAttention(w.B, w.T_txt, w.grid_h, w.grid_w, w.H, device=dev)
    out_f, lse_f = ja.forward(q, k, v, gains, vl)
    torch.cuda.synchronize()
    n_txt = -(-w.T_txt // 128)
    # the oracle on the same inputs (every head of the small cases; heads 0
    # and H - 1 of the full-size one)
    heads = list(range(w.H)) if w.S <= 1024 else [0, w.H - 1]
    sub = {n: batch[n][:, :, heads] for n in ("q", "k", "v")}
    sub["gains"] = batch["gains"]
    Q, K, V, _, g = Hh.oracle_inputs(sub)
    ro, rl = O.joint_attn_forward(Q, K, V, g, w.T_txt, w.grid_h, w.grid_w, batch["valid_len"], store_bf16=True)
    for bounds in _splits(ja.n_key_blocks(), n_txt, 7):
        out, lse = ja.forward_sharded(q, k, v, gains, vl, bounds)
        torch.cuda.synchronize()
        pkg.rlk_joint_attn_check_status()
        Hh.assert_forward_close(Hh.f64(out[:, :, heads]), Hh.f64(lse[:, heads]), ro, rl,
                                f"{w.name} shards {bounds}", scale=w.scale)
        assert Hh.bits_equal(out, out_f), (w.name, bounds)
        assert Hh.bits_equal(lse, lse_f), (w.name, bounds)


def test_shard_calls_are_traced(dev):
    import torch
    w = W.TINY
    batch = W.make_batch(w, 32, with_dout=False)
    q, k, v = (Hh.to_dev(batch[n], dev) for n in ("q", "k", "v"))
    gains = torch.from_numpy(batch["gains"]).to(dev)
    ja = pkg.JointAttention(w.B, w.T_txt, w.grid_h, w.grid_w, w.H, device=dev)
    with pkg.op_trace() as t:
        ja.forward_sharded(q, k, v, gains, [int(x) for x in batch["valid_len"]], [1])
        torch.cuda.synchronize()
    assert [(r["entry_point"], r["kernels"]) for r in t.records] == [
        ("rlk_qk_norm_rope", ["rope_table_kernel", "prologue_kernel"]),
        ("rlk_joint_attn_fwd_shard", ["attn_fwd_tc_kernel<shard>"]),
        ("rlk_joint_attn_fwd_shard", ["attn_fwd_tc_kernel<shard>"]),
    ]

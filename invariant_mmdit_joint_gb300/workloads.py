"""Seeded synthetic workloads for the joint attention path.

This module only draws random numbers and names shapes. It holds none of the
attention arithmetic, so the CUDA path, the tests, the benchmark and the CPU
oracle can all take their inputs from it without sharing any of the method.

Shapes follow the Qwen-Image model contract (RFC #386, "Model contract" table:
24 heads x 128, joint attention over [text, image], reference shapes 1024^2,
1328^2 and 1664x928). An image of W x H pixels becomes a (H/16) x (W/16) token
grid after the 8x VAE and the 2x2 packing.

Draw recipe (one independent PCG64 substream per logical row, so that stacking
rows into any batch gives the same bytes per row):
  * row r of seed s uses ``numpy.random.default_rng([s, r])`` and draws, in this
    order, Q, K, V and dO, each [S, H, D] standard normal in float32, times the
    config's scale, rounded to bfloat16 (round to nearest, ties to even);
  * the four RMSNorm gains (q_txt, k_txt, q_img, k_img) are model weights, not
    per-row data: they come from ``default_rng([s, GAIN_STREAM])`` as
    U(0.5, 1.5) float32 of shape [4, 128];
  * random valid text lengths (batch-invariance sweep) come from
    ``default_rng([s, LEN_STREAM])`` as integers in [1, T_txt].
bfloat16 values are carried as their uint16 bit patterns.
"""

from __future__ import annotations

import dataclasses
from typing import Sequence

import numpy as np

HEAD_DIM = 128
N_HEADS = 24
GAIN_STREAM = 1_000_003
LEN_STREAM = 1_000_033


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    T_txt: int
    grid_h: int
    grid_w: int
    valid_len: tuple
    scale: float = 1.0
    with_bwd: bool = True

    @property
    def T_img(self) -> int:
        return self.grid_h * self.grid_w

    @property
    def S(self) -> int:
        return self.T_txt + self.T_img

    def describe(self) -> dict:
        return {
            "workload": self.name,
            "B": self.B,
            "H": self.H,
            "D": HEAD_DIM,
            "T_txt": self.T_txt,
            "grid": [self.grid_h, self.grid_w],
            "T_img": self.T_img,
            "S": self.S,
            "valid_len": list(self.valid_len),
            "input_scale": self.scale,
        }


# The tiny sanity case: 8x8 image grid, 16 text tokens of which 11 are valid.
TINY = Workload("tiny", B=1, H=2, T_txt=16, grid_h=8, grid_w=8, valid_len=(11,))
# 1024x1024 image, CFG pair (cond, neg prompt rows).
CFG1024 = Workload("cfg1024", B=2, H=N_HEADS, T_txt=256, grid_h=64, grid_w=64,
                   valid_len=(87, 193))
# 1664 wide x 928 high image: 58 x 104 grid.
IMG1664x928 = Workload("img1664x928", B=2, H=N_HEADS, T_txt=512, grid_h=58,
                       grid_w=104, valid_len=(300, 512))
# 1328x1328 image, two prompts x CFG; inputs scaled by 3.
IMG1328 = Workload("img1328", B=4, H=N_HEADS, T_txt=256, grid_h=83, grid_w=83,
                   valid_len=(40, 40, 256, 129), scale=3.0)

WORKLOADS = {w.name: w for w in (TINY, CFG1024, IMG1664x928, IMG1328)}


def sweep_lengths(seed: int, n_rows: int = 8, T_txt: int = 256) -> np.ndarray:
    """Random valid text lengths in U{1..T_txt} for the batch-invariance sweep."""
    rng = np.random.default_rng([seed, LEN_STREAM])
    return rng.integers(1, T_txt + 1, size=n_rows).astype(np.int32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); return uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    # u + 0x7FFF + lsb, in place in 32 bits: a sum that wraps (only the
    # largest NaN payloads) loses 2^32, which the 16-bit result drops anyway
    r = (u >> np.uint32(16)) & np.uint32(1)
    r += np.uint32(0x7FFF)
    r += u
    r >>= np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bits to float32."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32)
            << np.uint32(16)).view(np.float32)


def gains(seed: int, D: int = HEAD_DIM) -> np.ndarray:
    """The four RMSNorm gains [q_txt, k_txt, q_img, k_img], float32 [4, D]."""
    rng = np.random.default_rng([seed, GAIN_STREAM])
    return rng.uniform(0.5, 1.5, size=(4, D)).astype(np.float32)


def make_row(S: int, H: int, seed: int, row: int, scale: float = 1.0,
             with_dout: bool = True, D: int = HEAD_DIM) -> dict:
    """Q, K, V (and dO) of one logical row as bfloat16 bits, each [S, H, D]."""
    rng = np.random.default_rng([seed, row])
    out = {}
    names = ("q", "k", "v", "do") if with_dout else ("q", "k", "v")
    for name in names:
        x = rng.standard_normal((S, H, D), dtype=np.float32)
        if scale != 1.0:
            x *= np.float32(scale)
        out[name] = f32_to_bf16_bits(x)
    return out


def make_batch(w: Workload, seed: int, rows: Sequence[int] | None = None,
               valid_len: Sequence[int] | None = None,
               with_dout: bool | None = None) -> dict:
    """Stack logical rows into one batch.

    Returns uint16 bf16 bits q, k, v, do of shape [B, S, H, D], float32 gains
    [4, D] and int32 valid_len [B]. ``rows`` names the logical rows (default
    0..B-1); ``valid_len`` overrides the workload's lengths.
    """
    rows = list(range(w.B)) if rows is None else list(rows)
    vl = list(w.valid_len) if valid_len is None else list(valid_len)
    if len(vl) != len(rows):
        raise ValueError("one valid length per row")
    wd = w.with_bwd if with_dout is None else with_dout
    per = [make_row(w.S, w.H, seed, r, w.scale, wd) for r in rows]
    out = {k: np.stack([p[k] for p in per]) for k in per[0]}
    out["gains"] = gains(seed)
    out["valid_len"] = np.asarray(vl, dtype=np.int32)
    return out


def credited_flops(w: Workload, valid_len: Sequence[int] | None = None,
                   D: int = HEAD_DIM) -> dict:
    """Algorithmic FLOPs of one forward / backward over valid keys only.

    A (b, h) pair costs two S x S_v x D GEMMs forward (S_v = T_img + L_b, the
    keys that are not masked) and five backward (recomputed scores, dP, dV, dK
    and dQ). Masked keys are work the method skips, so they are not counted.
    """
    vl = list(w.valid_len) if valid_len is None else list(valid_len)
    gemm = sum(2.0 * D * w.S * (w.T_img + L) for L in vl) * w.H
    return {"gemm": gemm, "fwd": 2 * gemm, "bwd": 5 * gemm, "fwd_bwd": 7 * gemm}


QKV_STREAM = 1_000_081


def make_qkv_inputs(w: Workload, seed: int) -> dict:
    """Seeded inputs of the per-stream QKV projection (bf16 bits, uint16):
    activations x_txt [B, T_txt, C] and x_img [B, T_img, C] ~ N(0, 1),
    weights w_txt, w_img [3C, C] ~ N(0, 1/C) (the usual initial scale, so
    the projections are O(1)) and biases b_txt, b_img [3C] ~ N(0, 0.02^2),
    C = H * D, all drawn from ``default_rng([seed, QKV_STREAM])``."""
    C = w.H * HEAD_DIM
    rng = np.random.default_rng([seed, QKV_STREAM])
    out = {}
    for s, T in (("txt", w.T_txt), ("img", w.T_img)):
        out["x_" + s] = f32_to_bf16_bits(rng.standard_normal((w.B, T, C), dtype=np.float32))
        out["w_" + s] = f32_to_bf16_bits(rng.standard_normal((3 * C, C), dtype=np.float32) / np.float32(np.sqrt(C)))
        out["b_" + s] = f32_to_bf16_bits(rng.standard_normal(3 * C, dtype=np.float32) * np.float32(0.02))
    return out


def qkv_flops(w: Workload) -> float:
    """FLOPs of the two streams' projections: 2 * tokens * 3C * C."""
    C = w.H * HEAD_DIM
    return 2.0 * w.B * w.S * 3 * C * C

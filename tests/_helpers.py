"""Shared helpers of the GPU tests: move seeded inputs to the device, run the
path through the C ABI, and compare with the oracle at the declared
tolerances: forward max abs <= 1e-2 and mean abs <= 1e-3 for N(0,1) inputs
(inputs drawn as sigma * N(0,1) scale both by sigma, since O is linear in
V), lse <= 1e-4 relative, gradients relative L2 <= 1e-2. The oracle is run
with the declared bf16 storage rounding of the normed, rotated q and k; the
exact-float64 oracle is also checked, at the looser lse bound that rounding
implies (PURE_LSE_ABS)."""

from __future__ import annotations

import numpy as np

from invariant_mmdit_joint_gb300 import workloads as W

FWD_MAX_ABS = 1e-2
FWD_MEAN_ABS = 1e-3
LSE_REL = 1e-4
GRAD_REL_L2 = 1e-2
# bf16 storage of q and k alone moves lse against exact float64 by up to
# ~1.5e-3 absolute at S = 80 and ~1.6e-3 at S = 4352 (measured with the
# oracle); little averaging over keys (S = 6) gives ~2.5e-3.
PURE_LSE_ABS = 5e-3


def to_dev(bits: np.ndarray, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)


def f64(t) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def run_gpu(ja, batch: dict, dev, with_bwd=True, dout_override=None):
    """Run the forward (and backward) on a workloads.make_batch() dict."""
    import torch
    q, k, v = (to_dev(batch[n], dev) for n in ("q", "k", "v"))
    gains = torch.from_numpy(batch["gains"]).to(dev)
    vl = [int(x) for x in batch["valid_len"]]
    out, lse = ja.forward(q, k, v, gains, vl)
    res = {"out": out, "lse": lse}
    if with_bwd:
        do = to_dev(batch["do"], dev) if dout_override is None else dout_override
        dq, dk, dv, dgp, dg = ja.backward(q, k, v, gains, vl, out, do, lse)
        res.update(dq=dq, dk=dk, dv=dv, dgp=dgp, dg=dg)
    torch.cuda.synchronize()
    return res


def oracle_inputs(batch: dict):
    from oracle import joint_attn as O
    Q, K, V = (O.widen_bf16(batch[n]) for n in ("q", "k", "v"))
    dO = O.widen_bf16(batch["do"]) if "do" in batch else None
    return Q, K, V, dO, batch["gains"].astype(np.float64)


def assert_forward_close(out, lse, ref_o, ref_lse, where="", scale=1.0, lse_abs=None):
    err = np.abs(out - ref_o)
    if lse_abs is not None:
        # against exact float64 the bf16 rounding of the stored q and k adds
        # to the output rounding; with few keys |O| is large and the bf16
        # output rounding alone reaches ~1e-3 mean: the bound doubles
        scale = 2.0 * scale
    assert err.max() <= FWD_MAX_ABS * scale, (where, "O max abs", err.max())
    assert err.mean() <= FWD_MEAN_ABS * scale, (where, "O mean abs", err.mean())
    if lse_abs is None:
        rel = np.abs(lse - ref_lse) / np.abs(ref_lse)
        assert rel.max() <= LSE_REL, (where, "lse rel", rel.max())
    else:
        assert np.max(np.abs(lse - ref_lse)) <= lse_abs, (where, "lse abs", np.max(np.abs(lse - ref_lse)))


def rel_l2(a, b) -> float:
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / nb) if nb > 0 else float(np.linalg.norm(a))


def assert_grad_close(name, a, b, where=""):
    r = rel_l2(a, b)
    assert r <= GRAD_REL_L2, (where, name, "rel L2", r)


def bits_equal(a, b) -> bool:
    """Byte equality of two device tensors (bf16 compared as int16 bits)."""
    import torch
    if a.dtype == torch.bfloat16:
        a, b = a.view(torch.int16), b.view(torch.int16)
    elif a.dtype == torch.float32:
        a, b = a.view(torch.int32), b.view(torch.int32)
    return a.shape == b.shape and bool(torch.equal(a, b))


def workload(name, B, H, T_txt, gh, gw, valid_len, scale=1.0):
    return W.Workload(name, B=B, H=H, T_txt=T_txt, grid_h=gh, grid_w=gw, valid_len=tuple(valid_len), scale=scale)

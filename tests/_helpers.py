"""Shared helpers of the GPU tests: move seeded inputs to the device, run the
path through the C ABI, and compare with the oracle at the declared
tolerances: forward max abs <= 1e-2 and mean abs <= 1e-3 for N(0,1) inputs
(inputs drawn as sigma * N(0,1) scale both by sigma, since O is linear in
V), lse <= 1e-4 relative, gradients relative L2 <= 1e-2.

These bounds are applied against the oracle run with the declared bf16
storage of the normed, rotated q and k (``store_bf16=True``): the prologue
is its own kernel whose output is stored as bf16, and the tensor cores take
no fp32 operand. Against the exact float64 oracle the bound is derived, not
chosen (``assert_forward_close_exact``): by the triangle inequality

    |gpu - exact| <= |gpu - stored| + |stored - exact|,

where the first term is held to the declared bounds and the second is the
change the storage rounding itself makes, which the oracle computes exactly,
element by element. The declared 1e-4 lse bound therefore holds against the
storage-rounded oracle; against exact float64 the lse differs by the
storage term as well (a few 1e-4 relative).
"""

from __future__ import annotations

import numpy as np

from invariant_mmdit_joint_gb300 import workloads as W

FWD_MAX_ABS = 1e-2
FWD_MEAN_ABS = 1e-3
LSE_REL = 1e-4
GRAD_REL_L2 = 1e-2


def to_dev(bits: np.ndarray, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)


def f64(t) -> np.ndarray:
    # (blocks an operator leaves unwritten, such as a text tile with no
    # valid key, may hold any bytes; the tests read only written ones, and a
    # NaN there fails every bound)
    with np.errstate(invalid="ignore"):
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


def assert_forward_close(out, lse, ref_o, ref_lse, where="", scale=1.0):
    """The declared bounds against the storage-rounded oracle."""
    err = np.abs(out - ref_o)
    assert err.max() <= FWD_MAX_ABS * scale, (where, "O max abs", err.max())
    assert err.mean() <= FWD_MEAN_ABS * scale, (where, "O mean abs", err.mean())
    rel = np.abs(lse - ref_lse) / np.abs(ref_lse)
    assert rel.max() <= LSE_REL, (where, "lse rel", rel.max())


def assert_forward_close_exact(out, lse, stored, exact, where="", scale=1.0):
    """Against the exact float64 oracle, at the bound the storage reading
    implies: per element, the declared bound plus the oracle's own change
    under bf16 storage of q and k (``stored`` = (O, lse) with storage
    rounding, ``exact`` = (O, lse) without). Records the measured errors
    when RLK_PARITY_REPORT names a file."""
    so, sl = stored
    eo, el = exact
    store_o = np.abs(so - eo)
    store_l = np.abs(sl - el)
    err = np.abs(out - eo)
    lerr = np.abs(lse - el)
    assert np.all(err <= FWD_MAX_ABS * scale + store_o), (where, "O abs vs exact", float(np.max(err - store_o)))
    assert err.mean() <= FWD_MEAN_ABS * scale + store_o.mean(), (where, "O mean abs vs exact", err.mean(),
                                                                 store_o.mean())
    assert np.all(lerr <= LSE_REL * np.abs(sl) + store_l), (where, "lse vs exact",
                                                          float(np.max(lerr - store_l)))
    report(where, {"o_max_abs": float(err.max()), "o_mean_abs": float(err.mean()),
                   "lse_max_rel": float(np.max(lerr / np.abs(el))),
                   "storage_o_max_abs": float(store_o.max()), "storage_o_mean_abs": float(store_o.mean()),
                   "storage_lse_max_rel": float(np.max(store_l / np.abs(el))),
                   "gpu_vs_stored_lse_max_rel": float(np.max(np.abs(lse - sl) / np.abs(sl))),
                   "n": int(err.size)})


def report(where, values: dict):
    """Append one JSON line to the file RLK_PARITY_REPORT names, if any."""
    import json
    import os
    path = os.environ.get("RLK_PARITY_REPORT")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"case": where, **values}) + "\n")


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

"""Benchmark of the joint attention forward + backward on GB300.

A step is one pass of the whole path -- forward (RoPE table, fused
RMSNorm+RoPE prologue, attention) and backward (Delta, dK/dV, dQ, RoPE/RMSNorm
backward, gain-gradient fold) -- over one batch of the 1024^2 CFG-pair
workload (B=2, 24 heads x 128, 4096 image + 256 text tokens, valid text
lengths 87 and 193), synthetic seeded inputs. Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   (the CPU oracle on a bounded sample)

value = credited algorithmic TFLOP/s (valid keys only; backward credited at
2.5x the forward) of the whole job. Under torchrun each rank runs its own
replica of the workload (the path has no exchange step) and value sums the
ranks' work over the slowest rank's time.

Timed regions, each of K steps after W warm-up steps, inputs resident in HBM
and larger than L2:
  value, ms_per_step        the API calls as a caller makes them
  kernels, roofline         the same with a CUDA event pair around every
                            launch (ms_per_step_instrumented); phases splits
                            it into forward and backward
  graph                     the step captured once into a CUDA graph, replayed
  e2e (e2e_serial)          with each step's inputs copied from pinned host
                            memory and its results read back, pipelined over
                            three streams (serial on one stream)
dense_convention restates value with every key counted, masked or not.
Outside those regions: the standalone operators (unfused_forward), the QKV
producer and output projection (qkv_producer), and the key-shard forward and
separate-stream step (shards_and_streams), each byte-compared with the fused
calls.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from invariant_mmdit_joint_gb300 import workloads as W  # noqa: E402

METRIC = "joint-attn fwd+bwd TFLOP/s and % of BF16 tensor peak at 1024² (4096 img+256 txt)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# fwd: table, prologue, attention; bwd: pre, key norm/rope, 2 folds, and a
# dK/dV + dQ pair per workspace group (one group with the full workspace)
LAUNCHES_FIXED, LAUNCHES_PER_GROUP = 7, 2
THROTTLE_BITS = {
    0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
    0x10: "sync_boost", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
    0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting",
}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")), ws


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest of every rank's value (timing is reported for the
    slowest rank); the identity with one rank."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_step: float, world: int, ms_per_step_slowest: float) -> float:
    """Whole-job TFLOP/s: every rank runs its own replica of the workload
    (weak scaling, no data-path collective), timed by the slowest rank."""
    return world * flops_per_step / (ms_per_step_slowest * 1e-3) / 1e12


def bench_config(w: W.Workload) -> dict:
    """The workload a line measures; both arms print exactly this."""
    return {**w.describe(), "credited_gflop_per_step": round(W.credited_flops(w)["fwd_bwd"] / 1e9, 2)}


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    def __init__(self, gpu_index: int):
        import tempfile
        self.proc = None
        fd, self.path = tempfile.mkstemp(suffix=".csv", prefix="rlk_clocks_")
        os.close(fd)
        self.gpu = gpu_index

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu),
                 "--query-gpu=clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.fh.close()

    def summary(self):
        if self.proc is None:
            return None
        sm, mx, reasons = [], None, set()
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 4:
                    continue
                try:
                    sm.append(float(parts[0]))
                    mx = float(parts[1])
                    bits = int(parts[3], 16)
                except ValueError:
                    continue
                for bit, name in THROTTLE_BITS.items():
                    if bits & bit:
                        reasons.add(name)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not sm:
            return None
        loaded = [s for s in sm if s > 0]
        return {"sm_mhz": statistics.median(loaded or sm), "sm_max_mhz": mx, "samples": len(sm),
                "reasons": sorted(reasons - {"gpu_idle"})}


# ---------------------------------------------------------------- per-kernel bytes / flops
def kernel_work(w: W.Workload):
    """Algorithmic work per launch of each kernel: ("tensor", flops) or ("hbm", bytes)."""
    fl = W.credited_flops(w)
    G = fl["gemm"]
    rows = w.B * w.H * w.S
    D = W.HEAD_DIM
    n_pos = (max(w.grid_h // 2, w.grid_w // 2) + w.T_txt) + max((w.grid_h + 1) // 2, (w.grid_w + 1) // 2)
    # bf16 dS^T tiles (128 x 128) the dK/dV kernel writes and the dQ kernel
    # reads: every query tile against the key tiles holding a valid key
    ntq_txt, ntq_img = -(-w.T_txt // 128), -(-w.T_img // 128)
    ds_bytes = sum(w.H * (ntq_txt + ntq_img) * (-(-L // 128) + ntq_img) * 128 * 128 * 2 for L in w.valid_len)
    return {
        "rope_table": ("hbm", n_pos * 64 * 8),
        # read Q, K (bf16), write qh, kh (bf16) and r (fp32) of both
        "prologue": ("hbm", 4 * rows * D * 2 + 2 * rows * 4),
        # QK^T and PV
        "attn_fwd": ("tensor", 2 * G),
        # read O, dO (bf16) and lse; write Delta and lse2 (fp32)
        "bwd_pre": ("hbm", 2 * rows * D * 2 + 3 * rows * 4),
        # recomputed S^T, dV, dP^T, dK: four of the five credited backward GEMMs
        # (it also writes the dS^T tiles, ds_bytes)
        "bwd_dkdv": ("tensor", 4 * G),
        # dQ = dS K, the fifth GEMM, streams the dS^T tiles: read them and K
        # once; its epilogue runs the RoPE / RMSNorm backward of the query
        # rows from TMEM: read q (bf16) and rq, write dQ (bf16) and the q
        # gain-gradient partials (one per 32-row quarter of a tile)
        "bwd_dq": ("hbm", ds_bytes + rows * D * 2 + rows * D * 2 + rows * 4 + rows * D * 2 + rows // 32 * D * 4),
        # read dk^ (fp32), k (bf16), rk; write dK (bf16) and the k partials
        "norm_rope_bwd_k": ("hbm", rows * D * 4 + rows * D * 2 + rows * 4 + rows * D * 2 + rows // 32 * D * 4),
        # read both operands' tile partials, write the (b, h) folds
        "dg_fold": ("hbm", 2 * rows // 32 * D * 4 + w.B * w.H * 4 * D * 4),
    }


def unfused_work(w: W.Workload):
    """Algorithmic HBM bytes per launch of the standalone operators: each
    reads its inputs once and writes its outputs once; the intermediates
    cover the key tiles each sample visits."""
    rows = w.B * w.H * w.S
    D = W.HEAD_DIM
    ntq_img = -(-w.T_img // 128)
    blocks = sum(w.H * w.S * (-(-L // 128) + ntq_img) for L in w.valid_len)  # (row, key tile) pairs
    scores, p, alpha = blocks * 128 * 4, blocks * 128 * 2, blocks * 4
    return {
        "qk_gemm": 2 * rows * D * 2 + scores,
        "softmax": scores + p + alpha + 2 * rows * 4,
        "av_gemm": p + alpha + rows * 4 + 2 * rows * D * 2,
    }


def measure_unfused(pkg, ja, w, q, k, v, gains, vl, fused_out, fused_ms, peaks, n_steps):
    """The forward as the four standalone operators (prologue, qk_gemm,
    softmax, av_gemm): time per forward, byte equality with the fused
    forward's output on the same inputs, and each operator's HBM rate."""
    import torch
    stream = torch.cuda.current_stream()
    u = ja.forward_unfused(q, k, v, gains, vl)  # warm-up; allocates the intermediates once
    torch.cuda.synchronize()
    byte_equal = bool(torch.equal(u["out"].view(torch.int16), fused_out.view(torch.int16)))
    del u
    pkg.rlk_kernel_timing(True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(n_steps):
        ja.forward_unfused(q, k, v, gains, vl)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / n_steps
    work = unfused_work(w)
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    ops = {}
    for name in ("qk_gemm", "softmax", "av_gemm"):
        tot, n = pkg.rlk_kernel_timing_read(name)
        if n:
            avg = tot / n
            gbs = work[name] / (avg * 1e-3) / 1e9
            ops[name] = {"avg_ms": round(avg, 4), "algorithmic_bytes": work[name], "achieved": round(gbs, 1),
                         "unit": "GB/s", "frac": round(gbs / hbm, 4)}
    pkg.rlk_kernel_timing(False)
    return {"ms_per_forward": round(ms, 4), "fused_forward_ms": round(fused_ms, 4),
            "byte_equal_to_fused": byte_equal, "steps": n_steps, "operators": ops,
            "peak": f"hbm_gbs {hbm}"}


def unfused_bwd_work(w: W.Workload):
    """Algorithmic HBM bytes per step of the standalone backward's kernels
    (each reads its inputs once and writes its outputs once; the [query,
    key] intermediates cover the key tiles each sample visits)."""
    rows = w.B * w.H * w.S
    D = W.HEAD_DIM
    ntq_img = -(-w.T_img // 128)
    blocks = sum(w.H * w.S * (-(-L // 128) + ntq_img) for L in w.valid_len)
    f32, b16 = blocks * 128 * 4, blocks * 128 * 2
    slots = w.B * w.H * 128 * (-(-w.T_txt // 128) + ntq_img)
    return {
        # P pass: scores, lse2 in; P out. dS pass: scores, dP, lse2, Delta in; dS out
        "softmax_bwd": (f32 + b16 + slots * 4) + (2 * f32 + b16 + 2 * slots * 4),
        # dO and V in, dP out
        "dp_gemm": 2 * rows * D * 2 + f32,
        # dV: P, dO in, dV out (bf16); dk^: dS, q^ in, dk^ out (fp32)
        "key_gemm": (b16 + rows * D * 2 + rows * D * 2) + (b16 + rows * D * 2 + rows * D * 4),
        # dq^: dS, k^ in, dq^ out (fp32)
        "query_gemm": b16 + rows * D * 2 + rows * D * 4,
    }


def measure_unfused_bwd(pkg, ja, w, q, k, v, do, gains, vl, fused, fused_ms, peaks, n_steps):
    """The backward as the standalone operators' backward calls (stats,
    softmax_bwd for P, av_gemm_bwd, softmax_bwd for dS, qk_gemm_bwd,
    qk_norm_rope_bwd) after a standalone forward: time per backward, byte
    equality with the fused backward on the same inputs (fused = its dq, dk,
    dv, dg_partial, dg) and the HBM rate of the materialising kernels."""
    import torch
    stream = torch.cuda.current_stream()
    u = ja.forward_unfused(q, k, v, gains, vl)
    ub = ja.backward_unfused(q, k, v, gains, vl, u["out"], do, u["lse"], u["scores"])  # warm-up
    torch.cuda.synchronize()
    byte_equal = all(bool(torch.equal(ub[n].view(torch.int32 if ub[n].dtype == torch.float32 else torch.int16),
                                      f.view(torch.int32 if f.dtype == torch.float32 else torch.int16)))
                     for n, f in zip(("dq", "dk", "dv", "dgp", "dg"), fused))
    del ub
    pkg.rlk_kernel_timing(True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(n_steps):
        ja.backward_unfused(q, k, v, gains, vl, u["out"], do, u["lse"], u["scores"])
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / n_steps
    work = unfused_bwd_work(w)
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    ops = {}
    for name in ("softmax_bwd", "dp_gemm", "key_gemm", "query_gemm", "norm_rope_bwd_q"):
        tot, n = pkg.rlk_kernel_timing_read(name)
        if n:
            per_step = tot / n_steps
            entry = {"ms_per_step": round(per_step, 4), "launches_per_step": n // n_steps}
            if name in work:
                gbs = work[name] / (per_step * 1e-3) / 1e9
                entry.update(algorithmic_bytes=work[name], achieved=round(gbs, 1), unit="GB/s",
                             frac=round(gbs / hbm, 4))
            ops[name] = entry
    pkg.rlk_kernel_timing(False)
    del u
    return {"ms_per_backward": round(ms, 4), "fused_backward_ms": round(fused_ms, 4),
            "byte_equal_to_fused": byte_equal, "steps": n_steps, "operators": ops, "peak": f"hbm_gbs {hbm}"}


def _time_ms(fn, n_steps):
    import torch
    stream = torch.cuda.current_stream()
    fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n_steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / n_steps


def measure_shards_streams(ja, w, q, k, v, do, gains, vl, flops, n_steps):
    """The key-shard forward (ring order: the softmax state handed from shard
    to shard) with the key blocks split into 2 and 4 equal shards, and the
    forward + backward on separately allocated text and image buffers; each
    timed per call with CUDA events and compared byte for byte with the
    fused calls on the concatenated buffers."""
    import torch

    def eq(a, b):
        return bool(torch.equal(a.contiguous().view(torch.int16), b.contiguous().view(torch.int16)))

    out_f, lse_f = ja.forward(q, k, v, gains, vl)
    res_f = ja.backward(q, k, v, gains, vl, out_f, do, lse_f)
    fwd_ms = _time_ms(lambda: ja.forward(q, k, v, gains, vl), n_steps)
    nb = ja.n_key_blocks()
    shards = {}
    for n in (2, 4):
        bounds = [round(i * nb / n) for i in range(1, n)]
        out_s, lse_s = ja.forward_sharded(q, k, v, gains, vl, bounds)
        ms = _time_ms(lambda: ja.forward_sharded(q, k, v, gains, vl, bounds), n_steps)
        shards[str(n)] = {"bounds": bounds, "ms": round(ms, 4),
                          "tflops": round(flops["fwd"] / (ms * 1e-3) / 1e12, 1),
                          "bytes_equal_to_fused": eq(out_s, out_f) and bool(torch.equal(lse_s, lse_f))}
    T = w.T_txt
    split = lambda t: (t[:, :T].contiguous() if T > 0 else None, t[:, T:].contiguous())  # noqa: E731
    qs, ks, vs, dos = split(q), split(k), split(v), split(do)

    def step_streams():
        o, l = ja.forward_streams(qs, ks, vs, gains, vl)
        return o, l, ja.backward_streams(qs, ks, vs, gains, vl, o, dos, l)

    o_s, l_s, r_s = step_streams()
    cat = lambda pair: torch.cat([x for x in pair if x is not None], dim=1)  # noqa: E731
    same = eq(cat(o_s), out_f) and bool(torch.equal(l_s, lse_f))
    for a, b in zip(r_s[:3], res_f[:3]):
        same = same and eq(cat(a), b)
    same = same and bool(torch.equal(r_s[3], res_f[3])) and bool(torch.equal(r_s[4], res_f[4]))
    ms_streams = _time_ms(step_streams, n_steps)
    def step_cat():
        o, l = ja.forward(q, k, v, gains, vl)
        return ja.backward(q, k, v, gains, vl, o, do, l)

    ms_cat = _time_ms(step_cat, n_steps)
    return {"fused_forward_ms": round(fwd_ms, 4), "key_shards": shards, "steps": n_steps,
            "separate_streams": {"ms_per_step": round(ms_streams, 4), "concatenated_ms_per_step": round(ms_cat, 4),
                                 "tflops": round(flops["fwd_bwd"] / (ms_streams * 1e-3) / 1e12, 1),
                                 "bytes_equal_to_concatenated": same}}


def measure_qkv(pkg, w, peaks, n_steps):
    """The attention's producer: the per-stream QKV projection with the
    QK-RMSNorm + RoPE epilogue (writing the attention context), against the
    plain projection followed by the prologue kernel; seeded bf16 inputs."""
    import torch
    dev = torch.device("cuda", torch.cuda.current_device())
    d = W.make_qkv_inputs(w, 0)

    def t(name):
        return None if d[name].size == 0 else torch.from_numpy(d[name].view(np.int16)).view(torch.bfloat16).to(dev)
    x, wt, b = ((t(p + "_txt"), t(p + "_img")) for p in ("x", "w", "b"))
    gains = torch.from_numpy(W.gains(0)).to(dev)
    shape = pkg.Shape.make(w.B, w.T_txt, w.grid_h, w.grid_w, w.H)
    ja = pkg.JointAttention(w.B, w.T_txt, w.grid_h, w.grid_w, w.H, device=dev)

    def pair():
        return tuple(None if T == 0 else torch.empty((w.B, T, w.H, 128), dtype=torch.bfloat16, device=dev)
                     for T in (w.T_txt, w.T_img))
    q, k, v = pair(), pair(), pair()
    none = (None, None)

    def fused():
        pkg.rlk_qkv_bias_gemm(shape, x, wt, b, gains, ja.ctx, none, none, v)

    def plain_then_prologue():
        pkg.rlk_qkv_bias_gemm(shape, x, wt, b, None, None, q, k, v)
        qc = q[1] if q[0] is None else torch.cat(q, dim=1)
        kc = k[1] if k[0] is None else torch.cat(k, dim=1)
        pkg.rlk_qk_norm_rope(shape, qc, kc, gains[0], gains[1], gains[2], gains[3], ja.ctx)

    C = w.H * W.HEAD_DIM
    o = tuple(None if t is None else t.view(w.B, -1, w.H, W.HEAD_DIM) for t in x)
    wo = tuple(t[:C].contiguous() for t in wt)
    bo = tuple(t[:C].contiguous() for t in b)
    y = tuple(None if t is None else torch.empty_like(t) for t in x)

    def out_proj():
        pkg.rlk_attn_out_bias_gemm(shape, o, wo, bo, y)

    res = {}
    stream = torch.cuda.current_stream()
    for name, fn in (("fused", fused), ("plain_then_prologue", plain_then_prologue), ("out_proj", out_proj)):
        for _ in range(3):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(n_steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        res[name] = e0.elapsed_time(e1) / n_steps
    pkg.rlk_joint_attn_check_status()
    flops = W.qkv_flops(w)
    peak = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    tf = flops / (res["fused"] * 1e-3) / 1e12
    return {"op": "qkv_bias_gemm + qk_rmsnorm + multi_axis_rope (both streams)", "gflop": round(flops / 1e9, 2),
            "ms_fused": round(res["fused"], 4), "ms_plain_then_prologue": round(res["plain_then_prologue"], 4),
            "achieved": round(tf, 1), "unit": "TFLOP/s", "peak": peak, "frac": round(tf / peak, 4),
            "peak_source": "bf16_tflops (burst: the projection is timed alone)", "steps": n_steps,
            "attn_out_bias_gemm": {"gflop": round(flops / 3e9, 2), "ms": round(res["out_proj"], 4),
                                   "achieved": round(flops / 3 / (res["out_proj"] * 1e-3) / 1e12, 1),
                                   "frac": round(flops / 3 / (res["out_proj"] * 1e-3) / 1e12 / peak, 4)}}


def load_traffic(source_hash: str):
    """dram bytes per launch from the committed ncu summary, if it was taken
    on this exact source tree."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return {}
    with open(path) as f:
        t = json.load(f)
    if t.get("source_hash") != source_hash:
        return {}
    return t.get("kernels", {})


# ---------------------------------------------------------------- our arm
def selected_workload(args) -> W.Workload:
    """The named workload; with --heads, the same shape on fewer heads (a
    reduced case for profiler section captures, reported as such)."""
    w = W.WORKLOADS[args.workload]
    if getattr(args, "heads", None):
        import dataclasses
        w = dataclasses.replace(w, name=f"{w.name}_h{args.heads}", H=int(args.heads))
    return w


def run_ours(args):
    import torch

    import invariant_mmdit_joint_gb300 as pkg
    from invariant_mmdit_joint_gb300 import _build

    rank, local_rank, world = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = selected_workload(args)
    batch = W.make_batch(w, seed=0)
    flops = W.credited_flops(w)

    def to_host(bits):
        t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
        return t.pin_memory()

    h_q, h_k, h_v, h_do = (to_host(batch[n]) for n in ("q", "k", "v", "do"))
    h_g = torch.from_numpy(batch["gains"]).pin_memory()
    q, k, v, do = (t.to(dev) for t in (h_q, h_k, h_v, h_do))
    gains = h_g.to(dev)
    vl = [int(x) for x in batch["valid_len"]]
    budget = None if args.ws_budget_gb is None else int(args.ws_budget_gb * 1e9)
    ja = pkg.JointAttention(w.B, w.T_txt, w.grid_h, w.grid_w, w.H, device=dev, ws_budget_bytes=budget)
    ws_full = pkg.rlk_joint_attn_bwd_workspace_bytes(ja.shape)
    ws_min = pkg.rlk_joint_attn_bwd_workspace_min_bytes(ja.shape)
    per_pair = (ws_full - ws_min) // max(1, w.B * w.H - 1) if w.B * w.H > 1 else 0
    ws_bytes = ja.workspace.numel()
    pairs_per_group = w.B * w.H if ws_bytes >= ws_full else 1 + (ws_bytes - ws_min) // per_pair
    workspace = {"bytes": ws_bytes, "full_bytes": ws_full, "min_bytes": ws_min, "pairs_per_group": pairs_per_group,
                 "groups": -(-(w.B * w.H) // pairs_per_group)}
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dgp = torch.empty((w.B, w.H, 4, W.HEAD_DIM), dtype=torch.float32, device=dev)
    dg = torch.empty((4, W.HEAD_DIM), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        ja.forward(q, k, v, gains, vl, out=out, lse=lse)
        ja.backward(q, k, v, gains, vl, out, do, lse, dq=dq, dk=dk, dv=dv, dg_partial=dgp, dg=dg)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    for _ in range(args.warmup):
        step()
    pkg.rlk_joint_attn_check_status()

    # ---- device-resident timed region (inputs in HBM; working set > L2) ----
    # the step exactly as a caller runs it: no per-kernel instrumentation
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clk:
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
    barrier()
    ms_total = e0.elapsed_time(e1)
    pkg.rlk_joint_attn_check_status()
    eager_result = [t.clone() for t in (out, lse, dq, dk, dv, dgp, dg)]

    # ---- the same steps again with a CUDA event pair around every launch
    # (rlk_kernel_timing): each kernel's average duration for the roofline.
    # The events lengthen the step a little (ms_per_step_instrumented). ----
    pkg.rlk_kernel_timing(True)
    torch.cuda.synchronize()
    i0, i1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    i0.record(stream)
    for _ in range(args.steps):
        step()
    i1.record(stream)
    torch.cuda.synchronize()
    kern = {}
    for name in pkg.KERNEL_IDS:
        tot, n = pkg.rlk_kernel_timing_read(name)
        kern[name] = (tot, n)
    pkg.rlk_kernel_timing(False)
    pkg.rlk_joint_attn_check_status()
    ms_instrumented = i0.elapsed_time(i1) / args.steps

    # ---- the step captured once into a CUDA graph and replayed ----
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            step()
    stream.wait_stream(cap)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for _ in range(args.steps):
        graph.replay()
    g1.record(stream)
    torch.cuda.synchronize()
    pkg.rlk_joint_attn_check_status()
    graph_bytes_equal = all(
        torch.equal(a.view(torch.uint8), b.view(torch.uint8))
        for a, b in zip(eager_result, (out, lse, dq, dk, dv, dgp, dg)))
    ms_graph = max_over_ranks(g0.elapsed_time(g1), world, dev) / args.steps

    ms_step = max_over_ranks(ms_total, world, dev) / args.steps
    value = job_throughput(flops["fwd_bwd"], world, ms_step)

    # ---- end to end through the public API with host buffers ----
    # Every step copies its own inputs from pinned host memory to the device
    # and reads all of its results back. Serial: copies and compute on one
    # stream. Pipelined (the reported e2e): double-buffered device inputs and
    # outputs and three streams, so step i's compute overlaps step i+1's
    # host-to-device copies and step i-1's device-to-host copies, as a
    # training loop would; the same bytes move every step.
    h_in = (h_q, h_k, h_v, h_do, h_g)
    slots = [{"in": (q, k, v, do, gains), "out": (out, dq, dk, dv, lse, dg), "dgp": dgp}]
    slots.append({"in": tuple(torch.empty_like(t) for t in slots[0]["in"]),
                  "out": tuple(torch.empty_like(t) for t in slots[0]["out"]), "dgp": torch.empty_like(dgp)})
    for sl in slots:
        sl["host"] = tuple(torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in sl["out"])
    h2d = sum(t.numel() * t.element_size() for t in h_in)
    d2h = sum(t.numel() * t.element_size() for t in slots[0]["host"])

    def compute(sl):
        q_, k_, v_, do_, g_ = sl["in"]
        out_, dq_, dk_, dv_, lse_, dg_ = sl["out"]
        ja.forward(q_, k_, v_, g_, vl, out=out_, lse=lse_)
        ja.backward(q_, k_, v_, g_, vl, out_, do_, lse_, dq=dq_, dk=dk_, dv=dv_, dg_partial=sl["dgp"], dg=dg_)

    def e2e_serial_step():
        sl = slots[0]
        for dst, src in zip(sl["in"], h_in):
            dst.copy_(src, non_blocking=True)
        compute(sl)
        for dst, src in zip(sl["host"], sl["out"]):
            dst.copy_(src, non_blocking=True)

    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def e2e_pipelined(n, start_event):
        comp_ev, out_ev = [], []
        s_in.wait_event(start_event)
        for i in range(n):
            sl = slots[i % 2]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(comp_ev[i - 2])  # the slot's inputs are free again
                for dst, src in zip(sl["in"], h_in):
                    dst.copy_(src, non_blocking=True)
                ev_in = torch.cuda.Event()
                ev_in.record(s_in)
            stream.wait_event(ev_in)
            if i >= 2:
                stream.wait_event(out_ev[i - 2])     # the slot's results were read back
            compute(sl)
            ev_c = torch.cuda.Event()
            ev_c.record(stream)
            comp_ev.append(ev_c)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_c)
                for dst, src in zip(sl["host"], sl["out"]):
                    dst.copy_(src, non_blocking=True)
                ev_o = torch.cuda.Event()
                ev_o.record(s_out)
                out_ev.append(ev_o)
        stream.wait_stream(s_in)
        stream.wait_stream(s_out)

    # as many steps as the device-resident region, so that filling and
    # draining the pipeline (the first step's uploads, the last step's
    # read-back) weigh as they would in a training run of K steps
    n_e2e = max(3, args.steps)
    e2e_serial_step()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(n_e2e):
        e2e_serial_step()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    ms_e2e_serial = max_over_ranks(e0.elapsed_time(e1) / n_e2e, world, dev)

    warm = torch.cuda.Event()
    warm.record(stream)
    e2e_pipelined(2, warm)
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as e2e_clk:
        e0.record(stream)
        e2e_pipelined(n_e2e, e0)
        e1.record(stream)
        torch.cuda.synchronize()
    barrier()
    ms_e2e = max_over_ranks(e0.elapsed_time(e1) / n_e2e, world, dev)
    e2e_value = job_throughput(flops["fwd_bwd"], world, ms_e2e)
    e2e_serial_value = job_throughput(flops["fwd_bwd"], world, ms_e2e_serial)
    # both buffer slots read back the same bytes (same inputs every step)
    for a_, b_ in zip(slots[1]["host"], slots[0]["host"]):
        if not torch.equal(a_.view(torch.int16) if a_.dtype == torch.bfloat16 else a_.view(torch.int32),
                           b_.view(torch.int16) if b_.dtype == torch.bfloat16 else b_.view(torch.int32)):
            raise RuntimeError("pipelined end-to-end results differ from the serial path")

    # ---- roofline of the dominant kernel ----
    peaks, peak_src = load_peaks()
    work = kernel_work(w)
    traffic = load_traffic(_build.source_hash())
    total_kernel_ms = sum(t for t, _ in kern.values()) or 1.0
    per_kernel = {}
    for name, (tot, n) in kern.items():
        if n == 0:
            continue
        avg_ms = tot / n
        bound, units = work[name]
        if bound == "tensor":
            ach = units / (avg_ms * 1e-3) / 1e12
            peak = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
            unit = "TFLOP/s"
        else:
            ach = units / (avg_ms * 1e-3) / 1e9
            peak = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
            unit = "GB/s"
        per_kernel[name] = {"bound": bound, "avg_ms": round(avg_ms, 4), "launches": n,
                            "share": round(tot / total_kernel_ms, 4), "achieved": round(ach, 2),
                            "peak": peak, "unit": unit, "frac": round(ach / peak, 4)}
    dom = max(per_kernel, key=lambda k: per_kernel[k]["share"])
    d = per_kernel[dom]
    tr = traffic.get(dom)
    roofline = {"kernel": dom, "bound": d["bound"], "achieved": d["achieved"], "peak": d["peak"],
                "unit": d["unit"], "frac": d["frac"], "traffic": tr,
                "peak_source": f"{peak_src} ({'bf16_tflops_sustained' if d['bound'] == 'tensor' else 'hbm_gbs'})",
                "algorithmic_per_launch": work[dom][1]}
    bf16_peak = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    bf16_burst = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])

    # forward and backward apart (sums of the instrumented per-kernel
    # averages), and the step under the dense convention that counts every
    # key, masked or not, as FlashAttention-style reports do
    fwd_names = ("rope_table", "prologue", "attn_fwd")
    bwd_names = ("bwd_pre", "bwd_dkdv", "bwd_dq", "norm_rope_bwd_k", "dg_fold")
    dense_gemm = 2.0 * W.HEAD_DIM * w.S * w.S * w.H * w.B
    phases = {"source": "instrumented region: CUDA events around each launch"}
    for ph, names, fl in (("fwd", fwd_names, flops["fwd"]), ("bwd", bwd_names, flops["bwd"])):
        ms = sum(per_kernel[n]["avg_ms"] for n in names if n in per_kernel)
        phases[ph] = {"ms": round(ms, 4), "credited_gflop": round(fl / 1e9, 2),
                      "tflops": round(fl / (ms * 1e-3) / 1e12, 1) if ms > 0 else None}
    dense = {"fwd_gflop": round(2 * dense_gemm / 1e9, 2), "fwd_bwd_gflop": round(7 * dense_gemm / 1e9, 2),
             "value": round(job_throughput(7 * dense_gemm, world, ms_step), 2), "unit": "TFLOP/s",
             "what": "every key counted (masked text keys included), same timed step as value"}

    clocks = clk.summary()
    unfused = unfused_bwd = None
    if not args.no_unfused:
        fwd_ms = sum(per_kernel[n]["avg_ms"] for n in ("rope_table", "prologue", "attn_fwd") if n in per_kernel)
        unfused = measure_unfused(pkg, ja, w, q, k, v, gains, vl, out, fwd_ms, peaks, max(3, min(args.steps, 10)))
        bwd_ms = sum(per_kernel[n]["avg_ms"] for n in bwd_names if n in per_kernel)
        unfused_bwd = measure_unfused_bwd(pkg, ja, w, q, k, v, do, gains, vl, eager_result[2:], bwd_ms, peaks,
                                          max(3, min(args.steps, 10)))
    qkv = rows23 = None
    if not args.no_unfused:
        qkv = measure_qkv(pkg, w, peaks, max(3, min(args.steps, 20)))
        rows23 = measure_shards_streams(ja, w, q, k, v, do, gains, vl, flops, max(3, min(args.steps, 20)))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank != 0:
        return
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, batch, budget_s=args.cpu_seconds)
    trace = pkg.rlk_joint_attn_trace()
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 inputs, U(0.5,1.5) gains)",
        "pct_of_bf16_peak": round(100.0 * value / world / bf16_peak, 2),
        "pct_of_bf16_peak_basis": f"{peak_src} sustained {bf16_peak} TFLOP/s (burst {bf16_burst})",
        "config": bench_config(w),
        "execution": f"replicas x{world}" if world > 1 else "single GPU",
        "l2": "inputs larger than L2 (no flush): q,k,v,dO total "
              f"{(4 * w.B * w.S * w.H * 128 * 2) / 1e6:.0f} MB, plus ctx and workspace, against 129 MB of L2",
        "roofline": roofline, "kernels": per_kernel, "phases": phases, "dense_convention": dense,
        "workspace": workspace,
        "unfused_forward": unfused, "unfused_backward": unfused_bwd, "qkv_producer": qkv,
        "shards_and_streams": rows23,
        "cpu_baseline": cpu,
        "e2e": {"value": round(e2e_value, 2), "unit": "TFLOP/s", "ms_per_step": round(ms_e2e, 4),
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n_e2e,
                "pipelined": "step i's compute overlaps step i+1's H2D and step i-1's D2H (3 streams, "
                             "double-buffered device buffers)", "clocks": e2e_clk.summary()},
        "e2e_serial": {"value": round(e2e_serial_value, 2), "unit": "TFLOP/s",
                       "ms_per_step": round(ms_e2e_serial, 4)},
        "ms_per_step_instrumented": round(ms_instrumented, 4),
        "graph": {"value": round(job_throughput(flops["fwd_bwd"], world, ms_graph), 2), "unit": "TFLOP/s",
                  "ms_per_step": round(ms_graph, 4), "bytes_equal_to_eager": graph_bytes_equal,
                  "what": "the forward+backward step captured once into a CUDA graph and replayed"},
        "gpu_launches": (LAUNCHES_FIXED + LAUNCHES_PER_GROUP * workspace["groups"]) * args.steps,
        "clocks": clocks,
        "backend": trace["backend"], "fingerprint": trace["fingerprint"],
    }
    print(json.dumps(line))


# ---------------------------------------------------------------- oracle arm
def _oracle_sample(w, batch, rows_per_sample, n_samples, seed=0):
    """Time the CPU oracle on (sample, head, query-row block) samples of w."""
    from oracle import joint_attn as O
    rng = np.random.default_rng(seed)
    g = batch["gains"].astype(np.float64)
    done_flops, t_total = 0.0, 0.0
    for i in range(n_samples):
        b = i % w.B
        h = int(rng.integers(0, w.H))
        r0 = int(rng.integers(0, max(1, w.S - rows_per_sample)))
        rows = np.arange(r0, min(w.S, r0 + rows_per_sample))
        Q = O.widen_bf16(batch["q"][b:b + 1, :, h:h + 1])
        K = O.widen_bf16(batch["k"][b:b + 1, :, h:h + 1])
        V = O.widen_bf16(batch["v"][b:b + 1, :, h:h + 1])
        dO = O.widen_bf16(batch["do"][b:b + 1, :, h:h + 1])
        t0 = time.perf_counter()
        O.pair_rows_forward_backward(Q, K, V, g, dO, w.T_txt, w.grid_h, w.grid_w, batch["valid_len"][b],
                                     0, 0, rows)
        t_total += time.perf_counter() - t0
        done_flops += 7 * 2.0 * W.HEAD_DIM * len(rows) * (w.T_img + int(batch["valid_len"][b]))
    return done_flops, t_total


def cpu_model() -> str:
    """The host CPU's model name as lscpu prints it, else the machine type."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.machine()


def oracle_one_thread(w, timeout_s: float = 180.0):
    """One full (sample, head) pair of w through the oracle with BLAS held to
    one thread. It runs in a child process, since a BLAS library fixes its
    thread count when numpy loads it."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-one-thread", "--workload", w.name]
    try:
        r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=timeout_s)
        res = json.loads(r.stdout.strip().splitlines()[-1])
    except (OSError, subprocess.SubprocessError, ValueError, IndexError) as e:
        return {"value": None, "error": type(e).__name__}
    res.update(unit="TFLOP/s", cores=1,
               sample=f"one full (sample, head) pair of {w.name}, forward+backward, BLAS on one thread")
    return res


def _one_thread_child(w):
    batch = W.make_batch(w, seed=0, rows=[0], valid_len=[w.valid_len[0]])  # sample 0 only
    fl, t = _oracle_sample(w, batch, w.S, 1)
    print(json.dumps({"value": round(fl / t / 1e12, 6), "seconds": round(t, 3)}))


def cpu_baseline(w, batch, budget_s=20.0):
    """The oracle as it stands, on the host cores, then one pair on one thread.

    At the 1024^2 CFG pair: full (sample, head) pairs of the workload until
    about ``budget_s`` seconds of work are done. At the larger shapes: every
    sample's heads 0 and H-1 (forward + backward each), the time per head
    scaled to all H heads and labelled as extrapolated."""
    if w.name == "cfg1024":
        fl, t = _oracle_sample(w, batch, w.S, 1)
        n = 1
        while t < budget_s and n < 2 * w.B * w.H:
            f2, t2 = _oracle_sample(w, batch, w.S, 1, seed=n)
            fl += f2
            t += t2
            n += 1
        res = {"value": round(fl / t / 1e12, 6), "extrapolated": False,
               "sample": f"{n} full (sample, head) pairs of {w.name}, forward+backward, float64 numpy "
                         f"(BLAS threads = host cores); credited flops of the sample / wall time"}
    else:
        heads = [0, w.H - 1] if w.H > 2 else list(range(w.H))
        fl, t = _oracle_pairs(w, batch, heads)
        per_head_s = t / len(heads)
        full_s = per_head_s * w.H
        full_flops = W.credited_flops(w)["fwd_bwd"]
        res = {"value": round(full_flops / full_s / 1e12, 6), "extrapolated": len(heads) < w.H,
               "measured_seconds": round(t, 3), "seconds_per_head": round(per_head_s, 3),
               "extrapolated_step_seconds": round(full_s, 2),
               "measured_value": round(fl / t / 1e12, 6),
               "sample": f"heads {heads} of every sample of {w.name} (all {w.B} samples, forward+backward, "
                         f"float64 numpy, BLAS threads = host cores); the time per head x {w.H} heads is the "
                         f"extrapolated step time, value = credited flops of the whole step / that time"}
    res.update({"unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle", "cpu_model": cpu_model(),
                "one_thread": oracle_one_thread(w)})
    return res


def _oracle_pairs(w, batch, heads):
    """Time the CPU oracle on full (sample, head) pairs: every sample of w,
    the given heads; returns (credited flops, seconds)."""
    from oracle import joint_attn as O
    g = batch["gains"].astype(np.float64)
    done_flops, t_total = 0.0, 0.0
    for b in range(w.B):
        for h in heads:
            Q, K, V, dO = (O.widen_bf16(batch[n][b:b + 1, :, h:h + 1]) for n in ("q", "k", "v", "do"))
            t0 = time.perf_counter()
            O.pair_rows_forward_backward(Q, K, V, g, dO, w.T_txt, w.grid_h, w.grid_w, batch["valid_len"][b],
                                         0, 0, np.arange(w.S))
            t_total += time.perf_counter() - t0
            done_flops += 7 * 2.0 * W.HEAD_DIM * w.S * (w.T_img + int(batch["valid_len"][b]))
    return done_flops, t_total


def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return
    w = selected_workload(args)
    batch = W.make_batch(w, seed=0)
    # size each step so the whole run stays within about two minutes
    per_step_budget = 120.0 / max(1, args.steps + args.warmup)
    f1, t1 = _oracle_sample(w, batch, 64, 1)
    rows = int(max(16, min(w.S, 64 * per_step_budget / max(t1, 1e-3))))
    for i in range(args.warmup):
        _oracle_sample(w, batch, rows, 1, seed=1000 + i)
    fl_tot, t_tot = 0.0, 0.0
    for i in range(args.steps):
        f, t = _oracle_sample(w, batch, rows, 1, seed=i)
        fl_tot += f
        t_tot += t
    value = fl_tot / t_tot / 1e12
    sample = (f"each step: forward+backward of {rows} consecutive query rows of one (sample, head) "
              f"pair of {w.name} against all keys, float64 numpy oracle")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * t_tot / args.steps, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": bench_config(w),
        "execution": "host cores",
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": os.cpu_count(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(W.WORKLOADS), default="cfg1024")
    ap.add_argument("--heads", type=int, default=None,
                    help="run the workload's shape on this many heads (a reduced profiling case)")
    ap.add_argument("--ws-budget-gb", type=float, default=None,
                    help="cap the backward workspace (the backward then runs its (sample, head) pairs in groups)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-unfused", action="store_true",
                    help="skip timing the standalone operators and the QKV producer")
    ap.add_argument("--oracle-one-thread", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.oracle_one_thread:
        _one_thread_child(W.WORKLOADS[args.workload])
        return
    if args.impl == "ours":
        args.warmup = max(3, args.warmup)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

"""Deterministic, batch-invariant joint attention of a Qwen-Image MMDiT block
(forward and backward, with the QK-RMSNorm + three-axis RoPE prologue) for one
NVIDIA GB300.

This module is a thin binding over the C ABI of ``librlk_joint_attn.so``
(declared in ``include/rlk_joint_attn.h``): it marshals arguments and checks
shapes so that no bad pointer reaches the library. Every step of the path runs
in the library's CUDA kernels; there is no CPU or PyTorch fallback. If the
library is missing, loading it raises.

PyTorch is used only for device memory and streams.
"""

from __future__ import annotations

import ctypes
import os
from typing import Sequence

__all__ = [
    "Shape", "RlkError", "lib", "library_path", "load_library",
    "rlk_joint_attn_ctx_bytes", "rlk_joint_attn_bwd_workspace_bytes", "rlk_joint_attn_bwd_workspace_min_bytes",
    "rlk_joint_attn_fwd", "rlk_joint_attn_bwd", "rlk_joint_attn_check_status",
    "rlk_strict_math_compiled", "rlk_joint_attn_trace", "rlk_strerror",
    "rlk_kernel_timing", "rlk_kernel_timing_read", "rlk_joint_attn_fwd_noalloc",
    "rlk_joint_attn_unfused_bytes", "rlk_qk_norm_rope", "rlk_joint_attn_qk_gemm",
    "rlk_joint_attn_softmax", "rlk_joint_attn_av_gemm", "UNFUSED", "JointAttention",
    "rlk_op_trace_enable", "rlk_op_trace_count", "rlk_op_trace_read", "op_trace", "OP_TRACE_CAP",
    "rlk_joint_attn_state_bytes", "rlk_joint_attn_fwd_shard", "rlk_joint_attn_fwd_streams",
    "rlk_joint_attn_bwd_streams", "rlk_qkv_bias_gemm", "rlk_joint_attn_fwd_ctx",
    "rlk_attn_out_bias_gemm", "rlk_selftest_wait_timeout", "rlk_fwd_tile_schedule", "FWD_TILES",
    "rlk_joint_attn_bwd_stats", "rlk_joint_attn_softmax_bwd", "rlk_joint_attn_av_gemm_bwd",
    "rlk_joint_attn_qk_gemm_bwd", "rlk_qk_norm_rope_bwd",
    "EXPORTED_SYMBOLS", "KERNEL_IDS",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_NAME = "librlk_joint_attn.so"
HEAD_DIM = 128
AXES = (16, 56, 56)
MAX_BATCH = 256

RLK_OK = 0
STATUS_NAMES = {
    0: "RLK_OK", 1: "RLK_ERR_INVALID_ARG", 2: "RLK_ERR_UNSUPPORTED", 3: "RLK_ERR_ALIGNMENT",
    4: "RLK_ERR_WORKSPACE", 5: "RLK_ERR_CUDA", 6: "RLK_ERR_DEVICE_TIMEOUT",
}
KERNEL_IDS = {
    "rope_table": 0, "prologue": 1, "attn_fwd": 2, "bwd_pre": 3,
    "bwd_dkdv": 4, "bwd_dq": 5, "norm_rope_bwd_k": 6, "dg_fold": 7,
    "qk_gemm": 8, "softmax": 9, "av_gemm": 10, "attn_fwd_shard": 11, "qkv_gemm": 12, "out_gemm": 13,
    "dp_gemm": 14, "softmax_bwd": 15, "key_gemm": 16, "query_gemm": 17, "norm_rope_bwd_q": 18,
}
# which intermediate rlk_joint_attn_unfused_bytes() sizes
UNFUSED = {"scores": 0, "p": 1, "alpha": 2, "rows": 3, "dp": 4, "ds": 5, "stats": 6, "dhat": 7, "gain_tiles": 8}
# Every symbol include/rlk_joint_attn.h declares.
EXPORTED_SYMBOLS = (
    "rlk_joint_attn_ctx_bytes", "rlk_joint_attn_bwd_workspace_bytes", "rlk_joint_attn_bwd_workspace_min_bytes",
    "rlk_joint_attn_fwd", "rlk_joint_attn_bwd", "rlk_joint_attn_check_status",
    "rlk_strict_math_compiled", "rlk_joint_attn_trace", "rlk_strerror",
    "rlk_kernel_timing", "rlk_kernel_timing_read", "rlk_joint_attn_fwd_noalloc",
    "rlk_joint_attn_unfused_bytes", "rlk_qk_norm_rope", "rlk_joint_attn_qk_gemm",
    "rlk_joint_attn_softmax", "rlk_joint_attn_av_gemm",
    "rlk_op_trace_enable", "rlk_op_trace_count", "rlk_op_trace_read",
    "rlk_joint_attn_state_bytes", "rlk_joint_attn_fwd_shard",
    "rlk_joint_attn_fwd_streams", "rlk_joint_attn_bwd_streams", "rlk_qkv_bias_gemm",
    "rlk_joint_attn_fwd_ctx", "rlk_attn_out_bias_gemm", "rlk_selftest_wait_timeout",
    "rlk_fwd_tile_schedule",
    "rlk_joint_attn_bwd_stats", "rlk_joint_attn_softmax_bwd", "rlk_joint_attn_av_gemm_bwd",
    "rlk_joint_attn_qk_gemm_bwd", "rlk_qk_norm_rope_bwd",
)
OP_TRACE_CAP = 256
OP_TRACE_MAX_KERNELS = 8


class Shape(ctypes.Structure):
    """rlk_ja_shape."""
    _fields_ = [
        ("B", ctypes.c_int32), ("T_txt", ctypes.c_int32), ("grid_h", ctypes.c_int32),
        ("grid_w", ctypes.c_int32), ("H", ctypes.c_int32), ("D", ctypes.c_int32),
        ("eps", ctypes.c_float), ("theta", ctypes.c_float), ("axes", ctypes.c_int32 * 3),
    ]

    @classmethod
    def make(cls, B, T_txt, grid_h, grid_w, H, D=HEAD_DIM, eps=1e-6, theta=10000.0, axes=AXES):
        s = cls()
        s.B, s.T_txt, s.grid_h, s.grid_w, s.H, s.D = B, T_txt, grid_h, grid_w, H, D
        s.eps, s.theta = eps, theta
        s.axes[0], s.axes[1], s.axes[2] = axes
        return s

    @property
    def S(self) -> int:
        return self.T_txt + self.grid_h * self.grid_w


class Trace(ctypes.Structure):
    """rlk_ja_trace."""
    _fields_ = [
        ("backend", ctypes.c_char * 32), ("reduction_order", ctypes.c_char * 160),
        ("accumulator", ctypes.c_char * 16), ("split_k", ctypes.c_int32),
        ("atomics", ctypes.c_int32), ("tf32", ctypes.c_int32), ("strict_math", ctypes.c_int32),
        ("block_q", ctypes.c_int32), ("block_kv", ctypes.c_int32),
        ("fingerprint", ctypes.c_char * 96),
    ]


class RlkError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)} ({_strerror(code)})")


class OpRecord(ctypes.Structure):
    """rlk_op_record: one operator-trace record."""
    _fields_ = [
        ("seq", ctypes.c_uint64), ("op", ctypes.c_char * 48), ("entry_point", ctypes.c_char * 40),
        ("requested_backend", ctypes.c_char * 24), ("actual_backend", ctypes.c_char * 24),
        ("status", ctypes.c_int32), ("fallback", ctypes.c_int32), ("split_k", ctypes.c_int32),
        ("atomics", ctypes.c_int32), ("tf32", ctypes.c_int32), ("n_kernels", ctypes.c_int32),
        ("kernels", (ctypes.c_char * 32) * OP_TRACE_MAX_KERNELS), ("kernel_fingerprint", ctypes.c_char * 96),
        ("accumulator", ctypes.c_char * 16), ("arithmetic_policy", ctypes.c_char * 192),
        ("reduction_order", ctypes.c_char * 160), ("B", ctypes.c_int32), ("H", ctypes.c_int32),
        ("T_txt", ctypes.c_int32), ("grid_h", ctypes.c_int32), ("grid_w", ctypes.c_int32),
    ]

    def to_dict(self) -> dict:
        d = {}
        for f, _ in self._fields_:
            v = getattr(self, f)
            if f == "kernels":
                d[f] = [v[i].value.decode() for i in range(self.n_kernels)]
            elif isinstance(v, bytes):
                d[f] = v.decode()
            else:
                d[f] = v
        return d


_lib = None


def library_path() -> str:
    return os.path.join(_PKG, LIB_NAME)


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load a build of the library and declare its signatures."""
    path = path or library_path()
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`. "
            "There is no fallback implementation.")
    L = ctypes.CDLL(path)
    vp, sz, i32, f32p = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.POINTER(ctypes.c_float)
    shp = ctypes.POINTER(Shape)
    L.rlk_joint_attn_ctx_bytes.argtypes = [shp]
    L.rlk_joint_attn_ctx_bytes.restype = sz
    L.rlk_joint_attn_bwd_workspace_bytes.argtypes = [shp]
    L.rlk_joint_attn_bwd_workspace_bytes.restype = sz
    L.rlk_joint_attn_bwd_workspace_min_bytes.argtypes = [shp]
    L.rlk_joint_attn_bwd_workspace_min_bytes.restype = sz
    L.rlk_joint_attn_fwd.argtypes = [shp, vp, vp, vp, vp, vp, vp, vp, ctypes.POINTER(ctypes.c_int32),
                                     vp, vp, vp, vp]
    L.rlk_joint_attn_fwd.restype = i32
    L.rlk_joint_attn_bwd.argtypes = [shp, vp, vp, vp, vp, vp, vp, vp, ctypes.POINTER(ctypes.c_int32),
                                     vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.rlk_joint_attn_bwd.restype = i32
    L.rlk_joint_attn_check_status.argtypes = [vp]
    L.rlk_joint_attn_check_status.restype = i32
    L.rlk_strict_math_compiled.argtypes = []
    L.rlk_strict_math_compiled.restype = i32
    L.rlk_selftest_wait_timeout.argtypes = [i32, vp]
    L.rlk_selftest_wait_timeout.restype = i32
    L.rlk_fwd_tile_schedule.argtypes = [i32]
    L.rlk_fwd_tile_schedule.restype = i32
    L.rlk_joint_attn_trace.argtypes = [ctypes.POINTER(Trace)]
    L.rlk_joint_attn_trace.restype = i32
    L.rlk_strerror.argtypes = [i32]
    L.rlk_strerror.restype = ctypes.c_char_p
    L.rlk_kernel_timing.argtypes = [i32]
    L.rlk_kernel_timing.restype = i32
    L.rlk_kernel_timing_read.argtypes = [i32, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int32)]
    L.rlk_kernel_timing_read.restype = i32
    L.rlk_joint_attn_fwd_noalloc.argtypes = [shp, vp, vp, vp, vp, vp, vp, vp, ctypes.POINTER(ctypes.c_int32),
                                             vp, vp, vp]
    L.rlk_joint_attn_fwd_noalloc.restype = i32
    L.rlk_joint_attn_unfused_bytes.argtypes = [shp, i32]
    L.rlk_joint_attn_unfused_bytes.restype = sz
    L.rlk_qk_norm_rope.argtypes = [shp, vp, vp, vp, vp, vp, vp, vp, vp]
    L.rlk_qk_norm_rope.restype = i32
    i32p = ctypes.POINTER(ctypes.c_int32)
    L.rlk_joint_attn_qk_gemm.argtypes = [shp, vp, i32p, vp, vp]
    L.rlk_joint_attn_qk_gemm.restype = i32
    L.rlk_joint_attn_softmax.argtypes = [shp, vp, i32p, vp, vp, vp, vp, vp]
    L.rlk_joint_attn_softmax.restype = i32
    L.rlk_joint_attn_av_gemm.argtypes = [shp, vp, vp, vp, vp, i32p, vp, vp]
    L.rlk_joint_attn_av_gemm.restype = i32
    L.rlk_joint_attn_bwd_stats.argtypes = [shp, vp, vp, vp, vp, vp]
    L.rlk_joint_attn_bwd_stats.restype = i32
    L.rlk_joint_attn_softmax_bwd.argtypes = [shp, vp, vp, vp, i32p, vp, vp, vp]
    L.rlk_joint_attn_softmax_bwd.restype = i32
    L.rlk_joint_attn_av_gemm_bwd.argtypes = [shp, vp, vp, vp, i32p, vp, vp, vp]
    L.rlk_joint_attn_av_gemm_bwd.restype = i32
    L.rlk_joint_attn_qk_gemm_bwd.argtypes = [shp, vp, vp, i32p, vp, vp, vp]
    L.rlk_joint_attn_qk_gemm_bwd.restype = i32
    L.rlk_qk_norm_rope_bwd.argtypes = [shp] + [vp] * 15
    L.rlk_qk_norm_rope_bwd.restype = i32
    L.rlk_joint_attn_state_bytes.argtypes = [shp]
    L.rlk_joint_attn_state_bytes.restype = sz
    L.rlk_joint_attn_fwd_shard.argtypes = [shp, vp, vp, i32p, ctypes.c_int32, ctypes.c_int32, vp, vp, vp, vp, vp]
    L.rlk_joint_attn_fwd_shard.restype = i32
    L.rlk_joint_attn_fwd_streams.argtypes = [shp] + [vp] * 10 + [i32p] + [vp] * 5
    L.rlk_joint_attn_fwd_streams.restype = i32
    L.rlk_joint_attn_bwd_streams.argtypes = [shp] + [vp] * 10 + [i32p] + [vp] * 14 + [sz, vp]
    L.rlk_joint_attn_bwd_streams.restype = i32
    L.rlk_qkv_bias_gemm.argtypes = [shp] + [vp] * 18
    L.rlk_qkv_bias_gemm.restype = i32
    L.rlk_joint_attn_fwd_ctx.argtypes = [shp, vp, vp, vp, i32p, vp, vp, vp, vp]
    L.rlk_joint_attn_fwd_ctx.restype = i32
    L.rlk_attn_out_bias_gemm.argtypes = [shp] + [vp] * 9
    L.rlk_attn_out_bias_gemm.restype = i32
    L.rlk_op_trace_enable.argtypes = [i32]
    L.rlk_op_trace_enable.restype = i32
    L.rlk_op_trace_count.argtypes = []
    L.rlk_op_trace_count.restype = ctypes.c_int32
    L.rlk_op_trace_read.argtypes = [ctypes.c_int32, ctypes.POINTER(OpRecord)]
    L.rlk_op_trace_read.restype = i32
    return L


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = load_library()
    return _lib


def _strerror(code: int) -> str:
    try:
        return lib().rlk_strerror(code).decode()
    except Exception:  # the library itself failed to load
        return "?"


def _check(code: int, where: str) -> None:
    if code != RLK_OK:
        raise RlkError(code, where)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream_handle(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _lengths(valid_len: Sequence[int], shape: Shape):
    """The host array of valid text lengths the C ABI reads: exactly B of
    them (the library reads B entries, so a shorter list is refused here)."""
    vals = [int(x) for x in valid_len]
    if len(vals) != shape.B:
        raise ValueError(f"expected {shape.B} valid text lengths (one per sample), got {len(vals)}")
    return (ctypes.c_int32 * max(1, len(vals)))(*vals)


def rlk_joint_attn_ctx_bytes(shape: Shape) -> int:
    return int(lib().rlk_joint_attn_ctx_bytes(ctypes.byref(shape)))


def rlk_joint_attn_bwd_workspace_bytes(shape: Shape) -> int:
    return int(lib().rlk_joint_attn_bwd_workspace_bytes(ctypes.byref(shape)))


def rlk_joint_attn_bwd_workspace_min_bytes(shape: Shape) -> int:
    return int(lib().rlk_joint_attn_bwd_workspace_min_bytes(ctypes.byref(shape)))


def rlk_joint_attn_fwd(shape, q, k, v, g_q_txt, g_k_txt, g_q_img, g_k_img, txt_valid_len,
                       out, lse, ctx, stream=None) -> None:
    """Enqueue the forward; tensors or raw device pointers (ints)."""
    rc = lib().rlk_joint_attn_fwd(
        ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g_q_txt), _ptr(g_k_txt),
        _ptr(g_q_img), _ptr(g_k_img), _lengths(txt_valid_len, shape), _ptr(out), _ptr(lse), _ptr(ctx),
        _stream_handle(stream))
    _check(rc, "rlk_joint_attn_fwd")


def rlk_joint_attn_fwd_noalloc(shape, q, k, v, g_q_txt, g_k_txt, g_q_img, g_k_img, txt_valid_len,
                               out, lse, stream=None) -> None:
    """Enqueue the forward with the library's built-in device scratch (for
    callers that cannot allocate); forward-only, calls must not overlap."""
    rc = lib().rlk_joint_attn_fwd_noalloc(
        ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g_q_txt), _ptr(g_k_txt),
        _ptr(g_q_img), _ptr(g_k_img), _lengths(txt_valid_len, shape), _ptr(out), _ptr(lse),
        _stream_handle(stream))
    _check(rc, "rlk_joint_attn_fwd_noalloc")


def rlk_joint_attn_bwd(shape, q, k, v, g_q_txt, g_k_txt, g_q_img, g_k_img, txt_valid_len,
                       out, dout, lse, ctx, dq, dk, dv, dg_partial, dg, workspace,
                       workspace_bytes=None, stream=None) -> None:
    """Enqueue the backward; tensors or raw device pointers (ints)."""
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    rc = lib().rlk_joint_attn_bwd(
        ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g_q_txt), _ptr(g_k_txt),
        _ptr(g_q_img), _ptr(g_k_img), _lengths(txt_valid_len, shape), _ptr(out), _ptr(dout), _ptr(lse),
        _ptr(ctx), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg_partial), _ptr(dg), _ptr(workspace),
        int(workspace_bytes), _stream_handle(stream))
    _check(rc, "rlk_joint_attn_bwd")


def rlk_joint_attn_unfused_bytes(shape: Shape, which: str | int) -> int:
    w = UNFUSED[which] if isinstance(which, str) else int(which)
    return int(lib().rlk_joint_attn_unfused_bytes(ctypes.byref(shape), w))


def rlk_qk_norm_rope(shape, q, k, g_q_txt, g_k_txt, g_q_img, g_k_img, ctx, stream=None) -> None:
    """Enqueue qk_rmsnorm + multi_axis_rope into ctx."""
    rc = lib().rlk_qk_norm_rope(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(g_q_txt), _ptr(g_k_txt),
                                _ptr(g_q_img), _ptr(g_k_img), _ptr(ctx), _stream_handle(stream))
    _check(rc, "rlk_qk_norm_rope")


def rlk_joint_attn_qk_gemm(shape, ctx, txt_valid_len, scores, stream=None) -> None:
    rc = lib().rlk_joint_attn_qk_gemm(ctypes.byref(shape), _ptr(ctx), _lengths(txt_valid_len, shape), _ptr(scores),
                                      _stream_handle(stream))
    _check(rc, "rlk_joint_attn_qk_gemm")


def rlk_joint_attn_softmax(shape, scores, txt_valid_len, p, alpha, l, lse, stream=None) -> None:
    rc = lib().rlk_joint_attn_softmax(ctypes.byref(shape), _ptr(scores), _lengths(txt_valid_len, shape), _ptr(p),
                                      _ptr(alpha), _ptr(l), _ptr(lse), _stream_handle(stream))
    _check(rc, "rlk_joint_attn_softmax")


def rlk_joint_attn_av_gemm(shape, p, alpha, l, v, txt_valid_len, out, stream=None) -> None:
    rc = lib().rlk_joint_attn_av_gemm(ctypes.byref(shape), _ptr(p), _ptr(alpha), _ptr(l), _ptr(v),
                                      _lengths(txt_valid_len, shape), _ptr(out), _stream_handle(stream))
    _check(rc, "rlk_joint_attn_av_gemm")


def rlk_joint_attn_bwd_stats(shape, out, dout, lse, stats, stream=None) -> None:
    _check(lib().rlk_joint_attn_bwd_stats(ctypes.byref(shape), _ptr(out), _ptr(dout), _ptr(lse), _ptr(stats),
                                          _stream_handle(stream)), "rlk_joint_attn_bwd_stats")


def rlk_joint_attn_softmax_bwd(shape, scores, stats, dp, txt_valid_len, p, ds, stream=None) -> None:
    _check(lib().rlk_joint_attn_softmax_bwd(ctypes.byref(shape), _ptr(scores), _ptr(stats), _ptr(dp),
                                            _lengths(txt_valid_len, shape), _ptr(p), _ptr(ds),
                                            _stream_handle(stream)), "rlk_joint_attn_softmax_bwd")


def rlk_joint_attn_av_gemm_bwd(shape, p, v, dout, txt_valid_len, dv, dp, stream=None) -> None:
    _check(lib().rlk_joint_attn_av_gemm_bwd(ctypes.byref(shape), _ptr(p), _ptr(v), _ptr(dout),
                                            _lengths(txt_valid_len, shape), _ptr(dv), _ptr(dp),
                                            _stream_handle(stream)), "rlk_joint_attn_av_gemm_bwd")


def rlk_joint_attn_qk_gemm_bwd(shape, ds, ctx, txt_valid_len, dqh, dkh, stream=None) -> None:
    _check(lib().rlk_joint_attn_qk_gemm_bwd(ctypes.byref(shape), _ptr(ds), _ptr(ctx),
                                            _lengths(txt_valid_len, shape), _ptr(dqh), _ptr(dkh),
                                            _stream_handle(stream)), "rlk_joint_attn_qk_gemm_bwd")


def rlk_qk_norm_rope_bwd(shape, q, k, g_q_txt, g_k_txt, g_q_img, g_k_img, ctx, dqh, dkh, dq, dk, dg_partial, dg,
                         gain_tiles, stream=None) -> None:
    _check(lib().rlk_qk_norm_rope_bwd(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(g_q_txt), _ptr(g_k_txt),
                                      _ptr(g_q_img), _ptr(g_k_img), _ptr(ctx), _ptr(dqh), _ptr(dkh), _ptr(dq),
                                      _ptr(dk), _ptr(dg_partial), _ptr(dg), _ptr(gain_tiles),
                                      _stream_handle(stream)), "rlk_qk_norm_rope_bwd")


def rlk_joint_attn_state_bytes(shape: Shape) -> int:
    return int(lib().rlk_joint_attn_state_bytes(ctypes.byref(shape)))


def rlk_joint_attn_fwd_shard(shape, ctx, v, txt_valid_len, blk_begin, blk_end, state_in, state_out, out, lse,
                             stream=None) -> None:
    """Enqueue the forward over key column blocks [blk_begin, blk_end),
    handing the online-softmax state on (see the header)."""
    rc = lib().rlk_joint_attn_fwd_shard(ctypes.byref(shape), _ptr(ctx), _ptr(v), _lengths(txt_valid_len, shape),
                                        int(blk_begin), int(blk_end), _ptr(state_in), _ptr(state_out), _ptr(out),
                                        _ptr(lse), _stream_handle(stream))
    _check(rc, "rlk_joint_attn_fwd_shard")


def rlk_joint_attn_fwd_streams(shape, q, k, v, g_q_txt, g_k_txt, g_q_img, g_k_img, txt_valid_len, out, lse, ctx,
                               stream=None) -> None:
    """Forward on separate streams: q, k, v and out are (text, image) pairs
    of tensors or device pointers (the text one may be None if T_txt == 0)."""
    args = [_ptr(x) for pair in (q, k, v) for x in pair]
    rc = lib().rlk_joint_attn_fwd_streams(
        ctypes.byref(shape), *args, _ptr(g_q_txt), _ptr(g_k_txt), _ptr(g_q_img), _ptr(g_k_img),
        _lengths(txt_valid_len, shape), _ptr(out[0]), _ptr(out[1]), _ptr(lse), _ptr(ctx), _stream_handle(stream))
    _check(rc, "rlk_joint_attn_fwd_streams")


def rlk_joint_attn_bwd_streams(shape, q, k, v, g_q_txt, g_k_txt, g_q_img, g_k_img, txt_valid_len, out, dout, lse,
                               ctx, dq, dk, dv, dg_partial, dg, workspace, workspace_bytes=None, stream=None) -> None:
    """Backward on separate streams; activations as (text, image) pairs."""
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    ins = [_ptr(x) for pair in (q, k, v) for x in pair]
    rc = lib().rlk_joint_attn_bwd_streams(
        ctypes.byref(shape), *ins, _ptr(g_q_txt), _ptr(g_k_txt), _ptr(g_q_img), _ptr(g_k_img),
        _lengths(txt_valid_len, shape), _ptr(out[0]), _ptr(out[1]), _ptr(dout[0]), _ptr(dout[1]), _ptr(lse), _ptr(ctx),
        _ptr(dq[0]), _ptr(dq[1]), _ptr(dk[0]), _ptr(dk[1]), _ptr(dv[0]), _ptr(dv[1]), _ptr(dg_partial), _ptr(dg),
        _ptr(workspace), int(workspace_bytes), _stream_handle(stream))
    _check(rc, "rlk_joint_attn_bwd_streams")


def rlk_qkv_bias_gemm(shape, x, w, b, gains, ctx, q, k, v, stream=None) -> None:
    """Per-stream QKV projection; x, w, b, q, k, v are (text, image) pairs
    (q, k may be (None, None) when ctx is given); gains a [4, 128] tensor or
    None (plain mode, ctx None)."""
    g = [None] * 4 if gains is None else [gains[0], gains[1], gains[2], gains[3]]
    rc = lib().rlk_qkv_bias_gemm(
        ctypes.byref(shape), _ptr(x[0]), _ptr(x[1]), _ptr(w[0]), _ptr(w[1]), _ptr(b[0]), _ptr(b[1]),
        *[_ptr(t) for t in g], _ptr(ctx), _ptr(q[0]), _ptr(q[1]), _ptr(k[0]), _ptr(k[1]), _ptr(v[0]), _ptr(v[1]),
        _stream_handle(stream))
    _check(rc, "rlk_qkv_bias_gemm")


def rlk_joint_attn_fwd_ctx(shape, ctx, v, txt_valid_len, out, lse, stream=None) -> None:
    """Attention from a prepared context; v and out are (text, image) pairs."""
    rc = lib().rlk_joint_attn_fwd_ctx(ctypes.byref(shape), _ptr(ctx), _ptr(v[0]), _ptr(v[1]),
                                      _lengths(txt_valid_len, shape), _ptr(out[0]), _ptr(out[1]), _ptr(lse),
                                      _stream_handle(stream))
    _check(rc, "rlk_joint_attn_fwd_ctx")


def rlk_attn_out_bias_gemm(shape, o, w, b, y, stream=None) -> None:
    """Per-stream output projection; o, w, b, y are (text, image) pairs."""
    rc = lib().rlk_attn_out_bias_gemm(ctypes.byref(shape), _ptr(o[0]), _ptr(o[1]), _ptr(w[0]), _ptr(w[1]),
                                      _ptr(b[0]), _ptr(b[1]), _ptr(y[0]), _ptr(y[1]), _stream_handle(stream))
    _check(rc, "rlk_attn_out_bias_gemm")


def rlk_op_trace_enable(enable: bool) -> None:
    _check(lib().rlk_op_trace_enable(1 if enable else 0), "rlk_op_trace_enable")


def rlk_op_trace_count() -> int:
    return int(lib().rlk_op_trace_count())


def rlk_op_trace_read() -> list[dict]:
    """Every record kept, oldest first, as dicts."""
    out = []
    for i in range(rlk_op_trace_count()):
        r = OpRecord()
        _check(lib().rlk_op_trace_read(i, ctypes.byref(r)), "rlk_op_trace_read")
        out.append(r.to_dict())
    return out


class op_trace:
    """Context manager: records every library call made inside it.
    ``with op_trace() as t: ...``; afterwards ``t.records`` holds the records."""

    def __enter__(self):
        rlk_op_trace_enable(True)
        self.records = []
        return self

    def __exit__(self, *exc):
        self.records = rlk_op_trace_read()
        rlk_op_trace_enable(False)
        return False


def rlk_joint_attn_check_status(stream=None) -> None:
    _check(lib().rlk_joint_attn_check_status(_stream_handle(stream)), "rlk_joint_attn_check_status")


def rlk_strict_math_compiled() -> int:
    return int(lib().rlk_strict_math_compiled())


def rlk_selftest_wait_timeout(limit_ms: int, stream=None) -> None:
    """Enqueue one warp whose bounded wait on a barrier nothing completes
    gives up after limit_ms: the next rlk_joint_attn_check_status() raises
    RlkError(RLK_ERR_DEVICE_TIMEOUT)."""
    _check(lib().rlk_selftest_wait_timeout(int(limit_ms), _stream_handle(stream)), "rlk_selftest_wait_timeout")


def rlk_joint_attn_trace() -> dict:
    t = Trace()
    _check(lib().rlk_joint_attn_trace(ctypes.byref(t)), "rlk_joint_attn_trace")
    return {f: (getattr(t, f).decode() if isinstance(getattr(t, f), bytes) else getattr(t, f))
            for f, _ in Trace._fields_}


FWD_TILES = {"auto": 0, "pairs": 1, "single": 2}


def rlk_fwd_tile_schedule(policy: str) -> str:
    """Set the fused forward's query-tile schedule ("auto", "pairs" or
    "single"; time only, never bytes); returns the previous one."""
    if policy not in FWD_TILES:
        raise ValueError(f"unknown tile schedule {policy!r}")
    prev = lib().rlk_fwd_tile_schedule(FWD_TILES[policy])
    if prev < 0:
        raise RuntimeError("rlk_fwd_tile_schedule refused the policy")
    return {v: k for k, v in FWD_TILES.items()}[prev]


def rlk_strerror(code: int) -> str:
    return _strerror(code)


def rlk_kernel_timing(enable: bool) -> None:
    _check(lib().rlk_kernel_timing(1 if enable else 0), "rlk_kernel_timing")


def rlk_kernel_timing_read(kernel: str | int) -> tuple[float, int]:
    kid = KERNEL_IDS[kernel] if isinstance(kernel, str) else int(kernel)
    ms, n = ctypes.c_double(), ctypes.c_int32()
    _check(lib().rlk_kernel_timing_read(kid, ctypes.byref(ms), ctypes.byref(n)), "rlk_kernel_timing_read")
    return ms.value, n.value


class JointAttention:
    """Buffers + calls for one geometry: allocates the caller-owned tensors
    with PyTorch and passes them to the C ABI. Inputs are bf16 [B, S, H, 128]
    CUDA tensors; gains a float32 [4, 128] tensor (q_txt, k_txt, q_img, k_img)."""

    def __init__(self, B: int, T_txt: int, grid_h: int, grid_w: int, H: int, device="cuda",
                 eps: float = 1e-6, theta: float = 10000.0, ws_budget_bytes: int | None = None):
        """ws_budget_bytes caps the backward workspace: with less than the
        full size the backward runs its (sample, head) pairs in groups (same
        bytes, more launches); below the minimum it raises."""
        import torch
        self.shape = Shape.make(B, T_txt, grid_h, grid_w, H, eps=eps, theta=theta)
        self.device = torch.device(device)
        n_ctx = rlk_joint_attn_ctx_bytes(self.shape)
        n_ws = rlk_joint_attn_bwd_workspace_bytes(self.shape)
        if n_ctx == 0 or n_ws == 0:
            raise RlkError(1, "JointAttention: invalid shape")
        if ws_budget_bytes is not None:
            n_min = rlk_joint_attn_bwd_workspace_min_bytes(self.shape)
            if ws_budget_bytes < n_min:
                raise RlkError(4, f"JointAttention: workspace budget {ws_budget_bytes} below the minimum {n_min}")
            n_ws = min(n_ws, int(ws_budget_bytes))
        self.ctx = torch.empty(n_ctx, dtype=torch.uint8, device=self.device)
        self.workspace = torch.empty(n_ws, dtype=torch.uint8, device=self.device)

    def _check_inputs(self, *ts):
        import torch
        sh = self.shape
        want = (sh.B, sh.S, sh.H, HEAD_DIM)
        for t in ts:
            if t.dtype != torch.bfloat16 or tuple(t.shape) != want or not t.is_contiguous() or t.device != self.device:
                raise ValueError(f"expected contiguous bf16 {want} on {self.device}, got {t.dtype} "
                                 f"{tuple(t.shape)} on {t.device}")

    def _check_f32(self, t, want, name):
        import torch
        if t.dtype != torch.float32 or tuple(t.shape) != tuple(want) or not t.is_contiguous() \
                or t.device != self.device:
            raise ValueError(f"{name} must be a contiguous float32 {tuple(want)} tensor on {self.device}, got "
                             f"{t.dtype} {tuple(t.shape)} on {t.device}")

    def _check_gains(self, gains):
        import torch
        if gains.dtype != torch.float32 or tuple(gains.shape) != (4, HEAD_DIM) or not gains.is_contiguous() \
                or gains.device != self.device:
            raise ValueError("gains must be a contiguous float32 [4, 128] tensor on the device")

    def forward(self, q, k, v, gains, valid_len, out=None, lse=None, want_lse=True, stream=None):
        import torch
        self._check_inputs(q, k, v)
        self._check_gains(gains)
        if len(valid_len) != self.shape.B:
            raise ValueError("one valid length per sample")
        sh = self.shape
        if out is None:
            out = torch.empty_like(q)
        else:
            self._check_inputs(out)
        if lse is None and want_lse:
            lse = torch.empty((sh.B, sh.H, sh.S), dtype=torch.float32, device=self.device)
        elif lse is not None:
            self._check_f32(lse, (sh.B, sh.H, sh.S), "lse")
        rlk_joint_attn_fwd(self.shape, q, k, v, gains[0], gains[1], gains[2], gains[3], valid_len,
                           out, lse, self.ctx, stream)
        return out, lse

    def backward(self, q, k, v, gains, valid_len, out, dout, lse, dq=None, dk=None, dv=None,
                 dg_partial=None, dg=None, stream=None):
        import torch
        self._check_inputs(q, k, v, out, dout)
        self._check_gains(gains)
        sh = self.shape
        self._check_f32(lse, (sh.B, sh.H, sh.S), "lse")
        dq = torch.empty_like(q) if dq is None else dq
        dk = torch.empty_like(k) if dk is None else dk
        dv = torch.empty_like(v) if dv is None else dv
        self._check_inputs(dq, dk, dv)
        if dg_partial is None:
            dg_partial = torch.empty((sh.B, sh.H, 4, HEAD_DIM), dtype=torch.float32, device=self.device)
        if dg is None:
            dg = torch.empty((4, HEAD_DIM), dtype=torch.float32, device=self.device)
        self._check_f32(dg_partial, (sh.B, sh.H, 4, HEAD_DIM), "dg_partial")
        self._check_f32(dg, (4, HEAD_DIM), "dg")
        rlk_joint_attn_bwd(sh, q, k, v, gains[0], gains[1], gains[2], gains[3], valid_len, out, dout,
                           lse, self.ctx, dq, dk, dv, dg_partial, dg, self.workspace, stream=stream)
        return dq, dk, dv, dg_partial, dg

    def forward_unfused(self, q, k, v, gains, valid_len, stream=None):
        """The forward as the four standalone operators (qk_rmsnorm +
        multi_axis_rope, joint_attn_qk_gemm, joint_attn_softmax,
        joint_attn_av_gemm) with materialised intermediates. Returns a dict
        with out, lse and the intermediates scores [B, H, S, n_tiles*128]
        fp32, p (same shape, bf16), alpha [B, H, S, n_tiles] fp32 and l."""
        import torch
        self._check_inputs(q, k, v)
        self._check_gains(gains)
        if len(valid_len) != self.shape.B:
            raise ValueError("one valid length per sample")
        sh = self.shape
        n_tiles = -(-sh.T_txt // 128) + -(-(sh.grid_h * sh.grid_w) // 128)
        dev = self.device
        scores = torch.empty((sh.B, sh.H, sh.S, n_tiles * 128), dtype=torch.float32, device=dev)
        p = torch.empty((sh.B, sh.H, sh.S, n_tiles * 128), dtype=torch.bfloat16, device=dev)
        alpha = torch.empty((sh.B, sh.H, sh.S, n_tiles), dtype=torch.float32, device=dev)
        l = torch.empty((sh.B, sh.H, sh.S), dtype=torch.float32, device=dev)
        lse = torch.empty((sh.B, sh.H, sh.S), dtype=torch.float32, device=dev)
        out = torch.empty_like(q)
        rlk_qk_norm_rope(sh, q, k, gains[0], gains[1], gains[2], gains[3], self.ctx, stream)
        rlk_joint_attn_qk_gemm(sh, self.ctx, valid_len, scores, stream)
        rlk_joint_attn_softmax(sh, scores, valid_len, p, alpha, l, lse, stream)
        rlk_joint_attn_av_gemm(sh, p, alpha, l, v, valid_len, out, stream)
        return {"out": out, "lse": lse, "l": l, "scores": scores, "p": p, "alpha": alpha}

    def backward_unfused(self, q, k, v, gains, valid_len, out, dout, lse, scores, stream=None):
        """The backward as the standalone operators' backward calls, after a
        forward (fused or standalone) on the same inputs left its context in
        this object; scores from rlk_joint_attn_qk_gemm. Returns a dict with
        dq, dk, dv, dgp, dg (bytes equal to backward()) and the intermediates
        stats, p, dp, ds, dqh, dkh."""
        import torch
        self._check_inputs(q, k, v, out, dout)
        self._check_gains(gains)
        if len(valid_len) != self.shape.B:
            raise ValueError("one valid length per sample")
        sh = self.shape
        n_tiles = -(-sh.T_txt // 128) + -(-(sh.grid_h * sh.grid_w) // 128)
        dev = self.device
        stats = torch.empty((2, sh.B, sh.H, n_tiles * 128), dtype=torch.float32, device=dev)
        p = torch.empty((sh.B, sh.H, sh.S, n_tiles * 128), dtype=torch.bfloat16, device=dev)
        ds = torch.empty_like(p)
        dp = torch.empty((sh.B, sh.H, sh.S, n_tiles * 128), dtype=torch.float32, device=dev)
        dqh = torch.empty((sh.B, sh.H, sh.S, HEAD_DIM), dtype=torch.float32, device=dev)
        dkh = torch.empty_like(dqh)
        gain_tiles = torch.empty(rlk_joint_attn_unfused_bytes(sh, UNFUSED["gain_tiles"]) // 4, dtype=torch.float32,
                                 device=dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        dgp = torch.empty((sh.B, sh.H, 4, HEAD_DIM), dtype=torch.float32, device=dev)
        dg = torch.empty((4, HEAD_DIM), dtype=torch.float32, device=dev)
        rlk_joint_attn_bwd_stats(sh, out, dout, lse, stats, stream)
        rlk_joint_attn_softmax_bwd(sh, scores, stats, None, valid_len, p, None, stream)
        rlk_joint_attn_av_gemm_bwd(sh, p, v, dout, valid_len, dv, dp, stream)
        rlk_joint_attn_softmax_bwd(sh, scores, stats, dp, valid_len, None, ds, stream)
        rlk_joint_attn_qk_gemm_bwd(sh, ds, self.ctx, valid_len, dqh, dkh, stream)
        rlk_qk_norm_rope_bwd(sh, q, k, gains[0], gains[1], gains[2], gains[3], self.ctx, dqh, dkh, dq, dk, dgp, dg,
                             gain_tiles, stream)
        return {"dq": dq, "dk": dk, "dv": dv, "dgp": dgp, "dg": dg, "stats": stats, "p": p, "dp": dp, "ds": ds,
                "dqh": dqh, "dkh": dkh}

    def forward_streams(self, q, k, v, gains, valid_len, stream=None):
        """Forward on separate text/image tensors: q, k, v are (txt, img)
        pairs, txt [B, T_txt, H, 128] and img [B, grid_h*grid_w, H, 128]
        bf16. Returns ((out_txt, out_img), lse)."""
        import torch
        sh = self.shape
        out = tuple(None if x is None else torch.empty_like(x) for x in q)
        lse = torch.empty((sh.B, sh.H, sh.S), dtype=torch.float32, device=self.device)
        rlk_joint_attn_fwd_streams(sh, q, k, v, gains[0], gains[1], gains[2], gains[3], valid_len, out, lse,
                                   self.ctx, stream)
        return out, lse

    def backward_streams(self, q, k, v, gains, valid_len, out, dout, lse, stream=None):
        """Backward on separate text/image tensors (pairs as in
        forward_streams). Returns dq, dk, dv pairs, dg_partial and dg."""
        import torch
        sh = self.shape
        like = lambda pair: tuple(None if x is None else torch.empty_like(x) for x in pair)  # noqa: E731
        dq, dk, dv = like(q), like(k), like(v)
        dgp = torch.empty((sh.B, sh.H, 4, HEAD_DIM), dtype=torch.float32, device=self.device)
        dg = torch.empty((4, HEAD_DIM), dtype=torch.float32, device=self.device)
        rlk_joint_attn_bwd_streams(sh, q, k, v, gains[0], gains[1], gains[2], gains[3], valid_len, out, dout, lse,
                                   self.ctx, dq, dk, dv, dgp, dg, self.workspace, stream=stream)
        return dq, dk, dv, dgp, dg

    def n_key_blocks(self) -> int:
        sh = self.shape
        return -(-sh.T_txt // 128) + -(-(sh.grid_h * sh.grid_w) // 128)

    def forward_sharded(self, q, k, v, gains, valid_len, bounds, stream=None):
        """The forward run as consecutive key shards handing the softmax
        state on (ring order). ``bounds`` are the shard boundaries inside
        (0, n_key_blocks()), ascending. Returns out and lse."""
        import torch
        self._check_inputs(q, k, v)
        self._check_gains(gains)
        sh = self.shape
        edges = [0] + [int(x) for x in bounds] + [self.n_key_blocks()]
        out = torch.empty_like(q)
        lse = torch.empty((sh.B, sh.H, sh.S), dtype=torch.float32, device=self.device)
        n_state = rlk_joint_attn_state_bytes(sh) // 4
        states = [torch.empty(n_state, dtype=torch.float32, device=self.device) for _ in range(2)]
        rlk_qk_norm_rope(sh, q, k, gains[0], gains[1], gains[2], gains[3], self.ctx, stream)
        for i in range(len(edges) - 1):
            last = i == len(edges) - 2
            st_in = None if i == 0 else states[(i - 1) % 2]
            st_out = None if last else states[i % 2]
            rlk_joint_attn_fwd_shard(sh, self.ctx, v, valid_len, edges[i], edges[i + 1], st_in, st_out,
                                     out if last else None, lse if last else None, stream)
        return out, lse

    def ctx_views(self):
        """Views of the forward context: qh, kh bf16 [B, H, S, 128]; rq, rk fp32 [B, H, S].
        The offsets follow the library's ctx layout (regions aligned to 256 bytes)."""
        import torch
        sh = self.shape
        rows = sh.B * sh.H * sh.S

        def up(x):
            return (x + 255) // 256 * 256
        o_kh = up(rows * HEAD_DIM * 2)
        o_rq = up(o_kh + rows * HEAD_DIM * 2)
        o_rk = up(o_rq + rows * 4)
        c = self.ctx
        qh = c[:rows * HEAD_DIM * 2].view(torch.bfloat16).view(sh.B, sh.H, sh.S, HEAD_DIM)
        kh = c[o_kh:o_kh + rows * HEAD_DIM * 2].view(torch.bfloat16).view(sh.B, sh.H, sh.S, HEAD_DIM)
        rq = c[o_rq:o_rq + rows * 4].view(torch.float32).view(sh.B, sh.H, sh.S)
        rk = c[o_rk:o_rk + rows * 4].view(torch.float32).view(sh.B, sh.H, sh.S)
        return qh, kh, rq, rk

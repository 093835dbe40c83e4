"""CPU tests of the C ABI boundary: the library loads, exports every symbol
the header declares, sizes its buffers as documented and fails closed on bad
arguments before touching the GPU. No compute call is made here."""

import ctypes
import os
import re

import pytest

import invariant_mmdit_joint_gb300 as pkg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(pkg.library_path()):
        from invariant_mmdit_joint_gb300 import _build
        _build.build()
    return pkg.lib()


def declared_functions():
    names = set()
    for f in os.listdir(HEADER_DIR):
        if not f.endswith(".h"):
            continue
        text = open(os.path.join(HEADER_DIR, f)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b(rlk_[a-z0-9_]+)\s*\(", text):
            names.add(m.group(1))
    return names


def test_library_exports_every_declared_symbol(L):
    declared = declared_functions()
    assert declared, "no declarations found"
    assert declared == set(pkg.EXPORTED_SYMBOLS)
    for name in declared:
        assert hasattr(L, name), name


def test_buffer_sizes_match_documented_layout(L):
    s = pkg.Shape.make(2, 256, 64, 64, 24)
    S, rows = 4352, 2 * 24 * 4352

    def up(x):
        return (x + 255) // 256 * 256
    n_pos = (32 + 256 - 1) - (-32) + 1
    ctx = up(up(up(up(rows * 256) + rows * 256) + rows * 4) + rows * 4) + n_pos * 64 * 8
    assert pkg.rlk_joint_attn_ctx_bytes(s) == up(ctx)
    nt = 256 // 128 + 4096 // 128
    slots = 2 * 24 * 128 * nt  # tile-padded lse2 and Delta
    # dk^ (fp32), gain-gradient partials per (b, h, q|k, tile, 32-row quarter), then per (b, h)
    ws = up(up(up(up(slots * 4) + slots * 4) + rows * 512) + 2 * 24 * 2 * nt * 4 * 512)
    ws = up(ws + 2 * 24 * 4 * 512)
    ws += 2 * 24 * 34 * 34 * 32768  # bf16 dS tiles, 128 x 128 per (query tile, key tile)
    assert pkg.rlk_joint_attn_bwd_workspace_bytes(s) == up(ws)
    assert S == s.S


@pytest.mark.parametrize("mutate,code", [
    (dict(D=64), 2), (dict(axes=(16, 48, 64)), 2), (dict(B=0), 1), (dict(B=257), 1),
    (dict(grid_h=0), 1), (dict(H=0), 1), (dict(eps=0.0), 1), (dict(theta=1.0), 1), (dict(T_txt=-1), 1),
])
def test_invalid_shapes_fail_closed(L, mutate, code):
    base = dict(B=1, T_txt=16, grid_h=8, grid_w=8, H=2)
    args = {**base, **{k: v for k, v in mutate.items() if k in base}}
    extra = {k: v for k, v in mutate.items() if k not in base}
    s = pkg.Shape.make(**args, **extra)
    assert pkg.rlk_joint_attn_ctx_bytes(s) == 0
    fake = 1 << 20  # an aligned fake address: validation must stop before any use
    rc = L.rlk_joint_attn_fwd(ctypes.byref(s), fake, fake, fake, fake, fake, fake, fake,
                              (ctypes.c_int32 * 1)(0), fake, fake, fake, None)
    assert rc == code


def test_row_count_limit(L):
    """B * H * (tile-padded S) must stay below 2^31 rows (the device indexes
    rows in 32 bits); a shape just under the limit is accepted."""
    rows_per_bh = 128 * (2 + 32)  # 256 text + 64 x 64 image tokens in tiles of 128
    ok = pkg.Shape.make(B=256, T_txt=256, grid_h=64, grid_w=64, H=1900)
    assert 256 * 1900 * rows_per_bh < 2 ** 31 and pkg.rlk_joint_attn_ctx_bytes(ok) > 0
    bad = pkg.Shape.make(B=256, T_txt=256, grid_h=64, grid_w=64, H=1928)
    assert 256 * 1928 * rows_per_bh >= 2 ** 31 and pkg.rlk_joint_attn_ctx_bytes(bad) == 0


def _fwd(L, s, vl, ptr=1 << 20, lse=1 << 20, **over):
    p = dict(q=ptr, k=ptr, v=ptr, a=ptr, b=ptr, c=ptr, d=ptr, out=ptr, ctx=ptr)
    p.update(over)
    arr = (ctypes.c_int32 * len(vl))(*vl)
    return L.rlk_joint_attn_fwd(ctypes.byref(s), p["q"], p["k"], p["v"], p["a"], p["b"], p["c"], p["d"],
                                arr, p["out"], lse, p["ctx"], None)


def test_argument_checks_fail_closed_without_a_gpu(L):
    s = pkg.Shape.make(2, 16, 8, 8, 2)
    assert _fwd(L, s, [3, 17]) == 1            # valid length beyond T_txt
    assert _fwd(L, s, [-1, 3]) == 1            # negative valid length
    assert _fwd(L, s, [3, 3], q=None) == 1     # null input
    assert _fwd(L, s, [3, 3], ctx=None) == 1   # null ctx
    assert _fwd(L, s, [3, 3], k=(1 << 20) + 8) == 3   # misaligned pointer
    assert _fwd(L, s, [3, 3], lse=(1 << 20) + 4) == 3
    # a well-formed call reaches the device check: with no GPU it reports a
    # CUDA error -- it never falls back to another implementation
    import torch
    if not torch.cuda.is_available():
        assert _fwd(L, s, [3, 3]) == 5


def test_backward_checks_workspace_size(L):
    """Below the minimum (one (sample, head) pair's dS tiles) the backward
    refuses before any launch; from the minimum up it reaches the device
    check (on this machine: no GPU)."""
    s = pkg.Shape.make(2, 16, 8, 8, 3)
    full = pkg.rlk_joint_attn_bwd_workspace_bytes(s)
    least = pkg.rlk_joint_attn_bwd_workspace_min_bytes(s)
    nt = 1 + 1
    assert full - least == (2 * 3 - 1) * nt * nt * 32768
    p = 1 << 20
    vl = (ctypes.c_int32 * 2)(4, 9)

    def bwd(n):
        return L.rlk_joint_attn_bwd(ctypes.byref(s), p, p, p, p, p, p, p, vl, p, p, p, p, p, p, p, None, p, p,
                                    n, None)
    assert bwd(least - 1) == 4
    import torch
    if not torch.cuda.is_available():
        assert bwd(least) == 5 and bwd(full) == 5
    assert pkg.rlk_joint_attn_bwd_workspace_min_bytes(pkg.Shape.make(1, 16, 8, 8, 2, D=64)) == 0
    # 1024^2: one pair's 34 x 34 tiles of 32 KiB above the fixed part
    big = pkg.Shape.make(2, 256, 64, 64, 24)
    assert (pkg.rlk_joint_attn_bwd_workspace_bytes(big) - pkg.rlk_joint_attn_bwd_workspace_min_bytes(big)
            == 47 * 34 * 34 * 32768)
    rc = L.rlk_joint_attn_bwd(ctypes.byref(s), p, p, p, p, p, p, p, vl, p, p, None, p, p, p, p, None, p, p,
                              full, None)
    assert rc == 1  # lse is required by the backward


def test_strerror_and_trace(L):
    assert pkg.rlk_strerror(0) == "ok"
    assert "fails closed" in pkg.rlk_strerror(2)
    t = pkg.rlk_joint_attn_trace()
    assert t["split_k"] == 0 and t["atomics"] == 0 and t["tf32"] == 0
    assert t["accumulator"] == "fp32"
    assert t["backend"].startswith("sm_103a")
    assert "fast_math" not in t["fingerprint"] and "-prec-div=true" in t["fingerprint"]


def test_product_never_imports_the_oracle():
    pkg_dir = os.path.join(ROOT, "invariant_mmdit_joint_gb300")
    for dirpath, _, files in os.walk(pkg_dir):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(from|import)\s+oracle\b", text, re.M), f
                assert "oracle/" not in text, f


def test_binding_rejects_missing_library(tmp_path):
    with pytest.raises(ImportError):
        pkg.load_library(str(tmp_path / "absent.so"))


def test_unfused_intermediate_sizes(L):
    s = pkg.Shape.make(2, 256, 64, 64, 24)
    rows, n_tiles = 2 * 24 * 4352, 2 + 32
    assert pkg.rlk_joint_attn_unfused_bytes(s, "scores") == rows * n_tiles * 128 * 4
    assert pkg.rlk_joint_attn_unfused_bytes(s, "p") == rows * n_tiles * 128 * 2
    assert pkg.rlk_joint_attn_unfused_bytes(s, "alpha") == rows * n_tiles * 4
    assert pkg.rlk_joint_attn_unfused_bytes(s, "rows") == rows * 4
    # the standalone backward's intermediates
    assert pkg.rlk_joint_attn_unfused_bytes(s, "dp") == rows * n_tiles * 128 * 4
    assert pkg.rlk_joint_attn_unfused_bytes(s, "ds") == rows * n_tiles * 128 * 2
    assert pkg.rlk_joint_attn_unfused_bytes(s, "stats") == 2 * 2 * 24 * n_tiles * 128 * 4
    assert pkg.rlk_joint_attn_unfused_bytes(s, "dhat") == rows * 128 * 4
    assert pkg.rlk_joint_attn_unfused_bytes(s, "gain_tiles") == 2 * 24 * 2 * n_tiles * 4 * 128 * 4
    assert L.rlk_joint_attn_unfused_bytes(ctypes.byref(s), 9) == 0
    assert L.rlk_joint_attn_unfused_bytes(ctypes.byref(s), -1) == 0
    # a ragged image side: ceil(83 * 83 / 128) = 54 image tiles, 2 text tiles
    s2 = pkg.Shape.make(4, 256, 83, 83, 24)
    assert pkg.rlk_joint_attn_unfused_bytes(s2, "alpha") == 4 * 24 * (256 + 83 * 83) * 56 * 4
    bad = pkg.Shape.make(1, 16, 8, 8, 2, D=64)
    assert pkg.rlk_joint_attn_unfused_bytes(bad, "scores") == 0


def test_unfused_operators_fail_closed_without_a_gpu(L):
    s = pkg.Shape.make(2, 16, 8, 8, 2)
    p = 1 << 20
    vl = (ctypes.c_int32 * 2)(3, 3)
    bad_vl = (ctypes.c_int32 * 2)(3, 17)
    assert L.rlk_qk_norm_rope(ctypes.byref(s), p, p, p, p, p, None, p, None) == 1
    assert L.rlk_qk_norm_rope(ctypes.byref(s), p, p + 8, p, p, p, p, p, None) == 3
    assert L.rlk_joint_attn_qk_gemm(ctypes.byref(s), p, bad_vl, p, None) == 1
    assert L.rlk_joint_attn_qk_gemm(ctypes.byref(s), p, vl, None, None) == 1
    assert L.rlk_joint_attn_softmax(ctypes.byref(s), p, vl, p, p, None, None, None) == 1   # l required
    assert L.rlk_joint_attn_softmax(ctypes.byref(s), p, vl, p, p, p, p + 4, None) == 3     # lse misaligned
    assert L.rlk_joint_attn_av_gemm(ctypes.byref(s), p, p, p, None, vl, p, None) == 1      # v required
    assert L.rlk_joint_attn_av_gemm(ctypes.byref(s), p, p, p, p, None, p, None) == 1      # lengths required
    bad = pkg.Shape.make(1, 16, 8, 8, 2, D=64)
    assert L.rlk_joint_attn_qk_gemm(ctypes.byref(bad), p, vl, p, None) == 2
    import torch
    if not torch.cuda.is_available():
        assert L.rlk_joint_attn_softmax(ctypes.byref(s), p, vl, p, p, p, None, None) == 5


def test_op_trace_records_refused_calls(L):
    s = pkg.Shape.make(2, 16, 8, 8, 2)
    p = 1 << 20
    vl = (ctypes.c_int32 * 2)(3, 5)
    bad_vl = (ctypes.c_int32 * 2)(3, 17)
    pkg.rlk_op_trace_enable(True)
    try:
        assert L.rlk_joint_attn_qk_gemm(ctypes.byref(s), p, bad_vl, p, None) == 1
        assert L.rlk_joint_attn_softmax(ctypes.byref(s), p, vl, p, p, None, None, None) == 1
        assert L.rlk_joint_attn_av_gemm(ctypes.byref(s), p, p, p, p, vl, p + 8, None) == 3
        assert L.rlk_qk_norm_rope(None, p, p, p, p, p, p, p, None) == 1
        assert _fwd(L, s, [3, 3], q=None) == 1
        big = pkg.Shape.make(2, 256, 64, 64, 24)  # context beyond the fixed scratch
        assert L.rlk_joint_attn_fwd_noalloc(ctypes.byref(big), p, p, p, p, p, p, p, vl, p, p, None) == 4
        recs = pkg.rlk_op_trace_read()
    finally:
        pkg.rlk_op_trace_enable(False)
    assert [r["entry_point"] for r in recs] == [
        "rlk_joint_attn_qk_gemm", "rlk_joint_attn_softmax", "rlk_joint_attn_av_gemm", "rlk_qk_norm_rope",
        "rlk_joint_attn_fwd", "rlk_joint_attn_fwd_noalloc"]
    assert [r["status"] for r in recs] == [1, 1, 3, 1, 1, 4]
    assert [r["seq"] for r in recs] == [1, 2, 3, 4, 5, 6]
    for r in recs:
        # nothing was enqueued and there is no other path to fall back to
        assert r["actual_backend"] == "none" and r["kernels"] == [] and r["fallback"] == 0
        assert r["requested_backend"] == "cuda"
        assert r["split_k"] == 0 and r["atomics"] == 0 and r["tf32"] == 0 and r["accumulator"] == "fp32"
        assert "-prec-div=true" in r["kernel_fingerprint"] and r["reduction_order"] and r["arithmetic_policy"]
    assert recs[0]["op"] == "joint_attn_qk_gemm" and (recs[0]["B"], recs[0]["T_txt"]) == (2, 16)
    assert recs[3]["B"] == 0  # no shape given
    assert recs[5]["B"] == 2 and recs[5]["grid_h"] == 64
    assert "no fast math" in recs[4]["arithmetic_policy"]
    # off: nothing is recorded, and enabling clears the log
    assert _fwd(L, s, [3, 3], q=None) == 1
    assert pkg.rlk_op_trace_count() == 0


def test_op_trace_ring_keeps_the_newest_records(L):
    s = pkg.Shape.make(1, 16, 8, 8, 2)
    bad = (ctypes.c_int32 * 1)(99)
    n = pkg.OP_TRACE_CAP + 44
    with pkg.op_trace() as t:
        for _ in range(n):
            assert L.rlk_joint_attn_qk_gemm(ctypes.byref(s), 1 << 20, bad, 1 << 20, None) == 1
    assert len(t.records) == pkg.OP_TRACE_CAP
    assert t.records[0]["seq"] == n - pkg.OP_TRACE_CAP + 1 and t.records[-1]["seq"] == n
    rec = pkg.OpRecord()
    pkg.rlk_op_trace_enable(True)
    try:
        assert L.rlk_op_trace_read(0, ctypes.byref(rec)) == 1   # empty log
        assert L.rlk_op_trace_read(-1, ctypes.byref(rec)) == 1
        assert L.rlk_op_trace_read(0, None) == 1
    finally:
        pkg.rlk_op_trace_enable(False)


def test_op_trace_is_whole_per_call_across_threads(L):
    import threading
    s = pkg.Shape.make(1, 16, 8, 8, 2)
    p = 1 << 20

    def worker(kind):
        vl = (ctypes.c_int32 * 1)(99)
        for _ in range(50):
            if kind == 0:
                L.rlk_joint_attn_qk_gemm(ctypes.byref(s), p, vl, p, None)
            else:
                L.rlk_joint_attn_av_gemm(ctypes.byref(s), p, p, p, p, vl, p, None)

    with pkg.op_trace() as t:
        ths = [threading.Thread(target=worker, args=(i % 2,)) for i in range(4)]
        for th in ths:
            th.start()
        for th in ths:
            th.join()
    assert len(t.records) == 200
    assert sorted(r["seq"] for r in t.records) == list(range(1, 201))
    for r in t.records:
        assert r["op"] == r["entry_point"].replace("rlk_", "") and r["status"] == 1


def test_op_record_layout_matches_the_header(tmp_path):
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "layout.c"
    src.write_text(
        '#include <stdio.h>\n#include <stddef.h>\n#include "rlk_joint_attn.h"\n'
        'int main(void) { printf("%zu %zu %zu %zu\\n", sizeof(rlk_op_record), offsetof(rlk_op_record, kernels), '
        'offsetof(rlk_op_record, arithmetic_policy), offsetof(rlk_op_record, grid_w)); return 0; }\n')
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", HEADER_DIR, str(src), "-o", str(exe)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()]
    R = pkg.OpRecord
    assert got == [ctypes.sizeof(R), R.kernels.offset, R.arithmetic_policy.offset, R.grid_w.offset]


def test_key_shard_forward_fails_closed(L):
    s = pkg.Shape.make(2, 200, 13, 21, 2)  # 2 text + 3 image key blocks
    assert pkg.rlk_joint_attn_state_bytes(s) == 2 * 2 * (200 + 273) * (2 + 128) * 4
    p = 1 << 20
    vl = (ctypes.c_int32 * 2)(3, 150)

    def shard(b0, b1, st_in=p, st_out=p, out=None, lse=None, ctx=p, lens=vl):
        return L.rlk_joint_attn_fwd_shard(ctypes.byref(s), ctx, p, lens, b0, b1, st_in, st_out, out, lse, None)
    assert shard(2, 2) == 1                       # empty shard
    assert shard(3, 6, st_out=None, out=p) == 1   # past the last block
    assert shard(0, 2) == 1                       # the first shard takes no state
    assert shard(1, 3, st_in=None) == 1           # a later shard needs one
    assert shard(1, 5, st_out=p, out=p) == 1      # the last shard hands no state on...
    assert shard(1, 5, st_out=None) == 1          # ...and writes out
    assert shard(1, 3, lse=p) == 1                # only the last shard writes lse
    assert shard(1, 3, st_out=p + 4) == 3         # misaligned state
    assert shard(1, 3, lens=(ctypes.c_int32 * 2)(3, 201)) == 1
    import torch
    if not torch.cuda.is_available():
        assert shard(0, 2, st_in=None) == 5 and shard(2, 5, st_out=None, out=p, lse=p) == 5


def test_stream_pair_calls_fail_closed(L):
    s = pkg.Shape.make(2, 16, 8, 8, 2)
    p = 1 << 20
    vl = (ctypes.c_int32 * 2)(3, 5)

    def fwd(qt=p, qi=p, vt=p, ot=p, oi=p, lse=p, shape=s, lens=vl):
        return L.rlk_joint_attn_fwd_streams(ctypes.byref(shape), qt, qi, p, p, vt, p, p, p, p, p, lens, ot, oi, lse,
                                            p, None)
    assert fwd(qi=None) == 1          # the image buffer is required
    assert fwd(qt=None) == 1          # the text buffer too, when T_txt > 0
    assert fwd(oi=p + 8) == 3
    assert fwd(vt=p + 2) == 3
    assert fwd(lse=p + 4) == 3
    assert fwd(lens=(ctypes.c_int32 * 2)(3, 17)) == 1
    no_text = pkg.Shape.make(2, 0, 8, 8, 2)
    zero = (ctypes.c_int32 * 2)(0, 0)
    ws = pkg.rlk_joint_attn_bwd_workspace_bytes(s)
    least = pkg.rlk_joint_attn_bwd_workspace_min_bytes(s)

    def bwd(wsb=ws, dvt=p):
        return L.rlk_joint_attn_bwd_streams(ctypes.byref(s), p, p, p, p, p, p, p, p, p, p, vl, p, p, p, p, p, p,
                                            p, p, p, p, dvt, p, None, p, p, wsb, None)
    assert bwd(wsb=least - 1) == 4
    assert bwd(dvt=None) == 1
    import torch
    if not torch.cuda.is_available():
        # well formed (text buffers may be absent without text) up to the device check
        assert fwd(qt=None, vt=None, ot=None, shape=no_text, lens=zero) != 1
        assert fwd() == 5 and bwd() == 5


def test_qkv_projection_and_context_forward_fail_closed(L):
    s = pkg.Shape.make(2, 16, 8, 8, 2)
    p = 1 << 20
    vl = (ctypes.c_int32 * 2)(3, 5)

    def qkv(ctx=None, q=(p, p), k=(p, p), x_img=p, b_txt=p, gq=p):
        return L.rlk_qkv_bias_gemm(ctypes.byref(s), p, x_img, p, p, b_txt, p, gq, p, p, p, ctx, q[0], q[1], k[0],
                                   k[1], p, p, None)
    assert qkv(x_img=None) == 1                       # inputs required
    assert qkv(b_txt=p + 2) == 3                      # misaligned bias
    assert qkv(q=(None, None)) == 1                   # plain mode needs Q and K
    assert qkv(q=(None, p)) == 1                      # a text buffer is needed when T_txt > 0
    assert qkv(ctx=p, gq=None) == 1                   # the fused epilogue needs the gains
    assert L.rlk_joint_attn_fwd_ctx(ctypes.byref(s), None, p, p, vl, p, p, p, None) == 1
    assert L.rlk_joint_attn_fwd_ctx(ctypes.byref(s), p, p, p, vl, p, p + 8, p, None) == 3
    import torch
    if not torch.cuda.is_available():
        assert qkv() == 5 and qkv(ctx=p, q=(None, None), k=(None, None)) == 5


def test_output_projection_fails_closed(L):
    s = pkg.Shape.make(2, 16, 8, 8, 2)
    p = 1 << 20
    assert L.rlk_attn_out_bias_gemm(ctypes.byref(s), p, None, p, p, p, p, p, p, None) == 1
    assert L.rlk_attn_out_bias_gemm(ctypes.byref(s), None, p, p, p, p, p, p, p, None) == 1
    assert L.rlk_attn_out_bias_gemm(ctypes.byref(s), p, p, p, p, p, p, p + 2, p, None) == 3
    no_text = pkg.Shape.make(2, 0, 8, 8, 2)
    import torch
    if not torch.cuda.is_available():
        assert L.rlk_attn_out_bias_gemm(ctypes.byref(no_text), None, p, None, p, None, p, None, p, None) == 5


def test_binding_refuses_a_wrong_number_of_valid_lengths(L):
    shape = pkg.Shape.make(2, 16, 8, 8, 2)
    for bad in ([3], [3, 4, 5], []):
        with pytest.raises(ValueError):
            pkg._lengths(bad, shape)
    assert list(pkg._lengths([3, 4], shape)) == [3, 4]


def test_joint_attention_checks_caller_supplied_buffers(L):
    """Wrongly shaped outputs are refused in Python, before the library is
    called (CPU tensors: nothing reaches a device)."""
    torch = pytest.importorskip("torch")
    ja = pkg.JointAttention(1, 16, 8, 8, 2, device="cpu")
    x = torch.zeros((1, 80, 2, 128), dtype=torch.bfloat16)
    gains = torch.ones((4, 128), dtype=torch.float32)
    with pytest.raises(ValueError):
        ja.forward(x, x, x, gains, [11], out=torch.zeros((1, 80, 2, 127), dtype=torch.bfloat16))
    with pytest.raises(ValueError):
        ja.forward(x, x, x, gains, [11], lse=torch.zeros((1, 2, 79)))
    lse = torch.zeros((1, 2, 80))
    with pytest.raises(ValueError):
        ja.backward(x, x, x, gains, [11], x, x, lse, dq=torch.zeros((1, 80, 2, 128)))
    with pytest.raises(ValueError):
        ja.backward(x, x, x, gains, [11], x, x, lse, dg_partial=torch.zeros((1, 2, 4, 127)))
    with pytest.raises(ValueError):
        ja.backward(x, x, x, gains, [11], x, x, lse, dg=torch.zeros((4, 127)))
    with pytest.raises(ValueError):
        ja.backward(x, x, x, gains, [11], x, x, torch.zeros((1, 2, 80), dtype=torch.float64))


def _noalloc(L, s, vl, ptr=1 << 20, lse=1 << 20, **over):
    p = dict(q=ptr, k=ptr, v=ptr, a=ptr, b=ptr, c=ptr, d=ptr, out=ptr)
    p.update(over)
    arr = (ctypes.c_int32 * len(vl))(*vl) if vl is not None else None
    return L.rlk_joint_attn_fwd_noalloc(ctypes.byref(s) if s is not None else None, p["q"], p["k"], p["v"],
                                        p["a"], p["b"], p["c"], p["d"], arr, p["out"], lse, None)


def test_noalloc_refuses_what_the_regular_forward_refuses(L):
    """The allocation-free forward runs the regular forward's checks first:
    every refusal gives the same status on both entry points, before any
    device work (the scratch address is looked up only after them)."""
    s = pkg.Shape.make(2, 16, 8, 8, 2)
    cases = [
        (dict(), [3, 17]), (dict(), [-1, 3]),
        (dict(q=None), [3, 3]), (dict(v=None), [3, 3]), (dict(d=None), [3, 3]), (dict(out=None), [3, 3]),
        (dict(k=(1 << 20) + 8), [3, 3]), (dict(out=(1 << 20) + 2), [3, 3]), (dict(lse=(1 << 20) + 4), [3, 3]),
        (dict(q=None, k=(1 << 20) + 8), [3, 3]),
    ]
    for over, vl in cases:
        lse = over.pop("lse", 1 << 20)
        a = _fwd(L, s, vl, lse=lse, **over)
        b = _noalloc(L, s, vl, lse=lse, **over)
        assert a == b and a != 0, (over, vl, a, b)
    for mutate in (dict(D=64), dict(B=0), dict(grid_h=0), dict(eps=0.0), dict(axes=(16, 48, 64))):
        base = dict(B=1, T_txt=16, grid_h=8, grid_w=8, H=2)
        sh = pkg.Shape.make(**{**base, **{k: v for k, v in mutate.items() if k in base}},
                            **{k: v for k, v in mutate.items() if k not in base})
        assert _fwd(L, sh, [0]) == _noalloc(L, sh, [0]) != 0, mutate
    assert L.rlk_joint_attn_fwd_noalloc(None, 0, 0, 0, 0, 0, 0, 0, None, 0, 0, None) == 1
    assert _noalloc(L, s, None) == 1
    # a shape beyond the fixed scratch is refused before the device check
    big = pkg.Shape.make(2, 256, 64, 64, 24)
    assert pkg.rlk_joint_attn_ctx_bytes(big) > (64 << 20)
    assert _noalloc(L, big, [87, 193]) == 4
    import torch
    if not torch.cuda.is_available():
        # a well-formed call reaches the device check on both entry points
        assert _fwd(L, s, [3, 3]) == _noalloc(L, s, [3, 3]) == 5


def test_forward_tile_schedule_setting(L):
    """Three schedules are accepted and the previous one returned; an
    unknown one changes nothing."""
    prev = L.rlk_fwd_tile_schedule(1)
    try:
        assert L.rlk_fwd_tile_schedule(2) == 1
        assert L.rlk_fwd_tile_schedule(7) == -1
        assert L.rlk_fwd_tile_schedule(-1) == -1
        assert L.rlk_fwd_tile_schedule(0) == 2
        assert pkg.rlk_fwd_tile_schedule("pairs") == "auto"
        assert pkg.rlk_fwd_tile_schedule("auto") == "pairs"
        with pytest.raises(ValueError):
            pkg.rlk_fwd_tile_schedule("halves")
    finally:
        L.rlk_fwd_tile_schedule(prev)


def test_backward_operators_fail_closed_without_a_gpu(L):
    """The standalone backward calls refuse bad arguments before any launch
    and otherwise reach the device check."""
    s = pkg.Shape.make(2, 16, 8, 8, 2)
    p = 1 << 20
    vl = (ctypes.c_int32 * 2)(3, 5)
    bad_vl = (ctypes.c_int32 * 2)(3, 17)
    sb = ctypes.byref(s)
    # stats
    assert L.rlk_joint_attn_bwd_stats(sb, p, p, p, None, None) == 1
    assert L.rlk_joint_attn_bwd_stats(sb, p, p + 8, p, p, None) == 3
    # softmax_bwd: P alone needs p; dS needs dp and ds together
    assert L.rlk_joint_attn_softmax_bwd(sb, p, p, None, vl, None, None, None) == 1
    assert L.rlk_joint_attn_softmax_bwd(sb, p, p, p, vl, p, None, None) == 1
    assert L.rlk_joint_attn_softmax_bwd(sb, p, p, None, vl, p, p, None) == 1
    assert L.rlk_joint_attn_softmax_bwd(sb, p, p, None, bad_vl, p, None, None) == 1
    assert L.rlk_joint_attn_softmax_bwd(sb, p, p, p, vl, None, p + 2, None) == 3
    # av_gemm_bwd: at least one output; dV needs P
    assert L.rlk_joint_attn_av_gemm_bwd(sb, p, p, p, vl, None, None, None) == 1
    assert L.rlk_joint_attn_av_gemm_bwd(sb, None, p, p, vl, p, None, None) == 1
    assert L.rlk_joint_attn_av_gemm_bwd(sb, p, p, p, vl, p, p + 4, None) == 3
    # qk_gemm_bwd and the norm/rope backward
    assert L.rlk_joint_attn_qk_gemm_bwd(sb, p, None, vl, p, p, None) == 1
    assert L.rlk_qk_norm_rope_bwd(sb, p, p, p, p, p, p, p, p, p, p, p, p, p, None, None) == 1
    bad = pkg.Shape.make(2, 16, 8, 8, 2, D=64)
    assert L.rlk_joint_attn_qk_gemm_bwd(ctypes.byref(bad), p, p, vl, p, p, None) == 2
    import torch
    if not torch.cuda.is_available():
        assert L.rlk_joint_attn_bwd_stats(sb, p, p, p, p, None) == 5
        assert L.rlk_joint_attn_softmax_bwd(sb, p, p, None, vl, p, None, None) == 5
        assert L.rlk_joint_attn_av_gemm_bwd(sb, p, p, p, vl, p, p, None) == 5
        assert L.rlk_joint_attn_qk_gemm_bwd(sb, p, p, vl, p, p, None) == 5
        assert L.rlk_qk_norm_rope_bwd(sb, p, p, p, p, p, p, p, p, p, p, p, p, p, p, None) == 5

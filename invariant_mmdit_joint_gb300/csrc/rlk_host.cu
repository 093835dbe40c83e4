// Host side of the C ABI declared in include/rlk_joint_attn.h: argument
// validation (fail closed, nothing launched on error), the layout of the
// caller-owned ctx and workspace buffers, kernel sequencing, the device
// status word, the trace record of the "WS1 Single-GPU Kernel List" (rule 7)
// and launch timing for benchmarks.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <initializer_list>
#include <utility>
#include <mutex>
#include <vector>

#include "rlk_device.cuh"
#include "rlk_internal.h"

RLK_DEFINE_STRICT_PROBE(probe_host_tu)

#ifndef RLK_SOURCE_HASH
#define RLK_SOURCE_HASH "unknown"
#endif
#ifndef RLK_BUILD_FLAGS
#define RLK_BUILD_FLAGS "unknown"
#endif

namespace rlk {
namespace {

constexpr size_t kAlign = 256;
constexpr int kMaxDevices = 64;
constexpr long long kMaxTokens = 1 << 20;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool shape_ok(const rlk_ja_shape* sh, rlk_status* why) {
    if (sh == nullptr) { *why = RLK_ERR_INVALID_ARG; return false; }
    if (sh->D != kHeadDim || sh->axes[0] != 16 || sh->axes[1] != 56 || sh->axes[2] != 56) {
        *why = RLK_ERR_UNSUPPORTED;
        return false;
    }
    if (sh->B < 1 || sh->B > RLK_MAX_BATCH || sh->T_txt < 0 || sh->grid_h < 1 || sh->grid_w < 1 ||
        sh->H < 1 || sh->H > 4096 || !(sh->eps > 0.0f) || !std::isfinite(sh->eps) || !(sh->theta > 1.0f) ||
        !std::isfinite(sh->theta)) {
        *why = RLK_ERR_INVALID_ARG;
        return false;
    }
    const long long t_img = (long long)sh->grid_h * sh->grid_w;
    const long long s = t_img + sh->T_txt;
    // rows (b, h, tile-padded token) are indexed in 32 bits on the device
    const long long s_pad = 128 * ((sh->T_txt + 127) / 128 + (t_img + 127) / 128);
    if (t_img > kMaxTokens || s > kMaxTokens || (long long)sh->B * sh->H * s_pad >= (1LL << 31)) {
        *why = RLK_ERR_INVALID_ARG;
        return false;
    }
    return true;
}

Geom make_geom(const rlk_ja_shape* sh) {
    Geom g{};
    g.B = sh->B;
    g.H = sh->H;
    g.T_txt = sh->T_txt;
    g.gh = sh->grid_h;
    g.gw = sh->grid_w;
    g.T_img = sh->grid_h * sh->grid_w;
    g.S = g.T_txt + g.T_img;
    g.txt_off = std::max(g.gh / 2, g.gw / 2);
    g.ctr_h = (g.gh + 1) / 2;
    g.ctr_w = (g.gw + 1) / 2;
    const int p_lo = -std::max(g.ctr_h, g.ctr_w);
    int p_hi = std::max(g.gh - 1 - g.ctr_h, g.gw - 1 - g.ctr_w);
    p_hi = std::max(p_hi, 0);
    if (g.T_txt > 0) p_hi = std::max(p_hi, g.txt_off + g.T_txt - 1);
    g.p_lo = p_lo;
    g.n_pos = p_hi - p_lo + 1;
    g.eps = sh->eps;
    g.theta = sh->theta;
    g.ntq_txt = (g.T_txt + 127) / 128;
    g.ntq_img = (g.T_img + 127) / 128;
    g.nq_pad = 128 * (g.ntq_txt + g.ntq_img);
    return g;
}

struct CtxLayout {
    size_t qh, kh, rq, rk, tab, total;
};
CtxLayout ctx_layout(const Geom& g) {
    const size_t rows = (size_t)g.B * g.H * g.S;
    CtxLayout l{};
    l.qh = 0;
    l.kh = align_up(l.qh + rows * kHeadDim * 2);
    l.rq = align_up(l.kh + rows * kHeadDim * 2);
    l.rk = align_up(l.rq + rows * 4);
    l.tab = align_up(l.rk + rows * 4);
    l.total = align_up(l.tab + (size_t)g.n_pos * kPairs * sizeof(float2));
    return l;
}

struct WsLayout {
    size_t lse2, delta, dkh, dgt, dgp, dst, total;
    size_t image_pair;  // bytes of one (sample, head) pair's dS^T images
};
// The workspace with room for the dS^T images of image_pairs (sample, head)
// pairs (all B * H by default: one dK/dV and one dQ launch).
WsLayout ws_layout(const Geom& g, long long image_pairs = -1) {
    const size_t rows = (size_t)g.B * g.H * g.S;
    const size_t slots = (size_t)g.B * g.H * g.nq_pad;
    const size_t ntiles = (size_t)g.ntq_txt + g.ntq_img;
    WsLayout l{};
    l.lse2 = 0;
    l.delta = align_up(l.lse2 + slots * 4);
    // dk^ (fp32 [B, H, S, 128]), from the dK/dV kernel to norm_rope_bwd_k
    l.dkh = align_up(l.delta + slots * 4);
    // gain-gradient partials [B, H, 2, n_tiles, 4, 128] and their per-(b, h) folds
    l.dgt = align_up(l.dkh + rows * kHeadDim * 4);
    l.dgp = align_up(l.dgt + (size_t)g.B * g.H * 2 * ntiles * 4 * kHeadDim * 4);
    // bf16 dS^T tile images, one 32 KB image per (query tile, key tile)
    l.dst = align_up(l.dgp + (size_t)g.B * g.H * 4 * kHeadDim * 4);
    l.image_pair = ntiles * ntiles * 32768;
    const size_t pairs = image_pairs < 0 ? (size_t)g.B * g.H : (size_t)image_pairs;
    l.total = align_up(l.dst + pairs * l.image_pair);
    return l;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Per-device one-time checks: compute capability 10.3 and strict math.
std::mutex g_dev_mu;
int g_dev_state[kMaxDevices];  // 0 unknown, 1 ok, 2 wrong arch, 3 fast math, 4 cuda error

int strict_all_units() {
    const int r[7] = {probe_host_tu(), probe_prologue_tu(), probe_fwd_tu(), probe_bwd_tu(), probe_unfused_tu(),
                      probe_qkv_tu(), probe_unfused_bwd_tu()};
    for (int v : r)
        if (v < 0) return -1;
    for (int v : r)
        if (v == 0) return 0;
    return 1;
}

// The first call on a device runs the probes, which launch and synchronise:
// inside a stream capture that would break the caller's capture, so such a
// call fails closed instead (one eager call first makes later calls
// capturable).
rlk_status device_ok(void* stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return RLK_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (g_dev_state[dev] == 0) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &cs) != cudaSuccess ||
            cs != cudaStreamCaptureStatusNone)
            return RLK_ERR_UNSUPPORTED;
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
            g_dev_state[dev] = 4;
        } else if (major != 10 || minor != 3) {
            g_dev_state[dev] = 2;
        } else {
            const int s = strict_all_units();
            g_dev_state[dev] = s == 1 ? 1 : (s == 0 ? 3 : 4);
        }
    }
    switch (g_dev_state[dev]) {
        case 1: return RLK_OK;
        case 2: case 3: return RLK_ERR_UNSUPPORTED;
        default: return RLK_ERR_CUDA;
    }
}

rlk_status common_checks(const rlk_ja_shape* sh, const int32_t* vl, Geom* g, ValidLen* v) {
    rlk_status why = RLK_OK;
    if (!shape_ok(sh, &why)) return why;
    if (vl == nullptr) return RLK_ERR_INVALID_ARG;
    for (int b = 0; b < sh->B; ++b)
        if (vl[b] < 0 || vl[b] > sh->T_txt) return RLK_ERR_INVALID_ARG;
    *g = make_geom(sh);
    std::memset(v, 0, sizeof(*v));
    for (int b = 0; b < sh->B; ++b) v->L[b] = vl[b];
    return RLK_OK;
}

// Rows qk_rmsnorm + multi_axis_rope: cos/sin table and normed, rotated q^, k^
// (with the RMSNorm factors) into ctx.
rlk_status run_prologue(const Geom& g, const SegBf16& q, const SegBf16& k, const float* const gains[4], void* ctx,
                        cudaStream_t s) {
    const CtxLayout l = ctx_layout(g);
    uint8_t* c = static_cast<uint8_t*>(ctx);
    float2* tab = reinterpret_cast<float2*>(c + l.tab);
    if (launch_rope_table(g, tab, s) != cudaSuccess) return RLK_ERR_CUDA;
    if (launch_prologue(g, q, k, gains, tab, reinterpret_cast<uint16_t*>(c + l.qh),
                        reinterpret_cast<uint16_t*>(c + l.kh), reinterpret_cast<float*>(c + l.rq),
                        reinterpret_cast<float*>(c + l.rk), s) != cudaSuccess)
        return RLK_ERR_CUDA;
    return RLK_OK;
}

// The forward and backward on segmented activations (arguments checked).
rlk_status fwd_core(const Geom& g, const ValidLen& vl, const SegBf16& q, const SegBf16& k, const SegBf16& v,
                    const float* const gains[4], const SegBf16& out, float* lse, void* ctx, cudaStream_t s) {
    const CtxLayout l = ctx_layout(g);
    const uint8_t* c = static_cast<const uint8_t*>(ctx);
    const rlk_status st = run_prologue(g, q, k, gains, ctx, s);
    if (st != RLK_OK) return st;
    if (launch_attn_fwd(g, vl, reinterpret_cast<const uint16_t*>(c + l.qh), reinterpret_cast<const uint16_t*>(c + l.kh),
                        v, out, lse, s) != cudaSuccess)
        return RLK_ERR_CUDA;
    return RLK_OK;
}

rlk_status bwd_core(const Geom& g, const ValidLen& vl, const SegBf16& q, const SegBf16& k, const SegBf16& v,
                    const float* const gains[4], const SegBf16& out, const SegBf16& dout, const float* lse,
                    const void* ctx, const SegBf16& dq, const SegBf16& dk, const SegBf16& dv, float* dg_partial,
                    float* dg, void* workspace, size_t workspace_bytes, cudaStream_t s);

// Sizes of the standalone operators' intermediates.// Sizes of the standalone operators' intermediates.
size_t unfused_bytes(const Geom& g, int which) {
    const size_t rows = (size_t)g.B * g.H * g.S;
    const size_t nblk = (size_t)g.ntq_txt + g.ntq_img;
    switch (which) {
        case RLK_UNFUSED_SCORES: return rows * nblk * 128 * 4;
        case RLK_UNFUSED_P: return rows * nblk * 128 * 2;
        case RLK_UNFUSED_ALPHA: return rows * nblk * 4;
        case RLK_UNFUSED_ROWS: return rows * 4;
        case RLK_UNFUSED_DP: return rows * nblk * 128 * 4;
        case RLK_UNFUSED_DS: return rows * nblk * 128 * 2;
        case RLK_UNFUSED_STATS: return (size_t)2 * g.B * g.H * g.nq_pad * 4;
        case RLK_UNFUSED_DHAT: return rows * kHeadDim * 4;
        case RLK_UNFUSED_GAIN_TILES: return (size_t)g.B * g.H * 2 * nblk * 4 * kHeadDim * 4;
        default: return 0;
    }
}

// Common argument checks of the standalone entry points: valid shape and
// lengths, non-null and 16-byte-aligned device pointers, a supported device.
rlk_status check_ptrs(std::initializer_list<const void*> required, std::initializer_list<const void*> optional) {
    for (const void* p : required)
        if (p == nullptr) return RLK_ERR_INVALID_ARG;
    for (const void* p : required)
        if (!aligned16(p)) return RLK_ERR_ALIGNMENT;
    for (const void* p : optional)
        if (p != nullptr && !aligned16(p)) return RLK_ERR_ALIGNMENT;
    return RLK_OK;
}

// ---- launch timing ----
constexpr int kMaxTimed = 4096;
struct Timing {
    std::mutex mu;
    bool on = false;
    std::vector<cudaEvent_t> ev[kNumKernelIds];
    int count[kNumKernelIds] = {};
};
Timing g_timing;

// ---- operator trace ----
struct OpInfo {
    const char* op;
    const char* entry;
    const char* policy;
    const char* order;
};
constexpr const char* kFwdPolicy =
    "bf16 q^ k^ v and bf16 P operands, fp32 TMEM accumulators, scores*log2(e)/sqrt(128) in one fmaf, "
    "exp2f numerators, lazy max (2^8), IEEE div/sqrt, one bf16 cast of O; no TF32, no fast math";
constexpr const char* kFwdOrder =
    "key tiles of 128: text tiles with a valid key, then image tiles, ascending; row sums: 8 partials "
    "by column mod 8, fixed tree";
const OpInfo kOps[] = {
    {"qk_rmsnorm+multi_axis_rope+joint_attention_fused", "rlk_joint_attn_fwd", kFwdPolicy, kFwdOrder},
    {"joint_attention_fused backward", "rlk_joint_attn_bwd",
     "bf16 operands with P and dS rounded to bf16, fp32 TMEM accumulators, exp2f numerators, dK and dQ "
     "from the same bf16 dS, one bf16 cast of dQ dK dV; no TF32, no fast math",
     "dK/dV: query tiles ascending; dQ: key tiles in the forward order; dg: 64-token chunks, then h, "
     "then b ascending"},
    {"qk_rmsnorm+multi_axis_rope+joint_attention_fused", "rlk_joint_attn_fwd_noalloc", kFwdPolicy, kFwdOrder},
    {"qk_rmsnorm+multi_axis_rope", "rlk_qk_norm_rope",
     "fp32 math, r = 1/sqrt(mean(x^2)+eps) with IEEE sqrt and division, fp32 cos/sin from fp64 angles, "
     "one bf16 cast of q^ k^",
     "sum of squares: 8 per lane in order, then xor butterfly 8,4,2,1"},
    {"joint_attn_qk_gemm", "rlk_joint_attn_qk_gemm",
     "bf16 q^ k^ operands, fp32 TMEM accumulators, raw scores stored fp32, -inf at masked keys",
     "k-steps of 16 in order; key tiles in the fused order"},
    {"joint_attn_softmax", "rlk_joint_attn_softmax", kFwdPolicy, kFwdOrder},
    {"joint_attn_av_gemm", "rlk_joint_attn_av_gemm",
     "bf16 P and v operands, fp32 TMEM accumulator rescaled by alpha per tile, O*(1/l), one bf16 cast",
     "key tiles in the fused order; k-steps of 16 in order"},
    {"joint_attention_fused key shard", "rlk_joint_attn_fwd_shard", kFwdPolicy,
     "key tiles of 128 in the fused order, shards in ascending block order, the online-softmax state "
     "handed from shard to shard"},
    {"qk_rmsnorm+multi_axis_rope+joint_attention_fused", "rlk_joint_attn_fwd_streams", kFwdPolicy, kFwdOrder},
    {"joint_attention_fused backward", "rlk_joint_attn_bwd_streams",
     "bf16 operands with P and dS rounded to bf16, fp32 TMEM accumulators, exp2f numerators, dK and dQ "
     "from the same bf16 dS, one bf16 cast of dQ dK dV; no TF32, no fast math",
     "dK/dV: query tiles ascending; dQ: key tiles in the forward order; dg: 64-token chunks, then h, "
     "then b ascending"},
    {"qkv_bias_gemm(+qk_rmsnorm+multi_axis_rope)", "rlk_qkv_bias_gemm",
     "bf16 X W operands, fp32 TMEM accumulators, + bf16 bias, one bf16 rounding of Q K V; the fused epilogue "
     "then runs the prologue arithmetic (IEEE sqrt and division)",
     "K in ascending steps of 64 (16 per MMA); no split-K; norm: 16 partials of 8 then a fixed tree"},
    {"joint_attention_fused (from context)", "rlk_joint_attn_fwd_ctx", kFwdPolicy, kFwdOrder},
    {"attn_out_bias_gemm", "rlk_attn_out_bias_gemm",
     "bf16 O W operands, fp32 TMEM accumulators, + bf16 bias, one bf16 rounding of the output",
     "K in ascending steps of 64 (16 per MMA); no split-K"},
    {"joint_attn_softmax backward preprocess", "rlk_joint_attn_bwd_stats",
     "fp32 lse * log2(e) and rowsum(dO * O), tile-padded", "row sums: 16 partials of 8 products, then xor 8,4,2,1"},
    {"joint_attn_softmax backward", "rlk_joint_attn_softmax_bwd",
     "P = exp2f(fmaf(s, log2(e)/sqrt(128), -lse2)) fp32, one bf16 rounding; dS = P * (dP - Delta), one bf16 "
     "rounding; no fast math",
     "elementwise"},
    {"joint_attn_av_gemm backward", "rlk_joint_attn_av_gemm_bwd",
     "bf16 dO V P operands, fp32 TMEM accumulators; dP fp32, dV one bf16 rounding",
     "dP: k-steps of 16 dims in order; dV: query tiles ascending, k-steps of 16 queries"},
    {"joint_attn_qk_gemm backward", "rlk_joint_attn_qk_gemm_bwd",
     "bf16 dS q^ k^ operands, fp32 TMEM accumulators, times 1/sqrt(128); dq^ dk^ fp32",
     "dk^: query tiles ascending; dq^: key tiles in the forward order; k-steps of 16"},
    {"qk_rmsnorm+multi_axis_rope backward", "rlk_qk_norm_rope_bwd",
     "fp32 inverse rotation and RMSNorm backward, one bf16 cast of dQ dK",
     "row dot products: 4 products per lane then xor 16..1; gain partials per 32-row quarter, then tiles, h, b "
     "ascending"},
};
const char* const kKernelNames[kNumKernelIds] = {
    "rope_table_kernel", "prologue_kernel", "attn_fwd_tc_kernel", "bwd_pre_kernel",
    "attn_bwd_dkdv_tc_kernel", "attn_bwd_dq_tc_kernel", "norm_rope_bwd_k_kernel", "dg_fold_kernels",
    "qk_gemm_kernel", "softmax_kernel", "av_gemm_kernel", "attn_fwd_tc_kernel<shard>", "qkv_gemm_kernel",
    "qkv_gemm_kernel<out_proj>", "qk_gemm_kernel<dp>", "softmax_bwd_kernel", "acc_gemm_kernel<key>",
    "acc_gemm_kernel<query>", "norm_rope_bwd_q_kernel"};

struct OpLog {
    std::mutex mu;
    std::atomic<bool> on{false};
    std::vector<rlk_op_record> ring;
    int head = 0, count = 0;
    uint64_t seq = 0;
};
OpLog g_op;
thread_local int t_op_depth = 0;
thread_local bool t_op_open = false;
thread_local rlk_op_record t_op_rec;

void copy_str(char* dst, size_t n, const char* src) { std::snprintf(dst, n, "%s", src); }

void op_trace_kernel(int id) {
    if (!t_op_open || id < 0 || id >= kNumKernelIds) return;
    if (t_op_rec.n_kernels < RLK_OP_TRACE_MAX_KERNELS)
        copy_str(t_op_rec.kernels[t_op_rec.n_kernels++], sizeof(t_op_rec.kernels[0]), kKernelNames[id]);
    copy_str(t_op_rec.actual_backend, sizeof(t_op_rec.actual_backend), "sm_103a tcgen05");
}

}  // namespace

OpScope::OpScope(OpKind kind, const rlk_ja_shape* sh) {
    if (t_op_depth++ > 0 || !g_op.on.load()) return;
    owner_ = true;
    t_op_open = true;
    rlk_op_record& r = t_op_rec;
    std::memset(&r, 0, sizeof(r));
    const OpInfo& info = kOps[kind];
    copy_str(r.op, sizeof(r.op), info.op);
    copy_str(r.entry_point, sizeof(r.entry_point), info.entry);
    copy_str(r.requested_backend, sizeof(r.requested_backend), "cuda");
    copy_str(r.actual_backend, sizeof(r.actual_backend), "none");
    std::snprintf(r.kernel_fingerprint, sizeof(r.kernel_fingerprint), "%s %s", RLK_SOURCE_HASH, RLK_BUILD_FLAGS);
    copy_str(r.accumulator, sizeof(r.accumulator), "fp32");
    copy_str(r.arithmetic_policy, sizeof(r.arithmetic_policy), info.policy);
    copy_str(r.reduction_order, sizeof(r.reduction_order), info.order);
    if (sh != nullptr) {
        r.B = sh->B;
        r.H = sh->H;
        r.T_txt = sh->T_txt;
        r.grid_h = sh->grid_h;
        r.grid_w = sh->grid_w;
    }
}

rlk_status OpScope::finish(rlk_status st) {
    if (owner_ && !done_) {
        t_op_rec.status = st;
        std::lock_guard<std::mutex> lk(g_op.mu);
        if (g_op.on.load()) {
            if ((int)g_op.ring.size() < RLK_OP_TRACE_CAP) g_op.ring.resize(RLK_OP_TRACE_CAP);
            t_op_rec.seq = ++g_op.seq;
            g_op.ring[(g_op.head + g_op.count) % RLK_OP_TRACE_CAP] = t_op_rec;
            if (g_op.count < RLK_OP_TRACE_CAP)
                ++g_op.count;
            else
                g_op.head = (g_op.head + 1) % RLK_OP_TRACE_CAP;
        }
        t_op_open = false;
    }
    done_ = true;
    return st;
}

OpScope::~OpScope() {
    if (owner_ && !done_) t_op_open = false;
    --t_op_depth;
}

void timing_begin(int id, cudaStream_t s) {
    op_trace_kernel(id);
    if (!g_timing.on) return;
    std::lock_guard<std::mutex> lk(g_timing.mu);
    const int i = g_timing.count[id];
    if (i >= kMaxTimed) return;
    auto& ev = g_timing.ev[id];
    while ((int)ev.size() < 2 * i + 2) {
        cudaEvent_t e;
        if (cudaEventCreate(&e) != cudaSuccess) return;
        ev.push_back(e);
    }
    cudaEventRecord(ev[2 * i], s);
}

void timing_end(int id, cudaStream_t s) {
    if (!g_timing.on) return;
    std::lock_guard<std::mutex> lk(g_timing.mu);
    const int i = g_timing.count[id];
    if (i >= kMaxTimed || (int)g_timing.ev[id].size() < 2 * i + 2) return;
    cudaEventRecord(g_timing.ev[id][2 * i + 1], s);
    g_timing.count[id] = i + 1;
}

}  // namespace rlk


namespace rlk {
namespace {
rlk_status bwd_core(const Geom& g, const ValidLen& vl, const SegBf16& q, const SegBf16& k, const SegBf16& v,
                    const float* const gains[4], const SegBf16& out, const SegBf16& dout, const float* lse,
                    const void* ctx, const SegBf16& dq, const SegBf16& dk, const SegBf16& dv, float* dg_partial,
                    float* dg, void* workspace, size_t workspace_bytes, cudaStream_t s) {
    const CtxLayout l = ctx_layout(g);
    const WsLayout w = ws_layout(g);
    const uint8_t* c = static_cast<const uint8_t*>(ctx);
    const uint16_t* qh = reinterpret_cast<const uint16_t*>(c + l.qh);
    const uint16_t* kh = reinterpret_cast<const uint16_t*>(c + l.kh);
    const float* rq = reinterpret_cast<const float*>(c + l.rq);
    const float* rk = reinterpret_cast<const float*>(c + l.rk);
    const float2* tab = reinterpret_cast<const float2*>(c + l.tab);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    float* lse2_p = reinterpret_cast<float*>(ws + w.lse2);
    float* delta_p = reinterpret_cast<float*>(ws + w.delta);
    float* dkh = reinterpret_cast<float*>(ws + w.dkh);
    float* dgt = reinterpret_cast<float*>(ws + w.dgt);
    float* dgp = dg_partial != nullptr ? dg_partial : reinterpret_cast<float*>(ws + w.dgp);
    uint8_t* ds_tiles = ws + w.dst;
    const NormRopeBwdIo nr{q, dq, rq, {gains[0], gains[1], gains[2], gains[3]}, tab, dgt};
    if (launch_bwd_pre(g, out, dout, lse, lse2_p, delta_p, s) != cudaSuccess) return RLK_ERR_CUDA;
    // dK/dV then dQ over consecutive groups of (sample, head) pairs, as many
    // per group as the workspace holds images for (every pair at once when
    // it holds them all); a pair's arithmetic never depends on its group
    const int n_pairs = g.B * g.H;
    const int group = (int)std::min<size_t>((size_t)n_pairs, (workspace_bytes - w.dst) / w.image_pair);
    for (int bh0 = 0; bh0 < n_pairs; bh0 += group) {
        const int n = std::min(group, n_pairs - bh0);
        if (launch_attn_bwd_dkdv(g, vl, qh, kh, v, dout, lse2_p, delta_p, dv, dkh, ds_tiles, bh0, n, s) !=
            cudaSuccess)
            return RLK_ERR_CUDA;
        if (launch_attn_bwd_dq(g, vl, kh, ds_tiles, nr, bh0, n, s) != cudaSuccess) return RLK_ERR_CUDA;
    }
    if (launch_norm_rope_bwd_k(g, k, gains[1], gains[3], tab, rk, dkh, dk, dgt, s) != cudaSuccess)
        return RLK_ERR_CUDA;
    if (launch_dg_fold(g, dgt, dgp, dg, s) != cudaSuccess) return RLK_ERR_CUDA;
    return RLK_OK;
}
}  // namespace
}  // namespace rlk

namespace rlk {

rlk_status fwd_validate(const rlk_ja_shape* shape, const void* q, const void* k, const void* v,
                        const float* g_q_txt, const float* g_k_txt, const float* g_q_img, const float* g_k_img,
                        const int32_t* txt_valid_len, const void* out, const float* lse, const void* ctx,
                        bool ctx_required, Geom* g, ValidLen* vl) {
    rlk_status st = common_checks(shape, txt_valid_len, g, vl);
    if (st != RLK_OK) return st;
    // without a ctx argument the slot repeats q, which changes no outcome
    const void* ptrs[] = {q, k, v, g_q_txt, g_k_txt, g_q_img, g_k_img, out, ctx_required ? ctx : q};
    for (const void* p : ptrs)
        if (p == nullptr) return RLK_ERR_INVALID_ARG;
    for (const void* p : ptrs)
        if (!aligned16(p)) return RLK_ERR_ALIGNMENT;
    if (lse != nullptr && !aligned16(lse)) return RLK_ERR_ALIGNMENT;
    return RLK_OK;
}

rlk_status device_check(void* stream) { return device_ok(stream); }

rlk_status fwd_run(const Geom& g, const ValidLen& vl, const void* q, const void* k, const void* v,
                   const float* g_q_txt, const float* g_k_txt, const float* g_q_img, const float* g_k_img,
                   void* out, float* lse, void* ctx, void* stream) {
    const float* gains[4] = {g_q_txt, g_k_txt, g_q_img, g_k_img};
    return fwd_core(g, vl, seg_concat(q, g), seg_concat(k, g), seg_concat(v, g), gains, seg_concat(out, g), lse, ctx,
                    static_cast<cudaStream_t>(stream));
}

size_t ctx_bytes_of(const Geom& g) { return ctx_layout(g).total; }

}  // namespace rlk

using namespace rlk;

extern "C" {

size_t rlk_joint_attn_ctx_bytes(const rlk_ja_shape* shape) {
    rlk_status why;
    if (!shape_ok(shape, &why)) return 0;
    return ctx_layout(make_geom(shape)).total;
}

size_t rlk_joint_attn_bwd_workspace_bytes(const rlk_ja_shape* shape) {
    rlk_status why;
    if (!shape_ok(shape, &why)) return 0;
    return ws_layout(make_geom(shape)).total;
}

size_t rlk_joint_attn_bwd_workspace_min_bytes(const rlk_ja_shape* shape) {
    rlk_status why;
    if (!shape_ok(shape, &why)) return 0;
    return ws_layout(make_geom(shape), 1).total;
}

static rlk_status rlk_joint_attn_fwd_impl(const rlk_ja_shape* shape, const void* q, const void* k, const void* v,
                              const float* g_q_txt, const float* g_k_txt, const float* g_q_img,
                              const float* g_k_img, const int32_t* txt_valid_len, void* out, float* lse,
                              void* ctx, void* stream) {
    Geom g;
    ValidLen vl;
    rlk_status st = fwd_validate(shape, q, k, v, g_q_txt, g_k_txt, g_q_img, g_k_img, txt_valid_len, out, lse, ctx,
                                 true, &g, &vl);
    if (st != RLK_OK) return st;
    st = device_ok(stream);
    if (st != RLK_OK) return st;
    return fwd_run(g, vl, q, k, v, g_q_txt, g_k_txt, g_q_img, g_k_img, out, lse, ctx, stream);
}

rlk_status rlk_joint_attn_fwd(const rlk_ja_shape* shape, const void* q, const void* k, const void* v,
                              const float* g_q_txt, const float* g_k_txt, const float* g_q_img,
                              const float* g_k_img, const int32_t* txt_valid_len, void* out, float* lse,
                              void* ctx, void* stream) {
    OpScope sc(kOpFwd, shape);
    return sc.finish(rlk_joint_attn_fwd_impl(shape, q, k, v, g_q_txt, g_k_txt, g_q_img, g_k_img, txt_valid_len,
                                             out, lse, ctx, stream));
}

static rlk_status rlk_joint_attn_bwd_impl(const rlk_ja_shape* shape, const void* q, const void* k, const void* v,
                              const float* g_q_txt, const float* g_k_txt, const float* g_q_img,
                              const float* g_k_img, const int32_t* txt_valid_len, const void* out,
                              const void* dout, const float* lse, const void* ctx, void* dq, void* dk, void* dv,
                              float* dg_partial, float* dg, void* workspace, size_t workspace_bytes,
                              void* stream) {
    Geom g;
    ValidLen vl;
    rlk_status st = common_checks(shape, txt_valid_len, &g, &vl);
    if (st != RLK_OK) return st;
    const void* ptrs[] = {q, k, v, g_q_txt, g_k_txt, g_q_img, g_k_img, out, dout, lse, ctx, dq, dk, dv, dg,
                          workspace};
    for (const void* p : ptrs)
        if (p == nullptr) return RLK_ERR_INVALID_ARG;
    for (const void* p : ptrs)
        if (!aligned16(p)) return RLK_ERR_ALIGNMENT;
    if (dg_partial != nullptr && !aligned16(dg_partial)) return RLK_ERR_ALIGNMENT;
    if (workspace_bytes < ws_layout(g, 1).total) return RLK_ERR_WORKSPACE;
    st = device_ok(stream);
    if (st != RLK_OK) return st;

    const float* gains[4] = {g_q_txt, g_k_txt, g_q_img, g_k_img};
    return bwd_core(g, vl, seg_concat(q, g), seg_concat(k, g), seg_concat(v, g), gains, seg_concat(out, g),
                    seg_concat(dout, g), lse, ctx, seg_concat(dq, g), seg_concat(dk, g), seg_concat(dv, g), dg_partial,
                    dg, workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

rlk_status rlk_joint_attn_bwd(const rlk_ja_shape* shape, const void* q, const void* k, const void* v,
                              const float* g_q_txt, const float* g_k_txt, const float* g_q_img,
                              const float* g_k_img, const int32_t* txt_valid_len, const void* out,
                              const void* dout, const float* lse, const void* ctx, void* dq, void* dk, void* dv,
                              float* dg_partial, float* dg, void* workspace, size_t workspace_bytes,
                              void* stream) {
    OpScope sc(kOpBwd, shape);
    return sc.finish(rlk_joint_attn_bwd_impl(shape, q, k, v, g_q_txt, g_k_txt, g_q_img, g_k_img, txt_valid_len,
                                             out, dout, lse, ctx, dq, dk, dv, dg_partial, dg, workspace,
                                             workspace_bytes, stream));
}

// Separate text and image buffers: an image pointer is required, a text
// pointer only when T_txt > 0; all 16-byte aligned.
static rlk_status check_pairs(const Geom& g, std::initializer_list<std::pair<const void*, const void*>> pairs) {
    for (const auto& pr : pairs) {
        if (pr.second == nullptr || (g.T_txt > 0 && pr.first == nullptr)) return RLK_ERR_INVALID_ARG;
        if (!aligned16(pr.second) || (pr.first != nullptr && !aligned16(pr.first))) return RLK_ERR_ALIGNMENT;
    }
    return RLK_OK;
}

static rlk_status rlk_joint_attn_fwd_streams_impl(const rlk_ja_shape* shape, const void* q_txt, const void* q_img,
                                                  const void* k_txt, const void* k_img, const void* v_txt,
                                                  const void* v_img, const float* g_q_txt, const float* g_k_txt,
                                                  const float* g_q_img, const float* g_k_img,
                                                  const int32_t* txt_valid_len, void* out_txt, void* out_img,
                                                  float* lse, void* ctx, void* stream) {
    Geom g;
    ValidLen vl;
    rlk_status st = common_checks(shape, txt_valid_len, &g, &vl);
    if (st != RLK_OK) return st;
    st = check_pairs(g, {{q_txt, q_img}, {k_txt, k_img}, {v_txt, v_img}, {out_txt, out_img}});
    if (st != RLK_OK) return st;
    st = check_ptrs({g_q_txt, g_k_txt, g_q_img, g_k_img, ctx}, {lse});
    if (st != RLK_OK) return st;
    st = device_ok(stream);
    if (st != RLK_OK) return st;
    const float* gains[4] = {g_q_txt, g_k_txt, g_q_img, g_k_img};
    return fwd_core(g, vl, seg_split(q_txt, q_img, g), seg_split(k_txt, k_img, g), seg_split(v_txt, v_img, g), gains,
                    seg_split(out_txt, out_img, g), lse, ctx, static_cast<cudaStream_t>(stream));
}

rlk_status rlk_joint_attn_fwd_streams(const rlk_ja_shape* shape, const void* q_txt, const void* q_img,
                                      const void* k_txt, const void* k_img, const void* v_txt, const void* v_img,
                                      const float* g_q_txt, const float* g_k_txt, const float* g_q_img,
                                      const float* g_k_img, const int32_t* txt_valid_len, void* out_txt,
                                      void* out_img, float* lse, void* ctx, void* stream) {
    OpScope sc(kOpFwdStreams, shape);
    return sc.finish(rlk_joint_attn_fwd_streams_impl(shape, q_txt, q_img, k_txt, k_img, v_txt, v_img, g_q_txt,
                                                     g_k_txt, g_q_img, g_k_img, txt_valid_len, out_txt, out_img,
                                                     lse, ctx, stream));
}

static rlk_status rlk_joint_attn_bwd_streams_impl(
    const rlk_ja_shape* shape, const void* q_txt, const void* q_img, const void* k_txt, const void* k_img,
    const void* v_txt, const void* v_img, const float* g_q_txt, const float* g_k_txt, const float* g_q_img,
    const float* g_k_img, const int32_t* txt_valid_len, const void* out_txt, const void* out_img,
    const void* dout_txt, const void* dout_img, const float* lse, const void* ctx, void* dq_txt, void* dq_img,
    void* dk_txt, void* dk_img, void* dv_txt, void* dv_img, float* dg_partial, float* dg, void* workspace,
    size_t workspace_bytes, void* stream) {
    Geom g;
    ValidLen vl;
    rlk_status st = common_checks(shape, txt_valid_len, &g, &vl);
    if (st != RLK_OK) return st;
    st = check_pairs(g, {{q_txt, q_img}, {k_txt, k_img}, {v_txt, v_img}, {out_txt, out_img}, {dout_txt, dout_img},
                         {dq_txt, dq_img}, {dk_txt, dk_img}, {dv_txt, dv_img}});
    if (st != RLK_OK) return st;
    st = check_ptrs({g_q_txt, g_k_txt, g_q_img, g_k_img, lse, ctx, dg, workspace}, {dg_partial});
    if (st != RLK_OK) return st;
    if (workspace_bytes < ws_layout(g, 1).total) return RLK_ERR_WORKSPACE;
    st = device_ok(stream);
    if (st != RLK_OK) return st;
    const float* gains[4] = {g_q_txt, g_k_txt, g_q_img, g_k_img};
    return bwd_core(g, vl, seg_split(q_txt, q_img, g), seg_split(k_txt, k_img, g), seg_split(v_txt, v_img, g), gains,
                    seg_split(out_txt, out_img, g), seg_split(dout_txt, dout_img, g), lse, ctx,
                    seg_split(dq_txt, dq_img, g), seg_split(dk_txt, dk_img, g), seg_split(dv_txt, dv_img, g),
                    dg_partial, dg, workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

rlk_status rlk_joint_attn_bwd_streams(const rlk_ja_shape* shape, const void* q_txt, const void* q_img,
                                      const void* k_txt, const void* k_img, const void* v_txt, const void* v_img,
                                      const float* g_q_txt, const float* g_k_txt, const float* g_q_img,
                                      const float* g_k_img, const int32_t* txt_valid_len, const void* out_txt,
                                      const void* out_img, const void* dout_txt, const void* dout_img,
                                      const float* lse, const void* ctx, void* dq_txt, void* dq_img, void* dk_txt,
                                      void* dk_img, void* dv_txt, void* dv_img, float* dg_partial, float* dg,
                                      void* workspace, size_t workspace_bytes, void* stream) {
    OpScope sc(kOpBwdStreams, shape);
    return sc.finish(rlk_joint_attn_bwd_streams_impl(
        shape, q_txt, q_img, k_txt, k_img, v_txt, v_img, g_q_txt, g_k_txt, g_q_img, g_k_img, txt_valid_len, out_txt,
        out_img, dout_txt, dout_img, lse, ctx, dq_txt, dq_img, dk_txt, dk_img, dv_txt, dv_img, dg_partial, dg,
        workspace, workspace_bytes, stream));
}

static rlk_status rlk_qkv_bias_gemm_impl(const rlk_ja_shape* shape, const void* x_txt, const void* x_img,
                                         const void* w_txt, const void* w_img, const void* b_txt, const void* b_img,
                                         const float* g_q_txt, const float* g_k_txt, const float* g_q_img,
                                         const float* g_k_img, void* ctx, void* q_txt, void* q_img, void* k_txt,
                                         void* k_img, void* v_txt, void* v_img, void* stream) {
    rlk_status why = RLK_OK;
    if (!shape_ok(shape, &why)) return why;
    const Geom g = make_geom(shape);
    const bool fused = ctx != nullptr;
    // inputs and V are required; Q and K outputs are required without a
    // context and optional with one (a stream pair, or neither)
    rlk_status st = check_pairs(g, {{x_txt, x_img}, {w_txt, w_img}, {b_txt, b_img}, {v_txt, v_img}});
    if (st != RLK_OK) return st;
    const bool store_q = q_img != nullptr || q_txt != nullptr;
    const bool store_k = k_img != nullptr || k_txt != nullptr;
    if (!fused && (!store_q || !store_k)) return RLK_ERR_INVALID_ARG;
    if (store_q && (st = check_pairs(g, {{q_txt, q_img}})) != RLK_OK) return st;
    if (store_k && (st = check_pairs(g, {{k_txt, k_img}})) != RLK_OK) return st;
    if (fused && (st = check_ptrs({g_q_txt, g_k_txt, g_q_img, g_k_img, ctx}, {})) != RLK_OK) return st;
    st = device_ok(stream);
    if (st != RLK_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const uint16_t* x[2] = {static_cast<const uint16_t*>(x_txt), static_cast<const uint16_t*>(x_img)};
    const uint16_t* w[2] = {static_cast<const uint16_t*>(w_txt), static_cast<const uint16_t*>(w_img)};
    const uint16_t* bias[2] = {static_cast<const uint16_t*>(b_txt), static_cast<const uint16_t*>(b_img)};
    const float* gains[4] = {g_q_txt, g_k_txt, g_q_img, g_k_img};
    uint16_t *qh = nullptr, *kh = nullptr;
    float *rq = nullptr, *rk = nullptr;
    const float2* tab = nullptr;
    if (fused) {
        const CtxLayout l = ctx_layout(g);
        uint8_t* c = static_cast<uint8_t*>(ctx);
        qh = reinterpret_cast<uint16_t*>(c + l.qh);
        kh = reinterpret_cast<uint16_t*>(c + l.kh);
        rq = reinterpret_cast<float*>(c + l.rq);
        rk = reinterpret_cast<float*>(c + l.rk);
        float2* t = reinterpret_cast<float2*>(c + l.tab);
        if (launch_rope_table(g, t, s) != cudaSuccess) return RLK_ERR_CUDA;
        tab = t;
    }
    const SegBf16 none = seg_split(nullptr, nullptr, g);
    if (launch_proj_gemm(g, false, x, w, bias, gains, qh, kh, rq, rk, tab, store_q ? seg_split(q_txt, q_img, g) : none,
                        store_k ? seg_split(k_txt, k_img, g) : none, seg_split(v_txt, v_img, g), store_q, store_k,
                        s) != cudaSuccess)
        return RLK_ERR_CUDA;
    return RLK_OK;
}

rlk_status rlk_qkv_bias_gemm(const rlk_ja_shape* shape, const void* x_txt, const void* x_img, const void* w_txt,
                             const void* w_img, const void* b_txt, const void* b_img, const float* g_q_txt,
                             const float* g_k_txt, const float* g_q_img, const float* g_k_img, void* ctx,
                             void* q_txt, void* q_img, void* k_txt, void* k_img, void* v_txt, void* v_img,
                             void* stream) {
    OpScope sc(kOpQkvGemm, shape);
    return sc.finish(rlk_qkv_bias_gemm_impl(shape, x_txt, x_img, w_txt, w_img, b_txt, b_img, g_q_txt, g_k_txt,
                                            g_q_img, g_k_img, ctx, q_txt, q_img, k_txt, k_img, v_txt, v_img, stream));
}

static rlk_status rlk_joint_attn_fwd_ctx_impl(const rlk_ja_shape* shape, const void* ctx, const void* v_txt,
                                             const void* v_img, const int32_t* txt_valid_len, void* out_txt,
                                             void* out_img, float* lse, void* stream) {
    Geom g;
    ValidLen vl;
    rlk_status st = common_checks(shape, txt_valid_len, &g, &vl);
    if (st != RLK_OK) return st;
    st = check_pairs(g, {{v_txt, v_img}, {out_txt, out_img}});
    if (st != RLK_OK) return st;
    st = check_ptrs({ctx}, {lse});
    if (st != RLK_OK) return st;
    st = device_ok(stream);
    if (st != RLK_OK) return st;
    const CtxLayout l = ctx_layout(g);
    const uint8_t* c = static_cast<const uint8_t*>(ctx);
    if (launch_attn_fwd(g, vl, reinterpret_cast<const uint16_t*>(c + l.qh), reinterpret_cast<const uint16_t*>(c + l.kh),
                        seg_split(v_txt, v_img, g), seg_split(out_txt, out_img, g), lse,
                        static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return RLK_ERR_CUDA;
    return RLK_OK;
}

rlk_status rlk_joint_attn_fwd_ctx(const rlk_ja_shape* shape, const void* ctx, const void* v_txt, const void* v_img,
                                  const int32_t* txt_valid_len, void* out_txt, void* out_img, float* lse,
                                  void* stream) {
    OpScope sc(kOpFwdCtx, shape);
    return sc.finish(rlk_joint_attn_fwd_ctx_impl(shape, ctx, v_txt, v_img, txt_valid_len, out_txt, out_img, lse,
                                                 stream));
}

static rlk_status rlk_attn_out_bias_gemm_impl(const rlk_ja_shape* shape, const void* o_txt, const void* o_img,
                                              const void* w_txt, const void* w_img, const void* b_txt,
                                              const void* b_img, void* y_txt, void* y_img, void* stream) {
    rlk_status why = RLK_OK;
    if (!shape_ok(shape, &why)) return why;
    const Geom g = make_geom(shape);
    rlk_status st = check_pairs(g, {{o_txt, o_img}, {w_txt, w_img}, {b_txt, b_img}, {y_txt, y_img}});
    if (st != RLK_OK) return st;
    st = device_ok(stream);
    if (st != RLK_OK) return st;
    const uint16_t* x[2] = {static_cast<const uint16_t*>(o_txt), static_cast<const uint16_t*>(o_img)};
    const uint16_t* w[2] = {static_cast<const uint16_t*>(w_txt), static_cast<const uint16_t*>(w_img)};
    const uint16_t* bias[2] = {static_cast<const uint16_t*>(b_txt), static_cast<const uint16_t*>(b_img)};
    const float* gains[4] = {nullptr, nullptr, nullptr, nullptr};
    const SegBf16 none = seg_split(nullptr, nullptr, g);
    if (launch_proj_gemm(g, true, x, w, bias, gains, nullptr, nullptr, nullptr, nullptr, nullptr, none, none,
                         seg_split(y_txt, y_img, g), false, false, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return RLK_ERR_CUDA;
    return RLK_OK;
}

rlk_status rlk_attn_out_bias_gemm(const rlk_ja_shape* shape, const void* o_txt, const void* o_img, const void* w_txt,
                                  const void* w_img, const void* b_txt, const void* b_img, void* y_txt, void* y_img,
                                  void* stream) {
    OpScope sc(kOpOutGemm, shape);
    return sc.finish(
        rlk_attn_out_bias_gemm_impl(shape, o_txt, o_img, w_txt, w_img, b_txt, b_img, y_txt, y_img, stream));
}

size_t rlk_joint_attn_unfused_bytes(const rlk_ja_shape* shape, int which) {
    rlk_status why;
    if (!shape_ok(shape, &why)) return 0;
    return unfused_bytes(make_geom(shape), which);
}

static rlk_status rlk_qk_norm_rope_impl(const rlk_ja_shape* shape, const void* q, const void* k, const float* g_q_txt,
                            const float* g_k_txt, const float* g_q_img, const float* g_k_img, void* ctx,
                            void* stream) {
    rlk_status why = RLK_OK;
    if (!shape_ok(shape, &why)) return why;
    rlk_status st = check_ptrs({q, k, g_q_txt, g_k_txt, g_q_img, g_k_img, ctx}, {});
    if (st != RLK_OK) return st;
    st = device_ok(stream);
    if (st != RLK_OK) return st;
    const Geom g = make_geom(shape);
    const float* gains[4] = {g_q_txt, g_k_txt, g_q_img, g_k_img};
    return run_prologue(g, seg_concat(q, g), seg_concat(k, g), gains, ctx, static_cast<cudaStream_t>(stream));
}

rlk_status rlk_qk_norm_rope(const rlk_ja_shape* shape, const void* q, const void* k, const float* g_q_txt,
                            const float* g_k_txt, const float* g_q_img, const float* g_k_img, void* ctx,
                            void* stream) {
    OpScope sc(kOpNormRope, shape);
    return sc.finish(rlk_qk_norm_rope_impl(shape, q, k, g_q_txt, g_k_txt, g_q_img, g_k_img, ctx, stream));
}

static rlk_status rlk_joint_attn_qk_gemm_impl(const rlk_ja_shape* shape, const void* ctx, const int32_t* txt_valid_len,
                                  float* scores, void* stream) {
    Geom g;
    ValidLen vl;
    rlk_status st = common_checks(shape, txt_valid_len, &g, &vl);
    if (st != RLK_OK) return st;
    st = check_ptrs({ctx, scores}, {});
    if (st != RLK_OK) return st;
    st = device_ok(stream);
    if (st != RLK_OK) return st;
    const CtxLayout l = ctx_layout(g);
    const uint8_t* c = static_cast<const uint8_t*>(ctx);
    if (launch_qk_gemm(g, vl, reinterpret_cast<const uint16_t*>(c + l.qh), reinterpret_cast<const uint16_t*>(c + l.kh),
                       scores, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return RLK_ERR_CUDA;
    return RLK_OK;
}

rlk_status rlk_joint_attn_qk_gemm(const rlk_ja_shape* shape, const void* ctx, const int32_t* txt_valid_len,
                                  float* scores, void* stream) {
    OpScope sc(kOpQkGemm, shape);
    return sc.finish(rlk_joint_attn_qk_gemm_impl(shape, ctx, txt_valid_len, scores, stream));
}

static rlk_status rlk_joint_attn_softmax_impl(const rlk_ja_shape* shape, const float* scores, const int32_t* txt_valid_len,
                                  void* p, float* alpha, float* l, float* lse, void* stream) {
    Geom g;
    ValidLen vl;
    rlk_status st = common_checks(shape, txt_valid_len, &g, &vl);
    if (st != RLK_OK) return st;
    st = check_ptrs({scores, p, alpha, l}, {lse});
    if (st != RLK_OK) return st;
    st = device_ok(stream);
    if (st != RLK_OK) return st;
    if (launch_softmax(g, vl, scores, static_cast<uint16_t*>(p), alpha, l, lse, static_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return RLK_ERR_CUDA;
    return RLK_OK;
}

rlk_status rlk_joint_attn_softmax(const rlk_ja_shape* shape, const float* scores, const int32_t* txt_valid_len,
                                  void* p, float* alpha, float* l, float* lse, void* stream) {
    OpScope sc(kOpSoftmax, shape);
    return sc.finish(rlk_joint_attn_softmax_impl(shape, scores, txt_valid_len, p, alpha, l, lse, stream));
}

static rlk_status rlk_joint_attn_av_gemm_impl(const rlk_ja_shape* shape, const void* p, const float* alpha, const float* l,
                                  const void* v, const int32_t* txt_valid_len, void* out, void* stream) {
    Geom g;
    ValidLen vl;
    rlk_status st = common_checks(shape, txt_valid_len, &g, &vl);
    if (st != RLK_OK) return st;
    st = check_ptrs({p, alpha, l, v, out}, {});
    if (st != RLK_OK) return st;
    st = device_ok(stream);
    if (st != RLK_OK) return st;
    if (launch_av_gemm(g, vl, static_cast<const uint16_t*>(p), alpha, l, seg_concat(v, g), seg_concat(out, g),
                       static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return RLK_ERR_CUDA;
    return RLK_OK;
}

rlk_status rlk_joint_attn_av_gemm(const rlk_ja_shape* shape, const void* p, const float* alpha, const float* l,
                                  const void* v, const int32_t* txt_valid_len, void* out, void* stream) {
    OpScope sc(kOpAvGemm, shape);
    return sc.finish(rlk_joint_attn_av_gemm_impl(shape, p, alpha, l, v, txt_valid_len, out, stream));
}

// ---- the standalone backward operators (k_attn_unfused_bwd.cu) ----
static rlk_status bwd_stats_impl(const rlk_ja_shape* shape, const void* out, const void* dout, const float* lse,
                                 float* stats, void* stream) {
    rlk_status why = RLK_OK;
    if (!shape_ok(shape, &why)) return why;
    const Geom g = make_geom(shape);
    rlk_status st = check_ptrs({out, dout, lse, stats}, {});
    if (st != RLK_OK) return st;
    st = device_ok(stream);
    if (st != RLK_OK) return st;
    const size_t half = (size_t)g.B * g.H * g.nq_pad;
    if (launch_bwd_pre(g, seg_concat(out, g), seg_concat(dout, g), lse, stats, stats + half,
                       static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return RLK_ERR_CUDA;
    return RLK_OK;
}

rlk_status rlk_joint_attn_bwd_stats(const rlk_ja_shape* shape, const void* out, const void* dout, const float* lse,
                                    float* stats, void* stream) {
    OpScope sc(kOpBwdStats, shape);
    return sc.finish(bwd_stats_impl(shape, out, dout, lse, stats, stream));
}

static rlk_status softmax_bwd_impl(const rlk_ja_shape* shape, const float* scores, const float* stats,
                                   const float* dp, const int32_t* txt_valid_len, void* p, void* ds, void* stream) {
    Geom g;
    ValidLen vl;
    rlk_status st = common_checks(shape, txt_valid_len, &g, &vl);
    if (st != RLK_OK) return st;
    // P alone (dp NULL), or dS (dp and ds given; P optional)
    if ((dp == nullptr) != (ds == nullptr) || (dp == nullptr && p == nullptr)) return RLK_ERR_INVALID_ARG;
    st = check_ptrs({scores, stats}, {dp, p, ds});
    if (st != RLK_OK) return st;
    st = device_ok(stream);
    if (st != RLK_OK) return st;
    const size_t half = (size_t)g.B * g.H * g.nq_pad;
    if (launch_softmax_bwd(g, vl, scores, stats, stats + half, dp, static_cast<uint16_t*>(p),
                           static_cast<uint16_t*>(ds), static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return RLK_ERR_CUDA;
    return RLK_OK;
}

rlk_status rlk_joint_attn_softmax_bwd(const rlk_ja_shape* shape, const float* scores, const float* stats,
                                      const float* dp, const int32_t* txt_valid_len, void* p, void* ds,
                                      void* stream) {
    OpScope sc(kOpSoftmaxBwd, shape);
    return sc.finish(softmax_bwd_impl(shape, scores, stats, dp, txt_valid_len, p, ds, stream));
}

static rlk_status av_gemm_bwd_impl(const rlk_ja_shape* shape, const void* p, const void* v, const void* dout,
                                   const int32_t* txt_valid_len, void* dv, float* dp, void* stream) {
    Geom g;
    ValidLen vl;
    rlk_status st = common_checks(shape, txt_valid_len, &g, &vl);
    if (st != RLK_OK) return st;
    if (dv == nullptr && dp == nullptr) return RLK_ERR_INVALID_ARG;
    if (dv != nullptr && p == nullptr) return RLK_ERR_INVALID_ARG;
    st = check_ptrs({v, dout}, {p, dv, dp});
    if (st != RLK_OK) return st;
    st = device_ok(stream);
    if (st != RLK_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dp != nullptr && launch_dp_gemm(g, vl, seg_concat(dout, g), seg_concat(v, g), dp, s) != cudaSuccess)
        return RLK_ERR_CUDA;
    if (dv != nullptr &&
        launch_dv_gemm(g, vl, static_cast<const uint16_t*>(p), seg_concat(dout, g), seg_concat(dv, g), s) !=
            cudaSuccess)
        return RLK_ERR_CUDA;
    return RLK_OK;
}

rlk_status rlk_joint_attn_av_gemm_bwd(const rlk_ja_shape* shape, const void* p, const void* v, const void* dout,
                                      const int32_t* txt_valid_len, void* dv, float* dp, void* stream) {
    OpScope sc(kOpAvGemmBwd, shape);
    return sc.finish(av_gemm_bwd_impl(shape, p, v, dout, txt_valid_len, dv, dp, stream));
}

static rlk_status qk_gemm_bwd_impl(const rlk_ja_shape* shape, const void* ds, const void* ctx,
                                   const int32_t* txt_valid_len, float* dqh, float* dkh, void* stream) {
    Geom g;
    ValidLen vl;
    rlk_status st = common_checks(shape, txt_valid_len, &g, &vl);
    if (st != RLK_OK) return st;
    st = check_ptrs({ds, ctx, dqh, dkh}, {});
    if (st != RLK_OK) return st;
    st = device_ok(stream);
    if (st != RLK_OK) return st;
    const CtxLayout l = ctx_layout(g);
    const uint8_t* c = static_cast<const uint8_t*>(ctx);
    if (launch_dhat_gemms(g, vl, static_cast<const uint16_t*>(ds), reinterpret_cast<const uint16_t*>(c + l.qh),
                          reinterpret_cast<const uint16_t*>(c + l.kh), dqh, dkh,
                          static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return RLK_ERR_CUDA;
    return RLK_OK;
}

rlk_status rlk_joint_attn_qk_gemm_bwd(const rlk_ja_shape* shape, const void* ds, const void* ctx,
                                      const int32_t* txt_valid_len, float* dqh, float* dkh, void* stream) {
    OpScope sc(kOpQkGemmBwd, shape);
    return sc.finish(qk_gemm_bwd_impl(shape, ds, ctx, txt_valid_len, dqh, dkh, stream));
}

static rlk_status norm_rope_bwd_impl(const rlk_ja_shape* shape, const void* q, const void* k, const float* g_q_txt,
                                     const float* g_k_txt, const float* g_q_img, const float* g_k_img,
                                     const void* ctx, const float* dqh, const float* dkh, void* dq, void* dk,
                                     float* dg_partial, float* dg, float* gain_tiles, void* stream) {
    rlk_status why = RLK_OK;
    if (!shape_ok(shape, &why)) return why;
    const Geom g = make_geom(shape);
    rlk_status st = check_ptrs({q, k, g_q_txt, g_k_txt, g_q_img, g_k_img, ctx, dqh, dkh, dq, dk, dg_partial, dg,
                                gain_tiles},
                               {});
    if (st != RLK_OK) return st;
    st = device_ok(stream);
    if (st != RLK_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const CtxLayout l = ctx_layout(g);
    const uint8_t* c = static_cast<const uint8_t*>(ctx);
    const float* rq = reinterpret_cast<const float*>(c + l.rq);
    const float* rk = reinterpret_cast<const float*>(c + l.rk);
    const float2* tab = reinterpret_cast<const float2*>(c + l.tab);
    if (launch_norm_rope_bwd_q(g, seg_concat(q, g), g_q_txt, g_q_img, tab, rq, dqh, seg_concat(dq, g), gain_tiles,
                               s) != cudaSuccess)
        return RLK_ERR_CUDA;
    if (launch_norm_rope_bwd_k(g, seg_concat(k, g), g_k_txt, g_k_img, tab, rk, dkh, seg_concat(dk, g), gain_tiles,
                               s) != cudaSuccess)
        return RLK_ERR_CUDA;
    if (launch_dg_fold(g, gain_tiles, dg_partial, dg, s) != cudaSuccess) return RLK_ERR_CUDA;
    return RLK_OK;
}

rlk_status rlk_qk_norm_rope_bwd(const rlk_ja_shape* shape, const void* q, const void* k, const float* g_q_txt,
                                const float* g_k_txt, const float* g_q_img, const float* g_k_img, const void* ctx,
                                const float* dqh, const float* dkh, void* dq, void* dk, float* dg_partial,
                                float* dg, float* gain_tiles, void* stream) {
    OpScope sc(kOpNormRopeBwd, shape);
    return sc.finish(norm_rope_bwd_impl(shape, q, k, g_q_txt, g_k_txt, g_q_img, g_k_img, ctx, dqh, dkh, dq, dk,
                                        dg_partial, dg, gain_tiles, stream));
}

size_t rlk_joint_attn_state_bytes(const rlk_ja_shape* shape) {
    rlk_status why;
    if (!shape_ok(shape, &why)) return 0;
    const Geom g = make_geom(shape);
    return (size_t)g.B * g.H * g.S * (2 + kHeadDim) * sizeof(float);
}

static rlk_status rlk_joint_attn_fwd_shard_impl(const rlk_ja_shape* shape, const void* ctx, const void* v,
                                                const int32_t* txt_valid_len, int32_t blk_begin, int32_t blk_end,
                                                const float* state_in, float* state_out, void* out, float* lse,
                                                void* stream) {
    Geom g;
    ValidLen vl;
    rlk_status st = common_checks(shape, txt_valid_len, &g, &vl);
    if (st != RLK_OK) return st;
    const int nblk = g.ntq_txt + g.ntq_img;
    if (blk_begin < 0 || blk_end > nblk || blk_begin >= blk_end) return RLK_ERR_INVALID_ARG;
    const bool first = blk_begin == 0, last = blk_end == nblk;
    // the state comes in unless this is the first shard and goes on unless
    // it is the last, which writes out (and lse if given)
    if ((state_in == nullptr) != first || (state_out == nullptr) != last || (out == nullptr) != !last ||
        (lse != nullptr && !last))
        return RLK_ERR_INVALID_ARG;
    st = check_ptrs({ctx, v}, {state_in, state_out, out, lse});
    if (st != RLK_OK) return st;
    st = device_ok(stream);
    if (st != RLK_OK) return st;
    const CtxLayout l = ctx_layout(g);
    const uint8_t* c = static_cast<const uint8_t*>(ctx);
    const SegBf16 out_seg = seg_concat(out, g);
    if (launch_attn_fwd_shard(g, vl, reinterpret_cast<const uint16_t*>(c + l.qh),
                              reinterpret_cast<const uint16_t*>(c + l.kh), seg_concat(v, g), blk_begin, blk_end,
                              state_in, state_out, out != nullptr ? &out_seg : nullptr, lse,
                              static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return RLK_ERR_CUDA;
    return RLK_OK;
}

rlk_status rlk_joint_attn_fwd_shard(const rlk_ja_shape* shape, const void* ctx, const void* v,
                                    const int32_t* txt_valid_len, int32_t blk_begin, int32_t blk_end,
                                    const float* state_in, float* state_out, void* out, float* lse, void* stream) {
    OpScope sc(kOpFwdShard, shape);
    return sc.finish(rlk_joint_attn_fwd_shard_impl(shape, ctx, v, txt_valid_len, blk_begin, blk_end, state_in,
                                                   state_out, out, lse, stream));
}

rlk_status rlk_joint_attn_check_status(void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return RLK_ERR_CUDA;
    const int a = read_and_clear_status_fwd(s);
    const int b = read_and_clear_status_bwd(s);
    const int c = read_and_clear_status_unfused(s);
    const int d = read_and_clear_status_qkv(s);
    const int e = read_and_clear_status_prologue(s);
    const int f = read_and_clear_status_unfused_bwd(s);
    if (a < 0 || b < 0 || c < 0 || d < 0 || e < 0 || f < 0) return RLK_ERR_CUDA;
    if (a != 0 || b != 0 || c != 0 || d != 0 || e != 0 || f != 0) return RLK_ERR_DEVICE_TIMEOUT;
    return RLK_OK;
}

int rlk_strict_math_compiled(void) { return strict_all_units(); }

rlk_status rlk_selftest_wait_timeout(int32_t limit_ms, void* stream) {
    if (limit_ms < 1 || limit_ms > 2000) return RLK_ERR_INVALID_ARG;
    return launch_wait_timeout_probe(limit_ms, static_cast<cudaStream_t>(stream)) == cudaSuccess ? RLK_OK
                                                                                                  : RLK_ERR_CUDA;
}

rlk_status rlk_joint_attn_trace(rlk_ja_trace* out) {
    if (out == nullptr) return RLK_ERR_INVALID_ARG;
    std::memset(out, 0, sizeof(*out));
    std::snprintf(out->backend, sizeof(out->backend), "sm_103a tcgen05");
    std::snprintf(out->reduction_order, sizeof(out->reduction_order),
                  "tiles of 128: text from 0 then image from T_txt, ascending; dkdv: q tiles ascending; "
                  "rows: lane order + xor butterfly; dg: 32-row quarters, (q0+q1)+(q2+q3), tiles, h, b ascending");
    std::snprintf(out->accumulator, sizeof(out->accumulator), "fp32");
    out->split_k = 0;
    out->atomics = 0;
    out->tf32 = 0;
    out->strict_math = strict_all_units();
    out->block_q = kFwdBlockQ;
    out->block_kv = kFwdBlockKV;
    std::snprintf(out->fingerprint, sizeof(out->fingerprint), "%s %s", RLK_SOURCE_HASH, RLK_BUILD_FLAGS);
    return RLK_OK;
}

rlk_status rlk_op_trace_enable(int enable) {
    std::lock_guard<std::mutex> lk(g_op.mu);
    g_op.on.store(enable != 0);
    g_op.head = g_op.count = 0;
    g_op.seq = 0;
    return RLK_OK;
}

int32_t rlk_op_trace_count(void) {
    std::lock_guard<std::mutex> lk(g_op.mu);
    return g_op.count;
}

rlk_status rlk_op_trace_read(int32_t i, rlk_op_record* out) {
    if (out == nullptr) return RLK_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(g_op.mu);
    if (i < 0 || i >= g_op.count) return RLK_ERR_INVALID_ARG;
    *out = g_op.ring[(g_op.head + i) % RLK_OP_TRACE_CAP];
    return RLK_OK;
}

const char* rlk_strerror(int status) {
    switch (status) {
        case RLK_OK: return "ok";
        case RLK_ERR_INVALID_ARG: return "invalid argument";
        case RLK_ERR_UNSUPPORTED: return "unsupported configuration (fails closed)";
        case RLK_ERR_ALIGNMENT: return "device pointer not 16-byte aligned";
        case RLK_ERR_WORKSPACE: return "workspace too small";
        case RLK_ERR_CUDA: return "CUDA error";
        case RLK_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
        default: return "unknown status";
    }
}

rlk_status rlk_kernel_timing(int enable) {
    std::lock_guard<std::mutex> lk(g_timing.mu);
    g_timing.on = enable != 0;
    for (int i = 0; i < kNumKernelIds; ++i) g_timing.count[i] = 0;
    return RLK_OK;
}

rlk_status rlk_kernel_timing_read(int kernel_id, double* total_ms, int32_t* launches) {
    if (kernel_id < 0 || kernel_id >= kNumKernelIds || total_ms == nullptr || launches == nullptr)
        return RLK_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(g_timing.mu);
    double sum = 0.0;
    const int n = g_timing.count[kernel_id];
    for (int i = 0; i < n; ++i) {
        float ms = 0.0f;
        if (cudaEventSynchronize(g_timing.ev[kernel_id][2 * i + 1]) != cudaSuccess) return RLK_ERR_CUDA;
        if (cudaEventElapsedTime(&ms, g_timing.ev[kernel_id][2 * i], g_timing.ev[kernel_id][2 * i + 1]) !=
            cudaSuccess)
            return RLK_ERR_CUDA;
        sum += ms;
    }
    *total_ms = sum;
    *launches = n;
    return RLK_OK;
}

}  // extern "C"

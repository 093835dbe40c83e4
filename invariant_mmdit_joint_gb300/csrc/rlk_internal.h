// Internal host/device interface between the translation units of
// librlk_joint_attn.so. Not part of the public ABI (include/rlk_joint_attn.h).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/rlk_joint_attn.h"

namespace rlk {

constexpr int kHeadDim = 128;
constexpr int kPairs = kHeadDim / 2;       // RoPE pairs per head row
constexpr int kAxis0Pairs = 8;             // frame axis: 16 dims
constexpr int kAxis1Pairs = 28;            // row axis: 56 dims

// Geometry of one call, derived from rlk_ja_shape on the host. Every kernel
// receives it by value. Tile boundaries are functions of (T_txt, grid) only.
struct Geom {
    int B, H, S, T_txt, T_img, gh, gw;
    int txt_off;        // o = max(gh/2, gw/2): position of text token 0
    int ctr_h, ctr_w;   // ceil(gh/2), ceil(gw/2): image centring
    int p_lo, n_pos;    // cos/sin table covers positions [p_lo, p_lo + n_pos)
    float eps, theta;
    // query / key tiles of 128, segment aligned: text tiles from token 0,
    // image tiles from token T_txt; nq_pad = 128 * (ntq_txt + ntq_img) slots
    // per (b, h) in the tile-padded layout of lse2 and Delta
    int ntq_txt, ntq_img, nq_pad;
};

// Per-sample valid text lengths travel by value as a kernel argument.
struct ValidLen {
    int32_t L[RLK_MAX_BATCH];
};

// A bf16 activation of shape [B, tokens, H, 128] given as its text rows and
// its image rows, each with its own batch stride in tokens: either one
// concatenated tensor (text then image; both strides S) or two separate
// tensors [B, T_txt, H, 128] and [B, T_img, H, 128] (strides T_txt, T_img),
// so a caller holding the two streams apart needs no concatenation copy.
struct SegBf16 {
    uint16_t* p[2];         // element 0 of the text rows / of the image rows
    long long bstride[2];   // tokens from sample b to sample b + 1
};

// Position of token n on axis a (0 frame, 1 row, 2 column).
__host__ __device__ inline int token_pos(const Geom& g, int n, int a) {
    if (n < g.T_txt) return g.txt_off + n;
    if (a == 0) return 0;
    int i = n - g.T_txt;
    int r = i / g.gw;
    return a == 1 ? r - g.ctr_h : (i - r * g.gw) - g.ctr_w;
}

// Address of (b, token n, head h, dim 0) in its segment's buffer.
// (Selects on constant indices, not t.p[seg]: a runtime index into a kernel
// parameter's array would make the compiler copy it to local memory.)
__host__ __device__ inline uint16_t* seg_row(const SegBf16& t, const Geom& g, int b, int n, int h) {
    const bool img = n >= g.T_txt;
    uint16_t* const base = img ? t.p[1] : t.p[0];
    const long long bs = img ? t.bstride[1] : t.bstride[0];
    const long long nn = img ? n - g.T_txt : n;
    return base + (((long long)b * bs + nn) * g.H + h) * kHeadDim;
}

// The two segment views of one concatenated [B, S, H, 128] tensor, and of
// two separate stream tensors.
inline SegBf16 seg_concat(const void* base, const Geom& g) {
    SegBf16 t;
    uint16_t* p = static_cast<uint16_t*>(const_cast<void*>(base));
    t.p[0] = p;
    t.p[1] = p + (size_t)g.T_txt * g.H * kHeadDim;
    t.bstride[0] = t.bstride[1] = g.S;
    return t;
}
inline SegBf16 seg_split(const void* txt, const void* img, const Geom& g) {
    SegBf16 t;
    t.p[0] = static_cast<uint16_t*>(const_cast<void*>(txt));
    t.p[1] = static_cast<uint16_t*>(const_cast<void*>(img));
    t.bstride[0] = g.T_txt;
    t.bstride[1] = g.T_img;
    return t;
}

// Axis owning RoPE pair k (dims 2k, 2k+1) of a 128-wide head row.
__host__ __device__ inline int pair_axis(int k) {
    return k < kAxis0Pairs ? 0 : (k < kAxis0Pairs + kAxis1Pairs ? 1 : 2);
}

// Kernel ids used by the launch timing hooks (see rlk_kernel_timing()).
enum KernelId {
    kKRopeTable = 0, kKPrologue = 1, kKAttnFwd = 2, kKBwdPre = 3,
    kKBwdDkDv = 4, kKBwdDq = 5, kKNormRopeBwd = 6, kKDgFold = 7,
    kKQkGemm = 8, kKSoftmax = 9, kKAvGemm = 10, kKAttnFwdShard = 11, kKQkvGemm = 12, kKOutGemm = 13,
    kKDpGemm = 14, kKSoftmaxBwd = 15, kKKeyGemm = 16, kKQueryGemm = 17, kKNormRopeBwdQ = 18, kNumKernelIds = 19
};

// Launch timing hooks (rlk_host.cu): bracket one launch with events.
// timing_begin also adds the kernel to the open operator-trace record.
void timing_begin(int kernel_id, cudaStream_t s);
void timing_end(int kernel_id, cudaStream_t s);

// Operator trace (rlk_host.cu). Every C ABI entry point that can launch work
// opens a scope; the outermost scope of a thread owns one record, which the
// launches inside it fill and finish() appends to the log.
enum OpKind {
    kOpFwd = 0, kOpBwd, kOpFwdNoalloc, kOpNormRope, kOpQkGemm, kOpSoftmax, kOpAvGemm, kOpFwdShard,
    kOpFwdStreams, kOpBwdStreams, kOpQkvGemm, kOpFwdCtx, kOpOutGemm,
    kOpBwdStats, kOpSoftmaxBwd, kOpAvGemmBwd, kOpQkGemmBwd, kOpNormRopeBwd
};
class OpScope {
   public:
    OpScope(OpKind kind, const rlk_ja_shape* shape);
    ~OpScope();
    rlk_status finish(rlk_status st);

   private:
    bool owner_ = false;
    bool done_ = false;
};

// Forward entry-point steps (rlk_host.cu), shared by the regular and the
// allocation-free forward so both refuse the same arguments with the same
// status, in the same order:
//   fwd_validate  shape, valid lengths, null and 16-byte alignment of every
//                 pointer (ctx too when ctx_required; lse may be null);
//                 touches no device
//   device_check  the per-device check (sm_103, strict math); its first run
//                 on a device launches probes and refuses a capturing stream
//   fwd_run       the launches, on checked arguments
rlk_status fwd_validate(const rlk_ja_shape* shape, const void* q, const void* k, const void* v,
                        const float* g_q_txt, const float* g_k_txt, const float* g_q_img, const float* g_k_img,
                        const int32_t* txt_valid_len, const void* out, const float* lse, const void* ctx,
                        bool ctx_required, Geom* g, ValidLen* vl);
rlk_status device_check(void* stream);
rlk_status fwd_run(const Geom& g, const ValidLen& vl, const void* q, const void* k, const void* v,
                   const float* g_q_txt, const float* g_k_txt, const float* g_q_img, const float* g_k_img,
                   void* out, float* lse, void* ctx, void* stream);
// Bytes of the forward context of a checked geometry.
size_t ctx_bytes_of(const Geom& g);

// ---- launchers (each returns the cudaGetLastError() of its launch) ----
// k_prologue.cu
cudaError_t launch_rope_table(const Geom& g, float2* tab, cudaStream_t s);
cudaError_t launch_prologue(const Geom& g, const SegBf16& q, const SegBf16& k,
                            const float* const gains[4], const float2* tab,
                            uint16_t* qh, uint16_t* kh, float* rq, float* rk,
                            cudaStream_t s);
cudaError_t launch_bwd_pre(const Geom& g, const SegBf16& out, const SegBf16& dout,
                           const float* lse, float* lse2_p, float* delta_p, cudaStream_t s);
// dK from dk^ (fp32 [B, H, S, 128]) and the k gain-gradient partials into dgt
cudaError_t launch_norm_rope_bwd_k(const Geom& g, const SegBf16& k, const float* gk_txt, const float* gk_img,
                                   const float2* tab, const float* rk, const float* dkh, const SegBf16& dk,
                                   float* dgt, cudaStream_t s);
cudaError_t launch_dg_fold(const Geom& g, const float* dgt, float* dg_partial,
                           float* dg, cudaStream_t s);
int probe_prologue_tu(void);
int read_and_clear_status_prologue(cudaStream_t s);
// one warp whose bounded wait on a barrier nothing completes gives up after limit_ms
cudaError_t launch_wait_timeout_probe(int limit_ms, cudaStream_t s);

// k_attn_fwd.cu
cudaError_t launch_attn_fwd(const Geom& g, const ValidLen& vl, const uint16_t* qh,
                            const uint16_t* kh, const SegBf16& v, const SegBf16& out,
                            float* lse, cudaStream_t s);
// One key shard of the forward: column blocks [blk_begin, blk_end) of the
// fused order, with the online-softmax state passed from and to the
// neighbouring shards (state: m, l fp32 [rows] then O fp32 [rows, 128]);
// out is null except for the last shard.
cudaError_t launch_attn_fwd_shard(const Geom& g, const ValidLen& vl, const uint16_t* qh,
                                  const uint16_t* kh, const SegBf16& v, int blk_begin, int blk_end,
                                  const float* state_in, float* state_out, const SegBf16* out,
                                  float* lse, cudaStream_t s);
int probe_fwd_tu(void);
int read_and_clear_status_fwd(cudaStream_t s);

// k_attn_bwd.cu
// What the RoPE / RMSNorm backward of the query rows (in the dQ kernel's
// epilogue) reads and writes: the pre-norm q (bf16 [B, S, H, 128] per
// segment), its RMSNorm factors rq [B, H, S], the gains (q_txt, k_txt,
// q_img, k_img), the cos/sin table; dQ (bf16, per segment) and the q half
// of the gain-gradient partials dgt [B, H, 2 (q, k), n_tiles, 4 (32-row
// quarters), 128].
struct NormRopeBwdIo {
    SegBf16 q, dq;
    const float* rq;
    const float* gains[4];
    const float2* tab;
    float* dgt;
};
// dkh: dk^ (the gradient of the rotated, normalised keys, times 1/sqrt(128)),
// fp32 [B, H, S, 128], written by dkdv and read by norm_rope_bwd_k.
// Both run over the (sample, head) pairs bh0 .. bh0 + n_pairs - 1 (b * H + h
// order); ds_tiles holds the n_pairs x nq x nq dS^T images of that range.
cudaError_t launch_attn_bwd_dkdv(const Geom& g, const ValidLen& vl, const uint16_t* qh,
                                 const uint16_t* kh, const SegBf16& v,
                                 const SegBf16& dout, const float* lse2_p,
                                 const float* delta_p, const SegBf16& dv, float* dkh,
                                 uint8_t* ds_tiles, int bh0, int n_pairs, cudaStream_t s);
cudaError_t launch_attn_bwd_dq(const Geom& g, const ValidLen& vl, const uint16_t* kh,
                               const uint8_t* ds_tiles, const NormRopeBwdIo& nr, int bh0, int n_pairs,
                               cudaStream_t s);
int probe_bwd_tu(void);
int read_and_clear_status_bwd(cudaStream_t s);

// k_attn_unfused.cu: the standalone joint_attn_qk_gemm, joint_attn_softmax
// and joint_attn_av_gemm operators (layouts in that file's header)
cudaError_t launch_qk_gemm(const Geom& g, const ValidLen& vl, const uint16_t* qh, const uint16_t* kh,
                           float* scores, cudaStream_t s);
cudaError_t launch_softmax(const Geom& g, const ValidLen& vl, const float* scores, uint16_t* p,
                           float* alpha, float* l, float* lse, cudaStream_t s);
cudaError_t launch_av_gemm(const Geom& g, const ValidLen& vl, const uint16_t* p, const float* alpha,
                           const float* l, const SegBf16& v, const SegBf16& out, cudaStream_t s);
// dP = dO V^T in the qk_gemm tiling, fp32 [B, H, S, n_tiles * 128] (the
// backward of joint_attn_av_gemm, first half)
cudaError_t launch_dp_gemm(const Geom& g, const ValidLen& vl, const SegBf16& dout, const SegBf16& v, float* dp,
                           cudaStream_t s);
int probe_unfused_tu(void);
int read_and_clear_status_unfused(cudaStream_t s);

// k_attn_unfused_bwd.cu: the standalone backward operators (layouts in that
// file's header). lse2 / delta: the tile-padded arrays of launch_bwd_pre.
cudaError_t launch_softmax_bwd(const Geom& g, const ValidLen& vl, const float* scores, const float* lse2,
                               const float* delta, const float* dp, uint16_t* p, uint16_t* ds, cudaStream_t s);
cudaError_t launch_dv_gemm(const Geom& g, const ValidLen& vl, const uint16_t* p, const SegBf16& dout,
                           const SegBf16& dv, cudaStream_t s);
cudaError_t launch_dhat_gemms(const Geom& g, const ValidLen& vl, const uint16_t* ds, const uint16_t* qh,
                              const uint16_t* kh, float* dqh, float* dkh, cudaStream_t s);
cudaError_t launch_norm_rope_bwd_q(const Geom& g, const SegBf16& q, const float* gq_txt, const float* gq_img,
                                   const float2* tab, const float* rq, const float* dqh, const SegBf16& dq,
                                   float* dgt, cudaStream_t s);
int probe_unfused_bwd_tu(void);
int read_and_clear_status_unfused_bwd(cudaStream_t s);

// k_qkv_gemm.cu: per-stream projection Y = X W^T + b (both streams in one
// launch), stored as bf16. QKV (out_proj false): W is [3C, C]; with
// qh != null the epilogue also runs qk_rmsnorm + multi_axis_rope into the
// context (q^, k^, r) from the table tab, and writes the pre-norm Q / K only
// if store_q / store_k. Output projection (out_proj true): W is [C, C] and
// every column goes to v.
cudaError_t launch_proj_gemm(const Geom& g, bool out_proj, const uint16_t* const x[2], const uint16_t* const w[2],
                             const uint16_t* const bias[2], const float* const gains[4], uint16_t* qh,
                             uint16_t* kh, float* rq, float* rk, const float2* tab, const SegBf16& q,
                             const SegBf16& k, const SegBf16& v, bool store_q, bool store_k, cudaStream_t s);
int probe_qkv_tu(void);
int read_and_clear_status_qkv(cudaStream_t s);

// Tile geometry of the attention kernels (reported by the trace record).
extern const int kFwdBlockQ, kFwdBlockKV;

}  // namespace rlk

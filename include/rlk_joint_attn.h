/*
 * rlk_joint_attn.h -- C ABI of the deterministic, batch-invariant joint
 * attention of a Qwen-Image MMDiT block (forward and backward), with its
 * QK-RMSNorm + three-axis RoPE prologue, for one NVIDIA GB300 (sm_103).
 *
 * What the operation is (sources are the RL-Kernel GitHub threads):
 *   "[RFC][Qwen-Image][CUDA/ROCm] WS1/WS2 kernel roadmap ... #386",
 *     Model contract table: 24 heads x 128; joint non-causal attention over
 *     [text, image]; padded prompts need a key mask; learned-gain per-head
 *     RMSNorm (eps 1e-6) on Q and K before RoPE; RoPE axes [16, 56, 56],
 *     theta 10000, centred spatial indices, text offset max(H/2, W/2).
 *     Numerical requirements: fixed reduction trees, FP32 accumulators, no
 *     split-K / stream-K / split-KV / atomics, no TF32 or fast math, one
 *     FP32->BF16 cast at the output, batch invariance, fail closed.
 *     WS1 table rows qk_rmsnorm, multi_axis_rope, joint_attn_qk_gemm,
 *     joint_attn_softmax, joint_attn_av_gemm, joint_attention_fused.
 *   "[RFC] [Qwen-Image] WS1 Single-GPU Kernel List", Kernel table: the same
 *     rows with "fwd + bwd"; rule 7 (trace records).
 *
 * Notation: B samples, H heads, D = 128, T_txt text tokens (the padded text
 * length, equal for all samples), T_img = grid_h * grid_w image tokens,
 * S = T_txt + T_img. Token n < T_txt is text token n; token T_txt + r*grid_w + c
 * is image token (row r, column c). L_b = valid text length of sample b: text
 * keys L_b <= n < T_txt are masked (padded prompt tokens).
 *
 * Per (sample b, head h), with x a row of Q or K:
 *   qk_rmsnorm:      r = 1 / sqrt(mean_d(x_d^2) + eps);  y = x * r * g
 *                    (g = the stream's gain: text rows use *_txt, image *_img)
 *   multi_axis_rope: dims [0,16) follow the frame axis, [16,72) the row axis,
 *                    [72,128) the column axis; pair (2j, 2j+1) of an axis
 *                    block of width d_a turns by pos_a * theta^(-2j/d_a).
 *                    Image token (r, c): pos = (0, r - ceil(gh/2), c - ceil(gw/2));
 *                    text token t: pos = (o+t, o+t, o+t), o = max(gh/2, gw/2)
 *                    (integer halves).
 *   attention:       s_ij = qh_i . kh_j / sqrt(128) over valid keys j;
 *                    P = softmax_j(s); O = P V; lse_i = log sum_j exp(s_ij).
 *
 * Layouts (all row-major, innermost index last):
 *   q, k, v, out, dout, dq, dk, dv : bf16 [B, S, H, D]  (D contiguous, then H)
 *   lse                            : fp32 [B, H, S]      (natural log)
 *   gains                          : fp32 [D] each, four vectors
 *   dg_partial                     : fp32 [B, H, 4, D]   slots (q_txt, k_txt, q_img, k_img)
 *   dg                             : fp32 [4, D]         same slots
 *   txt_valid_len                  : int32 [B], HOST memory, 0 <= L_b <= T_txt
 *
 * Ownership and streams: the caller owns and allocates every buffer (inputs,
 * outputs, ctx, workspace) on the current CUDA device. The library never
 * allocates or frees device memory and never synchronises, except in
 * rlk_joint_attn_check_status(). Every call enqueues its kernels on `stream`
 * (a cudaStream_t passed as void*; NULL = the legacy default stream) and
 * returns as soon as they are enqueued. Host arrays are read before return.
 *
 * CUDA graphs: every entry point may be captured into a CUDA graph (stream
 * capture), and a replay performs the same arithmetic as the eager call, so
 * it gives the same bytes. Host arrays (txt_valid_len) and the tensor maps are
 * taken by value at capture time. The first call on a device runs one-time
 * checks that launch and synchronise; called inside a capture it returns
 * RLK_ERR_UNSUPPORTED instead, so make one eager call first.
 *
 * Errors: every entry point returns an rlk_status. On any validation error
 * nothing is launched and no output is touched. Unsupported configurations
 * fail closed with RLK_ERR_UNSUPPORTED; there is no fallback path.
 *
 * Determinism: each output tile is produced by exactly one CTA whose visit
 * order over the other operand is fixed (text tiles from token 0, then image
 * tiles from token T_txt, ascending; tiles with no valid key are skipped).
 * Tile geometry depends on nothing but (T_txt, grid_h, grid_w), so a row's
 * bytes are the same for any B, any batch position, any run, and whether or
 * not lse is requested.
 */
#ifndef RLK_JOINT_ATTN_H
#define RLK_JOINT_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum rlk_status {
    RLK_OK = 0,
    RLK_ERR_INVALID_ARG = 1,   /* null pointer, bad size, L_b outside [0, T_txt] */
    RLK_ERR_UNSUPPORTED = 2,   /* D != 128, axes != {16,56,56}, not sm_103, fast-math build */
    RLK_ERR_ALIGNMENT = 3,     /* a device pointer not 16-byte aligned */
    RLK_ERR_WORKSPACE = 4,     /* workspace below rlk_joint_attn_bwd_workspace_min_bytes() */
    RLK_ERR_CUDA = 5,          /* a CUDA runtime/driver call failed */
    RLK_ERR_DEVICE_TIMEOUT = 6 /* a bounded device-side wait gave up (see check_status) */
} rlk_status;

/* Largest batch one call accepts (valid lengths travel as kernel arguments). */
#define RLK_MAX_BATCH 256

/* Shape limits (otherwise RLK_ERR_INVALID_ARG): T_txt + grid_h * grid_w
 * <= 2^20 tokens, and B * H * 128 * (ceil(T_txt / 128) + ceil(grid_h *
 * grid_w / 128)) < 2^31 rows (q alone would then exceed 512 GB). */
typedef struct rlk_ja_shape {
    int32_t B;        /* samples, 1 .. RLK_MAX_BATCH */
    int32_t T_txt;    /* padded text length, >= 0 */
    int32_t grid_h;   /* image token rows, >= 1 */
    int32_t grid_w;   /* image token columns, >= 1 */
    int32_t H;        /* heads, >= 1 */
    int32_t D;        /* head dim; must be 128 */
    float eps;        /* RMSNorm epsilon (the model uses 1e-6), > 0 */
    float theta;      /* RoPE base (the model uses 10000), > 1 */
    int32_t axes[3];  /* RoPE axis split; must be {16, 56, 56} */
} rlk_ja_shape;

/* Bytes of the forward context `ctx`: normed+rotated q and k (bf16
 * [B, H, S, D] each), the RMSNorm factors r of q and k (fp32 [B, H, S] each)
 * and the cos/sin table. The forward writes it; the backward reads it. Returns
 * 0 for an invalid shape. */
size_t rlk_joint_attn_ctx_bytes(const rlk_ja_shape* shape);

/* Bytes of the backward scratch `workspace`: lse * log2(e) and
 * rowsum(dO * O) (fp32, one 128-slot block per query tile of each (sample,
 * head)), the fp32 gradient of the rotated k ([B, H, S, D]), the
 * gain-gradient partials (fp32 [B, H, 2, n_tiles, 4, D]: q and k, per
 * 128-token tile and 32-row quarter) and the bf16 score gradients dS as 128 x
 * 128 tiles (B * H * n_tiles^2 * 32 KiB, n_tiles = ceil(T_txt / 128) +
 * ceil(grid_h * grid_w / 128); 1.8 GB for B = 2, H = 24 at 1024 x 1024).
 * Returns 0 for an invalid shape. */
size_t rlk_joint_attn_bwd_workspace_bytes(const rlk_ja_shape* shape);

/* The smallest backward workspace: everything above but the dS tiles of a
 * single (sample, head) pair (n_tiles^2 * 32 KiB; 37.9 MB at 1024 x 1024,
 * 52.4 MB at 1328 x 1328). A backward given less than
 * rlk_joint_attn_bwd_workspace_bytes() but at least this runs its dK/dV and
 * dQ kernels over consecutive groups of (sample, head) pairs, in b * H + h
 * order, each group as large as the dS tiles the workspace holds, reusing
 * the one region; the results are byte-identical to the single-group run (a
 * pair's arithmetic never depends on its group), only the launch count and
 * the time change. Returns 0 for an invalid shape. */
size_t rlk_joint_attn_bwd_workspace_min_bytes(const rlk_ja_shape* shape);

/* Forward: rows qk_rmsnorm, multi_axis_rope, joint_attn_qk_gemm,
 * joint_attn_softmax and joint_attn_av_gemm of the RFC's WS1 table, fused.
 *   q, k, v         device bf16 [B, S, H, D], read only
 *   g_q_txt ... g_k_img  device fp32 [D] each, read only
 *   txt_valid_len   HOST int32 [B]
 *   out             device bf16 [B, S, H, D], written (every row, padded
 *                   text query rows included)
 *   lse             device fp32 [B, H, S] or NULL (then not written; `out`
 *                   bytes do not change)
 *   ctx             device, rlk_joint_attn_ctx_bytes() bytes, written; keep
 *                   it for the backward
 * All device pointers must be 16-byte aligned. */
rlk_status rlk_joint_attn_fwd(const rlk_ja_shape* shape,
                              const void* q, const void* k, const void* v,
                              const float* g_q_txt, const float* g_k_txt,
                              const float* g_q_img, const float* g_k_img,
                              const int32_t* txt_valid_len,
                              void* out, float* lse, void* ctx, void* stream);

/* Size of the fixed device scratch used by rlk_joint_attn_fwd_noalloc():
 * 64 MiB, enough for one 1024x1024 image with 24 heads and 256 text tokens
 * (rlk_joint_attn_ctx_bytes() of that shape is about 54 MB). */
#define RLK_NOALLOC_SCRATCH_BYTES (64u << 20)

/* Forward without any caller-provided scratch and without allocating.
 * The pages have no counterpart to this entry point; it exists for callers
 * that cannot or may not allocate device memory on the call path (a plugin
 * host that gives its plugins no workspace, a serving process whose memory
 * pool owns the whole device, code that must not pay the synchronisation a
 * cudaMalloc / cudaFree can bring).
 * Arguments, layouts and results are those of rlk_joint_attn_fwd() minus
 * `ctx`: the forward context lives in a file-scope device array of
 * RLK_NOALLOC_SCRATCH_BYTES that every GPU loading the library holds until
 * the process exits. Nothing is allocated or freed.
 *   - Arguments are checked exactly as rlk_joint_attn_fwd() checks them,
 *     in the same order and with the same status codes (ctx aside).
 *   - Shapes whose rlk_joint_attn_ctx_bytes() exceeds RLK_NOALLOC_SCRATCH_BYTES
 *     return RLK_ERR_WORKSPACE before anything is launched.
 *   - Every call looks the array's device address up on the current device
 *     (nothing is cached, so a reset device context leaves no stale
 *     address); the first lookup on a device also loads the library's
 *     device code there, so make the first call on each device before any
 *     stream capture.
 *   - All calls share the one array and keep the last call's contents, so
 *     calls whose kernels overlap on the GPU (other streams, other host
 *     threads) race: serialise them. The context is not kept for a backward:
 *     this entry point serves forward-only (inference) use. */
rlk_status rlk_joint_attn_fwd_noalloc(const rlk_ja_shape* shape,
                                      const void* q, const void* k, const void* v,
                                      const float* g_q_txt, const float* g_k_txt,
                                      const float* g_q_img, const float* g_k_img,
                                      const int32_t* txt_valid_len,
                                      void* out, float* lse, void* stream);

/* Backward of the whole path: gradients of sum(out * dout).
 *   q, k, v, gains, txt_valid_len  as in the forward (same values)
 *   out, lse, ctx   what the forward wrote for these inputs (lse required)
 *   dout            device bf16 [B, S, H, D]
 *   dq, dk, dv      device bf16 [B, S, H, D], written; masked keys get 0
 *   dg_partial      device fp32 [B, H, 4, D] or NULL: per (sample, head)
 *                   gain gradients, each summed over one stream's tokens in
 *                   a fixed order; these are batch invariant
 *   dg              device fp32 [4, D], written: dg_partial summed over h
 *                   ascending, then over b ascending
 *   workspace       device scratch of >= rlk_joint_attn_bwd_workspace_min_bytes()
 *                   (rlk_joint_attn_bwd_workspace_bytes() runs every pair in
 *                   one group; less runs the pairs in groups, same bytes);
 *                   below the minimum: RLK_ERR_WORKSPACE, nothing launched
 * Note: a padded text query row with nonzero dout feeds the key and value
 * gradients of the valid keys, as the mathematics says. */
rlk_status rlk_joint_attn_bwd(const rlk_ja_shape* shape,
                              const void* q, const void* k, const void* v,
                              const float* g_q_txt, const float* g_k_txt,
                              const float* g_q_img, const float* g_k_img,
                              const int32_t* txt_valid_len,
                              const void* out, const void* dout,
                              const float* lse, const void* ctx,
                              void* dq, void* dk, void* dv,
                              float* dg_partial, float* dg,
                              void* workspace, size_t workspace_bytes,
                              void* stream);

/* ---------------------------------------------------------------------------
 * The path's operators one at a time. The RFC's WS1 table lists
 * qk_rmsnorm, multi_axis_rope, joint_attn_qk_gemm, joint_attn_softmax and
 * joint_attn_av_gemm as separate rows and requires joint_attention_fused to
 * be a byte-equal fusion of the three attention operators; the WS1
 * Single-GPU Kernel List asks the same of the fused kernel. The four calls
 * below, chained as
 *     rlk_qk_norm_rope -> rlk_joint_attn_qk_gemm -> rlk_joint_attn_softmax
 *                      -> rlk_joint_attn_av_gemm
 * produce `out` and `lse` bytes identical to rlk_joint_attn_fwd() on the same
 * inputs, for every shape, batch composition and run.
 *
 * Intermediate layouts (n_tiles = ceil(T_txt/128) + ceil(grid_h*grid_w/128);
 * column block t holds key tile t: text tiles from token 0, then image tiles
 * from token T_txt, 128 keys each):
 *   scores  fp32 [B, H, S, n_tiles * 128]  raw q^ . k^ (the 1/sqrt(128)
 *           scale is applied inside the softmax, folded with log2(e) into
 *           the exponent's one rounding, exactly as the fused kernel does)
 *   P       bf16 [B, H, S, n_tiles * 128]  exp(s_ij - m_i(t)) where m_i(t)
 *           is row i's running reference maximum when key tile t is visited
 *   alpha   fp32 [B, H, S, n_tiles]        factor by which the running O and
 *           row sum are rescaled at key tile t (1 when the reference stays)
 *   l       fp32 [B, H, S]                 final row sum, so that
 *           O_i = sum_t (prod_{t' > t} alpha_i(t')) P_i(t) V(t) / l_i
 *   lse     fp32 [B, H, S]                 natural-log logsumexp
 * Column blocks of text tiles past ceil(L_b/128) are not written; inside a
 * visited block, masked key columns (and columns past the key's segment)
 * hold -inf in `scores` and exactly 0 in P, so every written byte depends
 * only on the sample's own inputs. Sizes come from
 * rlk_joint_attn_unfused_bytes(). Pointer rules, errors and streams are those
 * of the fused calls: every device pointer 16-byte aligned, validation errors
 * launch nothing. */
#define RLK_UNFUSED_SCORES 0
#define RLK_UNFUSED_P 1
#define RLK_UNFUSED_ALPHA 2
#define RLK_UNFUSED_ROWS 3 /* one of l or lse */
/* the standalone backward's intermediates (see rlk_joint_attn_softmax_bwd()) */
#define RLK_UNFUSED_DP 4         /* dP, fp32, the layout of `scores` */
#define RLK_UNFUSED_DS 5         /* P or dS, bf16, the layout of P */
#define RLK_UNFUSED_STATS 6      /* lse2 and Delta, fp32 [2][B, H, n_tiles * 128] */
#define RLK_UNFUSED_DHAT 7       /* dq^ or dk^, fp32 [B, H, S, D] */
#define RLK_UNFUSED_GAIN_TILES 8 /* gain-gradient partials, fp32 [B, H, 2, n_tiles, 4, D] */

/* Bytes of one intermediate (`which` = RLK_UNFUSED_*); 0 for an invalid
 * shape or `which`. 3.6 GB of scores for B = 2, H = 24 at 1024 x 1024. */
size_t rlk_joint_attn_unfused_bytes(const rlk_ja_shape* shape, int which);

/* Rows qk_rmsnorm + multi_axis_rope: writes the normed, rotated q^ and k^
 * (bf16), their RMSNorm factors and the cos/sin table into `ctx`
 * (rlk_joint_attn_ctx_bytes() bytes), exactly as rlk_joint_attn_fwd() does
 * before its attention. Inputs as in rlk_joint_attn_fwd(). */
rlk_status rlk_qk_norm_rope(const rlk_ja_shape* shape, const void* q, const void* k,
                            const float* g_q_txt, const float* g_k_txt,
                            const float* g_q_img, const float* g_k_img,
                            void* ctx, void* stream);

/* Row joint_attn_qk_gemm: scores = q^ k^T for every key tile holding a valid
 * key, read from `ctx` as written by rlk_qk_norm_rope() or the forward. */
rlk_status rlk_joint_attn_qk_gemm(const rlk_ja_shape* shape, const void* ctx,
                                  const int32_t* txt_valid_len, float* scores,
                                  void* stream);

/* Row joint_attn_softmax: masked online softmax of `scores` over the key
 * tiles in the fixed order; writes P, alpha, l and (if non-NULL) lse. */
rlk_status rlk_joint_attn_softmax(const rlk_ja_shape* shape, const float* scores,
                                  const int32_t* txt_valid_len, void* p,
                                  float* alpha, float* l, float* lse, void* stream);

/* Row joint_attn_av_gemm: out = O / l from P, alpha and l (above) and
 * v (bf16 [B, S, H, D]); out bf16 [B, S, H, D], every row written. */
rlk_status rlk_joint_attn_av_gemm(const rlk_ja_shape* shape, const void* p,
                                  const float* alpha, const float* l, const void* v,
                                  const int32_t* txt_valid_len, void* out,
                                  void* stream);

/* ---------------------------------------------------------------------------
 * The backward of the same operators, one call per row, byte-equal in
 * composition to rlk_joint_attn_bwd(): the RFC #386 WS1 table marks every
 * attention row "fwd + bwd", and the fused backward's bytes are those of
 *     rlk_joint_attn_bwd_stats -> rlk_joint_attn_softmax_bwd (P)
 *       -> rlk_joint_attn_av_gemm_bwd (dV, dP)
 *       -> rlk_joint_attn_softmax_bwd (dS)
 *       -> rlk_joint_attn_qk_gemm_bwd (dq^, dk^)
 *       -> rlk_qk_norm_rope_bwd (dQ, dK, gain gradients)
 * run after the forward operators above (or the fused forward) on the same
 * inputs: dq, dk, dv, dg_partial and dg are identical to the fused call's.
 * Each step repeats the fused backward's arithmetic in its order (tiles of
 * 128, k-steps of 16, the same roundings); the products are taken with the
 * query index first where the fused kernel takes the key index first, which
 * gives the same bits on the tensor cores.
 * Intermediates (sizes from rlk_joint_attn_unfused_bytes()):
 *   stats  fp32: lse2 = lse * log2(e) [B, H, n_tiles * 128] (one 128-slot
 *          block per query tile, +inf past a segment), then Delta =
 *          rowsum(dO * O) in the same layout (0 past a segment)
 *   P, dS  bf16, the layout of the forward's P (visited key blocks only):
 *          P = exp2(s * log2(e) / sqrt(128) - lse2), the normalised
 *          probability (not the forward's lazily rescaled one); dS =
 *          P * (dP - Delta) with P in fp32; masked keys: P = 0
 *   dP     fp32, the layout of `scores`: dO V^T, every key of a visited
 *          block (masked ones too)
 *   dq^, dk^  fp32 [B, H, S, D]: dS k^ / sqrt(128) and dS^T q^ / sqrt(128)
 *          (masked keys: 0)
 * Pointer rules, errors and streams are those of the fused calls. */

/* lse2 and Delta into `stats` (the fused backward's preprocess). */
rlk_status rlk_joint_attn_bwd_stats(const rlk_ja_shape* shape, const void* out, const void* dout,
                                    const float* lse, float* stats, void* stream);

/* Row joint_attn_softmax, backward. With dp NULL: P from `scores` and
 * `stats` into p (required). With dp given: dS into ds (required), and P
 * into p if p is not NULL. */
rlk_status rlk_joint_attn_softmax_bwd(const rlk_ja_shape* shape, const float* scores, const float* stats,
                                      const float* dp, const int32_t* txt_valid_len, void* p, void* ds,
                                      void* stream);

/* Row joint_attn_av_gemm, backward: dP = dO V^T into dp and dV = P^T dO
 * (bf16 [B, S, H, D], masked keys 0) into dv; either may be NULL (not
 * both); p (from rlk_joint_attn_softmax_bwd) is required with dv. */
rlk_status rlk_joint_attn_av_gemm_bwd(const rlk_ja_shape* shape, const void* p, const void* v,
                                      const void* dout, const int32_t* txt_valid_len, void* dv,
                                      float* dp, void* stream);

/* Row joint_attn_qk_gemm, backward: dq^ and dk^ (fp32 [B, H, S, D]) from dS
 * and the q^, k^ in `ctx`. */
rlk_status rlk_joint_attn_qk_gemm_bwd(const rlk_ja_shape* shape, const void* ds, const void* ctx,
                                      const int32_t* txt_valid_len, float* dqh, float* dkh, void* stream);

/* Rows multi_axis_rope and qk_rmsnorm, backward: dQ, dK (bf16 [B, S, H, D])
 * from dq^, dk^, the inputs q, k, the gains and the RMSNorm factors and
 * cos/sin table in `ctx`; gain gradients as rlk_joint_attn_bwd() gives
 * them. gain_tiles: scratch of rlk_joint_attn_unfused_bytes(
 * RLK_UNFUSED_GAIN_TILES) bytes. */
rlk_status rlk_qk_norm_rope_bwd(const rlk_ja_shape* shape, const void* q, const void* k,
                                const float* g_q_txt, const float* g_k_txt,
                                const float* g_q_img, const float* g_k_img, const void* ctx,
                                const float* dqh, const float* dkh, void* dq, void* dk,
                                float* dg_partial, float* dg, float* gain_tiles, void* stream);

/* ---------------------------------------------------------------------------
 * The same forward and backward with the text and image streams in separate
 * buffers, so a caller whose per-stream projections produce them apart (the
 * RFC's Streams row: text and image keep separate weights; its WS1 rows
 * qkv_bias_gemm and attn_out_bias_gemm run per stream) needs no
 * concatenation copy before the attention or split copy after it.
 * Every activation is a pair: *_txt bf16 [B, T_txt, H, D] and *_img bf16
 * [B, grid_h * grid_w, H, D], each densely packed. *_img must be non-NULL;
 * *_txt may be NULL only when T_txt == 0. All other arguments, the results
 * and their bytes are exactly those of rlk_joint_attn_fwd() /
 * rlk_joint_attn_bwd() on the concatenation [text, image]. */
rlk_status rlk_joint_attn_fwd_streams(const rlk_ja_shape* shape,
                                      const void* q_txt, const void* q_img,
                                      const void* k_txt, const void* k_img,
                                      const void* v_txt, const void* v_img,
                                      const float* g_q_txt, const float* g_k_txt,
                                      const float* g_q_img, const float* g_k_img,
                                      const int32_t* txt_valid_len,
                                      void* out_txt, void* out_img, float* lse, void* ctx,
                                      void* stream);
rlk_status rlk_joint_attn_bwd_streams(const rlk_ja_shape* shape,
                                      const void* q_txt, const void* q_img,
                                      const void* k_txt, const void* k_img,
                                      const void* v_txt, const void* v_img,
                                      const float* g_q_txt, const float* g_k_txt,
                                      const float* g_q_img, const float* g_k_img,
                                      const int32_t* txt_valid_len,
                                      const void* out_txt, const void* out_img,
                                      const void* dout_txt, const void* dout_img,
                                      const float* lse, const void* ctx,
                                      void* dq_txt, void* dq_img, void* dk_txt, void* dk_img,
                                      void* dv_txt, void* dv_img,
                                      float* dg_partial, float* dg,
                                      void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * The attention's adjacent producer: row qkv_bias_gemm of the RFC's WS1
 * table (each stream's Q, K and V projections packed in one GEMM with a
 * bias; the WS1 kernel list: 3072 -> 3 x 3072, one weight set per stream), with qk_rmsnorm and
 * multi_axis_rope fused into its epilogue.
 *   x_txt, x_img   bf16 [B, T_txt, C] and [B, grid_h*grid_w, C], C = H * 128
 *   w_txt, w_img   bf16 [3C, C]: output feature rows (the nn.Linear layout),
 *                  Q features first (head-major: feature h*128 + d), then K, V
 *   b_txt, b_img   bf16 [3C]
 * Q, K, V = bf16(x w^T + b) per stream (fp32 accumulation in a fixed order,
 * one rounding). With `ctx` non-NULL the epilogue also writes the context
 * rlk_joint_attn_fwd() would write for these Q, K (the normed, rotated q^
 * and k^, the RMSNorm factors and the cos/sin table), byte for byte what
 * rlk_qk_norm_rope() gives on the stored Q, K; the gains are then required,
 * and the pre-norm Q and K are stored only if their buffers are given
 * (a backward needs them). With `ctx` NULL, Q and K are required and the
 * gains ignored. V is always stored. Outputs q_*, k_*, v_* are bf16
 * [B, T_s, H, 128]; a *_txt pointer may be NULL only when T_txt == 0. */
rlk_status rlk_qkv_bias_gemm(const rlk_ja_shape* shape,
                             const void* x_txt, const void* x_img,
                             const void* w_txt, const void* w_img,
                             const void* b_txt, const void* b_img,
                             const float* g_q_txt, const float* g_k_txt,
                             const float* g_q_img, const float* g_k_img, void* ctx,
                             void* q_txt, void* q_img, void* k_txt, void* k_img,
                             void* v_txt, void* v_img, void* stream);

/* The forward's attention from a context already holding q^ and k^ (written
 * by rlk_qkv_bias_gemm(), rlk_qk_norm_rope() or the forward): out and lse
 * are those of rlk_joint_attn_fwd_streams() on the same inputs. */
rlk_status rlk_joint_attn_fwd_ctx(const rlk_ja_shape* shape, const void* ctx,
                                  const void* v_txt, const void* v_img,
                                  const int32_t* txt_valid_len,
                                  void* out_txt, void* out_img, float* lse, void* stream);

/* The attention's adjacent consumer: row attn_out_bias_gemm of the RFC's
 * WS1 table (per-stream attention output projection 3072 -> 3072 + bias).
 *   o_txt, o_img   bf16 [B, T_txt, H, 128] and [B, grid_h*grid_w, H, 128]
 *                  (the forward's separate-stream output, read as [B, T_s, C])
 *   w_txt, w_img   bf16 [C, C] (nn.Linear layout: output feature rows)
 *   b_txt, b_img   bf16 [C]
 *   y_txt, y_img   bf16 [B, T_s, C], written: bf16(o w^T + b), fp32
 *                  accumulation over the input features in a fixed order.
 * A *_txt pointer may be NULL only when T_txt == 0. */
rlk_status rlk_attn_out_bias_gemm(const rlk_ja_shape* shape,
                                  const void* o_txt, const void* o_img,
                                  const void* w_txt, const void* w_img,
                                  const void* b_txt, const void* b_img,
                                  void* y_txt, void* y_img, void* stream);

/* Synchronises `stream`, then reads and clears the device-side error word
 * that bounded waits in the kernels set when they give up. Returns RLK_OK,
 * RLK_ERR_DEVICE_TIMEOUT, or RLK_ERR_CUDA if the stream reported an error. */
rlk_status rlk_joint_attn_check_status(void* stream);

/* Schedule of the fused forward's query tiles. It changes launch shape and
 * time only, never a byte of the results. The forward runs one CTA per SM
 * on pairs of 128-row query tiles of one (sample, head); by default the pairs
 * past the last full wave of CTAs run as two single-tile CTAs each, which
 * spreads the partial wave over twice the SMs.
 *   RLK_FWD_TILES_AUTO    (0)  that default
 *   RLK_FWD_TILES_PAIRS   (1)  every pair as one CTA
 *   RLK_FWD_TILES_SINGLE  (2)  every query tile as its own CTA
 * A query tile's arithmetic never depends on the tile it shares a CTA with,
 * so all three give identical bytes; the setting exists so that this can be
 * shown on any GPU, whatever its SM count. It is process-wide and applies to
 * later calls of every entry point that runs the fused forward (the
 * key-shard forward always runs pairs). Returns the previous policy, or -1
 * (nothing changed) for an unknown one. */
#define RLK_FWD_TILES_AUTO 0
#define RLK_FWD_TILES_PAIRS 1
#define RLK_FWD_TILES_SINGLE 2
int32_t rlk_fwd_tile_schedule(int32_t policy);

/* Self-test of the failure path: enqueues on `stream` one warp that waits,
 * through the same bounded mbarrier wait the kernels use, on a barrier that
 * nothing completes. After limit_ms (1 .. 2000) it gives up and records the
 * failure in the device status word, so the next
 * rlk_joint_attn_check_status() returns RLK_ERR_DEVICE_TIMEOUT (and clears
 * it); nothing faults and the context stays usable. RLK_ERR_INVALID_ARG
 * for a limit out of range. */
rlk_status rlk_selftest_wait_timeout(int32_t limit_ms, void* stream);

/* Runs, on the current device, a probe kernel compiled in each translation
 * unit with that unit's flags: a subnormal product must survive, and
 * division, square root and expf must keep IEEE / library accuracy. These
 * all change under --use_fast_math (nvcc defines no macro for it in device
 * code). Returns 1 if every unit is strict, 0 if not, -1 on a CUDA error.
 * The first forward/backward call on a device runs it and fails closed with
 * RLK_ERR_UNSUPPORTED if it returns 0.
 * Source: PR #537 (adaln_mod_projection) review thread on the strict-math
 * check, which replaced a macro test by a probe kernel. */
int rlk_strict_math_compiled(void);

typedef struct rlk_ja_trace {
    char backend[32];          /* e.g. "sm_103a" + engine name */
    char reduction_order[160]; /* how each sum is ordered */
    char accumulator[16];      /* "fp32" */
    int32_t split_k;           /* 0: no split-K / stream-K / split-KV */
    int32_t atomics;           /* 0: no atomic accumulation */
    int32_t tf32;              /* 0: TF32 off */
    int32_t strict_math;       /* rlk_strict_math_compiled() at trace time */
    int32_t block_q;           /* query rows per forward tile */
    int32_t block_kv;          /* keys per forward tile */
    char fingerprint[96];      /* source hash and build flags */
} rlk_ja_trace;

/* Fills the trace record of the WS1 kernel list's rule 7 (reduction order,
 * accumulator precision, split-K state, TF32 state, kernel fingerprint,
 * selected backend). */
rlk_status rlk_joint_attn_trace(rlk_ja_trace* out);

/* ---------------------------------------------------------------------------
 * The fused forward over one key shard, for ring-ordered sequence
 * parallelism. The RFC's WS2 table asks sp_attention_ring to fix both the
 * order of the global blocks and the order of merging partial states, and its numerical
 * requirements ask strict replay and topology invariance to keep byte
 * equality. Here the global blocks are the forward's own key tiles (column
 * block t = key tile t: text tiles from token 0, then image tiles from token
 * T_txt, 128 keys each; n_tiles = ceil(T_txt/128) + ceil(grid_h*grid_w/128)),
 * and the partial state -- per query row the running reference maximum m,
 * the row sum l and the unnormalised output O -- is handed from shard to
 * shard in ascending block order. Any split of [0, n_tiles) into shards
 * [b_0 = 0, b_1), [b_1, b_2), ..., [b_k, n_tiles), run in that order, gives
 * `out` and `lse` bytes identical to rlk_joint_attn_fwd() (one GPU emulates
 * what ranks holding consecutive key shards would do).
 *   ctx           as written by rlk_qk_norm_rope() or the forward
 *   v             device bf16 [B, S, H, D]
 *   blk_begin, blk_end   the shard, 0 <= blk_begin < blk_end <= n_tiles
 *   state_in      the previous shard's state_out; NULL iff blk_begin == 0
 *   state_out     rlk_joint_attn_state_bytes() bytes; NULL iff this is the
 *                 last shard (blk_end == n_tiles). It may equal state_in.
 *   out, lse      written by the last shard only (out required there, lse
 *                 optional); NULL for the others
 * The state is opaque: fp32 m (log2 units) [B, H, S], l [B, H, S], then
 * O [B, H, S, D]. Text blocks past a sample's valid keys are skipped as in
 * the fused forward; a shard with no valid key for a sample passes its
 * state through. */
size_t rlk_joint_attn_state_bytes(const rlk_ja_shape* shape);
rlk_status rlk_joint_attn_fwd_shard(const rlk_ja_shape* shape, const void* ctx, const void* v,
                                    const int32_t* txt_valid_len, int32_t blk_begin,
                                    int32_t blk_end, const float* state_in, float* state_out,
                                    void* out, float* lse, void* stream);

/* ---------------------------------------------------------------------------
 * Operator trace: one record per call. The RFC's Foundation table asks for
 * an operator trace that records the requested and actual backend, kernel
 * identity, arithmetic policy and fallback state (qwenimage_operator_trace);
 * the WS1 kernel list's rule 7 asks trace records to carry the reduction
 * order, accumulator precision, Split-K / Stream-K state, TF32 state, kernel
 * fingerprint and selected backend, and says there is no silent fallback.
 * While tracing is on, every entry point that can launch work (the fused
 * forward and backward with concatenated or separate streams, the
 * allocation-free forward, the key-shard and from-context forwards, the
 * QKV and output projections and the standalone operators) appends one
 * record when it returns, including calls refused
 * during validation (status != RLK_OK, no kernel listed, actual backend
 * "none"). The kernels listed are the ones the call enqueued, in launch
 * order. Records live in a ring of RLK_OP_TRACE_CAP entries in host memory;
 * the oldest is dropped first. Thread safe; nested calls (the allocation-free
 * forward calling the regular one) produce one record. */
#define RLK_OP_TRACE_CAP 256
#define RLK_OP_TRACE_MAX_KERNELS 8

typedef struct rlk_op_record {
    uint64_t seq;                  /* 1, 2, ... since tracing was last enabled */
    char op[48];                   /* WS1 row(s) the call computes */
    char entry_point[40];          /* the C ABI function called */
    char requested_backend[24];    /* "cuda": the library's only backend */
    char actual_backend[24];       /* "sm_103a tcgen05", or "none" if nothing ran */
    int32_t status;                /* rlk_status returned */
    int32_t fallback;              /* 0: there is no fallback path */
    int32_t split_k;               /* 0: no Split-K / Stream-K / split-KV */
    int32_t atomics;               /* 0: no atomic accumulation */
    int32_t tf32;                  /* 0: TF32 off */
    int32_t n_kernels;             /* kernels enqueued (<= RLK_OP_TRACE_MAX_KERNELS) */
    char kernels[RLK_OP_TRACE_MAX_KERNELS][32];
    char kernel_fingerprint[96];   /* source hash of the library and its build flags */
    char accumulator[16];          /* "fp32" */
    char arithmetic_policy[192];   /* operand/accumulate/cast/transcendental policy */
    char reduction_order[160];
    int32_t B, H, T_txt, grid_h, grid_w;  /* the call's geometry (0 if the shape was null) */
} rlk_op_record;

/* Turns the operator trace on (1) or off (0); either way clears the log. */
rlk_status rlk_op_trace_enable(int enable);
/* Records currently kept (0 .. RLK_OP_TRACE_CAP). */
int32_t rlk_op_trace_count(void);
/* Copies record i (0 = oldest kept) into *out; RLK_ERR_INVALID_ARG if i is
 * out of range or out is NULL. */
rlk_status rlk_op_trace_read(int32_t i, rlk_op_record* out);

/* Human-readable text of a status code (static storage). */
const char* rlk_strerror(int status);

/* Kernel timing for benchmarks. kernel ids: 0 rope table, 1 prologue,
 * 2 attention forward, 3 backward preprocess, 4 dK/dV, 5 dQ,
 * 6 RoPE/RMSNorm backward of the keys (the queries' runs inside dQ),
 * 7 gain-gradient fold, 8 qk_gemm, 9 softmax,
 * 10 av_gemm, 11 forward key shard, 12 qkv_bias_gemm, 13 attn_out_bias_gemm.
 * rlk_kernel_timing(1) makes later calls record a CUDA event pair around
 * every launch (up to 4096 launches per kernel id); rlk_kernel_timing(0)
 * stops and clears. rlk_kernel_timing_read() waits for the recorded events
 * and returns the summed milliseconds and the launch count of one kernel id
 * since the last clear. */
rlk_status rlk_kernel_timing(int enable);
rlk_status rlk_kernel_timing_read(int kernel_id, double* total_ms, int32_t* launches);

#ifdef __cplusplus
}
#endif

#endif /* RLK_JOINT_ATTN_H */

// The backward of the three attention operators of the RFC #386 WS1 table on
// their own (the table's rows joint_attn_qk_gemm, joint_attn_softmax and
// joint_attn_av_gemm are "fwd + bwd", and the WS1 Single-GPU Kernel List
// asks every differentiable operator for a backward), and of the
// qk_rmsnorm + multi_axis_rope prologue, whose composition reproduces the
// fused backward (k_attn_bwd.cu) byte for byte:
//
//   stats      lse2 = lse * log2(e) and Delta = rowsum(dO * O)   (the fused
//              backward's preprocess kernel, k_prologue.cu)
//   softmax_bwd, first pass   P = exp2(fmaf(s, log2(e)/sqrt(128), -lse2))
//              rounded once to bf16 (exactly the fused dK/dV kernel's P)
//   av_gemm_bwd   dP = dO V^T (fp32; the fused kernel's dP^T product in the
//              same k-step order) and dV = P^T dO over the query tiles in
//              ascending order (bf16; masked keys 0)
//   softmax_bwd, second pass  dS = P * (dP - Delta), P recomputed in fp32
//              as above, rounded once to bf16
//   qk_gemm_bwd   dq^ = dS k^ / sqrt(128) over the key tiles in the
//              forward's order and dk^ = dS^T q^ / sqrt(128) over the query
//              tiles in ascending order (fp32; masked keys 0)
//   qk_norm_rope_bwd  the RoPE / RMSNorm backward of the query rows (the
//              fused dQ kernel's epilogue arithmetic, rlk_normrope_bwd.cuh)
//              and of the key rows (norm_rope_bwd_k), then the fixed-order
//              gain-gradient folds.
//
// The products use the fused kernel's tile shape (128 x 128 x 16) and k-step
// order. They are taken query-major here ([query][key] intermediates, as
// the forward operators store them) where the fused kernel takes them
// key-major; the tensor cores give the same bits either way (checked on the
// GPU over every score of two geometries, and by the byte-equality tests).
// Rows past a segment read zeros (per-segment tensor maps), so a padded
// query slot adds +0 exactly as in the fused kernel.
#include "rlk_device.cuh"
#include "rlk_internal.h"
#include "rlk_normrope_bwd.cuh"
#include "rlk_sm100.cuh"
#include "rlk_tmap.h"

RLK_DEFINE_STRICT_PROBE(probe_unfused_bwd_tu)

namespace rlk {
namespace {

using namespace sm100;

constexpr int kBoxBytes = 128 * 128;       // 128 rows x 64 bf16
constexpr int kTileBytes = 2 * kBoxBytes;  // 128 rows x 128 bf16
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr float kC = (float)(1.4426950408889634 * 0.08838834764831845);  // log2(e) / sqrt(128)
constexpr float kScale = 0.08838834764831845f;                          // 1 / sqrt(128)

__device__ int g_status_unf_bwd;

__device__ __forceinline__ void fail(volatile int* abort_flag) {
    *abort_flag = 1;
    atomicOr(&g_status_unf_bwd, 1);
}

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, kWaitLimitNs));
}

// Query tile i (segment aligned): first token and end of its segment.
__device__ __forceinline__ void query_tile(const Geom& g, int i, int& q0, int& q_end) {
    if (i < g.ntq_txt) {
        q0 = i * 128;
        q_end = g.T_txt;
    } else {
        q0 = g.T_txt + (i - g.ntq_txt) * 128;
        q_end = g.S;
    }
}

// Key tile j of the forward's order for a sample with L valid text keys:
// its column block and first key (text tiles holding a valid key, then the
// image tiles).
__device__ __forceinline__ void key_tile(const Geom& g, int L, int j, int& blk, int& k0) {
    const int nkt_txt = (L + 127) / 128;
    if (j < nkt_txt) {
        blk = j;
        k0 = j * 128;
    } else {
        blk = g.ntq_txt + (j - nkt_txt);
        k0 = g.T_txt + (j - nkt_txt) * 128;
    }
}

// ====================================================================== softmax_bwd
// One thread per 8 consecutive columns of one row of the visited key blocks
// (text blocks holding a valid key, then every image block). Masked keys
// score -inf, so their P is exactly +0, as the fused kernel's.
struct SmBwdArgs {
    Geom g;
    ValidLen vl;
    const float* scores;  // [B, H, S, ncols]
    const float* lse2;    // [B, H, nq_pad] tile-padded
    const float* delta;   // [B, H, nq_pad]
    const float* dp;      // [B, H, S, ncols] or null (first pass)
    uint16_t* p;          // [B, H, S, ncols] bf16 or null
    uint16_t* ds;         // [B, H, S, ncols] bf16 or null
    int ncols;
};

__global__ void __launch_bounds__(256) softmax_bwd_kernel(const __grid_constant__ SmBwdArgs a) {
    const Geom& g = a.g;
    const int h = blockIdx.y, b = blockIdx.z;
    const int L = a.vl.L[b];
    const int nblk_txt = (L + 127) / 128;
    const int nvis = nblk_txt + g.ntq_img;  // visited blocks of every row
    const long long per_row = (long long)nvis * 16;
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= per_row * g.S) return;
    const int n = (int)(idx / per_row);
    const int c16 = (int)(idx % per_row);
    const int vb = c16 >> 4;
    const int blk = vb < nblk_txt ? vb : g.ntq_txt + (vb - nblk_txt);
    const int col = blk * 128 + (c16 & 15) * 8;
    const size_t bh = (size_t)b * g.H + h;
    // tile-padded slot of query row n
    const int slot = n < g.T_txt ? n : g.ntq_txt * 128 + (n - g.T_txt);
    const float l2 = a.lse2[bh * g.nq_pad + slot];
    const size_t off = (bh * g.S + n) * (size_t)a.ncols + col;
    const float4 s0 = *reinterpret_cast<const float4*>(a.scores + off);
    const float4 s1 = *reinterpret_cast<const float4*>(a.scores + off + 4);
    const float sv[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
    float pf[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) pf[e] = exp2_num(fmaf(sv[e], kC, -l2));
    if (a.p != nullptr)
        *reinterpret_cast<uint4*>(a.p + off) = make_uint4(pack_bf16(pf[0], pf[1]), pack_bf16(pf[2], pf[3]),
                                                          pack_bf16(pf[4], pf[5]), pack_bf16(pf[6], pf[7]));
    if (a.dp != nullptr) {
        const float dl = a.delta[bh * g.nq_pad + slot];
        const float4 d0 = *reinterpret_cast<const float4*>(a.dp + off);
        const float4 d1 = *reinterpret_cast<const float4*>(a.dp + off + 4);
        const float dv[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
        float ds[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) ds[e] = pf[e] * (dv[e] - dl);
        *reinterpret_cast<uint4*>(a.ds + off) = make_uint4(pack_bf16(ds[0], ds[1]), pack_bf16(ds[2], ds[3]),
                                                           pack_bf16(ds[4], ds[5]), pack_bf16(ds[6], ds[7]));
    }
}

// ====================================================================== accumulating products
// One CTA = one 128-row output tile of one (sample, head); 6 warps: warp 0
// TMA, warp 1 MMA issuer and TMEM owner, warps 2-5 epilogue (one output
// row per thread). TMEM: the fp32 accumulator [0, 128).
//   key-major (kKeyMajor): out[key][d] = sum over the query tiles, in
//     ascending order, of X[q][key] Y[q][d]: X (P or dS, [q][key] bf16) is
//     the MN-major A operand, Y (dO per segment, or q^) the MN-major B
//     operand. dV = P^T dO and dk^ = dS^T q^ / sqrt(128).
//   query-major: out[q][d] = sum over the key tiles of the forward's order
//     of X[q][key] Y[key][d]: X (dS) the K-major A operand, Y (k^) the
//     MN-major B operand. dq^ = dS k^ / sqrt(128).
// Per step the copy warp loads X's 128 x 128 block and Y's 128-row tile
// into a stage of a three-stage ring.
struct AccArgs {
    CUtensorMap map_x[2];    // X per segment of its rows (queries) [B*H, rows, ncols], box 64 x 128
    CUtensorMap map_x_all;   // X as [B*H*S, ncols], box 64 x 128 (query-major: rows past a segment are not stored)
    CUtensorMap map_y_seg[2];  // Y = dO per segment, 4-D (d, h, token, b)
    CUtensorMap map_y_rows;  // Y = q^ or k^ as [B*H*S, 128]
    Geom g;
    ValidLen vl;
    int y_rows;              // 1: Y from map_y_rows; 0: from map_y_seg
    int out_bf16;            // 1: bf16 out (dV); 0: fp32 out times kScale
    SegBf16 out_b;           // bf16 [B, S, H, 128] per segment
    float* out_f;            // fp32 [B, H, S, 128]
};

constexpr int kAccThreads = 192;
constexpr int kAccWarpTma = 0, kAccWarpMma = 1;
constexpr int kAccStages = 3;
constexpr int kAccStageBytes = 2 * kTileBytes;  // X block, Y tile
constexpr int kAccSmemBytes = kAccStages * kAccStageBytes + 1024;
constexpr uint32_t kAccTmemCols = 128;
constexpr uint32_t kIdescMM = idesc_bf16(128, 128, true, true);   // A, B MN-major
constexpr uint32_t kIdescKM = idesc_bf16(128, 128, false, true);  // A K-major, B MN-major

template <bool kKeyMajor>
__global__ void __launch_bounds__(kAccThreads, 1) acc_gemm_kernel(const __grid_constant__ AccArgs a) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bars[2 * kAccStages + 2];
    __shared__ uint32_t tmem_slot;
    __shared__ volatile int abort_flag;

    const Geom& g = a.g;
    const int t = blockIdx.x, h = blockIdx.y, b = blockIdx.z;  // t: key tile (key-major) or query tile
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int L = a.vl.L[b];
    const int nq = g.ntq_txt + g.ntq_img;
    const size_t bh = (size_t)b * g.H + h;
    const int row_base = (int)(bh * g.S);
    // the output tile's rows: keys (key-major) or queries, segment aligned
    int r0, r_end;
    query_tile(g, t, r0, r_end);
    const bool r_txt = t < g.ntq_txt;
    const int kvalid_end = r_txt ? L : g.S;  // key-major: keys at or past it are masked
    const int nsteps = kKeyMajor ? nq : (L + 127) / 128 + g.ntq_img;

    if (kKeyMajor && r0 >= kvalid_end) {  // every key of the tile is masked: exact zeros
        const int rows = min(128, r_end - r0);
        for (int i = tid; i < rows * 16; i += kAccThreads) {
            const int r = i >> 4, c = i & 15;
            if (a.out_bf16) {
                *reinterpret_cast<uint4*>(seg_row(a.out_b, g, b, r0 + r, h) + c * 8) = make_uint4(0, 0, 0, 0);
            } else {
                float4* dst = reinterpret_cast<float4*>(a.out_f + (bh * g.S + r0 + r) * kHeadDim + c * 8);
                dst[0] = make_float4(0.f, 0.f, 0.f, 0.f);
                dst[1] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        return;
    }

    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    auto stage_x = [&](int s) { return sbase + s * kAccStageBytes; };
    auto stage_y = [&](int s) { return sbase + s * kAccStageBytes + kTileBytes; };
    const uint32_t bar_full = smem_u32(&bars[0]);            // [3] stage loaded
    const uint32_t bar_empty = smem_u32(&bars[kAccStages]);  // [3] stage's product done
    const uint32_t bar_done = smem_u32(&bars[2 * kAccStages]);
    const uint32_t bar_drain = smem_u32(&bars[2 * kAccStages + 1]);

    if (tid == 0) {
        abort_flag = 0;
        for (int s = 0; s < kAccStages; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
        }
        mbar_init(bar_done, 1);
        mbar_init(bar_drain, 1);
        fence_barrier_init();
    }
    if (warp == kAccWarpMma) {
        tmem_alloc(smem_u32(&tmem_slot), kAccTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    if (warp == kAccWarpTma) {
        if (lane == 0) {
            int issued = 0;
            for (int j = 0; j < nsteps && !abort_flag; ++j) {
                const int s = j % kAccStages;
                if (j >= kAccStages &&
                    !mbar_wait(bar_empty + 8 * s, ((j / kAccStages) + 1) & 1, &abort_flag, kWaitLimitNs)) {
                    fail(&abort_flag);
                    break;
                }
                const uint32_t bf = bar_full + 8 * s;
                mbar_expect_tx(bf, kAccStageBytes);
                if (kKeyMajor) {
                    // step j: query tile j; X block (its 128 query rows, this key
                    // tile's columns) clipped at the query segment; Y its rows
                    int q0, q_end;
                    query_tile(g, j, q0, q_end);
                    const int qseg = j < g.ntq_txt ? 0 : 1, qrow = qseg ? q0 - g.T_txt : q0;
                    tma_load_3d(stage_x(s), &a.map_x[qseg], bf, t * 128, qrow, (int)bh);
                    tma_load_3d(stage_x(s) + kBoxBytes, &a.map_x[qseg], bf, t * 128 + 64, qrow, (int)bh);
                    if (a.y_rows) {
                        tma_load_2d(stage_y(s), &a.map_y_rows, bf, 0, row_base + q0);
                        tma_load_2d(stage_y(s) + kBoxBytes, &a.map_y_rows, bf, 64, row_base + q0);
                    } else {
                        tma_load_4d(stage_y(s), &a.map_y_seg[qseg], bf, 0, h, qrow, b);
                        tma_load_4d(stage_y(s) + kBoxBytes, &a.map_y_seg[qseg], bf, 64, h, qrow, b);
                    }
                } else {
                    // step j: key tile j of the forward's order; X block (this
                    // query tile's rows, that key tile's columns); Y = k^ rows
                    int blk, k0;
                    key_tile(g, L, j, blk, k0);
                    tma_load_2d(stage_x(s), &a.map_x_all, bf, blk * 128, row_base + r0);
                    tma_load_2d(stage_x(s) + kBoxBytes, &a.map_x_all, bf, blk * 128 + 64, row_base + r0);
                    tma_load_2d(stage_y(s), &a.map_y_rows, bf, 0, row_base + k0);
                    tma_load_2d(stage_y(s) + kBoxBytes, &a.map_y_rows, bf, 64, row_base + k0);
                }
                issued = j + 1;
            }
            const volatile int no_abort = 0;
            for (int j = issued - kAccStages < 0 ? 0 : issued - kAccStages; j < issued; ++j)
                mbar_wait(bar_full + 8 * (j % kAccStages), (j / kAccStages) & 1, &no_abort, kWaitLimitNs);
        }
    } else if (warp == kAccWarpMma) {
        if (lane == 0) {
            bool ok = true;
            for (int j = 0; ok && j < nsteps; ++j) {
                const int s = j % kAccStages;
                ok = mbar_wait(bar_full + 8 * s, (j / kAccStages) & 1, &abort_flag, kWaitLimitNs);
                if (!ok) break;
                tc_fence_after();
                const uint32_t dx = stage_x(s), dy = stage_y(s);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    // B: Y's rows 16 kk .. 16 kk + 15 (the k-step) read MN-major
                    const uint64_t bdesc = sdesc_sw128(dy + kk * 2048, kBoxBytes, 1024);
                    if (kKeyMajor)  // A: X's query rows 16 kk .., keys along M (MN-major)
                        mma_ss(tmem, sdesc_sw128(dx + kk * 2048, kBoxBytes, 1024), bdesc, kIdescMM,
                               (j > 0 || kk > 0) ? 1u : 0u);
                    else            // A: X's key columns 16 kk .. (K-major)
                        mma_ss(tmem, sdesc_sw128(dx + (kk >> 2) * kBoxBytes + (kk & 3) * 32, 16, 1024), bdesc,
                               kIdescKM, (j > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(bar_empty + 8 * s);
            }
            if (ok)
                mma_commit(bar_done);
            else
                fail(&abort_flag);
            mma_commit(bar_drain);
            const volatile int no_abort = 0;
            mbar_wait(bar_drain, 0, &no_abort, kWaitLimitNs);
        }
    } else {
        const uint32_t lane_addr = (uint32_t)((warp & 3) * 32) << 16;
        const int row = (warp & 3) * 32 + lane;
        const int n = r0 + row;
        const bool in_seg = n < r_end;
        // key-major: masked keys get exact zeros, as the fused kernel writes
        const bool keep = !kKeyMajor || n < kvalid_end;
        if (warp_wait(bar_done, 0, &abort_flag)) {
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                uint32_t r[32];
                tmem_ld32(tmem + lane_addr + 32 * c, r);
                tmem_ld_wait();
                if (!in_seg) continue;
                if (a.out_bf16) {
                    uint4* orow = reinterpret_cast<uint4*>(seg_row(a.out_b, g, b, n, h));
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            w[e] = keep ? pack_bf16(__uint_as_float(r[8 * q + 2 * e]), __uint_as_float(r[8 * q + 2 * e + 1]))
                                        : 0u;
                        orow[4 * c + q] = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                } else {
                    float4* orow = reinterpret_cast<float4*>(a.out_f + (bh * g.S + n) * kHeadDim);
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        orow[8 * c + q] = keep ? make_float4(__uint_as_float(r[4 * q]) * kScale,
                                                             __uint_as_float(r[4 * q + 1]) * kScale,
                                                             __uint_as_float(r[4 * q + 2]) * kScale,
                                                             __uint_as_float(r[4 * q + 3]) * kScale)
                                               : make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
        } else {
            fail(&abort_flag);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kAccWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, kAccTmemCols);
    }
}

// ====================================================================== RoPE / RMSNorm backward, query rows
// One CTA = one query tile of one (sample, head), one row per thread: the
// fused dQ kernel's epilogue (nrb_row) fed from dq^ in memory instead of its
// TMEM accumulator, with the same gain-gradient partial per (tile, 32-row
// quarter).
struct NrbQArgs {
    Geom g;
    SegBf16 q, dq;
    const float* rq;
    const float* gq_txt;
    const float* gq_img;
    const float2* tab;
    const float* dqh;  // fp32 [B, H, S, 128]
    float* dgt;        // [B, H, 2, n_tiles, 4, 128]
};

__global__ void __launch_bounds__(128) norm_rope_bwd_q_kernel(const __grid_constant__ NrbQArgs a) {
    const Geom& g = a.g;
    const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nq = g.ntq_txt + g.ntq_img;
    int q0, q_end;
    query_tile(g, qt, q0, q_end);
    const int r = warp * 32 + lane;
    const bool row_ok = q0 + r < q_end;
    const int tok = row_ok ? q0 + r : q0;  // rows past the segment read a valid row, store nothing
    const size_t bh = (size_t)b * g.H + h;
    const float4* src = reinterpret_cast<const float4*>(a.dqh + (bh * g.S + tok) * kHeadDim);
    auto dq_chunk = [&](int c, float (&dy)[32]) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 v = src[8 * c + i];
            dy[4 * i] = row_ok ? v.x : 0.0f;
            dy[4 * i + 1] = row_ok ? v.y : 0.0f;
            dy[4 * i + 2] = row_ok ? v.z : 0.0f;
            dy[4 * i + 3] = row_ok ? v.w : 0.0f;
        }
    };
    nrb_row(dq_chunk, row_ok, reinterpret_cast<const uint4*>(seg_row(a.q, g, b, tok, h)), a.rq[bh * g.S + tok],
            qt < g.ntq_txt ? a.gq_txt : a.gq_img, tab_rows(a.tab, g, tok),
            reinterpret_cast<uint4*>(seg_row(a.dq, g, b, tok, h)),
            a.dgt + ((bh * 2 * nq + qt) * 4 + warp) * kHeadDim, lane);
}

}  // namespace

cudaError_t launch_softmax_bwd(const Geom& g, const ValidLen& vl, const float* scores, const float* lse2,
                               const float* delta, const float* dp, uint16_t* p, uint16_t* ds, cudaStream_t s) {
    SmBwdArgs a;
    a.g = g;
    a.vl = vl;
    a.scores = scores;
    a.lse2 = lse2;
    a.delta = delta;
    a.dp = dp;
    a.p = p;
    a.ds = ds;
    a.ncols = 128 * (g.ntq_txt + g.ntq_img);
    // the widest row (every block visited) sizes the grid; shorter samples
    // leave their tail threads idle
    const long long per_bh = (long long)g.S * (g.ntq_txt + g.ntq_img) * 16;
    const dim3 grid((unsigned)((per_bh + 255) / 256), g.H, g.B);
    timing_begin(kKSoftmaxBwd, s);
    softmax_bwd_kernel<<<grid, 256, 0, s>>>(a);
    timing_end(kKSoftmaxBwd, s);
    return cudaGetLastError();
}

namespace {
cudaError_t launch_acc(bool key_major, AccArgs& a, const Geom& g, int kernel_id, cudaStream_t s) {
    auto kern = key_major ? acc_gemm_kernel<true> : acc_gemm_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kAccSmemBytes);
    if (e != cudaSuccess) return e;
    const dim3 grid(g.ntq_txt + g.ntq_img, g.H, g.B);
    timing_begin(kernel_id, s);
    kern<<<grid, kAccThreads, kAccSmemBytes, s>>>(a);
    timing_end(kernel_id, s);
    return cudaGetLastError();
}
}  // namespace

cudaError_t launch_dv_gemm(const Geom& g, const ValidLen& vl, const uint16_t* p, const SegBf16& dout,
                           const SegBf16& dv, cudaStream_t s) {
    AccArgs a;
    memset(&a, 0, sizeof(a));
    const int ncols = 128 * (g.ntq_txt + g.ntq_img);
    for (int seg = 0; seg < 2; ++seg)
        if (!tmap::p_bf16_segment(&a.map_x[seg], p, g, ncols, seg, 128) || !tmap::seg_bf16(&a.map_y_seg[seg], dout, g, seg))
            return cudaErrorInvalidValue;
    a.g = g;
    a.vl = vl;
    a.y_rows = 0;
    a.out_bf16 = 1;
    a.out_b = dv;
    return launch_acc(true, a, g, kKKeyGemm, s);
}

cudaError_t launch_dhat_gemms(const Geom& g, const ValidLen& vl, const uint16_t* ds, const uint16_t* qh,
                              const uint16_t* kh, float* dqh, float* dkh, cudaStream_t s) {
    const int ncols = 128 * (g.ntq_txt + g.ntq_img);
    const uint64_t rows = (uint64_t)g.B * g.H * g.S;
    // dk^ = dS^T q^ / sqrt(128), key-major over the query tiles
    AccArgs a;
    memset(&a, 0, sizeof(a));
    for (int seg = 0; seg < 2; ++seg)
        if (!tmap::p_bf16_segment(&a.map_x[seg], ds, g, ncols, seg, 128)) return cudaErrorInvalidValue;
    if (!tmap::rows_bf16(&a.map_y_rows, qh, rows)) return cudaErrorInvalidValue;
    a.g = g;
    a.vl = vl;
    a.y_rows = 1;
    a.out_bf16 = 0;
    a.out_f = dkh;
    cudaError_t e = launch_acc(true, a, g, kKKeyGemm, s);
    if (e != cudaSuccess) return e;
    // dq^ = dS k^ / sqrt(128), query-major over the key tiles in the forward's order
    AccArgs c;
    memset(&c, 0, sizeof(c));
    if (!tmap::mat_bf16(&c.map_x_all, ds, (long long)rows, ncols, 128) || !tmap::rows_bf16(&c.map_y_rows, kh, rows))
        return cudaErrorInvalidValue;
    c.g = g;
    c.vl = vl;
    c.y_rows = 1;
    c.out_bf16 = 0;
    c.out_f = dqh;
    return launch_acc(false, c, g, kKQueryGemm, s);
}

cudaError_t launch_norm_rope_bwd_q(const Geom& g, const SegBf16& q, const float* gq_txt, const float* gq_img,
                                   const float2* tab, const float* rq, const float* dqh, const SegBf16& dq,
                                   float* dgt, cudaStream_t s) {
    NrbQArgs a;
    a.g = g;
    a.q = q;
    a.dq = dq;
    a.rq = rq;
    a.gq_txt = gq_txt;
    a.gq_img = gq_img;
    a.tab = tab;
    a.dqh = dqh;
    a.dgt = dgt;
    const dim3 grid(g.ntq_txt + g.ntq_img, g.H, g.B);
    timing_begin(kKNormRopeBwdQ, s);
    norm_rope_bwd_q_kernel<<<grid, 128, 0, s>>>(a);
    timing_end(kKNormRopeBwdQ, s);
    return cudaGetLastError();
}

int read_and_clear_status_unfused_bwd(cudaStream_t s) {
    int v = 0, zero = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_status_unf_bwd, sizeof(int), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return -1;
    if (cudaMemcpyToSymbolAsync(g_status_unf_bwd, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return -1;
    if (cudaStreamSynchronize(s) != cudaSuccess) return -1;
    return v;
}

}  // namespace rlk

// The three attention operators of the RFC #386 WS1 table on their own --
// joint_attn_qk_gemm, joint_attn_softmax and joint_attn_av_gemm -- whose
// composition reproduces the fused forward (joint_attention_fused,
// k_attn_fwd.cu) byte for byte: the table's joint_attention_fused row and
// the WS1 Single-GPU Kernel List both define the fused kernel as one whose
// bytes equal those of the three operators run one after another.
//
// Byte equality holds because each operator performs the fused kernel's
// arithmetic in the fused kernel's order:
//   qk_gemm   the same tcgen05 SS products (128 x 128 x 16, 128-byte-swizzled
//             K-major q^ and k^ tiles, k-steps 0..7 in order) into TMEM, read
//             out as raw FP32 scores s = q^ . k^ (-inf for masked keys,
//             which the fused kernel also sets to -inf). The 1/sqrt(128) scale is
//             not applied here: the fused kernel folds it, with log2(e),
//             into the one rounding of the softmax argument
//             fmaf(s, log2(e)/sqrt(128), -m), and so does the softmax
//             operator.
//   softmax   per query row, key tiles in the fused order (text tiles that
//             hold a valid key, then image tiles): the same masking, lazy
//             reference max (moves only past a 2^8 growth), exp2f
//             numerators, eight-way partial sums and a fixed tree per 64-key
//             half, the two halves' sums added; it
//             writes P (bf16, relative to the row's reference max at that
//             tile), the rescale factor alpha of every tile, the final row
//             sum l and lse.
//   av_gemm   the same tcgen05 products O += P V (k-steps of 16 keys in the
//             fused kernel's order 0, 1, 4, 5, 2, 3, 6, 7; V tiles MN-major
//             in shared memory), O rescaled in
//             TMEM by alpha before each tile's product, then O * (1 / l)
//             rounded once to bf16.
// The intermediates are materialised in caller-owned buffers:
//   scores  fp32 [B, H, S, n_tiles * 128]   column block t = key tile t
//   P       bf16 [B, H, S, n_tiles * 128]   (text tiles t < ceil(T_txt/128),
//   alpha   fp32 [B, H, S, n_tiles]          then image tiles)
//   l, lse  fp32 [B, H, S]
// Blocks of text tiles with no valid key are not written; inside a visited
// block the columns of masked keys hold -inf (scores) and exactly 0 (P).
// Each query row is written by its own segment's tile. Every wait is
// bounded (RLK_ERR_DEVICE_TIMEOUT).
#include "rlk_device.cuh"
#include "rlk_internal.h"
#include "rlk_sm100.cuh"
#include "rlk_tmap.h"

RLK_DEFINE_STRICT_PROBE(probe_unfused_tu)

namespace rlk {
namespace {

using namespace sm100;

constexpr int kBoxBytes = 128 * 128;       // 128 rows x 64 bf16
constexpr int kTileBytes = 2 * kBoxBytes;  // 128 rows x 128 bf16
constexpr uint32_t kTmemCols = 256;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr float kC = (float)(1.4426950408889634 * 0.08838834764831845);  // log2(e) / sqrt(128)
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint32_t kIdescS = idesc_bf16(128, 128, false, false);
constexpr uint32_t kIdescO = idesc_bf16(128, 128, false, true);
constexpr int kThreads = 192;  // warp 0 TMA, warp 1 MMA + TMEM owner, warps 2-5 one query row per thread
constexpr int kWarpTma = 0, kWarpMma = 1;

__device__ int g_status_unf;

__device__ __forceinline__ void fail(volatile int* abort_flag) {
    *abort_flag = 1;
    atomicOr(&g_status_unf, 1);
}

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, kWaitLimitNs));
}

// Key tile j of the fused order for a sample with L valid text keys: its
// column block in the materialised layout and its key range [k0, kend) of
// valid keys.
struct KeyTile {
    int blk, k0, kend;
};
__device__ __forceinline__ KeyTile key_tile(const Geom& g, int L, int j) {
    const int nkt_txt = (L + 127) / 128;
    KeyTile t;
    if (j < nkt_txt) {
        t.blk = j;
        t.k0 = j * 128;
        t.kend = L;
    } else {
        t.blk = g.ntq_txt + (j - nkt_txt);
        t.k0 = g.T_txt + (j - nkt_txt) * 128;
        t.kend = g.S;
    }
    return t;
}
__device__ __forceinline__ int n_key_tiles(const Geom& g, int L) { return (L + 127) / 128 + g.ntq_img; }

// Query tile qt (segment aligned): first token and end of its segment.
__device__ __forceinline__ void query_tile(const Geom& g, int qt, int& q0, int& q_end) {
    if (qt < g.ntq_txt) {
        q0 = qt * 128;
        q_end = g.T_txt;
    } else {
        q0 = g.T_txt + (qt - g.ntq_txt) * 128;
        q_end = g.S;
    }
}

// ====================================================================== qk_gemm
struct QkArgs {
    CUtensorMap map_q;  // qh [B*H*S, 128] bf16
    CUtensorMap map_k;  // kh [B*H*S, 128] bf16
    // the dP form (joint_attn_av_gemm's backward, dP = dO V^T): dO as the A
    // rows and V as the B rows, per segment (rows past a segment read zeros)
    CUtensorMap map_a_seg[2];
    CUtensorMap map_b_seg[2];
    Geom g;
    ValidLen vl;
    float* scores;      // [B, H, S, ncols]
    int ncols;
    CUtensorMap map_s[2];  // scores per segment (text, image rows), fp32 boxes of 32 x 32
};

// Q, two K slots, and the epilogue's staging: per epilogue warp its 32 rows
// as four 32-column boxes of 4 KB in the 128-byte-swizzled layout of map_s
constexpr int kQkStageBytes = 4 * 4 * 4096;
constexpr int kQkSmemBytes = 3 * kTileBytes + kQkStageBytes + 1024;

// kDp: the backward's dP = dO V^T in the same tiling -- the A rows come from
// dO and the B rows from V (per-segment maps), and no key is masked (dP of a
// masked key is finite; its P is 0).
template <bool kDp>
__global__ void __launch_bounds__(kThreads, 1) qk_gemm_kernel(const __grid_constant__ QkArgs a) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bars[10];
    __shared__ uint32_t tmem_slot;
    __shared__ volatile int abort_flag;

    const Geom& g = a.g;
    const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int q0, q_end;
    query_tile(g, qt, q0, q_end);
    const int L = a.vl.L[b];
    const int nkt = n_key_tiles(g, L);
    const size_t bh = (size_t)b * g.H + h;
    const int row_base = (int)(bh * g.S);

    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const uint32_t sQ = sbase, sK = sbase + kTileBytes;
    const uint32_t bar_q = smem_u32(&bars[0]);
    const uint32_t bar_kf = smem_u32(&bars[1]);  // [2] K slot loaded
    const uint32_t bar_ke = smem_u32(&bars[3]);  // [2] K slot free (its product done)
    const uint32_t bar_s = smem_u32(&bars[5]);   // [2] score buffer written
    const uint32_t bar_se = smem_u32(&bars[7]);  // [2] score buffer read out
    const uint32_t bar_drain = smem_u32(&bars[9]);

    if (tid == 0) {
        abort_flag = 0;
        mbar_init(bar_q, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar_kf + 8 * s, 1);
            mbar_init(bar_ke + 8 * s, 1);
            mbar_init(bar_s + 8 * s, 1);
            mbar_init(bar_se + 8 * s, 128);
        }
        mbar_init(bar_drain, 1);
        fence_barrier_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc(smem_u32(&tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    if (warp == kWarpTma) {
        if (lane == 0) {
            prefetch_tensormap(&a.map_q);
            prefetch_tensormap(&a.map_k);
            mbar_expect_tx(bar_q, kTileBytes);
            if (kDp) {
                const int aseg = q0 < g.T_txt ? 0 : 1, arow = aseg ? q0 - g.T_txt : q0;
                tma_load_4d(sQ, &a.map_a_seg[aseg], bar_q, 0, h, arow, b);
                tma_load_4d(sQ + kBoxBytes, &a.map_a_seg[aseg], bar_q, 64, h, arow, b);
            } else {
                tma_load_2d(sQ, &a.map_q, bar_q, 0, row_base + q0);
                tma_load_2d(sQ + kBoxBytes, &a.map_q, bar_q, 64, row_base + q0);
            }
            int issued = 0;
            for (int j = 0; j < nkt && !abort_flag; ++j) {
                const int s = j & 1;
                if (j >= 2 && !mbar_wait(bar_ke + 8 * s, ((j >> 1) + 1) & 1, &abort_flag, kWaitLimitNs)) {
                    fail(&abort_flag);
                    break;
                }
                const KeyTile kt = key_tile(g, L, j);
                mbar_expect_tx(bar_kf + 8 * s, kTileBytes);
                if (kDp) {
                    const int bseg = kt.k0 < g.T_txt ? 0 : 1, brow = bseg ? kt.k0 - g.T_txt : kt.k0;
                    tma_load_4d(sK + s * kTileBytes, &a.map_b_seg[bseg], bar_kf + 8 * s, 0, h, brow, b);
                    tma_load_4d(sK + s * kTileBytes + kBoxBytes, &a.map_b_seg[bseg], bar_kf + 8 * s, 64, h, brow, b);
                } else {
                    tma_load_2d(sK + s * kTileBytes, &a.map_k, bar_kf + 8 * s, 0, row_base + kt.k0);
                    tma_load_2d(sK + s * kTileBytes + kBoxBytes, &a.map_k, bar_kf + 8 * s, 64, row_base + kt.k0);
                }
                issued = j + 1;
            }
            const volatile int no_abort = 0;
            mbar_wait(bar_q, 0, &no_abort, kWaitLimitNs);
            for (int j = issued - 2 < 0 ? 0 : issued - 2; j < issued; ++j)
                mbar_wait(bar_kf + 8 * (j & 1), (j >> 1) & 1, &no_abort, kWaitLimitNs);
        }
    } else if (warp == kWarpMma) {
        if (lane == 0) {
            bool ok = mbar_wait(bar_q, 0, &abort_flag, kWaitLimitNs);
            for (int j = 0; ok && j < nkt; ++j) {
                const int s = j & 1;
                ok = mbar_wait(bar_kf + 8 * s, (j >> 1) & 1, &abort_flag, kWaitLimitNs) &&
                     (j < 2 || mbar_wait(bar_se + 8 * s, ((j >> 1) + 1) & 1, &abort_flag, kWaitLimitNs));
                if (!ok) break;
                tc_fence_after();
                const uint32_t dk = sK + s * kTileBytes;
                // the fused forward's score product, k-steps in the same order
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
                    mma_ss(tmem + 128 * s, sdesc_sw128(sQ + off, 16, 1024), sdesc_sw128(dk + off, 16, 1024), kIdescS,
                           kk > 0);
                }
                mma_commit(bar_s + 8 * s);
                mma_commit(bar_ke + 8 * s);
            }
            if (!ok) fail(&abort_flag);
            mma_commit(bar_drain);
            const volatile int no_abort = 0;
            mbar_wait(bar_drain, 0, &no_abort, kWaitLimitNs);
        }
    } else {
        // one query row per thread: TMEM lane quarter warp % 4. The warp
        // stages its 32 rows of a key tile as four 32 x 32 fp32 boxes and its
        // lane 0 stores them with TMA; the segment maps clip rows past the
        // query's segment.
        const int wq = warp & 3;
        const uint32_t lane_addr = (uint32_t)(wq * 32) << 16;
        const uint32_t stage = sbase + 3 * kTileBytes + wq * (4 * 4096);
        uint8_t* stage_p = smem_raw + (stage - smem_u32(smem_raw));
        const int seg = qt < g.ntq_txt ? 0 : 1;
        const int srow = (seg ? q0 - g.T_txt : q0) + 32 * wq;  // the warp's first row in its segment
        const int sw = lane & 7;
        if (lane == 0) prefetch_tensormap(&a.map_s[seg]);
        bool ok = true;
        for (int j = 0; j < nkt; ++j) {
            const int s = j & 1;
            if (!warp_wait(bar_s + 8 * s, (j >> 1) & 1, &abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t r[128];
#pragma unroll
            for (int c = 0; c < 4; ++c)
                tmem_ld32(tmem + lane_addr + 128 * s + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&r[32 * c]));
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive(bar_se + 8 * s);
            const KeyTile kt = key_tile(g, L, j);
            const int nvalid = kt.kend - kt.k0;  // masked keys (and keys past the segment) score -inf
            if (!kDp && nvalid < 128) {
#pragma unroll
                for (int i = 0; i < 128; ++i) r[i] = i < nvalid ? r[i] : 0xff800000u;
            }
            // the staging of the previous key tile has been read by its stores
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint8_t* rowp = stage_p + c * 4096 + lane * 128;
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    *reinterpret_cast<float4*>(rowp + ((k ^ sw) << 4)) =
                        make_float4(__uint_as_float(r[32 * c + 4 * k]), __uint_as_float(r[32 * c + 4 * k + 1]),
                                    __uint_as_float(r[32 * c + 4 * k + 2]), __uint_as_float(r[32 * c + 4 * k + 3]));
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
#pragma unroll
                for (int c = 0; c < 4; ++c) tma_store_3d(&a.map_s[seg], stage + c * 4096, kt.blk * 128 + 32 * c, srow, (int)bh);
                bulk_commit_group();
            }
        }
        if (lane == 0) bulk_wait_read_all();  // the staging must outlive the stores' reads
        __syncwarp();
        if (!ok) fail(&abort_flag);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ====================================================================== softmax
// One warp per 32 query rows (a CTA of one warp; four per query tile), one
// row per lane, the key tiles in the fused order. Lane 0 loads the warp's
// 32 x 128 fp32 scores of the next key tile by TMA into the other of two
// shared-memory slots (four 32 x 32 boxes, 128-byte swizzled) while the
// lanes work on the current one; each lane reads its row back from the slot,
// exactly the values the fused kernel reads from TMEM, and goes through the
// fused kernel's steps: mask, row max, lazy reference max, exp2f numerators,
// partial sums. P is staged as two 64 x 32 bf16 boxes and stored by TMA
// through per-segment maps, which clip rows past the query's segment.
struct SmArgs {
    CUtensorMap map_sc;    // scores [B*H*S, ncols] fp32, box 32 x 32
    CUtensorMap map_p[2];  // P per segment (text, image rows) [B*H, rows, ncols] bf16, box 64 x 32 x 1
    Geom g;
    ValidLen vl;
    float* alpha;          // [B, H, S, nblk]
    float* l;              // [B, H, S]
    float* lse;            // [B, H, S] or null
    int ncols, nblk;
};

constexpr int kSmSlotBytes = 4 * 4096;                          // 32 rows x 128 fp32
constexpr int kSmStageBytes = 2 * 4096;                         // 32 rows x 128 bf16
constexpr int kSmSmemBytes = 2 * kSmSlotBytes + kSmStageBytes + 1024;

__global__ void __launch_bounds__(32) softmax_kernel(const __grid_constant__ SmArgs a) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bars[2];  // score slot s loaded
    __shared__ volatile int abort_flag;

    const Geom& g = a.g;
    const int wq = (int)blockIdx.x & 3, qt = (int)blockIdx.x >> 2, h = blockIdx.y, b = blockIdx.z;
    const int lane = threadIdx.x;
    int q0, q_end;
    query_tile(g, qt, q0, q_end);
    const int r0 = q0 + 32 * wq;  // the warp's first row
    if (r0 >= q_end) return;      // the whole warp lies past the segment
    const int n = r0 + lane;
    const bool row_ok = n < q_end;
    const int L = a.vl.L[b];
    const int nkt = n_key_tiles(g, L);
    const size_t bh = (size_t)b * g.H + h;
    const size_t rowi = bh * g.S + n;
    const int seg = qt < g.ntq_txt ? 0 : 1;
    const int srow = seg ? r0 - g.T_txt : r0;  // the warp's first row in its segment

    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    auto slot = [&](int s) { return sbase + s * kSmSlotBytes; };
    const uint32_t stage = sbase + 2 * kSmSlotBytes;
    const uint8_t* base_p = smem_raw + (sbase - smem_u32(smem_raw));
    uint8_t* stage_p = smem_raw + (stage - smem_u32(smem_raw));
    const uint32_t bar = smem_u32(&bars[0]);
    const int sw = lane & 7;
    if (lane == 0) {
        abort_flag = 0;
        mbar_init(bar, 1);
        mbar_init(bar + 8, 1);
        fence_barrier_init();
        prefetch_tensormap(&a.map_sc);
        prefetch_tensormap(&a.map_p[seg]);
    }
    __syncwarp();
    auto issue = [&](int j) {  // lane 0: key tile j's scores into slot j & 1
        const KeyTile kt = key_tile(g, L, j);
        const uint32_t bs = bar + 8 * (j & 1);
        mbar_expect_tx(bs, kSmSlotBytes);
#pragma unroll
        for (int c = 0; c < 4; ++c)
            tma_load_2d(slot(j & 1) + c * 4096, &a.map_sc, bs, kt.blk * 128 + 32 * c, (int)(bh * g.S) + r0);
    };
    int issued = 0;  // key tiles whose loads lane 0 has issued
    if (lane == 0) {
        issue(0);
        issued = 1;
    }
    float m = -INFINITY, l = 0.0f;
    bool ok = true;
    for (int j = 0; j < nkt; ++j) {
        const int s = j & 1;
        // the other slot was read out by every lane in the previous tile
        __syncwarp();
        if (lane == 0 && j + 1 < nkt) {
            issue(j + 1);
            issued = j + 2;
        }
        if (!warp_wait(bar + 8 * s, (j >> 1) & 1, &abort_flag)) {
            ok = false;
            break;
        }
        const KeyTile kt = key_tile(g, L, j);
        const int nvalid = kt.kend - kt.k0;
        uint32_t r[128];
        const uint8_t* rowp = base_p + s * kSmSlotBytes + lane * 128;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint4 v = *reinterpret_cast<const uint4*>(rowp + c * 4096 + ((k ^ sw) << 4));
                r[32 * c + 4 * k] = v.x;
                r[32 * c + 4 * k + 1] = v.y;
                r[32 * c + 4 * k + 2] = v.z;
                r[32 * c + 4 * k + 3] = v.w;
            }
        }
        if (nvalid < 128) {
#pragma unroll
            for (int i = 0; i < 128; ++i) r[i] = i < nvalid ? r[i] : 0xff800000u;  // -inf
        }
        float mp[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mp[i] = __uint_as_float(r[i]);
#pragma unroll
        for (int i = 8; i < 128; ++i) mp[i & 7] = fmaxf(mp[i & 7], __uint_as_float(r[i]));
        const float mx = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])),
                               fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7])));
        const float m_cand = fmaxf(m, mx * kC);
        const bool move = m_cand > m + 8.0f;
        const float m_new = move ? m_cand : m;
        const float alpha = move ? exp2f(m - m_new) : 1.0f;
        // the row sum as the fused kernel's two threads of a row form it:
        // per 64-key half, column i into partial i % 8, partials in a fixed
        // tree; then half 0 + half 1
        float rs_half[2];
#pragma unroll
        for (int hc = 0; hc < 2; ++hc) {
            float sp[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int i = 32 * hc; i < 32 * hc + 32; ++i) {
                const float p0 = exp2_num(fmaf(__uint_as_float(r[2 * i]), kC, -m_new));
                const float p1 = exp2_num(fmaf(__uint_as_float(r[2 * i + 1]), kC, -m_new));
                sp[(2 * i) & 7] += p0;
                sp[(2 * i + 1) & 7] += p1;
                r[i] = pack_bf16(p0, p1);
            }
            rs_half[hc] = ((sp[0] + sp[1]) + (sp[2] + sp[3])) + ((sp[4] + sp[5]) + (sp[6] + sp[7]));
        }
        const float rs = rs_half[0] + rs_half[1];
        l = fmaf(l, alpha, rs);
        m = m_new;
        // P: the previous tile's stores have read the staging
        if (lane == 0) bulk_wait_read_all();
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            uint8_t* prow = stage_p + c * 4096 + lane * 128;
#pragma unroll
            for (int k = 0; k < 8; ++k)
                *reinterpret_cast<uint4*>(prow + ((k ^ sw) << 4)) =
                    make_uint4(r[32 * c + 4 * k], r[32 * c + 4 * k + 1], r[32 * c + 4 * k + 2], r[32 * c + 4 * k + 3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
#pragma unroll
            for (int c = 0; c < 2; ++c) tma_store_3d(&a.map_p[seg], stage + c * 4096, kt.blk * 128 + 64 * c, srow, (int)bh);
            bulk_commit_group();
        }
        if (row_ok) a.alpha[rowi * a.nblk + kt.blk] = alpha;
    }
    if (!ok) {
        if (lane == 0) fail(&abort_flag);
    } else if (row_ok) {
        a.l[rowi] = l;
        if (a.lse != nullptr) a.lse[rowi] = (m + log2f(l)) * kLn2;
    }
    // the slots' loads in flight and the staging's stores finish before exit
    if (lane == 0) {
        const volatile int no_abort = 0;
        for (int j = issued - 2 < 0 ? 0 : issued - 2; j < issued; ++j)
            mbar_wait(bar + 8 * (j & 1), (j >> 1) & 1, &no_abort, kWaitLimitNs);
        bulk_wait_read_all();
    }
    __syncwarp();
}

// ====================================================================== av_gemm
// One CTA = one query tile. TMEM: O [0, 128). Per key tile j of the fused
// order the copy warp loads V_j and the tile's P block (128 rows x 128 bf16,
// two 128-byte-swizzled boxes) by TMA into a stage of a three-stage ring;
// the row threads load alpha, wait for the previous product, rescale O by
// alpha (only in warps where a row's alpha differs from 1, as the fused
// kernel does; the other rows scale by exactly 1) and signal the MMA thread,
// which issues O += P V with P as the K-major A operand from shared memory.
struct AvArgs {
    CUtensorMap map_v[2];  // v per segment (0 text, 1 image) as 4-D (d, h, token, b)
    CUtensorMap map_p;     // P bf16 [B*H*S, ncols], box 64 x 128
    Geom g;
    ValidLen vl;
    const float* alpha;    // [B, H, S, nblk]
    const float* l;        // [B, H, S]
    SegBf16 out;           // [B, S, H, 128] (text rows, image rows)
    int ncols, nblk;
};

constexpr int kAvStages = 3;
constexpr int kAvStageBytes = 2 * kTileBytes;  // V tile, P block
constexpr int kAvSmemBytes = kAvStages * kAvStageBytes + 1024;

__global__ void __launch_bounds__(kThreads, 1) av_gemm_kernel(const __grid_constant__ AvArgs a) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bars[2 * kAvStages + 3];
    __shared__ uint32_t tmem_slot;
    __shared__ volatile int abort_flag;

    const Geom& g = a.g;
    const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int q0, q_end;
    query_tile(g, qt, q0, q_end);
    const int L = a.vl.L[b];
    const int nkt = n_key_tiles(g, L);
    const size_t bh = (size_t)b * g.H + h;

    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    auto stage_v = [&](int s) { return sbase + s * kAvStageBytes; };
    auto stage_p = [&](int s) { return sbase + s * kAvStageBytes + kTileBytes; };
    const uint32_t bar_full = smem_u32(&bars[0]);           // [kAvStages] V and P loaded
    const uint32_t bar_empty = smem_u32(&bars[kAvStages]);  // [kAvStages] stage's product done
    const uint32_t bar_p = smem_u32(&bars[2 * kAvStages]);      // O rescaled (128 row threads)
    const uint32_t bar_o = smem_u32(&bars[2 * kAvStages + 1]);  // product of tile j done (O updated)
    const uint32_t bar_drain = smem_u32(&bars[2 * kAvStages + 2]);

    if (tid == 0) {
        abort_flag = 0;
        for (int s = 0; s < kAvStages; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
        }
        mbar_init(bar_p, 128);
        mbar_init(bar_o, 1);
        mbar_init(bar_drain, 1);
        fence_barrier_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc(smem_u32(&tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    if (warp == kWarpTma) {
        if (lane == 0) {
            prefetch_tensormap(&a.map_v[0]);
            prefetch_tensormap(&a.map_v[1]);
            prefetch_tensormap(&a.map_p);
            const int prow = (int)(bh * g.S) + q0;  // the tile's first row of P
            int issued = 0;
            for (int j = 0; j < nkt && !abort_flag; ++j) {
                const int s = j % kAvStages;
                if (j >= kAvStages &&
                    !mbar_wait(bar_empty + 8 * s, ((j / kAvStages) + 1) & 1, &abort_flag, kWaitLimitNs)) {
                    fail(&abort_flag);
                    break;
                }
                const KeyTile kt = key_tile(g, L, j);
                const uint32_t bf = bar_full + 8 * s;
                mbar_expect_tx(bf, kAvStageBytes);
                const int vseg = kt.k0 < g.T_txt ? 0 : 1, vrow = vseg ? kt.k0 - g.T_txt : kt.k0;
                tma_load_4d(stage_v(s), &a.map_v[vseg], bf, 0, h, vrow, b);
                tma_load_4d(stage_v(s) + kBoxBytes, &a.map_v[vseg], bf, 64, h, vrow, b);
                tma_load_2d(stage_p(s), &a.map_p, bf, kt.blk * 128, prow);
                tma_load_2d(stage_p(s) + kBoxBytes, &a.map_p, bf, kt.blk * 128 + 64, prow);
                issued = j + 1;
            }
            const volatile int no_abort = 0;
            for (int j = issued - kAvStages < 0 ? 0 : issued - kAvStages; j < issued; ++j)
                mbar_wait(bar_full + 8 * (j % kAvStages), (j / kAvStages) & 1, &no_abort, kWaitLimitNs);
        }
    } else if (warp == kWarpMma) {
        if (lane == 0) {
            bool ok = true;
            for (int j = 0; ok && j < nkt; ++j) {
                const int s = j % kAvStages;
                ok = mbar_wait(bar_p, j & 1, &abort_flag, kWaitLimitNs) &&
                     mbar_wait(bar_full + 8 * s, (j / kAvStages) & 1, &abort_flag, kWaitLimitNs);
                if (!ok) break;
                tc_fence_after();
                // the fused forward's PV product: A = P (K-major, here from
                // shared memory), B = V MN-major, k-steps in the same order
                const uint32_t dv = stage_v(s), dp = stage_p(s);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    // the fused kernel's k-step order: 0, 1, 4, 5, then 2, 3, 6, 7
                    const int kk = 2 * (i >> 2) + (i & 1) + 4 * ((i >> 1) & 1);
                    mma_ss(tmem, sdesc_sw128(dp + (kk >> 2) * kBoxBytes + (kk & 3) * 32, 16, 1024),
                           sdesc_sw128(dv + kk * 2048, kBoxBytes, 1024), kIdescO, (j > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(bar_o);
                mma_commit(bar_empty + 8 * s);
            }
            if (!ok) fail(&abort_flag);
            mma_commit(bar_drain);
            const volatile int no_abort = 0;
            mbar_wait(bar_drain, 0, &no_abort, kWaitLimitNs);
        }
    } else {
        const uint32_t lane_addr = (uint32_t)((warp & 3) * 32) << 16;
        const int row = (warp & 3) * 32 + lane;
        const int n = q0 + row;
        const bool in_seg = n < q_end;
        const size_t rowi = bh * g.S + (in_seg ? n : q0);
        bool ok = true;
        for (int j = 0; j < nkt; ++j) {
            const KeyTile kt = key_tile(g, L, j);
            const float alpha = in_seg ? a.alpha[rowi * a.nblk + kt.blk] : 1.0f;
            if (j > 0) {
                // the product of tile j - 1 has finished writing O
                if (!warp_wait(bar_o, (j - 1) & 1, &abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (__any_sync(0xffffffffu, alpha != 1.0f)) {
                    uint32_t o32[32];
#pragma unroll 1
                    for (int c = 0; c < 4; ++c) {
                        tmem_ld32(tmem + lane_addr + 32 * c, o32);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o32[i] = __float_as_uint(__uint_as_float(o32[i]) * alpha);
                        tmem_st32(tmem + lane_addr + 32 * c, o32);
                    }
                    tmem_st_wait();
                }
            }
            tc_fence_before();
            mbar_arrive(bar_p);
        }
        if (ok && warp_wait(bar_o, (nkt - 1) & 1, &abort_flag)) {
            tc_fence_after();
            // the TMEM loads are warp-collective; only rows inside the
            // segment store
            const float inv = 1.0f / a.l[rowi];
            uint4* orow = reinterpret_cast<uint4*>(seg_row(a.out, g, b, in_seg ? n : q0, h));
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                uint32_t r[32];
                tmem_ld32(tmem + lane_addr + 32 * c, r);
                tmem_ld_wait();
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        w[e] = pack_bf16(__uint_as_float(r[8 * q + 2 * e]) * inv,
                                         __uint_as_float(r[8 * q + 2 * e + 1]) * inv);
                    if (in_seg) orow[4 * c + q] = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
        } else {
            fail(&abort_flag);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

cudaError_t launch_qk_gemm(const Geom& g, const ValidLen& vl, const uint16_t* qh, const uint16_t* kh, float* scores,
                           cudaStream_t s) {
    QkArgs a;
    memset(a.map_a_seg, 0, sizeof(a.map_a_seg));  // the dP form's maps: unused here
    memset(a.map_b_seg, 0, sizeof(a.map_b_seg));
    const uint64_t rows = (uint64_t)g.B * g.H * g.S;
    if (!tmap::rows_bf16(&a.map_q, qh, rows) || !tmap::rows_bf16(&a.map_k, kh, rows)) return cudaErrorInvalidValue;
    a.g = g;
    a.vl = vl;
    a.scores = scores;
    a.ncols = 128 * (g.ntq_txt + g.ntq_img);
    for (int seg = 0; seg < 2; ++seg)
        if (!tmap::scores_f32_segment(&a.map_s[seg], scores, g, a.ncols, seg)) return cudaErrorInvalidValue;
    cudaError_t e =
        cudaFuncSetAttribute(qk_gemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kQkSmemBytes);
    if (e != cudaSuccess) return e;
    const dim3 grid(g.ntq_txt + g.ntq_img, g.H, g.B);
    timing_begin(kKQkGemm, s);
    qk_gemm_kernel<false><<<grid, kThreads, kQkSmemBytes, s>>>(a);
    timing_end(kKQkGemm, s);
    return cudaGetLastError();
}

cudaError_t launch_dp_gemm(const Geom& g, const ValidLen& vl, const SegBf16& dout, const SegBf16& v, float* dp,
                           cudaStream_t s) {
    QkArgs a;
    memset(&a.map_q, 0, sizeof(a.map_q));
    memset(&a.map_k, 0, sizeof(a.map_k));
    for (int seg = 0; seg < 2; ++seg)
        if (!tmap::seg_bf16(&a.map_a_seg[seg], dout, g, seg) || !tmap::seg_bf16(&a.map_b_seg[seg], v, g, seg))
            return cudaErrorInvalidValue;
    a.g = g;
    a.vl = vl;
    a.scores = dp;
    a.ncols = 128 * (g.ntq_txt + g.ntq_img);
    for (int seg = 0; seg < 2; ++seg)
        if (!tmap::scores_f32_segment(&a.map_s[seg], dp, g, a.ncols, seg)) return cudaErrorInvalidValue;
    cudaError_t e =
        cudaFuncSetAttribute(qk_gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kQkSmemBytes);
    if (e != cudaSuccess) return e;
    const dim3 grid(g.ntq_txt + g.ntq_img, g.H, g.B);
    timing_begin(kKDpGemm, s);
    qk_gemm_kernel<true><<<grid, kThreads, kQkSmemBytes, s>>>(a);
    timing_end(kKDpGemm, s);
    return cudaGetLastError();
}

cudaError_t launch_softmax(const Geom& g, const ValidLen& vl, const float* scores, uint16_t* p, float* alpha,
                           float* l, float* lse, cudaStream_t s) {
    SmArgs a;
    a.g = g;
    a.vl = vl;
    a.alpha = alpha;
    a.l = l;
    a.lse = lse;
    a.nblk = g.ntq_txt + g.ntq_img;
    a.ncols = 128 * a.nblk;
    if (!tmap::mat_f32(&a.map_sc, scores, (long long)g.B * g.H * g.S, a.ncols, 32, 32)) return cudaErrorInvalidValue;
    for (int seg = 0; seg < 2; ++seg)
        if (!tmap::p_bf16_segment(&a.map_p[seg], p, g, a.ncols, seg)) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(softmax_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmSmemBytes);
    if (e != cudaSuccess) return e;
    const dim3 grid(4 * a.nblk, g.H, g.B);
    timing_begin(kKSoftmax, s);
    softmax_kernel<<<grid, 32, kSmSmemBytes, s>>>(a);
    timing_end(kKSoftmax, s);
    return cudaGetLastError();
}

cudaError_t launch_av_gemm(const Geom& g, const ValidLen& vl, const uint16_t* p, const float* alpha, const float* l,
                           const SegBf16& v, const SegBf16& out, cudaStream_t s) {
    AvArgs a;
    if (!tmap::seg_bf16(&a.map_v[0], v, g, 0) || !tmap::seg_bf16(&a.map_v[1], v, g, 1)) return cudaErrorInvalidValue;
    a.g = g;
    a.vl = vl;
    a.alpha = alpha;
    a.l = l;
    a.out = out;
    a.nblk = g.ntq_txt + g.ntq_img;
    a.ncols = 128 * a.nblk;
    if (!tmap::mat_bf16(&a.map_p, p, (long long)g.B * g.H * g.S, a.ncols, 128)) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(av_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kAvSmemBytes);
    if (e != cudaSuccess) return e;
    const dim3 grid(a.nblk, g.H, g.B);
    timing_begin(kKAvGemm, s);
    av_gemm_kernel<<<grid, kThreads, kAvSmemBytes, s>>>(a);
    timing_end(kKAvGemm, s);
    return cudaGetLastError();
}

int read_and_clear_status_unfused(cudaStream_t s) {
    int v = 0, zero = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_status_unf, sizeof(int), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return -1;
    if (cudaMemcpyToSymbolAsync(g_status_unf, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return -1;
    if (cudaStreamSynchronize(s) != cudaSuccess) return -1;
    return v;
}

}  // namespace rlk

// Joint attention backward on the tcgen05 tensor cores (the "bwd" half of
// the WS1 attention rows of RFC #386 and of the "WS1 Single-GPU Kernel
// List"): two atomic-free kernels with the forward's warp roles.
//
//   dkdv: one CTA = (key tile of 128, head, sample). Walks every query tile
//         of 128 in one fixed ascending order (text tiles from token 0, then
//         image tiles from token T_txt). Per query tile (dS^T is formed
//         while dV computes, the next tile's P^T while dK computes):
//           S^T  = K Q^T, dP^T = V dO^T            (tcgen05, A and B in smem)
//           P^T  = exp2(S^T * c - lse2), dS^T = P^T * (dP^T - Delta)
//                                                  (8 warps: key row = TMEM
//                                                   lane, 64 queries each;
//                                                   bf16 results into TMEM)
//           dV  += P^T dO,  dK += dS^T Q           (tcgen05, A from TMEM)
//         and stores the bf16 dS^T tile in the tensor cores' operand layout.
//   dq:   persistent; one unit = (query tile of 128, head, sample):
//         dQ += dS K over the key tiles in the forward's order, reading the
//         dS^T tiles back, so S and dP are computed once, not twice.
// Accumulators (dV, dK, dQ) stay in TMEM in FP32 for the whole unit and are
// written once. P and dS enter their products as bf16 (round to nearest
// even); dK and dQ use the same bf16 dS. lse2 = lse * log2(e) and Delta = rowsum(dO * O) come from the
// backward preprocess in a tile-padded layout (one 128-slot block per query
// tile; slots past a segment hold lse2 = +inf and Delta = 0, so their P is
// exactly 0). Every wait is bounded (RLK_ERR_DEVICE_TIMEOUT on give-up).
#include "rlk_device.cuh"
#include "rlk_internal.h"
#include "rlk_normrope_bwd.cuh"
#include "rlk_sm100.cuh"
#include "rlk_tmap.h"


RLK_DEFINE_STRICT_PROBE(probe_bwd_tu)

namespace rlk {
namespace {

using namespace sm100;

// warps 0-7: elementwise (warp w owns TMEM lane quarter w % 4 and the
// column half w / 4 of each row; kEwWarps below); warp 8: TMA producer;
// warps 9 and 10: MMA issuers of two independent chains (warp 9 owns TMEM).
constexpr int kEwWarps = 8;                       // elementwise warps (16 measured 3% slower)
constexpr int kEwThreads = 32 * kEwWarps;
constexpr int kThreads = kEwThreads + 96;         // + TMA producer + two MMA issuers
constexpr int kWarpTma = kEwWarps, kWarpMma = kEwWarps + 1;
constexpr int kGroupCols = 128 / (kEwWarps / 4);  // query columns per elementwise warp
constexpr int kBoxBytes = 128 * 128;       // 128 rows x 64 bf16
constexpr int kTileBytes = 2 * kBoxBytes;  // 128 rows x 128 bf16
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr float kC = (float)(1.4426950408889634 * 0.08838834764831845);  // log2(e) / sqrt(128)
constexpr float kScale = 0.08838834764831845f;                          // 1 / sqrt(128)
constexpr uint32_t kIdescKK = idesc_bf16(128, 128, false, false);
constexpr uint32_t kIdescKM = idesc_bf16(128, 128, false, true);

__device__ int g_status_bwd;

struct BwdArgs {
    CUtensorMap map_q;    // qh [B*H*S, 128]
    CUtensorMap map_k;    // kh [B*H*S, 128]
    CUtensorMap map_v[2];   // v per segment (0 text, 1 image), 4-D (d, h, token, b)
    CUtensorMap map_do[2];  // dO per segment
    Geom g;
    ValidLen vl;
    const float* lse2_p;  // [B, H, nq_pad]
    const float* delta_p; // [B, H, nq_pad]
    SegBf16 dv;           // [B, S, H, 128] (text rows, image rows)
    uint8_t* ds_tiles;    // [B, H, nq, nq] images of 32 KB (query tile major)
    // output maps per segment (0 text, 1 image) so a tile's rows past its
    // segment are clipped: dV [B, S, H, 128] bf16, dk^ [B*H, S, 128] fp32
    CUtensorMap map_dv[2];
    CUtensorMap map_dk[2];
    float* dkh;  // dk^ = dK of the rotated, normalised keys / sqrt(128), fp32 [B, H, S, 128]
    // the RoPE / RMSNorm backward of the query rows in the dQ epilogue:
    // input q (bf16 [B, S, H, 128]), its RMSNorm factors rq [B, H, S], the
    // gains (q_txt, k_txt, q_img, k_img), the cos/sin table; outputs dQ and
    // the q gain-gradient partials of every (b, h, 128-token tile, 32-row
    // quarter) in dgt [B, H, 2 (q, k), n_tiles, 4, 128]
    SegBf16 q_in, dq_out;
    const float* rq;
    const float* gains[4];
    const float2* tab;
    float* dgt;
};

__device__ __forceinline__ void fail(volatile int* abort_flag) {
    *abort_flag = 1;
    atomicOr(&g_status_bwd, 1);
}

// K-major operand (rows x 128 bf16 as two 64-column boxes), k-step kk of 16
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t tile, int kk) {
    return sdesc_sw128(tile + (kk >> 2) * kBoxBytes + (kk & 3) * 32, 16, 1024);
}
// MN-major operand: the same tile read with its rows as the K dimension
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t tile, int kk) {
    return sdesc_sw128(tile + kk * 2048, kBoxBytes, 1024);
}

// TMEM column of the bf16 A operand (P or dS) for k-step kk: the column
// half h = kk / 4 of the 128 fp32 columns is rewritten in place as 32 packed
// columns at the start of that half, so the two warps sharing a lane
// quarter never overwrite each other's unread scores.
__device__ __forceinline__ uint32_t a_col(int kk) {
    return (16 * kk / kGroupCols) * kGroupCols + (16 * kk % kGroupCols) / 2;
}
// A warp's packed bf16 pairs of its columns, kGroupCols / 2 TMEM columns.
__device__ __forceinline__ void tmem_st_packed(uint32_t taddr, const uint32_t (&r)[kGroupCols / 2]) {
    if constexpr (kGroupCols == 64)
        tmem_st32(taddr, *reinterpret_cast<const uint32_t(*)[32]>(&r[0]));
    else
        tmem_st16(taddr, *reinterpret_cast<const uint32_t(*)[16]>(&r[0]));
}

// dS^T tile image (128 keys x 128 queries, bf16, 32 KB): the non-swizzled
// MN-major operand layout of the tensor cores. Query chunk C (8 queries) is
// a 2 KB block of 128 key rows of 16 bytes, so 8 consecutive keys of one
// chunk form one 128-byte core matrix; chunks along MN are 2 KB apart,
// 8-key groups along K 128 bytes apart.
constexpr int kDsChunkBytes = 2048;
__device__ __forceinline__ int ds_image_offset(int query, int key) {
    return (query >> 3) * kDsChunkBytes + key * 16 + (query & 7) * 2;
}
__device__ __forceinline__ uint64_t desc_ds_image(uint32_t tile, int kk) {
    return sdesc_noswizzle(tile + kk * 2 * 128, 128, kDsChunkBytes);
}

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, kWaitLimitNs));
}

// Query tile i (segment aligned): first token and end of its segment.
__device__ __forceinline__ void q_tile(const Geom& g, int i, int& q0, int& q_end) {
    if (i < g.ntq_txt) {
        q0 = i * 128;
        q_end = g.T_txt;
    } else {
        q0 = g.T_txt + (i - g.ntq_txt) * 128;
        q_end = g.S;
    }
}

// ====================================================================== dK, dV
constexpr int kKvSmemK = 0, kKvSmemV = kTileBytes, kKvSmemStage = 2 * kTileBytes;
constexpr int kKvStageBytes = 2 * kTileBytes + 1024;  // Q, dO, lse2[128], delta[128]
constexpr int kKvSmemBytes = kKvSmemStage + 2 * kKvStageBytes + 1024;
constexpr uint32_t kColDV = 0, kColDK = 128, kColST = 256, kColDPT = 384;

__global__ void __launch_bounds__(kThreads, 1) attn_bwd_dkdv_tc_kernel(const __grid_constant__ BwdArgs a) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bars[12];  // bars[9]: second issuer's drain
    __shared__ uint32_t tmem_slot;
    __shared__ volatile int abort_flag;

    const Geom& g = a.g;
    const int kt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool k_txt = kt < g.ntq_txt;
    const int k0 = k_txt ? kt * 128 : g.T_txt + (kt - g.ntq_txt) * 128;
    const int seg_end = k_txt ? g.T_txt : g.S;
    const int L = a.vl.L[b];
    const int kvalid_end = k_txt ? L : g.S;
    const size_t bh = (size_t)b * g.H + h;
    const int row_base = (int)(bh * g.S);
    const int nq = g.ntq_txt + g.ntq_img;

    float* dkh = a.dkh + bh * g.S * kHeadDim;

    if (k0 >= kvalid_end) {  // every key of the tile is masked: exact zeros
        const int rows = min(128, seg_end - k0);
        for (int i = tid; i < rows * 16; i += kThreads) {
            const int r = i >> 4, c = i & 15;
            *reinterpret_cast<uint4*>(seg_row(a.dv, g, b, k0 + r, h) + c * 8) = make_uint4(0, 0, 0, 0);
            float4* dst = reinterpret_cast<float4*>(dkh + (size_t)(k0 + r) * kHeadDim + c * 8);
            dst[0] = make_float4(0.f, 0.f, 0.f, 0.f);
            dst[1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        return;
    }

    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const uint32_t sK = sbase + kKvSmemK, sV = sbase + kKvSmemV;
    auto stage_q = [&](int s) { return sbase + kKvSmemStage + s * kKvStageBytes; };
    auto stage_o = [&](int s) { return stage_q(s) + kTileBytes; };
    auto stage_l = [&](int s) { return stage_q(s) + 2 * kTileBytes; };
    const uint32_t bar_kv = smem_u32(&bars[0]);
    const uint32_t bar_full = smem_u32(&bars[1]);   // [2]
    const uint32_t bar_empty = smem_u32(&bars[3]);  // [2]
    const uint32_t bar_st = smem_u32(&bars[5]);   // S^T_i computed
    const uint32_t bar_dpt = smem_u32(&bars[6]);  // dP^T_i computed
    const uint32_t bar_p = smem_u32(&bars[10]);   // P^T_i written (bf16)
    const uint32_t bar_ds = smem_u32(&bars[11]);  // dS^T_i written (bf16)
    const uint32_t bar_done = smem_u32(&bars[7]);
    const uint32_t bar_drain = smem_u32(&bars[8]);

    if (tid == 0) {
        abort_flag = 0;
        mbar_init(bar_kv, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 2);  // one commit per issuer
        }
        mbar_init(bar_st, 1);
        mbar_init(bar_dpt, 1);
        mbar_init(bar_p, kEwThreads);
        mbar_init(bar_ds, kEwThreads);
        mbar_init(bar_done, 2);
        mbar_init(bar_drain, 1);
        mbar_init(smem_u32(&bars[9]), 1);
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
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tensormap(&a.map_q);
            prefetch_tensormap(&a.map_k);
            prefetch_tensormap(&a.map_v[0]);
            prefetch_tensormap(&a.map_v[1]);
            prefetch_tensormap(&a.map_do[0]);
            prefetch_tensormap(&a.map_do[1]);
            mbar_expect_tx(bar_kv, 2 * kTileBytes);
            tma_load_2d(sK, &a.map_k, bar_kv, 0, row_base + k0);
            tma_load_2d(sK + kBoxBytes, &a.map_k, bar_kv, 64, row_base + k0);
            // tiles never straddle the streams: rows counted from the segment start
            const int vseg = k_txt ? 0 : 1, vrow = k_txt ? k0 : k0 - g.T_txt;
            tma_load_4d(sV, &a.map_v[vseg], bar_kv, 0, h, vrow, b);
            tma_load_4d(sV + kBoxBytes, &a.map_v[vseg], bar_kv, 64, h, vrow, b);
            int issued = 0;
            for (int i = 0; i < nq && !abort_flag; ++i) {
                const int s = i & 1;
                if (i >= 2 && !mbar_wait(bar_empty + 8 * s, ((i >> 1) + 1) & 1, &abort_flag, kWaitLimitNs)) {
                    fail(&abort_flag);
                    break;
                }
                int q0, q_end;
                q_tile(g, i, q0, q_end);
                const uint32_t bf = bar_full + 8 * s;
                mbar_expect_tx(bf, 2 * kTileBytes + 1024);
                tma_load_2d(stage_q(s), &a.map_q, bf, 0, row_base + q0);
                tma_load_2d(stage_q(s) + kBoxBytes, &a.map_q, bf, 64, row_base + q0);
                const int oseg = i < g.ntq_txt ? 0 : 1, orow = oseg ? q0 - g.T_txt : q0;
                tma_load_4d(stage_o(s), &a.map_do[oseg], bf, 0, h, orow, b);
                tma_load_4d(stage_o(s) + kBoxBytes, &a.map_do[oseg], bf, 64, h, orow, b);
                const size_t slot = bh * g.nq_pad + (size_t)i * 128;
                bulk_load(stage_l(s), a.lse2_p + slot, 512, bf);
                bulk_load(stage_l(s) + 512, a.delta_p + slot, 512, bf);
                issued = i + 1;
            }
            const volatile int no_abort = 0;
            mbar_wait(bar_kv, 0, &no_abort, kWaitLimitNs);
            for (int i = issued - 2 < 0 ? 0 : issued - 2; i < issued; ++i)
                mbar_wait(bar_full + 8 * (i & 1), (i >> 1) & 1, &no_abort, kWaitLimitNs);
        }
    } else if (warp == kWarpMma || warp == kWarpMma + 1) {
        // ------------------------------------------------ MMA issuers
        // Two independent chains, one issuing thread each, so that one keeps
        // the tensor pipe fed while the other waits on a barrier:
        //   warp 9:  S^T_0; per query tile i: dV_i (after P^T_i), then
        //            S^T_{i+1} (after stage i+1 lands). S^T_{i+1} overwrites
        //            the columns holding P^T_i, which dV_i, issued before it
        //            on the same thread, has consumed.
        //   warp 10: per query tile i: dP^T_i, then dK_i (after dS^T_i).
        //            dP^T_{i+1} overwrites dS^T_i after dK_i, likewise.
        // The two write disjoint TMEM columns; a stage frees when both have
        // issued their last product reading it.
        if (lane == 0) {
            const bool chain_p = warp == kWarpMma;
            const uint32_t bar_my_drain = chain_p ? bar_drain : smem_u32(&bars[9]);
            auto issue_st = [&](int i) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_ss(tmem + kColST, desc_kmajor(sK, kk), desc_kmajor(stage_q(i & 1), kk), kIdescKK, kk > 0);
                mma_commit(bar_st);
            };
            bool ok = mbar_wait(bar_kv, 0, &abort_flag, kWaitLimitNs);
            if (chain_p) {
                ok = ok && mbar_wait(bar_full, 0, &abort_flag, kWaitLimitNs);
                if (ok) {
                    tc_fence_after();
                    issue_st(0);
                }
                for (int i = 0; ok && i < nq; ++i) {
                    const int s = i & 1;
                    if (!mbar_wait(bar_p, i & 1, &abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_ts(tmem + kColDV, tmem + kColST + a_col(kk), desc_mnmajor(stage_o(s), kk), kIdescKM,
                               (i > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(bar_empty + 8 * s);
                    if (i + 1 < nq) {
                        if (!mbar_wait(bar_full + 8 * (s ^ 1), ((i + 1) >> 1) & 1, &abort_flag, kWaitLimitNs)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        issue_st(i + 1);
                    }
                }
            } else {
                for (int i = 0; ok && i < nq; ++i) {
                    const int s = i & 1;
                    if (!mbar_wait(bar_full + 8 * s, (i >> 1) & 1, &abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_ss(tmem + kColDPT, desc_kmajor(sV, kk), desc_kmajor(stage_o(s), kk), kIdescKK, kk > 0);
                    mma_commit(bar_dpt);
                    if (!mbar_wait(bar_ds, i & 1, &abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_ts(tmem + kColDK, tmem + kColDPT + a_col(kk), desc_mnmajor(stage_q(s), kk), kIdescKM,
                               (i > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(bar_empty + 8 * s);
                }
            }
            if (ok)
                mma_commit(bar_done);
            else
                fail(&abort_flag);
            mma_commit(bar_my_drain);
            const volatile int no_abort = 0;
            mbar_wait(bar_my_drain, 0, &no_abort, kWaitLimitNs);
        }
    } else {
        // ------------------------------------------------ elementwise warps
        // warp w: key rows 32 * (w % 4) + lane, query columns
        // [kGroupCols * grp, kGroupCols * (grp + 1)), grp = w / 4. No row
        // reduction: every element of P^T and dS^T is the thread's own.
        const int lq = warp & 3, grp = warp >> 2;
        const uint32_t lane_addr = (uint32_t)(lq * 32) << 16;
        const int kr = lq * 32 + lane;
        const int c0 = kGroupCols * grp;
        const bool kvalid = k0 + kr < kvalid_end;
        bool ok = true;
        for (int i = 0; i < nq; ++i) {
            const int s = i & 1;
            if (!warp_wait(bar_full + 8 * s, (i >> 1) & 1, &abort_flag) || !warp_wait(bar_st, i & 1, &abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const float4* l2v =
                reinterpret_cast<const float4*>(smem_raw + (stage_l(s) - smem_u32(smem_raw))) + c0 / 4;
            const float4* dlv = l2v + 32;
            // P^T = exp2(S^T * c - lse2[query]) (masked keys: 0), kept in fp32 for dS
            uint32_t rs[kGroupCols];
#pragma unroll
            for (int c = 0; c < kGroupCols; c += 32)
                tmem_ld32(tmem + lane_addr + kColST + c0 + c, *reinterpret_cast<uint32_t(*)[32]>(&rs[c]));
            tmem_ld_wait();
            float pf[kGroupCols];
            uint32_t pk[kGroupCols / 2];
            if (kvalid) {  // the row's key is valid for the whole CTA: no per-element select
#pragma unroll
                for (int e4 = 0; e4 < kGroupCols / 4; ++e4) {
                    const float4 l4 = l2v[e4];
                    const float lq4[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        pf[4 * e4 + u] = exp2_num(fmaf(__uint_as_float(rs[4 * e4 + u]), kC, -lq4[u]));
                    pk[2 * e4] = pack_bf16(pf[4 * e4], pf[4 * e4 + 1]);
                    pk[2 * e4 + 1] = pack_bf16(pf[4 * e4 + 2], pf[4 * e4 + 3]);
                }
            } else {  // a masked key: P = 0
#pragma unroll
                for (int e = 0; e < kGroupCols; ++e) pf[e] = 0.0f;
#pragma unroll
                for (int e = 0; e < kGroupCols / 2; ++e) pk[e] = 0u;
            }
            tmem_st_packed(tmem + lane_addr + kColST + c0, pk);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bar_p);
            // dS^T = P^T * (dP^T - Delta[query])
            if (!warp_wait(bar_dpt, i & 1, &abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t rd[kGroupCols];
#pragma unroll
            for (int c = 0; c < kGroupCols; c += 32)
                tmem_ld32(tmem + lane_addr + kColDPT + c0 + c, *reinterpret_cast<uint32_t(*)[32]>(&rd[c]));
            tmem_ld_wait();
#pragma unroll
            for (int e4 = 0; e4 < kGroupCols / 4; ++e4) {
                const float4 d4 = dlv[e4];
                const float dq4[4] = {d4.x, d4.y, d4.z, d4.w};
                float ds[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) ds[u] = pf[4 * e4 + u] * (__uint_as_float(rd[4 * e4 + u]) - dq4[u]);
                pk[2 * e4] = pack_bf16(ds[0], ds[1]);
                pk[2 * e4 + 1] = pack_bf16(ds[2], ds[3]);
            }
            tmem_st_packed(tmem + lane_addr + kColDPT + c0, pk);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bar_ds);
            // the same bf16 dS^T row into the (query tile i, key tile kt)
            // image for the dQ product (see ds_image_offset): a warp's
            // store of one query chunk covers 512 contiguous bytes
            uint8_t* ds_img = a.ds_tiles + ((bh * nq + i) * nq + kt) * (size_t)kTileBytes + ds_image_offset(c0, kr);
#pragma unroll
            for (int c = 0; c < kGroupCols / 8; ++c)
                *reinterpret_cast<uint4*>(ds_img + c * kDsChunkBytes) =
                    make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        }
        if (ok && warp_wait(bar_done, 0, &abort_flag)) {
            tc_fence_after();
            // Stage dV (bf16) and dK (fp32, times 1/sqrt(D)) in the K, V and
            // first Q buffers (every product has finished) as six 128-row x
            // 128-byte boxes in the 128-byte-swizzled layout of the output
            // maps: dV boxes 0-1 (64 columns each), dK boxes 2-5 (32 columns
            // each). One thread then stores the tile with TMA; the segment
            // maps clip rows past the key's segment. Masked keys get zeros.
            uint8_t* stg = smem_raw + (sbase - smem_u32(smem_raw));
            const int sw = kr & 7;
#pragma unroll 1
            for (int c = 0; c < kGroupCols; c += 32) {
                uint32_t r[32];
                tmem_ld32(tmem + lane_addr + kColDV + c0 + c, r);
                tmem_ld_wait();
                // dV box (c0 + c) / 64, 16-byte chunks from ((c0 + c) % 64) / 8
                uint8_t* dvrow = stg + ((c0 + c) >> 6) * kBoxBytes + kr * 128;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        w[e] = kvalid ? pack_bf16(__uint_as_float(r[8 * q + 2 * e]), __uint_as_float(r[8 * q + 2 * e + 1]))
                                      : 0u;
                    *reinterpret_cast<uint4*>(dvrow + (((((c0 + c) & 63) >> 3) + q) ^ sw) * 16) =
                        make_uint4(w[0], w[1], w[2], w[3]);
                }
                tmem_ld32(tmem + lane_addr + kColDK + c0 + c, r);
                tmem_ld_wait();
                uint8_t* dkrow = stg + (2 + ((c0 + c) >> 5)) * kBoxBytes + kr * 128;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    float4 f;
                    f.x = kvalid ? __uint_as_float(r[4 * q]) * kScale : 0.0f;
                    f.y = kvalid ? __uint_as_float(r[4 * q + 1]) * kScale : 0.0f;
                    f.z = kvalid ? __uint_as_float(r[4 * q + 2]) * kScale : 0.0f;
                    f.w = kvalid ? __uint_as_float(r[4 * q + 3]) * kScale : 0.0f;
                    *reinterpret_cast<float4*>(dkrow + ((q ^ sw) << 4)) = f;
                }
            }
            fence_proxy_async_smem();
            named_barrier_sync(1, kEwThreads);
            if (tid == 0) {
                const int seg = k_txt ? 0 : 1;
                const int srow = k_txt ? k0 : k0 - g.T_txt;
                tma_store_4d(&a.map_dv[seg], sbase, 0, h, srow, b);
                tma_store_4d(&a.map_dv[seg], sbase + kBoxBytes, 64, h, srow, b);
#pragma unroll
                for (int q = 0; q < 4; ++q) tma_store_3d(&a.map_dk[seg], sbase + (2 + q) * kBoxBytes, 32 * q, srow, (int)bh);
                bulk_commit_group();
                bulk_wait_read_all();
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

// ====================================================================== dQ
// dQ_i = sum_j dS_ij K_j as a streaming tcgen05 GEMM over the bf16 dS^T
// images the dK/dV kernel wrote (one 32 KB image per (query tile, key tile)
// pair, query tile major, in the tensor cores' non-swizzled operand layout,
// so one bulk copy stages it and it enters the product as an MN-major A). Persistent: CTA c takes the units (query tile, head, sample)
// c, c + grid, ... in order; a unit sums its key tiles in the forward's
// order into one of two TMEM accumulators, so the epilogue of one unit
// overlaps the products of the next. No unit depends on which CTA runs it.
constexpr int kDqThreads = 192;  // warps 0-3 epilogue, 4 copies, 5 MMA
constexpr int kDqWarpTma = 4, kDqWarpMma = 5;
constexpr int kDqStages = 3;
constexpr int kDqStageBytes = 2 * kTileBytes;  // dS^T image, K tile
constexpr int kDqSmemBytes = kDqStages * kDqStageBytes + 1024;
constexpr uint32_t kDqTmemCols = 256;
constexpr uint32_t kIdescMM = idesc_bf16(128, 128, true, true);

struct DqUnit {
    int qt, h, b;
};
// Units run from the last (sample, head) down: the dK/dV kernel's last CTAs
// wrote those dS^T images, some still in L2 (317.0 -> 313.6 us measured).
__device__ __forceinline__ DqUnit dq_unit(const Geom& g, int nq, int u) {
    DqUnit r;
    u = nq * g.H * g.B - 1 - u;
    r.qt = u % nq;
    r.h = (u / nq) % g.H;
    r.b = u / (nq * g.H);
    return r;
}

__global__ void __launch_bounds__(kDqThreads, 1) attn_bwd_dq_tc_kernel(const __grid_constant__ BwdArgs a) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bars[2 * kDqStages + 5];
    __shared__ uint32_t tmem_slot;
    __shared__ volatile int abort_flag;

    const Geom& g = a.g;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nq = g.ntq_txt + g.ntq_img;
    const int n_units = nq * g.H * g.B;
    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    auto stage = [&](int s) { return sbase + s * kDqStageBytes; };
    const uint32_t bar_full = smem_u32(&bars[0]);                   // [3] stage loaded
    const uint32_t bar_empty = smem_u32(&bars[kDqStages]);          // [3] stage consumed
    const uint32_t bar_acc = smem_u32(&bars[2 * kDqStages]);        // [2] accumulator complete
    const uint32_t bar_free = smem_u32(&bars[2 * kDqStages + 2]);   // [2] accumulator read out
    const uint32_t bar_drain = smem_u32(&bars[2 * kDqStages + 4]);

    if (tid == 0) {
        abort_flag = 0;
        for (int s = 0; s < kDqStages; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar_acc + 8 * s, 1);
            mbar_init(bar_free + 8 * s, 128);
        }
        mbar_init(bar_drain, 1);
        fence_barrier_init();
    }
    if (warp == kDqWarpMma) {
        tmem_alloc(smem_u32(&tmem_slot), kDqTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    if (warp == kDqWarpTma) {
        // ------------------------------------------------ copies
        if (lane == 0) {
            prefetch_tensormap(&a.map_k);
            int t = 0;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < n_units && !abort_flag; u += gridDim.x) {
                const DqUnit w = dq_unit(g, nq, u);
                const int L = a.vl.L[w.b];
                const int nkt_txt = (L + 127) / 128;
                const int nkt = nkt_txt + g.ntq_img;
                const size_t bh = (size_t)w.b * g.H + w.h;
                const int row_base = (int)(bh * g.S);
                const uint8_t* tiles = a.ds_tiles + (bh * nq + w.qt) * nq * (size_t)kTileBytes;
                for (int j = 0; j < nkt; ++j, ++t) {
                    const int s = t % kDqStages;
                    if (t >= kDqStages &&
                        !mbar_wait(bar_empty + 8 * s, ((t / kDqStages) + 1) & 1, &abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    const int kt = j < nkt_txt ? j : g.ntq_txt + (j - nkt_txt);
                    const int kk0 = j < nkt_txt ? j * 128 : g.T_txt + (j - nkt_txt) * 128;
                    const uint32_t bf = bar_full + 8 * s;
                    mbar_expect_tx(bf, kDqStageBytes);
                    bulk_load(stage(s), tiles + (size_t)kt * kTileBytes, kTileBytes, bf);
                    tma_load_2d(stage(s) + kTileBytes, &a.map_k, bf, 0, row_base + kk0);
                    tma_load_2d(stage(s) + kTileBytes + kBoxBytes, &a.map_k, bf, 64, row_base + kk0);
                }
            }
            if (!ok) fail(&abort_flag);
            const volatile int no_abort = 0;
            for (int tt = t - kDqStages < 0 ? 0 : t - kDqStages; tt < t; ++tt)
                mbar_wait(bar_full + 8 * (tt % kDqStages), (tt / kDqStages) & 1, &no_abort, kWaitLimitNs);
        }
    } else if (warp == kDqWarpMma) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            int t = 0, n = 0;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < n_units; u += gridDim.x, ++n) {
                const DqUnit w = dq_unit(g, nq, u);
                const int nkt = (a.vl.L[w.b] + 127) / 128 + g.ntq_img;
                const int buf = n & 1;
                if (n >= 2 && !mbar_wait(bar_free + 8 * buf, ((n >> 1) + 1) & 1, &abort_flag, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int j = 0; j < nkt; ++j, ++t) {
                    const int s = t % kDqStages;
                    if (!mbar_wait(bar_full + 8 * s, (t / kDqStages) & 1, &abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_ss(tmem + 128 * buf, desc_ds_image(stage(s), kk), desc_mnmajor(stage(s) + kTileBytes, kk),
                               kIdescMM, (j > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(bar_empty + 8 * s);
                }
                if (ok) mma_commit(bar_acc + 8 * buf);
            }
            if (!ok) fail(&abort_flag);
            mma_commit(bar_drain);
            const volatile int no_abort = 0;
            mbar_wait(bar_drain, 0, &no_abort, kWaitLimitNs);
        }
    } else {
        // ------------------------------------------------ epilogue warps 0-3: query row 32 w + lane
        // Per unit: the RoPE / RMSNorm backward of the tile's query rows
        // from dq^ = acc / sqrt(128) (TMEM): bf16 dQ rows and this warp's
        // partial of the tile's q gain gradient (its 32 rows summed by a
        // transposing butterfly), stored for the fold.
        const uint32_t lane_addr = (uint32_t)(warp * 32) << 16;
        const int r = warp * 32 + lane;
        int n = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++n) {
            const DqUnit w = dq_unit(g, nq, u);
            const int buf = n & 1;
            if (!warp_wait(bar_acc + 8 * buf, (n >> 1) & 1, &abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            int q0, q_end;
            q_tile(g, w.qt, q0, q_end);
            const bool row_ok = q0 + r < q_end;
            const int tok = row_ok ? q0 + r : q0;  // rows past the segment read a valid row, store nothing
            const size_t bh = (size_t)w.b * g.H + w.h;
            const uint32_t acc_addr = tmem + lane_addr + 128 * buf;
            auto dq_chunk = [&](int c, float (&dy)[32]) {
                uint32_t acc[32];
                tmem_ld32(acc_addr + 32 * c, acc);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) dy[i] = row_ok ? __uint_as_float(acc[i]) * kScale : 0.0f;
            };
            nrb_row(dq_chunk, row_ok, reinterpret_cast<const uint4*>(seg_row(a.q_in, g, w.b, tok, w.h)),
                    a.rq[bh * g.S + tok], w.qt < g.ntq_txt ? a.gains[0] : a.gains[2], tab_rows(a.tab, g, tok),
                    reinterpret_cast<uint4*>(seg_row(a.dq_out, g, w.b, tok, w.h)),
                    a.dgt + ((bh * 2 * nq + w.qt) * 4 + warp) * kHeadDim, lane);
            tc_fence_before();
            mbar_arrive(bar_free + 8 * buf);
        }
        if (!ok) fail(&abort_flag);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kDqWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, kDqTmemCols);
    }
}

// ---------------------------------------------------------------- tensor maps
bool make_args(BwdArgs* a, const Geom& g, const ValidLen& vl, const uint16_t* qh, const uint16_t* kh,
               const SegBf16& v, const SegBf16& dout, const float* lse2_p, const float* delta_p) {
    const uint64_t rows = (uint64_t)g.B * g.H * g.S;
    if (!tmap::rows_bf16(&a->map_q, qh, rows) || !tmap::rows_bf16(&a->map_k, kh, rows))
        return false;
    for (int seg = 0; seg < 2; ++seg)
        if (!tmap::seg_bf16(&a->map_v[seg], v, g, seg) || !tmap::seg_bf16(&a->map_do[seg], dout, g, seg))
            return false;
    a->g = g;
    a->vl = vl;
    a->lse2_p = lse2_p;
    a->delta_p = delta_p;
    a->dv = SegBf16{{nullptr, nullptr}, {0, 0}};
    a->dkh = nullptr;
    a->ds_tiles = nullptr;
    return true;
}

void set_norm_rope_io(BwdArgs* a, const NormRopeBwdIo& nr) {
    a->q_in = nr.q;
    a->dq_out = nr.dq;
    a->rq = nr.rq;
    for (int i = 0; i < 4; ++i) a->gains[i] = nr.gains[i];
    a->tab = nr.tab;
    a->dgt = nr.dgt;
}

}  // namespace

cudaError_t launch_attn_bwd_dkdv(const Geom& g, const ValidLen& vl, const uint16_t* qh, const uint16_t* kh,
                                 const SegBf16& v, const SegBf16& dout, const float* lse2_p, const float* delta_p,
                                 const SegBf16& dv, float* dkh, uint8_t* ds_tiles, cudaStream_t s) {
    BwdArgs args;
    if (!make_args(&args, g, vl, qh, kh, v, dout, lse2_p, delta_p)) return cudaErrorInvalidValue;
    args.dv = dv;
    args.dkh = dkh;
    args.ds_tiles = ds_tiles;
    for (int seg = 0; seg < 2; ++seg)
        if (!tmap::seg_bf16(&args.map_dv[seg], dv, g, seg) || !tmap::bhsd_f32_segment(&args.map_dk[seg], dkh, g, seg))
            return cudaErrorInvalidValue;
    cudaError_t e =
        cudaFuncSetAttribute(attn_bwd_dkdv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kKvSmemBytes);
    if (e != cudaSuccess) return e;
    dim3 grid(g.ntq_txt + g.ntq_img, g.H, g.B);
    timing_begin(kKBwdDkDv, s);
    attn_bwd_dkdv_tc_kernel<<<grid, kThreads, kKvSmemBytes, s>>>(args);
    timing_end(kKBwdDkDv, s);
    return cudaGetLastError();
}

cudaError_t launch_attn_bwd_dq(const Geom& g, const ValidLen& vl, const uint16_t* kh, const uint8_t* ds_tiles,
                               const NormRopeBwdIo& nr, cudaStream_t s) {
    BwdArgs args;
    if (!tmap::rows_bf16(&args.map_k, kh, (uint64_t)g.B * g.H * g.S)) return cudaErrorInvalidValue;
    args.g = g;
    args.vl = vl;
    args.ds_tiles = const_cast<uint8_t*>(ds_tiles);
    set_norm_rope_io(&args, nr);
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(attn_bwd_dq_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDqSmemBytes);
    if (e != cudaSuccess) return e;
    const int n_units = (g.ntq_txt + g.ntq_img) * g.H * g.B;
    const int grid = n_units < sms ? n_units : sms;
    timing_begin(kKBwdDq, s);
    attn_bwd_dq_tc_kernel<<<grid, kDqThreads, kDqSmemBytes, s>>>(args);
    timing_end(kKBwdDq, s);
    return cudaGetLastError();
}

int read_and_clear_status_bwd(cudaStream_t s) {
    int v = 0, zero = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_status_bwd, sizeof(int), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return -1;
    if (cudaMemcpyToSymbolAsync(g_status_bwd, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return -1;
    if (cudaStreamSynchronize(s) != cudaSuccess) return -1;
    return v;
}

}  // namespace rlk

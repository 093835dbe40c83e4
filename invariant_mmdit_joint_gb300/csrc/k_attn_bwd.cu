// Joint attention backward on the tcgen05 tensor cores (the "bwd" half of
// the WS1 attention rows of RFC #386 and of the "WS1 Single-GPU Kernel
// List"): two atomic-free kernels with the forward's warp roles.
//
//   dkdv: one CTA = (key tile of 128, head, sample). Walks every query tile
//         of 128 in one fixed ascending order (text tiles from token 0, then
//         image tiles from token T_txt). Per query tile (P^T is formed while
//         dP^T computes, dS^T while dV computes):
//           S^T  = K Q^T, dP^T = V dO^T            (tcgen05, A and B in smem)
//           P^T  = exp2(S^T * c - lse2), dS^T = P^T * (dP^T - Delta)
//                                                  (4 warps, one key row each;
//                                                   bf16 results into TMEM)
//           dV  += P^T dO,  dK += dS^T Q           (tcgen05, A from TMEM)
//   dq:   one CTA = (query tile of 128, head, sample). Walks the key tiles of
//         128 in the forward's order: S = Q K^T, dP = dO V^T, dS as above,
//         dQ += dS K; the next tile's S and dP are computed while the
//         elementwise warps work on the current one.
// Accumulators (dV, dK, dQ) stay in TMEM in FP32 for the whole CTA and are
// written once. P and dS enter their products as bf16 (round to nearest
// even). lse2 = lse * log2(e) and Delta = rowsum(dO * O) come from the
// backward preprocess in a tile-padded layout (one 128-slot block per query
// tile; slots past a segment hold lse2 = +inf and Delta = 0, so their P is
// exactly 0). Every wait is bounded (RLK_ERR_DEVICE_TIMEOUT on give-up).
#include "rlk_device.cuh"
#include "rlk_internal.h"
#include "rlk_sm100.cuh"

#include <cudaTypedefs.h>

RLK_DEFINE_STRICT_PROBE(probe_bwd_tu)

namespace rlk {
namespace {

using namespace sm100;

// warps 0-7: elementwise (warp w owns TMEM lane quarter w % 4 and the
// column half w / 4 of each row); warp 8: TMA producer; warp 9: MMA issuer
// and TMEM owner.
constexpr int kThreads = 320;
constexpr int kEwThreads = 256;
constexpr int kWarpTma = 8, kWarpMma = 9;
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
    CUtensorMap map_v;    // v  [B, S, H, 128] 4-D
    CUtensorMap map_do;   // dO [B, S, H, 128] 4-D
    Geom g;
    ValidLen vl;
    const float* lse2_p;  // [B, H, nq_pad]
    const float* delta_p; // [B, H, nq_pad]
    uint16_t* dv;         // [B, S, H, 128]
    float* dkh;           // [B, H, S, 128]
    float* dqh;           // [B, H, S, 128]
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
__device__ __forceinline__ uint32_t a_col(int kk) { return (kk < 4) ? kk * 8 : 64 + (kk - 4) * 8; }

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
    __shared__ __align__(8) uint64_t bars[12];
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
    float* dkh = a.dkh + bh * g.S * kHeadDim;

    if (k0 >= kvalid_end) {  // every key of the tile is masked: exact zeros
        const int rows = min(128, seg_end - k0);
        for (int i = tid; i < rows * 16; i += kThreads) {
            const int r = i >> 4, c = i & 15;
            *reinterpret_cast<uint4*>(a.dv + (((size_t)b * g.S + k0 + r) * g.H + h) * kHeadDim + c * 8) =
                make_uint4(0, 0, 0, 0);
            float4* dst = reinterpret_cast<float4*>(dkh + (size_t)(k0 + r) * kHeadDim + c * 8);
            dst[0] = make_float4(0.f, 0.f, 0.f, 0.f);
            dst[1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        return;
    }
    const int nq = g.ntq_txt + g.ntq_img;

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
            mbar_init(bar_empty + 8 * s, 1);
        }
        mbar_init(bar_st, 1);
        mbar_init(bar_dpt, 1);
        mbar_init(bar_p, kEwThreads);
        mbar_init(bar_ds, kEwThreads);
        mbar_init(bar_done, 1);
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
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tensormap(&a.map_q);
            prefetch_tensormap(&a.map_k);
            prefetch_tensormap(&a.map_v);
            prefetch_tensormap(&a.map_do);
            mbar_expect_tx(bar_kv, 2 * kTileBytes);
            tma_load_2d(sK, &a.map_k, bar_kv, 0, row_base + k0);
            tma_load_2d(sK + kBoxBytes, &a.map_k, bar_kv, 64, row_base + k0);
            tma_load_4d(sV, &a.map_v, bar_kv, 0, h, k0, b);
            tma_load_4d(sV + kBoxBytes, &a.map_v, bar_kv, 64, h, k0, b);
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
                tma_load_4d(stage_o(s), &a.map_do, bf, 0, h, q0, b);
                tma_load_4d(stage_o(s) + kBoxBytes, &a.map_do, bf, 64, h, q0, b);
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
    } else if (warp == kWarpMma) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            bool ok = mbar_wait(bar_kv, 0, &abort_flag, kWaitLimitNs);
            for (int i = 0; ok && i < nq; ++i) {
                const int s = i & 1;
                if (!mbar_wait(bar_full + 8 * s, (i >> 1) & 1, &abort_flag, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_ss(tmem + kColST, desc_kmajor(sK, kk), desc_kmajor(stage_q(s), kk), kIdescKK, kk > 0);
                mma_commit(bar_st);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_ss(tmem + kColDPT, desc_kmajor(sV, kk), desc_kmajor(stage_o(s), kk), kIdescKK, kk > 0);
                mma_commit(bar_dpt);
                // dV needs only P (the warps form it while dP^T computes);
                // dK needs dS (formed while dV computes)
                if (!mbar_wait(bar_p, i & 1, &abort_flag, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_ts(tmem + kColDV, tmem + kColST + a_col(kk), desc_mnmajor(stage_o(s), kk), kIdescKM,
                           (i > 0 || kk > 0) ? 1u : 0u);
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
            if (ok)
                mma_commit(bar_done);
            else
                fail(&abort_flag);
            mma_commit(bar_drain);
            const volatile int no_abort = 0;
            mbar_wait(bar_drain, 0, &no_abort, kWaitLimitNs);
        }
    } else {
        // ------------------------------------------------ elementwise warps 0-7
        // warp w: key rows 32 * (w % 4) + lane, query columns [64 h, 64 h + 64), h = w / 4
        const int lq = warp & 3, half = warp >> 2;
        const uint32_t lane_addr = (uint32_t)(lq * 32) << 16;
        const int kr = lq * 32 + lane;
        const int c0 = 64 * half;
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
            uint32_t rs[64];
            tmem_ld32(tmem + lane_addr + kColST + c0, *reinterpret_cast<uint32_t(*)[32]>(&rs[0]));
            tmem_ld32(tmem + lane_addr + kColST + c0 + 32, *reinterpret_cast<uint32_t(*)[32]>(&rs[32]));
            tmem_ld_wait();
            float pf[64];
            uint32_t pk[32];
#pragma unroll
            for (int e4 = 0; e4 < 16; ++e4) {
                const float4 l4 = l2v[e4];
                const float lq4[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float pv = exp2f(fmaf(__uint_as_float(rs[4 * e4 + u]), kC, -lq4[u]));
                    pf[4 * e4 + u] = kvalid ? pv : 0.0f;
                }
                pk[2 * e4] = pack_bf16(pf[4 * e4], pf[4 * e4 + 1]);
                pk[2 * e4 + 1] = pack_bf16(pf[4 * e4 + 2], pf[4 * e4 + 3]);
            }
            tmem_st32(tmem + lane_addr + kColST + c0, pk);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bar_p);
            // dS^T = P^T * (dP^T - Delta[query])
            if (!warp_wait(bar_dpt, i & 1, &abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t rd[64];
            tmem_ld32(tmem + lane_addr + kColDPT + c0, *reinterpret_cast<uint32_t(*)[32]>(&rd[0]));
            tmem_ld32(tmem + lane_addr + kColDPT + c0 + 32, *reinterpret_cast<uint32_t(*)[32]>(&rd[32]));
            tmem_ld_wait();
#pragma unroll
            for (int e4 = 0; e4 < 16; ++e4) {
                const float4 d4 = dlv[e4];
                const float dq4[4] = {d4.x, d4.y, d4.z, d4.w};
                float ds[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) ds[u] = pf[4 * e4 + u] * (__uint_as_float(rd[4 * e4 + u]) - dq4[u]);
                pk[2 * e4] = pack_bf16(ds[0], ds[1]);
                pk[2 * e4 + 1] = pack_bf16(ds[2], ds[3]);
            }
            tmem_st32(tmem + lane_addr + kColDPT + c0, pk);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bar_ds);
        }
        if (ok && warp_wait(bar_done, 0, &abort_flag)) {
            tc_fence_after();
            const int j = k0 + kr;
            const bool row_ok = j < seg_end;
            uint16_t* dvrow = a.dv + (((size_t)b * g.S + j) * g.H + h) * kHeadDim;
            float* dkrow = dkh + (size_t)j * kHeadDim;
#pragma unroll 1
            for (int c = c0; c < c0 + 64; c += 32) {
                uint32_t r[32];
                tmem_ld32(tmem + lane_addr + kColDV + c, r);
                tmem_ld_wait();
                uint32_t w[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    w[e] = kvalid ? pack_bf16(__uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1])) : 0u;
                if (row_ok) {
                    uint4* dst = reinterpret_cast<uint4*>(dvrow + c);
#pragma unroll
                    for (int v4 = 0; v4 < 4; ++v4)
                        dst[v4] = make_uint4(w[4 * v4], w[4 * v4 + 1], w[4 * v4 + 2], w[4 * v4 + 3]);
                }
                tmem_ld32(tmem + lane_addr + kColDK + c, r);
                tmem_ld_wait();
                if (row_ok) {
                    float4* dst = reinterpret_cast<float4*>(dkrow + c);
#pragma unroll
                    for (int v4 = 0; v4 < 8; ++v4) {
                        float4 f;
                        f.x = kvalid ? __uint_as_float(r[4 * v4]) * kScale : 0.0f;
                        f.y = kvalid ? __uint_as_float(r[4 * v4 + 1]) * kScale : 0.0f;
                        f.z = kvalid ? __uint_as_float(r[4 * v4 + 2]) * kScale : 0.0f;
                        f.w = kvalid ? __uint_as_float(r[4 * v4 + 3]) * kScale : 0.0f;
                        dst[v4] = f;
                    }
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

// ====================================================================== dQ
// TMEM: R0, R1 (scores of alternate key tiles), dP, dQ. Per key tile j the
// elementwise warps pull S_j and dP_j into registers and report "consumed";
// the MMA thread then computes S_{j+1} into the other R region and dP_{j+1}
// over dP while the warps form dS_j = P (dP - Delta) and write it (bf16) over
// S_j; then dQ += dS_j K_j. Reduction order over keys: tiles ascending.
// K tiles live in a three-slot ring (each is read by S_j early and by the
// dQ product late); V tiles, read only by dP_j, in a two-slot ring released
// as soon as dP_j is done.
constexpr int kDqSmemQ = 0, kDqSmemO = kTileBytes, kDqSmemK = 2 * kTileBytes;  // K: 3 slots
constexpr int kDqSmemV = 5 * kTileBytes;                                           // V: 2 slots
constexpr int kDqSmemBytes = 7 * kTileBytes + 1024;
constexpr uint32_t kColR0 = 0, kColR1 = 128, kColDP = 256, kColDQ = 384;

__global__ void __launch_bounds__(kThreads, 1) attn_bwd_dq_tc_kernel(const __grid_constant__ BwdArgs a) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bars[19];
    __shared__ uint32_t tmem_slot;
    __shared__ volatile int abort_flag;

    const Geom& g = a.g;
    const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int q0, q_end;
    q_tile(g, qt, q0, q_end);
    const int L = a.vl.L[b];
    const int nkt_txt = (L + 127) / 128;
    const int nkt = nkt_txt + g.ntq_img;
    const size_t bh = (size_t)b * g.H + h;
    const int row_base = (int)(bh * g.S);

    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const uint32_t sQ = sbase + kDqSmemQ, sO = sbase + kDqSmemO;
    auto slot_k = [&](int j) { return sbase + kDqSmemK + (j % 3) * kTileBytes; };
    auto slot_v = [&](int j) { return sbase + kDqSmemV + (j & 1) * kTileBytes; };
    auto col_r = [&](int j) { return (j & 1) ? kColR1 : kColR0; };
    const uint32_t bar_qo = smem_u32(&bars[0]);
    const uint32_t bar_kf = smem_u32(&bars[1]);   // [3] K slot loaded
    const uint32_t bar_ke = smem_u32(&bars[4]);   // [3] K slot free (dQ_j done)
    const uint32_t bar_vf = smem_u32(&bars[7]);   // [2] V slot loaded
    const uint32_t bar_ve = smem_u32(&bars[9]);   // [2] V slot free (dP_j done)
    const uint32_t bar_sq = smem_u32(&bars[17]);  // [2] by tile parity: S_j computed
    const uint32_t bar_dp = smem_u32(&bars[11]);  // dP_j computed
    const uint32_t bar_c = smem_u32(&bars[12]);   // dP_j read into registers
    const uint32_t bar_p = smem_u32(&bars[13]);   // [2] by tile parity: dS_j written
    const uint32_t bar_done = smem_u32(&bars[15]);
    const uint32_t bar_drain = smem_u32(&bars[16]);

    if (tid == 0) {
        abort_flag = 0;
        mbar_init(bar_qo, 1);
        for (int s = 0; s < 3; ++s) {
            mbar_init(bar_kf + 8 * s, 1);
            mbar_init(bar_ke + 8 * s, 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar_vf + 8 * s, 1);
            mbar_init(bar_ve + 8 * s, 1);
            mbar_init(bar_p + 8 * s, kEwThreads);
        }
        mbar_init(bar_sq, 1);
        mbar_init(bar_sq + 8, 1);
        mbar_init(bar_dp, 1);
        mbar_init(bar_c, kEwThreads);
        mbar_init(bar_done, 1);
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
            prefetch_tensormap(&a.map_v);
            prefetch_tensormap(&a.map_do);
            mbar_expect_tx(bar_qo, 2 * kTileBytes);
            tma_load_2d(sQ, &a.map_q, bar_qo, 0, row_base + q0);
            tma_load_2d(sQ + kBoxBytes, &a.map_q, bar_qo, 64, row_base + q0);
            tma_load_4d(sO, &a.map_do, bar_qo, 0, h, q0, b);
            tma_load_4d(sO + kBoxBytes, &a.map_do, bar_qo, 64, h, q0, b);
            int k_issued = 0, v_issued = 0;
            for (int j = 0; j < nkt && !abort_flag; ++j) {
                const int kk0 = j < nkt_txt ? j * 128 : g.T_txt + (j - nkt_txt) * 128;
                const uint32_t kf = bar_kf + 8 * (j % 3), vf = bar_vf + 8 * (j & 1);
                if (j >= 3 && !mbar_wait(bar_ke + 8 * (j % 3), ((j / 3) + 1) & 1, &abort_flag, kWaitLimitNs)) {
                    fail(&abort_flag);
                    break;
                }
                mbar_expect_tx(kf, kTileBytes);
                tma_load_2d(slot_k(j), &a.map_k, kf, 0, row_base + kk0);
                tma_load_2d(slot_k(j) + kBoxBytes, &a.map_k, kf, 64, row_base + kk0);
                k_issued = j + 1;
                if (j >= 2 && !mbar_wait(bar_ve + 8 * (j & 1), ((j >> 1) + 1) & 1, &abort_flag, kWaitLimitNs)) {
                    fail(&abort_flag);
                    break;
                }
                mbar_expect_tx(vf, kTileBytes);
                tma_load_4d(slot_v(j), &a.map_v, vf, 0, h, kk0, b);
                tma_load_4d(slot_v(j) + kBoxBytes, &a.map_v, vf, 64, h, kk0, b);
                v_issued = j + 1;
            }
            const volatile int no_abort = 0;
            mbar_wait(bar_qo, 0, &no_abort, kWaitLimitNs);
            for (int j = k_issued - 3 < 0 ? 0 : k_issued - 3; j < k_issued; ++j)
                mbar_wait(bar_kf + 8 * (j % 3), (j / 3) & 1, &no_abort, kWaitLimitNs);
            for (int j = v_issued - 2 < 0 ? 0 : v_issued - 2; j < v_issued; ++j)
                mbar_wait(bar_vf + 8 * (j & 1), (j >> 1) & 1, &no_abort, kWaitLimitNs);
        }
    } else if (warp == kWarpMma) {
        if (lane == 0) {
            // S_j = Q K_j^T into R(j), dP_j = dO V_j^T into dP
            // S_j = Q K_j^T into R(j) (needs K_j), dP_j = dO V_j^T (needs V_j)
            auto issue_s = [&](int j) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_ss(tmem + col_r(j), desc_kmajor(sQ, kk), desc_kmajor(slot_k(j), kk), kIdescKK, kk > 0);
                mma_commit(bar_sq + 8 * (j & 1));
            };
            auto issue_dp = [&](int j) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_ss(tmem + kColDP, desc_kmajor(sO, kk), desc_kmajor(slot_v(j), kk), kIdescKK, kk > 0);
                mma_commit(bar_dp);
                mma_commit(bar_ve + 8 * (j & 1));
            };
            auto wait_kv = [&](int j) {
                return mbar_wait(bar_kf + 8 * (j % 3), (j / 3) & 1, &abort_flag, kWaitLimitNs) &&
                       mbar_wait(bar_vf + 8 * (j & 1), (j >> 1) & 1, &abort_flag, kWaitLimitNs);
            };
            bool ok = mbar_wait(bar_qo, 0, &abort_flag, kWaitLimitNs) && wait_kv(0);
            if (ok) {
                tc_fence_after();
                issue_s(0);
                issue_dp(0);
            }
            for (int j = 0; ok && j < nkt; ++j) {
                const int s = j & 1;
                if (j + 1 < nkt) {
                    // S_{j+1} goes to the other R region; dP_{j+1} waits until
                    // the warps hold dP_j in registers
                    if (!wait_kv(j + 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issue_s(j + 1);
                    if (!mbar_wait(bar_c, j & 1, &abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issue_dp(j + 1);
                }
                if (!mbar_wait(bar_p + 8 * s, (j >> 1) & 1, &abort_flag, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_ts(tmem + kColDQ, tmem + col_r(j) + a_col(kk), desc_mnmajor(slot_k(j), kk), kIdescKM,
                           (j > 0 || kk > 0) ? 1u : 0u);
                mma_commit(bar_ke + 8 * (j % 3));
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
        // ------------------------------------------------ elementwise warps 0-7
        // warp w: query rows 32 * (w % 4) + lane, key columns [64 hf, 64 hf + 64), hf = w / 4
        const int lq = warp & 3, hf = warp >> 2;
        const uint32_t lane_addr = (uint32_t)(lq * 32) << 16;
        const int r = lq * 32 + lane;
        const int c0 = 64 * hf;
        const size_t slot = bh * g.nq_pad + (size_t)qt * 128 + r;
        const float l2 = a.lse2_p[slot];
        const float dl = a.delta_p[slot];
        bool ok = true;
        for (int j = 0; j < nkt; ++j) {
            if (!warp_wait(bar_sq + 8 * (j & 1), (j >> 1) & 1, &abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t s_cols = tmem + lane_addr + col_r(j) + c0;
            const int kk0 = j < nkt_txt ? j * 128 : g.T_txt + (j - nkt_txt) * 128;
            const int nvalid = (j < nkt_txt ? L : g.S) - kk0 - c0;  // valid columns of this half
            // P = exp2(S * c - lse2) (masked keys: 0) while dP_j computes
            uint32_t rs[64];
            tmem_ld32(s_cols, *reinterpret_cast<uint32_t(*)[32]>(&rs[0]));
            tmem_ld32(s_cols + 32, *reinterpret_cast<uint32_t(*)[32]>(&rs[32]));
            tmem_ld_wait();
            float pf[64];
#pragma unroll
            for (int i = 0; i < 64; ++i) pf[i] = exp2f(fmaf(__uint_as_float(rs[i]), kC, -l2));
            if (nvalid < 64) {
#pragma unroll
                for (int i = 0; i < 64; ++i) pf[i] = i < nvalid ? pf[i] : 0.0f;
            }
            if (!warp_wait(bar_dp, j & 1, &abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t rd[64];
            tmem_ld32(tmem + lane_addr + kColDP + c0, *reinterpret_cast<uint32_t(*)[32]>(&rd[0]));
            tmem_ld32(tmem + lane_addr + kColDP + c0 + 32, *reinterpret_cast<uint32_t(*)[32]>(&rd[32]));
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive(bar_c);  // dP_j is in registers: the MMA may overwrite dP
            uint32_t pd[32];
#pragma unroll
            for (int i = 0; i < 32; ++i)
                pd[i] = pack_bf16(pf[2 * i] * (__uint_as_float(rd[2 * i]) - dl),
                                  pf[2 * i + 1] * (__uint_as_float(rd[2 * i + 1]) - dl));
            tmem_st32(s_cols, pd);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bar_p + 8 * (j & 1));
        }
        if (ok && warp_wait(bar_done, 0, &abort_flag)) {
            tc_fence_after();
            const bool row_ok = q0 + r < q_end;
            float* dqrow = a.dqh + (bh * g.S + q0 + r) * kHeadDim;
#pragma unroll 1
            for (int c = c0; c < c0 + 64; c += 32) {
                uint32_t rr[32];
                tmem_ld32(tmem + lane_addr + kColDQ + c, rr);
                tmem_ld_wait();
                if (row_ok) {
                    float4* dst = reinterpret_cast<float4*>(dqrow + c);
#pragma unroll
                    for (int v4 = 0; v4 < 8; ++v4)
                        dst[v4] = make_float4(__uint_as_float(rr[4 * v4]) * kScale, __uint_as_float(rr[4 * v4 + 1]) * kScale,
                                              __uint_as_float(rr[4 * v4 + 2]) * kScale,
                                              __uint_as_float(rr[4 * v4 + 3]) * kScale);
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

// ---------------------------------------------------------------- tensor maps
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (fn == nullptr) {
        cudaDriverEntryPointQueryResult q;
        void* p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

bool encode_rows(CUtensorMap* m, const void* base, uint64_t rows) {
    auto enc = get_encode();
    if (enc == nullptr) return false;
    cuuint64_t dims[2] = {128, rows};
    cuuint64_t strides[1] = {256};
    cuuint32_t box[2] = {64, 128};
    cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_bshd(CUtensorMap* m, const void* base, const Geom& g) {
    auto enc = get_encode();
    if (enc == nullptr) return false;
    cuuint64_t dims[4] = {128, (cuuint64_t)g.H, (cuuint64_t)g.S, (cuuint64_t)g.B};
    cuuint64_t strides[3] = {256, (cuuint64_t)g.H * 256, (cuuint64_t)g.S * g.H * 256};
    cuuint32_t box[4] = {64, 1, 128, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_args(BwdArgs* a, const Geom& g, const ValidLen& vl, const uint16_t* qh, const uint16_t* kh,
               const uint16_t* v, const uint16_t* dout, const float* lse2_p, const float* delta_p) {
    const uint64_t rows = (uint64_t)g.B * g.H * g.S;
    if (!encode_rows(&a->map_q, qh, rows) || !encode_rows(&a->map_k, kh, rows) || !encode_bshd(&a->map_v, v, g) ||
        !encode_bshd(&a->map_do, dout, g))
        return false;
    a->g = g;
    a->vl = vl;
    a->lse2_p = lse2_p;
    a->delta_p = delta_p;
    a->dv = nullptr;
    a->dkh = nullptr;
    a->dqh = nullptr;
    return true;
}

}  // namespace

cudaError_t launch_attn_bwd_dkdv(const Geom& g, const ValidLen& vl, const uint16_t* qh, const uint16_t* kh,
                                 const uint16_t* v, const uint16_t* dout, const float* lse2_p, const float* delta_p,
                                 uint16_t* dv, float* dkh, cudaStream_t s) {
    BwdArgs args;
    if (!make_args(&args, g, vl, qh, kh, v, dout, lse2_p, delta_p)) return cudaErrorInvalidValue;
    args.dv = dv;
    args.dkh = dkh;
    cudaError_t e =
        cudaFuncSetAttribute(attn_bwd_dkdv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kKvSmemBytes);
    if (e != cudaSuccess) return e;
    dim3 grid(g.ntq_txt + g.ntq_img, g.H, g.B);
    timing_begin(kKBwdDkDv, s);
    attn_bwd_dkdv_tc_kernel<<<grid, kThreads, kKvSmemBytes, s>>>(args);
    timing_end(kKBwdDkDv, s);
    return cudaGetLastError();
}

cudaError_t launch_attn_bwd_dq(const Geom& g, const ValidLen& vl, const uint16_t* qh, const uint16_t* kh,
                               const uint16_t* v, const uint16_t* dout, const float* lse2_p, const float* delta_p,
                               float* dqh, cudaStream_t s) {
    BwdArgs args;
    if (!make_args(&args, g, vl, qh, kh, v, dout, lse2_p, delta_p)) return cudaErrorInvalidValue;
    args.dqh = dqh;
    cudaError_t e =
        cudaFuncSetAttribute(attn_bwd_dq_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDqSmemBytes);
    if (e != cudaSuccess) return e;
    dim3 grid(g.ntq_txt + g.ntq_img, g.H, g.B);
    timing_begin(kKBwdDq, s);
    attn_bwd_dq_tc_kernel<<<grid, kThreads, kDqSmemBytes, s>>>(args);
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

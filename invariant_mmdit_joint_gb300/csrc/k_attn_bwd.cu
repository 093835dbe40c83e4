// Joint attention backward (the "bwd" half of the WS1 attention rows of
// RFC #386 and of the "WS1 Single-GPU Kernel List"): two atomic-free kernels.
//
//   dkdv: one CTA = (key tile of 128, head, sample). Walks every query tile of
//         64 in one fixed ascending order (text tiles from token 0, then image
//         tiles from token T_txt), recomputing P^T = exp(S^T - lse) and
//         accumulating dV += P^T dO and dK += dS^T Q in FP32, with
//         dS^T = P^T * (V dO^T - Delta).
//   dq:   one CTA = (query tile of 128, head, sample). Walks the key tiles of
//         64 in the forward's order, recomputing P and dP = dO V^T, and
//         accumulates dQ += dS K in FP32. No atomics, no split.
//
// Every output element is produced by one CTA with a fixed reduction order,
// so the bytes are independent of B, batch position and the SM count. P and
// dS enter their products as bf16 (round to nearest even).
#include "rlk_device.cuh"
#include "rlk_internal.h"

RLK_DEFINE_STRICT_PROBE(probe_bwd_tu)

namespace rlk {
namespace {

constexpr int kThreads = 256;
constexpr float kC = (float)(1.4426950408889634 * 0.08838834764831845);
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kScale = 0.08838834764831845f;  // 1 / sqrt(128)

__device__ int g_status_bwd;

struct BwdArgs {
    Geom g;
    ValidLen vl;
    const uint16_t* qh;    // [B, H, S, D]
    const uint16_t* kh;    // [B, H, S, D]
    const uint16_t* v;     // [B, S, H, D]
    const uint16_t* dout;  // [B, S, H, D]
    const float* lse;      // [B, H, S]
    const float* delta;    // [B, H, S]
    uint16_t* dv;          // [B, S, H, D]
    float* dkh;            // [B, H, S, D]
    float* dqh;            // [B, H, S, D]
};

__device__ __forceinline__ size_t bshd(const Geom& g, int b, int n, int h) {
    return (((size_t)b * g.S + n) * g.H + h) * kHeadDim;
}

// ---------------------------------------------------------------- dK, dV
constexpr int kKvBK = 128;  // keys per CTA (8 warps x 16)
constexpr int kKvBQ = 64;   // queries per step
constexpr int kKvSmem = 2 * kKvBK * 256 + 4 * kKvBQ * 256 + 4 * kKvBQ * 4;

__global__ void __launch_bounds__(kThreads, 1) attn_bwd_dkdv_kernel(const __grid_constant__ BwdArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const Geom& g = a.g;
    const int kt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gr = lane >> 2, gc = lane & 3;
    const int nkt_txt = (g.T_txt + kKvBK - 1) / kKvBK;
    const bool k_txt = kt < nkt_txt;
    const int k0 = k_txt ? kt * kKvBK : g.T_txt + (kt - nkt_txt) * kKvBK;
    const int seg_end = k_txt ? g.T_txt : g.S;
    const int L = a.vl.L[b];
    const int kvalid_end = k_txt ? L : g.S;
    const size_t bh = (size_t)b * g.H + h;
    const uint16_t* qh = a.qh + bh * g.S * kHeadDim;
    const uint16_t* kh = a.kh + bh * g.S * kHeadDim;
    float* dkh = a.dkh + bh * g.S * kHeadDim;

    if (k0 >= kvalid_end) {  // every key of the tile is masked: exact zeros
        const int rows = min(kKvBK, seg_end - k0);
        for (int i = tid; i < rows * 16; i += kThreads) {
            const int r = i >> 4, c = i & 15;
            *reinterpret_cast<uint4*>(a.dv + bshd(g, b, k0 + r, h) + c * 8) = make_uint4(0, 0, 0, 0);
            float4* dst = reinterpret_cast<float4*>(dkh + (size_t)(k0 + r) * kHeadDim + c * 8);
            dst[0] = make_float4(0.f, 0.f, 0.f, 0.f);
            dst[1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        return;
    }

    const uint32_t sK = smem_u32(smem);
    const uint32_t sV = sK + kKvBK * 256;
    const uint32_t sQ = sV + kKvBK * 256;          // 2 buffers
    const uint32_t sO = sQ + 2 * kKvBQ * 256;      // dO, 2 buffers
    float* sStat = reinterpret_cast<float*>(smem + 2 * kKvBK * 256 + 4 * kKvBQ * 256);  // [2][lse2 | delta][64]

    for (int i = tid; i < kKvBK * 16; i += kThreads) {
        const int r = i >> 4, c = i & 15, n = k0 + r;
        const bool ok = n < kvalid_end;
        const int nn = ok ? n : 0;
        cp_async16(tile_addr(sK, r, c), kh + (size_t)nn * kHeadDim + c * 8, ok);
        cp_async16(tile_addr(sV, r, c), a.v + bshd(g, b, nn, h) + c * 8, ok);
    }
    const int nqt_txt = (g.T_txt + kKvBQ - 1) / kKvBQ;
    const int nqt = nqt_txt + (g.T_img + kKvBQ - 1) / kKvBQ;
    auto load_q = [&](int t, int buf) {
        const bool txt = t < nqt_txt;
        const int q0 = txt ? t * kKvBQ : g.T_txt + (t - nqt_txt) * kKvBQ;
        const int qend = txt ? g.T_txt : g.S;
        for (int i = tid; i < kKvBQ * 16; i += kThreads) {
            const int r = i >> 4, c = i & 15, n = q0 + r;
            const bool ok = n < qend;
            const int nn = ok ? n : 0;
            cp_async16(tile_addr(sQ + buf * kKvBQ * 256, r, c), qh + (size_t)nn * kHeadDim + c * 8, ok);
            cp_async16(tile_addr(sO + buf * kKvBQ * 256, r, c), a.dout + bshd(g, b, nn, h) + c * 8, ok);
        }
        if (tid < kKvBQ) {
            const int n = q0 + tid;
            const bool ok = n < qend;
            // rows outside the segment get lse = +inf, so their P is exactly 0
            sStat[buf * 2 * kKvBQ + tid] = ok ? a.lse[bh * g.S + n] * kLog2e : INFINITY;
            sStat[buf * 2 * kKvBQ + kKvBQ + tid] = ok ? a.delta[bh * g.S + n] : 0.0f;
        }
    };
    load_q(0, 0);
    cp_async_commit();

    float dv[16][4], dk[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        dv[i][0] = dv[i][1] = dv[i][2] = dv[i][3] = 0.0f;
        dk[i][0] = dk[i][1] = dk[i][2] = dk[i][3] = 0.0f;
    }
    const bool kv0 = k0 + 16 * warp + gr < kvalid_end;
    const bool kv1 = k0 + 16 * warp + gr + 8 < kvalid_end;

    for (int t = 0; t < nqt; ++t) {
        if (t + 1 < nqt) load_q(t + 1, (t + 1) & 1);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        const uint32_t qb = sQ + (t & 1) * kKvBQ * 256;
        const uint32_t ob = sO + (t & 1) * kKvBQ * 256;
        const float* lse2 = sStat + (t & 1) * 2 * kKvBQ;
        const float* dlt = lse2 + kKvBQ;

        // S^T = K Q^T: 16 keys x 64 queries
        float p[8][4];
#pragma unroll
        for (int i = 0; i < 8; ++i) p[i][0] = p[i][1] = p[i][2] = p[i][3] = 0.0f;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            uint32_t ka[4];
            ldsm_x4(tile_addr(sK, 16 * warp + (lane & 15), 2 * ks + (lane >> 4)), ka[0], ka[1], ka[2], ka[3]);
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t r0, r1, r2, r3;
                ldsm_x4(tile_addr(qb, 16 * np + (lane & 7) + ((lane >> 4) << 3), 2 * ks + ((lane >> 3) & 1)), r0,
                        r1, r2, r3);
                mma_bf16(p[2 * np], ka, r0, r1);
                mma_bf16(p[2 * np + 1], ka, r2, r3);
            }
        }
        // P^T = exp2(S^T * kC - lse2[query]); masked keys -> 0
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const float l2 = lse2[8 * nt + 2 * gc + e];
                p[nt][e] = kv0 ? exp2f(p[nt][e] * kC - l2) : 0.0f;
                p[nt][2 + e] = kv1 ? exp2f(p[nt][2 + e] * kC - l2) : 0.0f;
            }
        }
        // dV += P^T dO
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const uint32_t pa[4] = {pack_bf16(p[2 * kk][0], p[2 * kk][1]), pack_bf16(p[2 * kk][2], p[2 * kk][3]),
                                    pack_bf16(p[2 * kk + 1][0], p[2 * kk + 1][1]),
                                    pack_bf16(p[2 * kk + 1][2], p[2 * kk + 1][3])};
#pragma unroll
            for (int dp = 0; dp < 8; ++dp) {
                uint32_t r0, r1, r2, r3;
                ldsm_x4_t(tile_addr(ob, 16 * kk + (lane & 7) + (((lane >> 3) & 1) << 3), 2 * dp + (lane >> 4)), r0,
                          r1, r2, r3);
                mma_bf16(dv[2 * dp], pa, r0, r1);
                mma_bf16(dv[2 * dp + 1], pa, r2, r3);
            }
        }
        // dP^T = V dO^T
        float ds[8][4];
#pragma unroll
        for (int i = 0; i < 8; ++i) ds[i][0] = ds[i][1] = ds[i][2] = ds[i][3] = 0.0f;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            uint32_t va[4];
            ldsm_x4(tile_addr(sV, 16 * warp + (lane & 15), 2 * ks + (lane >> 4)), va[0], va[1], va[2], va[3]);
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t r0, r1, r2, r3;
                ldsm_x4(tile_addr(ob, 16 * np + (lane & 7) + ((lane >> 4) << 3), 2 * ks + ((lane >> 3) & 1)), r0,
                        r1, r2, r3);
                mma_bf16(ds[2 * np], va, r0, r1);
                mma_bf16(ds[2 * np + 1], va, r2, r3);
            }
        }
        // dS^T = P^T * (dP^T - Delta[query])
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const float d = dlt[8 * nt + 2 * gc + e];
                ds[nt][e] = p[nt][e] * (ds[nt][e] - d);
                ds[nt][2 + e] = p[nt][2 + e] * (ds[nt][2 + e] - d);
            }
        }
        // dK += dS^T Q
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const uint32_t sa[4] = {pack_bf16(ds[2 * kk][0], ds[2 * kk][1]), pack_bf16(ds[2 * kk][2], ds[2 * kk][3]),
                                    pack_bf16(ds[2 * kk + 1][0], ds[2 * kk + 1][1]),
                                    pack_bf16(ds[2 * kk + 1][2], ds[2 * kk + 1][3])};
#pragma unroll
            for (int dp = 0; dp < 8; ++dp) {
                uint32_t r0, r1, r2, r3;
                ldsm_x4_t(tile_addr(qb, 16 * kk + (lane & 7) + (((lane >> 3) & 1) << 3), 2 * dp + (lane >> 4)), r0,
                          r1, r2, r3);
                mma_bf16(dk[2 * dp], sa, r0, r1);
                mma_bf16(dk[2 * dp + 1], sa, r2, r3);
            }
        }
        __syncthreads();
    }

    // epilogue: dV -> bf16 [B,S,H,D] (staged through the Q buffers); dkh -> fp32
    const int r_lo = 16 * warp + gr, r_hi = r_lo + 8;
    const uint32_t stage = sQ;  // 2 x 64 rows = 128 rows of 256 bytes
#pragma unroll
    for (int dt = 0; dt < 16; ++dt) {
        const uint32_t lo = kv0 ? pack_bf16(dv[dt][0], dv[dt][1]) : 0u;
        const uint32_t hi = kv1 ? pack_bf16(dv[dt][2], dv[dt][3]) : 0u;
        asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(tile_addr(stage, r_lo, dt) + 4 * gc), "r"(lo));
        asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(tile_addr(stage, r_hi, dt) + 4 * gc), "r"(hi));
        if (k0 + r_lo < seg_end) {
            const float2 v = kv0 ? make_float2(dk[dt][0] * kScale, dk[dt][1] * kScale) : make_float2(0.f, 0.f);
            *reinterpret_cast<float2*>(dkh + (size_t)(k0 + r_lo) * kHeadDim + 8 * dt + 2 * gc) = v;
        }
        if (k0 + r_hi < seg_end) {
            const float2 v = kv1 ? make_float2(dk[dt][2] * kScale, dk[dt][3] * kScale) : make_float2(0.f, 0.f);
            *reinterpret_cast<float2*>(dkh + (size_t)(k0 + r_hi) * kHeadDim + 8 * dt + 2 * gc) = v;
        }
    }
    __syncwarp();
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int i = lane + 32 * it;
        const int r = 16 * warp + (i >> 4), c = i & 15;
        const int n = k0 + r;
        if (n < seg_end) {
            uint4 v;
            asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];\n"
                         : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                         : "r"(tile_addr(stage, r, c)));
            *reinterpret_cast<uint4*>(a.dv + bshd(g, b, n, h) + c * 8) = v;
        }
    }
}

// ---------------------------------------------------------------- dQ
constexpr int kDqBQ = 128;  // query rows per CTA (8 warps x 16)
constexpr int kDqBN = 64;   // keys per step
constexpr int kDqSmem = 2 * kDqBQ * 256 + 4 * kDqBN * 256;

__global__ void __launch_bounds__(kThreads, 1) attn_bwd_dq_kernel(const __grid_constant__ BwdArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const Geom& g = a.g;
    const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gr = lane >> 2, gc = lane & 3;
    const int nqt_txt = (g.T_txt + kDqBQ - 1) / kDqBQ;
    const bool q_txt = qt < nqt_txt;
    const int q0 = q_txt ? qt * kDqBQ : g.T_txt + (qt - nqt_txt) * kDqBQ;
    const int q_end = q_txt ? g.T_txt : g.S;
    const int L = a.vl.L[b];
    const int nkt_txt = (L + kDqBN - 1) / kDqBN;
    const int nkt = nkt_txt + (g.T_img + kDqBN - 1) / kDqBN;
    const size_t bh = (size_t)b * g.H + h;
    const uint16_t* qh = a.qh + bh * g.S * kHeadDim;
    const uint16_t* kh = a.kh + bh * g.S * kHeadDim;

    const uint32_t sQ = smem_u32(smem);
    const uint32_t sO = sQ + kDqBQ * 256;
    const uint32_t sK = sO + kDqBQ * 256;          // 2 buffers
    const uint32_t sV = sK + 2 * kDqBN * 256;      // 2 buffers

    for (int i = tid; i < kDqBQ * 16; i += kThreads) {
        const int r = i >> 4, c = i & 15, n = q0 + r;
        const bool ok = n < q_end;
        const int nn = ok ? n : 0;
        cp_async16(tile_addr(sQ, r, c), qh + (size_t)nn * kHeadDim + c * 8, ok);
        cp_async16(tile_addr(sO, r, c), a.dout + bshd(g, b, nn, h) + c * 8, ok);
    }
    auto load_kv = [&](int t, int buf) {
        const bool txt = t < nkt_txt;
        const int k0 = txt ? t * kDqBN : g.T_txt + (t - nkt_txt) * kDqBN;
        const int kend = txt ? L : g.S;
        for (int i = tid; i < kDqBN * 16; i += kThreads) {
            const int r = i >> 4, c = i & 15, n = k0 + r;
            const bool ok = n < kend;
            const int nn = ok ? n : 0;
            cp_async16(tile_addr(sK + buf * kDqBN * 256, r, c), kh + (size_t)nn * kHeadDim + c * 8, ok);
            cp_async16(tile_addr(sV + buf * kDqBN * 256, r, c), a.v + bshd(g, b, nn, h) + c * 8, ok);
        }
    };
    load_kv(0, 0);
    cp_async_commit();

    const int r_lo = 16 * warp + gr, r_hi = r_lo + 8;
    const bool ok_lo = q0 + r_lo < q_end, ok_hi = q0 + r_hi < q_end;
    const float l2_lo = ok_lo ? a.lse[bh * g.S + q0 + r_lo] * kLog2e : 0.0f;
    const float l2_hi = ok_hi ? a.lse[bh * g.S + q0 + r_hi] * kLog2e : 0.0f;
    const float d_lo = ok_lo ? a.delta[bh * g.S + q0 + r_lo] : 0.0f;
    const float d_hi = ok_hi ? a.delta[bh * g.S + q0 + r_hi] : 0.0f;

    float dq[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) dq[i][0] = dq[i][1] = dq[i][2] = dq[i][3] = 0.0f;

    for (int t = 0; t < nkt; ++t) {
        if (t + 1 < nkt) load_kv(t + 1, (t + 1) & 1);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        const uint32_t kb = sK + (t & 1) * kDqBN * 256;
        const uint32_t vb = sV + (t & 1) * kDqBN * 256;
        const bool txt = t < nkt_txt;
        const int k0 = txt ? t * kDqBN : g.T_txt + (t - nkt_txt) * kDqBN;
        const int kend = txt ? L : g.S;

        // S = Q K^T and dP = dO V^T, 16 rows x 64 keys each
        float p[8][4], dp[8][4];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            p[i][0] = p[i][1] = p[i][2] = p[i][3] = 0.0f;
            dp[i][0] = dp[i][1] = dp[i][2] = dp[i][3] = 0.0f;
        }
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            uint32_t qa[4], oa[4];
            ldsm_x4(tile_addr(sQ, 16 * warp + (lane & 15), 2 * ks + (lane >> 4)), qa[0], qa[1], qa[2], qa[3]);
            ldsm_x4(tile_addr(sO, 16 * warp + (lane & 15), 2 * ks + (lane >> 4)), oa[0], oa[1], oa[2], oa[3]);
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t r0, r1, r2, r3;
                const int row = 16 * np + (lane & 7) + ((lane >> 4) << 3), ch = 2 * ks + ((lane >> 3) & 1);
                ldsm_x4(tile_addr(kb, row, ch), r0, r1, r2, r3);
                mma_bf16(p[2 * np], qa, r0, r1);
                mma_bf16(p[2 * np + 1], qa, r2, r3);
                ldsm_x4(tile_addr(vb, row, ch), r0, r1, r2, r3);
                mma_bf16(dp[2 * np], oa, r0, r1);
                mma_bf16(dp[2 * np + 1], oa, r2, r3);
            }
        }
        // dS = P * (dP - Delta); masked keys -> 0
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const bool ok = k0 + 8 * nt + 2 * gc + e < kend;
                const float p_lo = ok ? exp2f(p[nt][e] * kC - l2_lo) : 0.0f;
                const float p_hi = ok ? exp2f(p[nt][2 + e] * kC - l2_hi) : 0.0f;
                p[nt][e] = p_lo * (dp[nt][e] - d_lo);
                p[nt][2 + e] = p_hi * (dp[nt][2 + e] - d_hi);
            }
        }
        // dQ += dS K
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const uint32_t sa[4] = {pack_bf16(p[2 * kk][0], p[2 * kk][1]), pack_bf16(p[2 * kk][2], p[2 * kk][3]),
                                    pack_bf16(p[2 * kk + 1][0], p[2 * kk + 1][1]),
                                    pack_bf16(p[2 * kk + 1][2], p[2 * kk + 1][3])};
#pragma unroll
            for (int dd = 0; dd < 8; ++dd) {
                uint32_t r0, r1, r2, r3;
                ldsm_x4_t(tile_addr(kb, 16 * kk + (lane & 7) + (((lane >> 3) & 1) << 3), 2 * dd + (lane >> 4)), r0,
                          r1, r2, r3);
                mma_bf16(dq[2 * dd], sa, r0, r1);
                mma_bf16(dq[2 * dd + 1], sa, r2, r3);
            }
        }
        __syncthreads();
    }

    float* dqh = a.dqh + bh * g.S * kHeadDim;
#pragma unroll
    for (int dt = 0; dt < 16; ++dt) {
        if (ok_lo)
            *reinterpret_cast<float2*>(dqh + (size_t)(q0 + r_lo) * kHeadDim + 8 * dt + 2 * gc) =
                make_float2(dq[dt][0] * kScale, dq[dt][1] * kScale);
        if (ok_hi)
            *reinterpret_cast<float2*>(dqh + (size_t)(q0 + r_hi) * kHeadDim + 8 * dt + 2 * gc) =
                make_float2(dq[dt][2] * kScale, dq[dt][3] * kScale);
    }
}

}  // namespace

cudaError_t launch_attn_bwd_dkdv(const Geom& g, const ValidLen& vl, const uint16_t* qh, const uint16_t* kh,
                                 const uint16_t* v, const uint16_t* dout, const float* lse, const float* delta,
                                 uint16_t* dv, float* dkh, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_dkdv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kKvSmem);
    if (e != cudaSuccess) return e;
    BwdArgs args{g, vl, qh, kh, v, dout, lse, delta, dv, dkh, nullptr};
    const int nkt = (g.T_txt + kKvBK - 1) / kKvBK + (g.T_img + kKvBK - 1) / kKvBK;
    dim3 grid(nkt, g.H, g.B);
    timing_begin(kKBwdDkDv, s);
    attn_bwd_dkdv_kernel<<<grid, kThreads, kKvSmem, s>>>(args);
    timing_end(kKBwdDkDv, s);
    return cudaGetLastError();
}

cudaError_t launch_attn_bwd_dq(const Geom& g, const ValidLen& vl, const uint16_t* qh, const uint16_t* kh,
                               const uint16_t* v, const uint16_t* dout, const float* lse, const float* delta,
                               float* dqh, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDqSmem);
    if (e != cudaSuccess) return e;
    BwdArgs args{g, vl, qh, kh, v, dout, lse, delta, nullptr, nullptr, dqh};
    const int nqt = (g.T_txt + kDqBQ - 1) / kDqBQ + (g.T_img + kDqBQ - 1) / kDqBQ;
    dim3 grid(nqt, g.H, g.B);
    timing_begin(kKBwdDq, s);
    attn_bwd_dq_kernel<<<grid, kThreads, kDqSmem, s>>>(args);
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

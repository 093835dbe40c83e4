// Row qkv_bias_gemm of the RFC #386 WS1 table (each stream's Q, K and V
// projections in one GEMM with a bias; the WS1 Single-GPU Kernel List:
// 3072 -> 3 x 3072, one weight set per stream) on the tcgen05 tensor cores, with rows qk_rmsnorm and
// multi_axis_rope fused into its epilogue, so the normed, rotated q^ and k^
// go straight into the attention's context (the "adjacent producer" of the
// fused attention).
//
//   Y_s = X_s W_s^T + b_s      X_s bf16 [B * T_s, C], W_s bf16 [3C, C] (the
//                              Q rows, then K, then V), b_s bf16 [3C],
//                              C = H * 128, s = text or image stream
//   Q, K, V = bf16(Y)          one rounding: the declared storage of the
//                              projections (as the unfused operator stores them)
//   fused:  q^, k^ = bf16(RoPE(RMSNorm_g(Q, K)))   with the prologue kernel's
//           arithmetic step for step (so the bytes equal prologue(Q, K)); V
//           (and, if asked, Q and K for the backward) stored as bf16
//   plain:  Q, K, V stored as bf16 [B, T_s, H, 128]
//
// Persistent CTAs (grid <= SM count) take the tiles (stream, 128 rows, 256
// columns = two heads) t = blockIdx.x, blockIdx.x + gridDim.x, ... in one
// fixed order; each output tile is one CTA's FP32 TMEM accumulator summed
// over K in ascending 64-wide steps (no split-K, no atomics). Warps: 0 TMA
// producer (4 stages of a 128 x 64 A box and a 256 x 64 B box), 1 MMA issuer
// and TMEM owner (two 256-column accumulators, so a tile's epilogue overlaps
// the next tile's products), 2-5 epilogue (one output row per thread). Every
// wait is bounded (RLK_ERR_DEVICE_TIMEOUT).
#include "rlk_device.cuh"
#include "rlk_internal.h"
#include "rlk_sm100.cuh"
#include "rlk_tmap.h"

RLK_DEFINE_STRICT_PROBE(probe_qkv_tu)

namespace rlk {
namespace {

using namespace sm100;

constexpr int kBM = 128, kBN = 256, kBK = 64;
constexpr int kStages = 4;
constexpr int kABytes = kBM * kBK * 2;          // 16 KB
constexpr int kBBytes = kBN * kBK * 2;          // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;  // 48 KB
constexpr int kSmemBytes = kStages * kStageBytes + 1024;
constexpr int kThreads = 192;
constexpr int kWarpTma = 0, kWarpMma = 1;
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint32_t kIdesc = idesc_bf16(kBM, kBN, false, false);

__device__ int g_status_qkv;

__device__ __forceinline__ void fail(volatile int* abort_flag) {
    *abort_flag = 1;
    atomicOr(&g_status_qkv, 1);
}

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, kWaitLimitNs));
}

struct QkvArgs {
    CUtensorMap map_x[2];   // X_s as [B * T_s, C] bf16, box 64 x 128
    CUtensorMap map_w[2];   // W_s as [3C, C] bf16, box 64 x 256
    const uint16_t* bias[2];
    const float* gain[2][2];  // [stream][0 q, 1 k]
    Geom g;
    int C;                  // H * 128 (the input features)
    int ncols;              // output features: 3C (QKV) or C (output projection)
    bool out_proj;          // every column is one plain output, stored to v
    int m_tiles[2];         // ceil(B * T_s / 128)
    int n_tiles;            // ceil(ncols / 256)
    // fused mode (qh != null): q^, k^ [B*H*S, 128] and r [B*H*S] into the
    // context, the cos/sin table read from it; q, k optional pre-norm copies
    uint16_t* qh;
    uint16_t* kh;
    float* rq;
    float* rk;
    const float2* tab;
    SegBf16 q, k, v;        // [B, T_s, H, 128] per stream; q, k may be null in fused mode
    bool store_q, store_k;
};

struct Tile {
    int s, m0, n0;  // stream, first row of X_s, first column of Y_s
};
__device__ __forceinline__ Tile tile_of(const QkvArgs& a, int t) {
    Tile r;
    const int per0 = a.m_tiles[0] * a.n_tiles;
    r.s = t < per0 ? 0 : 1;
    const int tl = r.s == 0 ? t : t - per0;
    r.m0 = (tl / a.n_tiles) * kBM;  // consecutive tiles share their rows of X (L2 reuse)
    r.n0 = (tl % a.n_tiles) * kBN;
    return r;
}

// qk_rmsnorm + multi_axis_rope of one head row held by one thread (x: the
// row's 128 values, already bf16-rounded), with the prologue kernel's
// arithmetic: the prologue spreads the row over 16 lanes of 8 dims, each
// lane summing its 8 squares in order, then adds across lanes with a
// butterfly (xor 8, 4, 2, 1); addition is commutative, so every lane ends
// with ((a0 + a4) + (a2 + a6)) + ((a1 + a5) + (a3 + a7)), a_i = s_i + s_{i+8},
// which is the tree below. r = 1 / sqrt(ss / 128 + eps) (IEEE), y = (x r) g,
// pairs turned by the table's (cos, sin) of their axis.
__device__ __forceinline__ void norm_rope_full_row(const float (&x)[128], const float* __restrict__ gain,
                                                   const float2* __restrict__ tab, const Geom& g, int n,
                                                   uint16_t* __restrict__ dst, float& r_out) {
    float s[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        float v = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) v = fmaf(x[8 * j + i], x[8 * j + i], v);
        s[j] = v;
    }
    float a[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = s[i] + s[i + 8];
    const float b0 = a[0] + a[4], b1 = a[1] + a[5], b2 = a[2] + a[6], b3 = a[3] + a[7];
    const float ss = (b0 + b2) + (b1 + b3);
    const float r = 1.0f / sqrtf(fmaf(ss, 1.0f / 128.0f, g.eps));
    r_out = r;
    const float2* trow[3];
#pragma unroll
    for (int ax = 0; ax < 3; ++ax) trow[ax] = tab + (size_t)(token_pos(g, n, ax) - g.p_lo) * kPairs;
    uint4* out = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int c = 0; c < 16; ++c) {  // 8 dims = 4 pairs per 16-byte store
        const float4 g0 = __ldg(reinterpret_cast<const float4*>(gain) + 2 * c);
        const float4 g1 = __ldg(reinterpret_cast<const float4*>(gain) + 2 * c + 1);
        const float gv[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
        const int ax = pair_axis(4 * c);  // the 4 pairs of a 16-byte chunk share one axis
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 cs = trow[ax][4 * c + i];
            const float y0 = (x[8 * c + 2 * i] * r) * gv[2 * i];
            const float y1 = (x[8 * c + 2 * i + 1] * r) * gv[2 * i + 1];
            const float o0 = fmaf(y0, cs.x, -(y1 * cs.y));
            const float o1 = fmaf(y0, cs.y, y1 * cs.x);
            o[i] = pack_bf16(o0, o1);
        }
        out[c] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

__global__ void __launch_bounds__(kThreads, 1) qkv_gemm_kernel(const __grid_constant__ QkvArgs a) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bars[2 * kStages + 5];
    __shared__ uint32_t tmem_slot;
    __shared__ volatile int abort_flag;

    const Geom& g = a.g;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n_tiles_all = (a.m_tiles[0] + a.m_tiles[1]) * a.n_tiles;
    const int k_steps = a.C / kBK;
    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    auto stage_a = [&](int st) { return sbase + st * kStageBytes; };
    auto stage_b = [&](int st) { return sbase + st * kStageBytes + kABytes; };
    const uint32_t bar_full = smem_u32(&bars[0]);             // [kStages] stage loaded
    const uint32_t bar_empty = smem_u32(&bars[kStages]);      // [kStages] stage consumed
    const uint32_t bar_acc = smem_u32(&bars[2 * kStages]);    // [2] accumulator complete
    const uint32_t bar_free = smem_u32(&bars[2 * kStages + 2]);  // [2] accumulator read out
    const uint32_t bar_drain = smem_u32(&bars[2 * kStages + 4]);

    if (tid == 0) {
        abort_flag = 0;
        for (int st = 0; st < kStages; ++st) {
            mbar_init(bar_full + 8 * st, 1);
            mbar_init(bar_empty + 8 * st, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_acc + 8 * b, 1);
            mbar_init(bar_free + 8 * b, 128);
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
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            for (int s = 0; s < 2; ++s) {
                prefetch_tensormap(&a.map_x[s]);
                prefetch_tensormap(&a.map_w[s]);
            }
            long long it = 0;  // stage uses so far (phase tracking)
            bool ok = true;
            for (int t = blockIdx.x; ok && t < n_tiles_all && !abort_flag; t += gridDim.x) {
                const Tile tl = tile_of(a, t);
                for (int kk = 0; kk < k_steps; ++kk, ++it) {
                    const int st = (int)(it % kStages);
                    const uint32_t use = (uint32_t)(it / kStages);
                    if (use > 0 && !mbar_wait(bar_empty + 8 * st, (use - 1) & 1, &abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(bar_full + 8 * st, kStageBytes);
                    tma_load_2d(stage_a(st), &a.map_x[tl.s], bar_full + 8 * st, kk * kBK, tl.m0);
                    tma_load_2d(stage_b(st), &a.map_w[tl.s], bar_full + 8 * st, kk * kBK, tl.n0);
                }
            }
            if (!ok) fail(&abort_flag);
            // drain: every issued stage has landed (the last kStages uses)
            const volatile int no_abort = 0;
            for (long long u = it - kStages < 0 ? 0 : it - kStages; u < it; ++u)
                mbar_wait(bar_full + 8 * (int)(u % kStages), (uint32_t)(u / kStages) & 1, &no_abort, kWaitLimitNs);
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            long long it = 0;
            int local = 0;  // tiles taken by this CTA
            bool ok = true;
            for (int t = blockIdx.x; ok && t < n_tiles_all; t += gridDim.x, ++local) {
                const int buf = local & 1;
                const uint32_t use_b = (uint32_t)(local >> 1);
                // the epilogue has read this accumulator's previous tile
                if (use_b > 0 && !mbar_wait(bar_free + 8 * buf, (use_b - 1) & 1, &abort_flag, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t acc = tmem + (uint32_t)(buf * kBN);
                for (int kk = 0; kk < k_steps; ++kk, ++it) {
                    const int st = (int)(it % kStages);
                    if (!mbar_wait(bar_full + 8 * st, (uint32_t)(it / kStages) & 1, &abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int j = 0; j < kBK / 16; ++j)
                        mma_ss(acc, sdesc_sw128(stage_a(st) + 32 * j, 16, 1024), sdesc_sw128(stage_b(st) + 32 * j, 16, 1024),
                               kIdesc, (kk > 0 || j > 0) ? 1u : 0u);
                    mma_commit(bar_empty + 8 * st);
                }
                if (ok) mma_commit(bar_acc + 8 * buf);
            }
            if (!ok) fail(&abort_flag);
            mma_commit(bar_drain);
            const volatile int no_abort = 0;
            mbar_wait(bar_drain, 0, &no_abort, kWaitLimitNs);
        }
    } else {
        // ------------------------------------------------ epilogue: one output row per thread
        const uint32_t lane_addr = (uint32_t)((warp & 3) * 32) << 16;
        const int row = (warp & 3) * 32 + lane;
        int local = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < n_tiles_all; t += gridDim.x, ++local) {
            const int buf = local & 1;
            if (!warp_wait(bar_acc + 8 * buf, (uint32_t)(local >> 1) & 1, &abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const Tile tl = tile_of(a, t);
            const int T_s = tl.s == 0 ? g.T_txt : g.T_img;
            const int m = tl.m0 + row;  // row of X_s / Y_s
            const bool live = m < g.B * T_s;
            const int b = live ? m / T_s : 0;
            const int n = (live ? m % T_s : 0) + (tl.s == 0 ? 0 : g.T_txt);  // token in [0, S)
#pragma unroll 1
            for (int hl = 0; hl < 2; ++hl) {
                const int col0 = tl.n0 + 128 * hl;
                if (col0 >= a.ncols) break;             // past the last head (odd H): warp-uniform
                // 0 Q, 1 K, 2 V (the output projection stores like V)
                const int part = a.out_proj ? 2 : col0 / a.C;
                const int head = (col0 % a.C) / 128;
                float x[128];
                __syncwarp();  // the TMEM loads are warp-collective
                {
                    uint32_t r32[32];
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        tmem_ld32(tmem + lane_addr + (uint32_t)(buf * kBN + 128 * hl + 32 * c), r32);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) x[32 * c + i] = __uint_as_float(r32[i]);
                    }
                }
                // + bias, one bf16 rounding: the stored projection
                const uint4* bp = reinterpret_cast<const uint4*>(a.bias[tl.s] + col0);
                uint32_t y[64];
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const uint4 bv = __ldg(bp + c);
                    const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        y[4 * c + e] = pack_bf16(x[8 * c + 2 * e] + bf16_lo(bw[e]), x[8 * c + 2 * e + 1] + bf16_hi(bw[e]));
                        x[8 * c + 2 * e] = bf16_lo(y[4 * c + e]);
                        x[8 * c + 2 * e + 1] = bf16_hi(y[4 * c + e]);
                    }
                }
                if (!live) continue;
                const bool plain_out = part == 2 || (part == 0 ? a.store_q : a.store_k);
                if (plain_out) {
                    const SegBf16& dst = part == 0 ? a.q : (part == 1 ? a.k : a.v);
                    uint4* o = reinterpret_cast<uint4*>(seg_row(dst, g, b, n, head));
#pragma unroll
                    for (int c = 0; c < 16; ++c) o[c] = make_uint4(y[4 * c], y[4 * c + 1], y[4 * c + 2], y[4 * c + 3]);
                }
                if (part < 2 && a.qh != nullptr) {
                    const size_t ri = ((size_t)b * g.H + head) * g.S + n;
                    float r;
                    norm_rope_full_row(x, a.gain[tl.s][part], a.tab, g, n, (part == 0 ? a.qh : a.kh) + ri * kHeadDim, r);
                    (part == 0 ? a.rq : a.rk)[ri] = r;
                }
            }
            tc_fence_before();
            mbar_arrive(bar_free + 8 * buf);
        }
        if (!ok) fail(&abort_flag);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

cudaError_t launch_proj_gemm(const Geom& g, bool out_proj, const uint16_t* const x[2], const uint16_t* const w[2],
                             const uint16_t* const bias[2], const float* const gains[4], uint16_t* qh, uint16_t* kh,
                             float* rq, float* rk, const float2* tab, const SegBf16& q, const SegBf16& k,
                             const SegBf16& v, bool store_q, bool store_k, cudaStream_t s) {
    QkvArgs a;
    const int C = g.H * kHeadDim;
    const int ncols = out_proj ? C : 3 * C;
    const long long rows[2] = {(long long)g.B * g.T_txt, (long long)g.B * g.T_img};
    for (int st = 0; st < 2; ++st) {
        if (rows[st] == 0) {
            memset(&a.map_x[st], 0, sizeof(a.map_x[st]));
            memset(&a.map_w[st], 0, sizeof(a.map_w[st]));
        } else if (!tmap::mat_bf16(&a.map_x[st], x[st], rows[st], C, kBM) ||
                   !tmap::mat_bf16(&a.map_w[st], w[st], ncols, C, kBN)) {
            return cudaErrorInvalidValue;
        }
        a.bias[st] = bias[st];
        a.m_tiles[st] = (int)((rows[st] + kBM - 1) / kBM);
    }
    a.gain[0][0] = gains[0];  // q text
    a.gain[0][1] = gains[1];  // k text
    a.gain[1][0] = gains[2];  // q image
    a.gain[1][1] = gains[3];  // k image
    a.g = g;
    a.C = C;
    a.ncols = ncols;
    a.out_proj = out_proj;
    a.n_tiles = (ncols + kBN - 1) / kBN;
    a.qh = qh;
    a.kh = kh;
    a.rq = rq;
    a.rk = rk;
    a.tab = tab;
    a.q = q;
    a.k = k;
    a.v = v;
    a.store_q = store_q;
    a.store_k = store_k;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(qkv_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    const int tiles = (a.m_tiles[0] + a.m_tiles[1]) * a.n_tiles;
    const int grid = tiles < sms ? tiles : sms;
    if (grid == 0) return cudaSuccess;
    const int kid = out_proj ? kKOutGemm : kKQkvGemm;
    timing_begin(kid, s);
    qkv_gemm_kernel<<<grid, kThreads, kSmemBytes, s>>>(a);
    timing_end(kid, s);
    return cudaGetLastError();
}

int read_and_clear_status_qkv(cudaStream_t s) {
    int v = 0, zero = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_status_qkv, sizeof(int), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return -1;
    if (cudaMemcpyToSymbolAsync(g_status_qkv, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return -1;
    if (cudaStreamSynchronize(s) != cudaSuccess) return -1;
    return v;
}

}  // namespace rlk

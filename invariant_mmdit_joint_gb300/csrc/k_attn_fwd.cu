// Joint attention forward: rows joint_attn_qk_gemm, joint_attn_softmax and
// joint_attn_av_gemm of the RFC #386 WS1 table, fused
// ("joint_attention_fused"), with an online softmax over key tiles.
//
// One CTA = one (query tile of 128 rows, head, sample). Query tiles are
// segment aligned: text tiles start at token 0, image tiles at token T_txt,
// so no tile straddles the two streams. Key tiles of 64 are visited in one
// fixed order -- text tiles from key 0 (only those holding a valid key), then
// image tiles from key T_txt -- so a row's result depends only on its own
// sample's data, never on B, batch position, padding or the SM count. No
// split-KV, no atomics. Scores, running max/sum and the O accumulator are
// FP32; P enters the PV product as bf16 (round to nearest even); O is cast
// to bf16 once, at the output.
#include "rlk_device.cuh"
#include "rlk_internal.h"

RLK_DEFINE_STRICT_PROBE(probe_fwd_tu)

namespace rlk {

const int kFwdBlockQ = 128;
const int kFwdBlockKV = 64;

namespace {

constexpr int kBM = 128;             // query rows per CTA
constexpr int kBN = 64;              // keys per tile
constexpr int kThreads = 256;        // 8 warps x 16 query rows
constexpr int kTileBytesQ = kBM * 256;
constexpr int kTileBytesKV = kBN * 256;
constexpr int kSmemBytes = kTileBytesQ + 4 * kTileBytesKV;  // Q + 2 x (K, V)
// exp(s / sqrt(128)) = exp2(s * kC); kC = log2(e) / sqrt(128)
constexpr float kC = (float)(1.4426950408889634 * 0.08838834764831845);
constexpr float kLn2 = 0.6931471805599453f;

__device__ int g_status_fwd;

struct FwdArgs {
    Geom g;
    ValidLen vl;
    const uint16_t* qh;   // [B, H, S, D] normed + rotated q
    const uint16_t* kh;   // [B, H, S, D]
    const uint16_t* v;    // [B, S, H, D]
    uint16_t* out;        // [B, S, H, D]
    float* lse;           // [B, H, S] or null
};

__global__ void __launch_bounds__(kThreads, 1) attn_fwd_kernel(const __grid_constant__ FwdArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const Geom& g = a.g;
    const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gr = lane >> 2, gc = lane & 3;

    const int nqt_txt = (g.T_txt + kBM - 1) / kBM;
    const bool q_txt = qt < nqt_txt;
    const int q0 = q_txt ? qt * kBM : g.T_txt + (qt - nqt_txt) * kBM;
    const int q_end = q_txt ? g.T_txt : g.S;
    const int L = a.vl.L[b];
    const int nkt_txt = (L + kBN - 1) / kBN;
    const int nkt = nkt_txt + (g.T_img + kBN - 1) / kBN;
    const size_t bh = (size_t)b * g.H + h;
    const uint16_t* qh = a.qh + bh * g.S * kHeadDim;
    const uint16_t* kh = a.kh + bh * g.S * kHeadDim;

    const uint32_t sQ = smem_u32(smem);
    const uint32_t sK = sQ + kTileBytesQ;
    const uint32_t sV = sK + 2 * kTileBytesKV;

    for (int i = tid; i < kBM * 16; i += kThreads) {
        const int r = i >> 4, c = i & 15, n = q0 + r;
        const bool ok = n < q_end;
        cp_async16(tile_addr(sQ, r, c), qh + (size_t)(ok ? n : 0) * kHeadDim + c * 8, ok);
    }
    auto load_kv = [&](int t, int buf) {
        const bool txt = t < nkt_txt;
        const int k0 = txt ? t * kBN : g.T_txt + (t - nkt_txt) * kBN;
        const int kend = txt ? L : g.S;
        for (int i = tid; i < kBN * 16; i += kThreads) {
            const int r = i >> 4, c = i & 15, n = k0 + r;
            const bool ok = n < kend;
            const int nn = ok ? n : 0;
            cp_async16(tile_addr(sK + buf * kTileBytesKV, r, c), kh + (size_t)nn * kHeadDim + c * 8, ok);
            cp_async16(tile_addr(sV + buf * kTileBytesKV, r, c),
                       a.v + (((size_t)b * g.S + nn) * g.H + h) * kHeadDim + c * 8, ok);
        }
    };
    load_kv(0, 0);
    cp_async_commit();

    float o[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;
    uint32_t qf[8][4];

    for (int t = 0; t < nkt; ++t) {
        if (t + 1 < nkt) load_kv(t + 1, (t + 1) & 1);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        if (t == 0) {
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                ldsm_x4(tile_addr(sQ, 16 * warp + (lane & 15), 2 * ks + (lane >> 4)), qf[ks][0], qf[ks][1],
                        qf[ks][2], qf[ks][3]);
        }
        const uint32_t kb = sK + (t & 1) * kTileBytesKV;
        const uint32_t vb = sV + (t & 1) * kTileBytesKV;

        // S = Q K^T for this warp's 16 rows x 64 keys
        float s[8][4];
#pragma unroll
        for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.0f;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t r0, r1, r2, r3;
                ldsm_x4(tile_addr(kb, 16 * np + (lane & 7) + ((lane >> 4) << 3), 2 * ks + ((lane >> 3) & 1)), r0,
                        r1, r2, r3);
                mma_bf16(s[2 * np], qf[ks], r0, r1);
                mma_bf16(s[2 * np + 1], qf[ks], r2, r3);
            }
        }

        // mask, scale to log2 units, online softmax (rows gr and gr + 8)
        const bool txt = t < nkt_txt;
        const int k0 = txt ? t * kBN : g.T_txt + (t - nkt_txt) * kBN;
        const int kend = txt ? L : g.S;
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const bool ok = k0 + 8 * nt + 2 * gc + e < kend;
                s[nt][e] = ok ? s[nt][e] * kC : -INFINITY;
                s[nt][2 + e] = ok ? s[nt][2 + e] * kC : -INFINITY;
                mx0 = fmaxf(mx0, s[nt][e]);
                mx1 = fmaxf(mx1, s[nt][2 + e]);
            }
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float al0 = exp2f(m0 - mn0), al1 = exp2f(m1 - mn1);
        m0 = mn0;
        m1 = mn1;
        float rs0 = 0.0f, rs1 = 0.0f;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                s[nt][e] = exp2f(s[nt][e] - mn0);
                s[nt][2 + e] = exp2f(s[nt][2 + e] - mn1);
                rs0 += s[nt][e];
                rs1 += s[nt][2 + e];
            }
        }
        l0 = l0 * al0 + rs0;
        l1 = l1 * al1 + rs1;
#pragma unroll
        for (int dt = 0; dt < 16; ++dt) {
            o[dt][0] *= al0;
            o[dt][1] *= al0;
            o[dt][2] *= al1;
            o[dt][3] *= al1;
        }

        // O += P V
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const uint32_t pa[4] = {pack_bf16(s[2 * kk][0], s[2 * kk][1]), pack_bf16(s[2 * kk][2], s[2 * kk][3]),
                                    pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]),
                                    pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3])};
#pragma unroll
            for (int dp = 0; dp < 8; ++dp) {
                uint32_t r0, r1, r2, r3;
                ldsm_x4_t(tile_addr(vb, 16 * kk + (lane & 7) + (((lane >> 3) & 1) << 3), 2 * dp + (lane >> 4)), r0,
                          r1, r2, r3);
                mma_bf16(o[2 * dp], pa, r0, r1);
                mma_bf16(o[2 * dp + 1], pa, r2, r3);
            }
        }
        __syncthreads();
    }

    // epilogue: O / l, one bf16 cast, staged through this warp's Q rows
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    const float inv0 = 1.0f / l0, inv1 = 1.0f / l1;
    const int r_lo = 16 * warp + gr, r_hi = r_lo + 8;
#pragma unroll
    for (int dt = 0; dt < 16; ++dt) {
        const uint32_t lo = pack_bf16(o[dt][0] * inv0, o[dt][1] * inv0);
        const uint32_t hi = pack_bf16(o[dt][2] * inv1, o[dt][3] * inv1);
        asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(tile_addr(sQ, r_lo, dt) + 4 * gc), "r"(lo));
        asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(tile_addr(sQ, r_hi, dt) + 4 * gc), "r"(hi));
    }
    if (a.lse != nullptr && gc == 0) {
        if (q0 + r_lo < q_end) a.lse[bh * g.S + q0 + r_lo] = (m0 + log2f(l0)) * kLn2;
        if (q0 + r_hi < q_end) a.lse[bh * g.S + q0 + r_hi] = (m1 + log2f(l1)) * kLn2;
    }
    __syncwarp();
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int i = lane + 32 * it;
        const int r = 16 * warp + (i >> 4), c = i & 15;
        const int n = q0 + r;
        if (n < q_end) {
            uint4 v;
            asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];\n"
                         : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                         : "r"(tile_addr(sQ, r, c)));
            *reinterpret_cast<uint4*>(a.out + (((size_t)b * g.S + n) * g.H + h) * kHeadDim + c * 8) = v;
        }
    }
}

}  // namespace

cudaError_t launch_attn_fwd(const Geom& g, const ValidLen& vl, const uint16_t* qh, const uint16_t* kh,
                            const uint16_t* v, uint16_t* out, float* lse, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    FwdArgs args{g, vl, qh, kh, v, out, lse};
    const int nqt = (g.T_txt + kBM - 1) / kBM + (g.T_img + kBM - 1) / kBM;
    dim3 grid(nqt, g.H, g.B);
    timing_begin(kKAttnFwd, s);
    attn_fwd_kernel<<<grid, kThreads, kSmemBytes, s>>>(args);
    timing_end(kKAttnFwd, s);
    return cudaGetLastError();
}

int read_and_clear_status_fwd(cudaStream_t s) {
    int v = 0, zero = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_status_fwd, sizeof(int), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return -1;
    if (cudaMemcpyToSymbolAsync(g_status_fwd, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return -1;
    if (cudaStreamSynchronize(s) != cudaSuccess) return -1;
    return v;
}

}  // namespace rlk

// HBM-bound kernels of the joint attention path (CUDA cores, FP32 math):
//   rope_table      cos/sin of every (position, RoPE pair) the call needs
//   prologue        qk_rmsnorm + multi_axis_rope of Q and K, one bf16 cast
//   bwd_pre         Delta = rowsum(dO * O) and lse2 = lse * log2(e), tile padded
//   norm_rope_bwd_k inverse RoPE rotation + RMSNorm backward of the keys and
//                   their gain-gradient partials (the queries' runs in the
//                   dQ kernel's epilogue)
//   dg_fold         fixed-order folds of the gain-gradient partials
// Sources: RFC #386 "WS1/WS2 kernel roadmap", Model contract table (Q/K
// preprocessing and RoPE rows) and WS1 table (qk_rmsnorm, multi_axis_rope);
// "WS1 Single-GPU Kernel List", Kernel table (fwd + bwd for both rows) and
// Acceptance (gradients summed over several paths in one fixed order).
#include <cmath>

#include "rlk_device.cuh"
#include "rlk_internal.h"
#include "rlk_sm100.cuh"
#include "rlk_tmap.h"

RLK_DEFINE_STRICT_PROBE(probe_prologue_tu)

namespace rlk {
namespace {

using namespace sm100;

constexpr int kRowThreads = 16;  // a half warp covers one 128-wide row, 8 dims per lane

// ---------------------------------------------------------------- rope table
// tab[(p - p_lo) * 64 + k] = (cos, sin) of p * freq[k], freq[k] =
// theta^(-2j/d_a) for pair k = pair j of axis a (computed once on the host in
// FP64). Angles and cos/sin in FP64, rounded once to FP32.
struct PairFreqs {
    double f[kPairs];
};

__global__ void rope_table_kernel(Geom g, const PairFreqs fr, float2* __restrict__ tab) {
    int idx = blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= g.n_pos * kPairs) return;
    int k = idx % kPairs;
    int p = g.p_lo + idx / kPairs;
    double ang = (double)p * fr.f[k];
    double s, c;
    sincos(ang, &s, &c);
    tab[idx] = make_float2((float)c, (float)s);
}

// ---------------------------------------------------------------- prologue
// One half warp per (b, n, h) row; lane l owns dims [8l, 8l+8) = RoPE pairs
// [4l, 4l+4), which all lie on one axis (the axis blocks start at pairs 0,
// 8 and 36, multiples of 4), so a lane reads its four (cos, sin) from one
// table row with two 16-byte loads. Sum of squares: each lane adds its 8
// squares in order, then a butterfly over the 16 lanes (xor 8, 4, 2, 1).
// r = 1 / sqrt(ss/128 + eps) with IEEE sqrt and division. y = (x * r) * g;
// then each pair turns by its angle; one round to bf16 at the output.
__device__ __forceinline__ void norm_rope_row(const uint4 xv, const float* gain, const float4 t0, const float4 t1,
                                              int lane16, float eps, uint4& out, float& r_out) {
    float x[8] = {bf16_lo(xv.x), bf16_hi(xv.x), bf16_lo(xv.y), bf16_hi(xv.y),
                  bf16_lo(xv.z), bf16_hi(xv.z), bf16_lo(xv.w), bf16_hi(xv.w)};
    float ss = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) ss = fmaf(x[i], x[i], ss);
#pragma unroll
    for (int m = 8; m >= 1; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
    float r = 1.0f / sqrtf(fmaf(ss, 1.0f / 128.0f, eps));
    r_out = r;
    const float4 g0 = reinterpret_cast<const float4*>(gain)[2 * lane16];
    const float4 g1 = reinterpret_cast<const float4*>(gain)[2 * lane16 + 1];
    const float gv[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
    const float2 cs[4] = {make_float2(t0.x, t0.y), make_float2(t0.z, t0.w), make_float2(t1.x, t1.y),
                          make_float2(t1.z, t1.w)};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float y0 = (x[2 * i] * r) * gv[2 * i];
        float y1 = (x[2 * i + 1] * r) * gv[2 * i + 1];
        float o0 = fmaf(y0, cs[i].x, -(y1 * cs[i].y));
        float o1 = fmaf(y0, cs[i].y, y1 * cs[i].x);
        o[i] = pack_bf16(o0, o1);
    }
    out = make_uint4(o[0], o[1], o[2], o[3]);
}

// A CTA of 256 threads covers 32 rows: half warp w takes rows base + w and
// base + 16 + w (the two half warps of a warp read 512 contiguous bytes).
// Every global load of a lane (q, k and the (cos, sin) table row of both
// rows) is issued before any arithmetic; the four gain vectors are staged
// in shared memory first.
constexpr int kPrologueRowsPerCta = 32;

__global__ void __launch_bounds__(256, 4) prologue_kernel(
    Geom g, const SegBf16 q, const SegBf16 k,
    const float* __restrict__ gq_txt, const float* __restrict__ gk_txt,
    const float* __restrict__ gq_img, const float* __restrict__ gk_img,
    const float2* __restrict__ tab, uint16_t* __restrict__ qh, uint16_t* __restrict__ kh,
    float* __restrict__ rq, float* __restrict__ rk) {
    __shared__ __align__(16) float gs[4][kHeadDim];  // q_txt, k_txt, q_img, k_img
    {
        const int i = threadIdx.x;  // 256 threads, 512 gains
        const float* src0 = i < kHeadDim ? gq_txt : gk_txt;
        const float* src1 = i < kHeadDim ? gq_img : gk_img;
        gs[i / kHeadDim][i % kHeadDim] = __ldg(src0 + i % kHeadDim);
        gs[2 + i / kHeadDim][i % kHeadDim] = __ldg(src1 + i % kHeadDim);
    }
    // rows (b, n, h) of [B, S, H] in 32-bit arithmetic (B * S * H rows of
    // 256 bytes fit far below 2^31); the CTA's first row is divided out once,
    // each thread's row follows from it by carrying, not by division
    const int rows = g.B * g.S * g.H;
    const int lane16 = threadIdx.x % kRowThreads;
    const int axis = pair_axis(4 * lane16);
    const int base = (int)blockIdx.x * kPrologueRowsPerCta;
    const int bn0 = base / g.H, h0 = base - bn0 * g.H;
    const int b0 = bn0 / g.S, n0 = bn0 - b0 * g.S;
    uint4 xq[2], xk[2];
    float4 ta[2], tb[2];
    int hh[2], nn[2], bb[2];
    bool active[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        // a half warp past the end works on the last row and stores
        // nothing, so that every lane of the warp reaches the shuffles
        const int ro = (int)(threadIdx.x / kRowThreads) + 16 * u;  // row offset in the CTA
        active[u] = base + ro < rows;
        int h = h0 + ro, n = n0, b = b0;
        while (h >= g.H) {
            h -= g.H;
            if (++n == g.S) {
                n = 0;
                ++b;
            }
        }
        if (!active[u]) {
            h = g.H - 1;
            n = g.S - 1;
            b = g.B - 1;
        }
        hh[u] = h;
        nn[u] = n;
        bb[u] = b;
        // q and k share their segment strides (both calls pass them alike),
        // so one offset addresses both
        const bool img = nn[u] >= g.T_txt;
        const long long off =
            (((long long)bb[u] * (img ? q.bstride[1] : q.bstride[0]) + (img ? nn[u] - g.T_txt : nn[u])) * g.H +
             hh[u]) * kHeadDim + 8 * lane16;
        xq[u] = __ldg(reinterpret_cast<const uint4*>((img ? q.p[1] : q.p[0]) + off));
        xk[u] = __ldg(reinterpret_cast<const uint4*>((img ? k.p[1] : k.p[0]) + off));
        // lane l's four (cos, sin) pairs: two 16-byte loads from one table row
        const float4* trow =
            reinterpret_cast<const float4*>(tab + (size_t)(token_pos(g, nn[u], axis) - g.p_lo) * kPairs + 4 * lane16);
        ta[u] = __ldg(trow);
        tb[u] = __ldg(trow + 1);
    }
    __syncthreads();  // gains staged
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int h = hh[u], n = nn[u], b = bb[u];
        const bool txt = n < g.T_txt;
        uint4 oq, ok;
        float r_q, r_k;
        norm_rope_row(xq[u], gs[txt ? 0 : 2], ta[u], tb[u], lane16, g.eps, oq, r_q);
        norm_rope_row(xk[u], gs[txt ? 1 : 3], ta[u], tb[u], lane16, g.eps, ok, r_k);
        if (!active[u]) continue;
        const size_t bh = (size_t)b * g.H + h;
        const size_t dst = (bh * g.S + n) * kHeadDim + 8 * lane16;
        *reinterpret_cast<uint4*>(qh + dst) = oq;
        *reinterpret_cast<uint4*>(kh + dst) = ok;
        if (lane16 == 0) {
            rq[bh * g.S + n] = r_q;
            rk[bh * g.S + n] = r_k;
        }
    }
}

// ---------------------------------------------------------------- Delta, lse2
// Backward preprocess in the tile-padded layout: slot r of (b, h) belongs to
// query tile r / 128 (text tiles first, then image tiles) at offset r % 128.
// A slot holding a token gets Delta = sum_d dO * O and lse2 = lse * log2(e);
// a slot past its segment gets Delta = 0 and lse2 = +inf, so the backward
// kernels see P = 0 there. One warp (a CTA) per 32 consecutive slots of one
// (b, h), a slot per lane: the warp's 32 tokens of o and dout arrive by TMA
// as 128-byte-swizzled boxes of 64 dims x 32 tokens (tokens past the segment
// read zeros), and each lane sums its row in the order of a half warp
// holding 8 dims per lane: 16 partials of 8 products each in order, then the
// butterfly tree xor 8, 4, 2, 1.
__device__ int g_status_pro;
constexpr uint64_t kProWaitLimitNs = 2000000000ull;

struct PreArgs {
    CUtensorMap map_o[2];   // o per segment (text, image rows), box 64 x 1 x 32 x 1
    CUtensorMap map_do[2];  // dout likewise
    Geom g;
    const float* lse;
    float* lse2_p;
    float* delta_p;
};
constexpr int kPreSmemBytes = 4 * 4096 + 1024;  // o, dout: two boxes each

__global__ void __launch_bounds__(32) bwd_pre_kernel(const __grid_constant__ PreArgs a) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar_s;
    __shared__ volatile int abort_flag;
    const Geom& g = a.g;
    const int lane = threadIdx.x;
    const int bh = (int)blockIdx.x, r0 = 32 * (int)blockIdx.y;
    const int b = bh / g.H, h = bh - b * g.H;
    const int t = r0 >> 7;
    const int seg = t < g.ntq_txt ? 0 : 1;
    const int n_seg0 = seg ? 128 * (t - g.ntq_txt) + (r0 & 127) : r0;  // first token, counted in its segment
    const int seg_len = seg ? g.T_img : g.T_txt;
    const size_t slot = (size_t)bh * g.nq_pad + r0 + lane;
    const bool valid = n_seg0 + lane < seg_len;
    const int n = (seg ? g.T_txt : 0) + n_seg0 + lane;
    if (n_seg0 >= seg_len) {  // all 32 slots lie past the segment
        a.delta_p[slot] = 0.0f;
        a.lse2_p[slot] = INFINITY;
        return;
    }
    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const uint8_t* sp = smem_raw + (sbase - smem_u32(smem_raw));
    const uint32_t bar = smem_u32(&bar_s);
    if (lane == 0) {
        abort_flag = 0;
        mbar_init(bar, 1);
        fence_barrier_init();
        mbar_expect_tx(bar, 4 * 4096);
        tma_load_4d(sbase, &a.map_o[seg], bar, 0, h, n_seg0, b);
        tma_load_4d(sbase + 4096, &a.map_o[seg], bar, 64, h, n_seg0, b);
        tma_load_4d(sbase + 8192, &a.map_do[seg], bar, 0, h, n_seg0, b);
        tma_load_4d(sbase + 12288, &a.map_do[seg], bar, 64, h, n_seg0, b);
    }
    const float lse_n = valid ? __ldg(a.lse + (size_t)bh * g.S + n) : 0.0f;
    __syncwarp();
    if (!__all_sync(0xffffffffu, mbar_wait(bar, 0, &abort_flag, kProWaitLimitNs))) {
        if (lane == 0) atomicOr(&g_status_pro, 1);
        return;
    }
    const int sw = lane & 7;
    float s16[16];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {  // dims 64 c + 8 k .. + 7: one half-warp lane's share
            const uint4 ov = *reinterpret_cast<const uint4*>(sp + c * 4096 + lane * 128 + ((k ^ sw) << 4));
            const uint4 dv = *reinterpret_cast<const uint4*>(sp + 8192 + c * 4096 + lane * 128 + ((k ^ sw) << 4));
            const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w};
            const uint32_t dw[4] = {dv.x, dv.y, dv.z, dv.w};
            float acc = 0.0f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc = fmaf(bf16_lo(dw[i]), bf16_lo(ow[i]), acc);
                acc = fmaf(bf16_hi(dw[i]), bf16_hi(ow[i]), acc);
            }
            s16[8 * c + k] = acc;
        }
    }
    float t8[8], t4[4];
#pragma unroll
    for (int i = 0; i < 8; ++i) t8[i] = s16[i] + s16[i + 8];
#pragma unroll
    for (int i = 0; i < 4; ++i) t4[i] = t8[i] + t8[i + 4];
    const float delta = (t4[0] + t4[2]) + (t4[1] + t4[3]);
    a.delta_p[slot] = valid ? delta : 0.0f;
    a.lse2_p[slot] = valid ? lse_n * 1.4426950408889634f : INFINITY;
}

// ---------------------------------------------------------------- key-side norm/rope backward
// (The query side runs in the dQ kernel's epilogue, from its accumulator.)
// CTA = (128-token tile of one stream segment, h, b), 128 threads; warp w
// takes rows 32 w .. 32 w + 31 of the tile in ascending order, loading four
// rows at a time (measured against 256-thread CTAs of 16 rows per warp, and
// against groups of 2 or 8 rows or a cap of 64 registers: all slower). Lane l owns dims
// [4l, 4l+4) = pairs 2l, 2l+1. Per row:
//   u  = R(-angle) * dk^          (inverse rotation)
//   xh = k * r,  w = u * g,  c = (sum_d w_d xh_d) / 128   (lane order, then xor 16..1)
//   dK = r * (w - xh * c)  -> bf16
//   gain-gradient partial += u * xh (per lane, rows ascending)
// Warp w's partial is the tile's quarter w, dgt[b][h][1][tile][w][128]: the
// layout the dQ epilogue fills for q.
constexpr int kNrbWarps = 4;
constexpr int kNrbRowsPerWarp = 32;
constexpr int kNrbGroup = 4;

__global__ void __launch_bounds__(kNrbWarps * 32) norm_rope_bwd_k_kernel(
    Geom g, const SegBf16 k, const float* __restrict__ gk_txt, const float* __restrict__ gk_img,
    const float2* __restrict__ tab, const float* __restrict__ rk, const float* __restrict__ dkh, const SegBf16 dk,
    float* __restrict__ dgt) {
    const int tile = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const bool txt = tile < g.ntq_txt;
    const int t0 = txt ? tile * 128 : g.T_txt + (tile - g.ntq_txt) * 128;
    const int seg_end = txt ? g.T_txt : g.S;
    const size_t bh = (size_t)b * g.H + h;
    const float4 gv = __ldg(reinterpret_cast<const float4*>(txt ? gk_txt : gk_img) + lane);
    const int k0 = 2 * lane, k1 = 2 * lane + 1;
    const int ax = pair_axis(k0);  // both pairs of a lane share an axis
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    const int row0 = t0 + warp * kNrbRowsPerWarp;
    // the tile lies in one segment of one sample: consecutive tokens are
    // H * 128 elements apart in either layout. (Pointers are selected one by
    // one: a reference to a parameter chosen at run time would put the
    // parameters in local memory.)
    const int sg = txt ? 0 : 1;
    const uint16_t* x_seg = sg ? k.p[1] : k.p[0];
    uint16_t* dx_seg = sg ? dk.p[1] : dk.p[0];
    const long long x_bs = sg ? k.bstride[1] : k.bstride[0];
    const long long dx_bs = sg ? dk.bstride[1] : dk.bstride[0];
    const int row0c = min(row0, seg_end - 1);  // row0, or the segment's last row when the warp has none
    const long long n0 = row0c - (sg ? g.T_txt : 0);  // token of row0c inside its segment
    const uint16_t* x_row0 = x_seg + (((long long)b * x_bs + n0) * g.H + h) * kHeadDim + 4 * lane;
    uint16_t* dx_row0 = dx_seg + (((long long)b * dx_bs + n0) * g.H + h) * kHeadDim + 4 * lane;
    const size_t token_stride = (size_t)g.H * kHeadDim;
    // rows in groups of kNrbGroup: every load of a group is issued before
    // its arithmetic, so a warp keeps several rows in flight
    for (int i0 = 0; i0 < kNrbRowsPerWarp; i0 += kNrbGroup) {
        float4 dyv[kNrbGroup];
        uint2 xv[kNrbGroup];
        float rv[kNrbGroup];
        float2 c0v[kNrbGroup], c1v[kNrbGroup];
#pragma unroll
        for (int j = 0; j < kNrbGroup; ++j) {
            const int n = min(row0 + i0 + j, seg_end - 1);  // rows past the segment: a valid row, not stored
            const float2* trow = tab + (size_t)(token_pos(g, n, ax) - g.p_lo) * kPairs;
            c0v[j] = __ldg(trow + k0);
            c1v[j] = __ldg(trow + k1);
            dyv[j] = __ldg(reinterpret_cast<const float4*>(dkh + (bh * g.S + n) * kHeadDim + 4 * lane));
            xv[j] = __ldg(reinterpret_cast<const uint2*>(x_row0 + (size_t)(n - row0c) * token_stride));
            rv[j] = __ldg(rk + bh * g.S + n);
        }
#pragma unroll
        for (int j = 0; j < kNrbGroup; ++j) {
            const int i = i0 + j;
            if (row0 + i >= seg_end) break;
            const float4 dy = dyv[j];
            const float2 c0 = c0v[j], c1 = c1v[j];
            const float r = rv[j];
            float u[4];
            u[0] = fmaf(dy.x, c0.x, dy.y * c0.y);
            u[1] = fmaf(dy.y, c0.x, -(dy.x * c0.y));
            u[2] = fmaf(dy.z, c1.x, dy.w * c1.y);
            u[3] = fmaf(dy.w, c1.x, -(dy.z * c1.y));
            const float x[4] = {bf16_lo(xv[j].x), bf16_hi(xv[j].x), bf16_lo(xv[j].y), bf16_hi(xv[j].y)};
            const float gg[4] = {gv.x, gv.y, gv.z, gv.w};
            float xh[4], w[4];
            float dot = 0.0f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                xh[e] = x[e] * r;
                w[e] = u[e] * gg[e];
                dot = fmaf(w[e], xh[e], dot);
            }
#pragma unroll
            for (int m = 16; m >= 1; m >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, m);
            const float c = dot * (1.0f / 128.0f);
            float dx[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                dx[e] = r * fmaf(-xh[e], c, w[e]);
                acc[e] = fmaf(u[e], xh[e], acc[e]);
            }
            *reinterpret_cast<uint2*>(dx_row0 + (size_t)i * token_stride) =
                make_uint2(pack_bf16(dx[0], dx[1]), pack_bf16(dx[2], dx[3]));
        }
    }
    const int nt = g.ntq_txt + g.ntq_img;
    float* part = dgt + (((bh * 2 + 1) * nt + tile) * 4 + warp) * kHeadDim;
    *reinterpret_cast<float4*>(part + 4 * lane) = make_float4(acc[0], acc[1], acc[2], acc[3]);
}

// ---------------------------------------------------------------- gain-gradient folds
// The dQ kernel's epilogue (q) and norm_rope_bwd_k (k) leave one partial per (b, h, q|k, 128-token
// tile, 32-row quarter, dim): dgt[b][h][q|k][tile][quarter][128].
// dg_partial[b,h,slot,d] = sum over that stream's tiles, ascending, of
// ((quarter 0 + quarter 1) + (quarter 2 + quarter 3)).
// Slots: 0 q_txt, 1 k_txt, 2 q_img, 3 k_img.
__global__ void dg_fold_bh_kernel(Geom g, const float* __restrict__ dgt, float* __restrict__ dg_partial) {
    const int idx = blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= g.B * g.H * 4 * kHeadDim) return;
    const int d = idx % kHeadDim;
    const int slot = (idx / kHeadDim) % 4;
    const size_t bh = idx / (4 * kHeadDim);
    const int which = slot & 1;
    const bool img = slot >= 2;
    const int nt = g.ntq_txt + g.ntq_img;
    const int t_begin = img ? g.ntq_txt : 0;
    const int t_end = img ? nt : g.ntq_txt;
    const float* src = dgt + ((bh * 2 + which) * nt) * 4 * kHeadDim + d;
    float s = 0.0f;
#pragma unroll 8
    for (int t = t_begin; t < t_end; ++t) {  // unrolled so the loads of 8 tiles are in flight together
        const float* p = src + (size_t)t * 4 * kHeadDim;
        s += (p[0] + p[kHeadDim]) + (p[2 * kHeadDim] + p[3 * kHeadDim]);
    }
    dg_partial[idx] = s;
}

// dg[slot,d] = sum_b ( sum_h dg_partial[b,h,slot,d] ), both ascending.
__global__ void dg_fold_total_kernel(Geom g, const float* __restrict__ dg_partial,
                                     float* __restrict__ dg) {
    const int idx = threadIdx.x;  // slot * 128 + d, 512 threads
    float total = 0.0f;
    for (int b = 0; b < g.B; ++b) {
        float sb = 0.0f;
#pragma unroll 8
        for (int h = 0; h < g.H; ++h) sb += dg_partial[((size_t)b * g.H + h) * 4 * kHeadDim + idx];
        total += sb;
    }
    dg[idx] = total;
}

unsigned row_blocks(const Geom& g) {
    const int rows = g.B * g.S * g.H;
    return (unsigned)((rows + kPrologueRowsPerCta - 1) / kPrologueRowsPerCta);
}

// The failure path's self-test: one warp waits on an mbarrier that nothing
// completes; the bounded wait gives up after limit_ns and records the
// failure like every kernel's wait does.
__global__ void wait_timeout_probe_kernel(uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar_s;
    __shared__ volatile int abort_flag;
    const uint32_t bar = smem_u32(&bar_s);
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(bar, 1);
        fence_barrier_init();
    }
    __syncwarp();
    if (!__all_sync(0xffffffffu, mbar_wait(bar, 0, &abort_flag, limit_ns)) && threadIdx.x == 0)
        atomicOr(&g_status_pro, 1);
}

}  // namespace

cudaError_t launch_wait_timeout_probe(int limit_ms, cudaStream_t s) {
    wait_timeout_probe_kernel<<<1, 32, 0, s>>>((uint64_t)limit_ms * 1000000ull);
    return cudaGetLastError();
}

cudaError_t launch_rope_table(const Geom& g, float2* tab, cudaStream_t s) {
    const int n = g.n_pos * kPairs;
    PairFreqs fr;
    for (int k = 0; k < kPairs; ++k) {
        const int a = pair_axis(k);
        const int j = a == 0 ? k : (a == 1 ? k - kAxis0Pairs : k - kAxis0Pairs - kAxis1Pairs);
        const double d_a = a == 0 ? 16.0 : 56.0;
        fr.f[k] = std::pow((double)g.theta, -2.0 * (double)j / d_a);
    }
    timing_begin(kKRopeTable, s);
    rope_table_kernel<<<(n + 127) / 128, 128, 0, s>>>(g, fr, tab);
    timing_end(kKRopeTable, s);
    return cudaGetLastError();
}

cudaError_t launch_prologue(const Geom& g, const SegBf16& q, const SegBf16& k,
                            const float* const gains[4], const float2* tab, uint16_t* qh,
                            uint16_t* kh, float* rq, float* rk, cudaStream_t s) {
    timing_begin(kKPrologue, s);
    prologue_kernel<<<row_blocks(g), 256, 0, s>>>(g, q, k, gains[0], gains[1], gains[2], gains[3],
                                                  tab, qh, kh, rq, rk);
    timing_end(kKPrologue, s);
    return cudaGetLastError();
}

cudaError_t launch_bwd_pre(const Geom& g, const SegBf16& out, const SegBf16& dout, const float* lse,
                           float* lse2_p, float* delta_p, cudaStream_t s) {
    PreArgs a;
    for (int seg = 0; seg < 2; ++seg)
        if (!tmap::seg_bf16(&a.map_o[seg], out, g, seg, 32) || !tmap::seg_bf16(&a.map_do[seg], dout, g, seg, 32))
            return cudaErrorInvalidValue;
    a.g = g;
    a.lse = lse;
    a.lse2_p = lse2_p;
    a.delta_p = delta_p;
    const dim3 grid((unsigned)(g.B * g.H), (unsigned)(g.nq_pad / 32));
    timing_begin(kKBwdPre, s);
    bwd_pre_kernel<<<grid, 32, kPreSmemBytes, s>>>(a);
    timing_end(kKBwdPre, s);
    return cudaGetLastError();
}

cudaError_t launch_norm_rope_bwd_k(const Geom& g, const SegBf16& k, const float* gk_txt, const float* gk_img,
                                   const float2* tab, const float* rk, const float* dkh, const SegBf16& dk,
                                   float* dgt, cudaStream_t s) {
    dim3 grid(g.ntq_txt + g.ntq_img, g.H, g.B);
    timing_begin(kKNormRopeBwd, s);
    norm_rope_bwd_k_kernel<<<grid, kNrbWarps * 32, 0, s>>>(g, k, gk_txt, gk_img, tab, rk, dkh, dk, dgt);
    timing_end(kKNormRopeBwd, s);
    return cudaGetLastError();
}

cudaError_t launch_dg_fold(const Geom& g, const float* dgt, float* dg_partial, float* dg,
                           cudaStream_t s) {
    const int n = g.B * g.H * 4 * kHeadDim;
    timing_begin(kKDgFold, s);
    dg_fold_bh_kernel<<<(n + 255) / 256, 256, 0, s>>>(g, dgt, dg_partial);
    dg_fold_total_kernel<<<1, 4 * kHeadDim, 0, s>>>(g, dg_partial, dg);
    timing_end(kKDgFold, s);
    return cudaGetLastError();
}

int read_and_clear_status_prologue(cudaStream_t s) {
    int v = 0, zero = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_status_pro, sizeof(int), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return -1;
    if (cudaMemcpyToSymbolAsync(g_status_pro, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return -1;
    if (cudaStreamSynchronize(s) != cudaSuccess) return -1;
    return v;
}

}  // namespace rlk

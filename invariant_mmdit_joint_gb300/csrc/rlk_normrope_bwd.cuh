// Backward of rows multi_axis_rope and qk_rmsnorm for one head row held by
// one thread, in 32-dim chunks, for the epilogue of the dQ kernel (RFC #386
// WS1 rows qk_rmsnorm / multi_axis_rope, "fwd + bwd" in the WS1 Single-GPU
// Kernel List):
//   u  = R(-angle) dy                       inverse rotation of each pair
//   xh = x r,  w = u g,  c = (sum_d w_d xh_d) / 128
//   dx = r (w - xh c)                       one bf16 rounding
//   gain gradient contribution  u_d xh_d
// The sum over d uses the fixed tree of norm_rope_bwd_k's layout, in which
// lane l of a warp holds dims 4l .. 4l+3: each lane's four products in order,
// then the butterfly xor 16, 8, 4, 2, 1 (fp32 addition is commutative, so
// every lane of that butterfly ends with the value lane_tree() forms). Query
// and key rows therefore round identically whichever kernel forms them.
#pragma once

#include "rlk_device.cuh"
#include "rlk_internal.h"

namespace rlk {

// The (cos, sin) table rows of token n, one per axis.
struct TabRows {
    const float2* r[3];
};
__device__ __forceinline__ TabRows tab_rows(const float2* tab, const Geom& g, int n) {
    TabRows t;
#pragma unroll
    for (int ax = 0; ax < 3; ++ax) t.r[ax] = tab + (size_t)(token_pos(g, n, ax) - g.p_lo) * kPairs;
    return t;
}

// The table row of RoPE axis ax (selects: an index computed at run time into
// the struct would move it to local memory).
__device__ __forceinline__ const float2* tab_row(const TabRows& t, int ax) {
    return ax == 0 ? t.r[0] : (ax == 1 ? t.r[1] : t.r[2]);
}

// u, xh, w of dims 32 c .. 32 c + 31 (pairs 16 c .. 16 c + 15) from dy (the
// chunk's dq^ / dk^), x (the chunk's bf16 input row, widened), r and the
// gain g (the row's 128 gains).
__device__ __forceinline__ void nrb_chunk(int c, const float (&dy)[32], const float (&x)[32], float r,
                                          const float* __restrict__ g, const TabRows& t, float (&u)[32],
                                          float (&xh)[32], float (&w)[32]) {
#pragma unroll
    for (int p = 0; p < 16; ++p) {  // pair 16 c + p: dims 2p, 2p + 1 of the chunk
        const int k = 16 * c + p;
        const float2 cs = tab_row(t, pair_axis(k))[k];
        u[2 * p] = fmaf(dy[2 * p], cs.x, dy[2 * p + 1] * cs.y);
        u[2 * p + 1] = fmaf(dy[2 * p + 1], cs.x, -(dy[2 * p] * cs.y));
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        xh[j] = x[j] * r;
        w[j] = u[j] * __ldg(g + 32 * c + j);
    }
}

// The 8 lane partials of a chunk (lanes 8 c .. 8 c + 7 of norm_rope_bwd_k's
// layout): four products each, in order.
__device__ __forceinline__ void nrb_partials(const float (&w)[32], const float (&xh)[32], float* s8) {
#pragma unroll
    for (int l = 0; l < 8; ++l) {
        float d = 0.0f;
#pragma unroll
        for (int j = 0; j < 4; ++j) d = fmaf(w[4 * l + j], xh[4 * l + j], d);
        s8[l] = d;
    }
}

// The butterfly xor 16, 8, 4, 2, 1 over the 32 lane partials, as lane 0 forms it.
__device__ __forceinline__ float lane_tree(const float (&s)[32]) {
    float b[16], c[8], d[4];
#pragma unroll
    for (int i = 0; i < 16; ++i) b[i] = s[i] + s[i + 16];
#pragma unroll
    for (int i = 0; i < 8; ++i) c[i] = b[i] + b[i + 8];
#pragma unroll
    for (int i = 0; i < 4; ++i) d[i] = c[i] + c[i + 4];
    const float e0 = d[0] + d[2], e1 = d[1] + d[3];
    return e0 + e1;
}

// dx of a chunk, packed to bf16 pairs.
__device__ __forceinline__ void nrb_dx(const float (&w)[32], const float (&xh)[32], float r, float cdot,
                                       uint32_t (&out)[16]) {
#pragma unroll
    for (int i = 0; i < 16; ++i)
        out[i] = pack_bf16(r * fmaf(-xh[2 * i], cdot, w[2 * i]), r * fmaf(-xh[2 * i + 1], cdot, w[2 * i + 1]));
}

// Sum of v over the 32 lanes of the warp for each of the 32 dims, by a
// transposing butterfly (31 shuffles): on return lane L holds the sum of
// dim L in v[0]. A fixed order: the same bits on every run.
__device__ __forceinline__ float warp_transpose_sum(float (&v)[32], int lane) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) {
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int i = 0; i < m; ++i) {
            const float send = upper ? v[i] : v[i + m];
            const float keep = upper ? v[i + m] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
        }
    }
    return v[0];
}

// The backward of one row held by one thread of a warp: dy_chunk(c, dy)
// gives the row's dq^ / dk^ of dims 32 c .. 32 c + 31 (zero in rows that
// do not exist), xrow the bf16 input row. Pass 1 forms the dot product of
// the RMSNorm backward, pass 2 writes dx (bf16, 256 bytes, only when row_ok)
// and the warp's gain-gradient partial of every dim: the sum of u * xh over
// the warp's 32 rows, part[0 .. 127].
template <class DyChunk>
__device__ __forceinline__ void nrb_row(const DyChunk& dy_chunk, bool row_ok, const uint4* __restrict__ xrow, float r,
                                        const float* __restrict__ gain, const TabRows& t, uint4* dxrow,
                                        float* __restrict__ part, int lane) {
    auto x_chunk = [&](int c, float (&x)[32]) {
#pragma unroll
        for (int v4 = 0; v4 < 4; ++v4) {
            const uint4 xv = row_ok ? __ldg(xrow + 4 * c + v4) : make_uint4(0u, 0u, 0u, 0u);
            const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                x[8 * v4 + 2 * e] = bf16_lo(xw[e]);
                x[8 * v4 + 2 * e + 1] = bf16_hi(xw[e]);
            }
        }
    };
    float sp[32];
#pragma unroll
    for (int c = 0; c < 4; ++c) {  // unrolled: sp stays in registers
        float dy[32], x[32], u[32], xh[32], w[32];
        dy_chunk(c, dy);
        x_chunk(c, x);
        nrb_chunk(c, dy, x, r, gain, t, u, xh, w);
        nrb_partials(w, xh, &sp[8 * c]);
    }
    const float cdot = lane_tree(sp) * (1.0f / 128.0f);
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
        float dy[32], x[32], u[32], xh[32], w[32];
        dy_chunk(c, dy);
        x_chunk(c, x);
        nrb_chunk(c, dy, x, r, gain, t, u, xh, w);
        uint32_t o[16];
        nrb_dx(w, xh, r, cdot, o);
        if (row_ok) {
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4)
                dxrow[4 * c + v4] = make_uint4(o[4 * v4], o[4 * v4 + 1], o[4 * v4 + 2], o[4 * v4 + 3]);
        }
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = u[j] * xh[j];  // zero in rows that do not exist
        part[32 * c + lane] = warp_transpose_sum(v, lane);
    }
}

}  // namespace rlk

// Host-side TMA tensor-map encoders shared by the attention kernels' launch
// code. Every map uses the 128-byte swizzle: boxes are 128 rows of 128
// bytes, so a shared-memory tile is rows of 128 bytes whose 16-byte chunk c
// sits at position c ^ (row % 8).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <string.h>

#include "rlk_internal.h"

namespace rlk {
namespace tmap {

inline PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
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

inline bool encode(CUtensorMap* m, CUtensorMapDataType type, cuuint32_t rank, const void* base,
                   const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box) {
    auto enc = get_encode();
    if (enc == nullptr) return false;
    const cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return enc(m, type, rank, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 [rows, 128] (q^, k^ as one [B*H*S, 128] matrix), box 64 x 128
inline bool rows_bf16(CUtensorMap* m, const void* base, uint64_t rows) {
    const cuuint64_t dims[2] = {128, rows};
    const cuuint64_t strides[1] = {256};
    const cuuint32_t box[2] = {64, 128};
    return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box);
}

// bf16 row-major [rows, cols] (cols a multiple of 64), box 64 x box_rows
inline bool mat_bf16(CUtensorMap* m, const void* base, long long rows, int cols, int box_rows) {
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box);
}

// bf16 [B, S, H, 128] as 4-D (d, h, token, b), box 64 x 1 x 128 x 1; seg
// -1 = all S tokens, 0 = the text rows [0, T_txt), 1 = the image rows
// [T_txt, S) (a box reaching past the segment is clipped there). A
// segment with no rows gets a zeroed map that no kernel uses.
inline bool bshd_bf16(CUtensorMap* m, const void* base, const Geom& g, int seg = -1) {
    const int rows = seg < 0 ? g.S : (seg == 0 ? g.T_txt : g.T_img);
    if (rows == 0) {
        memset(m, 0, sizeof(*m));
        return true;
    }
    const uint16_t* p = static_cast<const uint16_t*>(base) + (seg == 1 ? (size_t)g.T_txt * g.H * kHeadDim : 0);
    const cuuint64_t dims[4] = {128, (cuuint64_t)g.H, (cuuint64_t)rows, (cuuint64_t)g.B};
    const cuuint64_t strides[3] = {256, (cuuint64_t)g.H * 256, (cuuint64_t)g.S * g.H * 256};
    const cuuint32_t box[4] = {64, 1, 128, 1};
    return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, p, dims, strides, box);
}

// One segment (0 text, 1 image) of a segmented bf16 activation as a 4-D
// map (d, h, token in the segment, b), box 64 x 1 x box_rows x 1: a box reaching
// past the segment is clipped there (loads read zeros, stores are dropped).
// A segment with no rows gets a zeroed map that no kernel uses.
inline bool seg_bf16(CUtensorMap* m, const SegBf16& t, const Geom& g, int seg, int box_rows = 128) {
    const int rows = seg == 0 ? g.T_txt : g.T_img;
    if (rows == 0) {
        memset(m, 0, sizeof(*m));
        return true;
    }
    const cuuint64_t dims[4] = {128, (cuuint64_t)g.H, (cuuint64_t)rows, (cuuint64_t)g.B};
    const cuuint64_t strides[3] = {256, (cuuint64_t)g.H * 256, (cuuint64_t)t.bstride[seg] * g.H * 256};
    const cuuint32_t box[4] = {64, 1, (cuuint32_t)box_rows, 1};
    return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, t.p[seg], dims, strides, box);
}

// fp32 [B*H, S, 128] per segment (as bshd_bf16), box 32 x 128 x 1
inline bool bhsd_f32_segment(CUtensorMap* m, const float* base, const Geom& g, int seg) {
    const int rows = seg == 0 ? g.T_txt : g.T_img;
    if (rows == 0) {
        memset(m, 0, sizeof(*m));
        return true;
    }
    const float* p = base + (seg == 0 ? 0 : (size_t)g.T_txt * kHeadDim);
    const cuuint64_t dims[3] = {128, (cuuint64_t)rows, (cuuint64_t)g.B * g.H};
    const cuuint64_t strides[2] = {512, (cuuint64_t)g.S * 512};
    const cuuint32_t box[3] = {32, 128, 1};
    return encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, p, dims, strides, box);
}

// fp32 scores [B*H, S, ncols] per segment (0 text, 1 image rows) as 3-D
// (col, row in the segment, b*H + h), box 32 x 32 x 1: a box reaching past
// the segment is clipped there.
inline bool scores_f32_segment(CUtensorMap* m, const float* base, const Geom& g, int ncols, int seg) {
    const int rows = seg == 0 ? g.T_txt : g.T_img;
    if (rows == 0) {
        memset(m, 0, sizeof(*m));
        return true;
    }
    const float* p = base + (seg == 0 ? 0 : (size_t)g.T_txt * ncols);
    const cuuint64_t dims[3] = {(cuuint64_t)ncols, (cuuint64_t)rows, (cuuint64_t)g.B * g.H};
    const cuuint64_t strides[2] = {(cuuint64_t)ncols * 4, (cuuint64_t)g.S * ncols * 4};
    const cuuint32_t box[3] = {32, 32, 1};
    return encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, p, dims, strides, box);
}

// fp32 row-major [rows, cols] (cols a multiple of 32), box box_cols x box_rows
inline bool mat_f32(CUtensorMap* m, const float* base, long long rows, int cols, int box_cols, int box_rows) {
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 4};
    const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    return encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box);
}

// bf16 P [B*H, S, ncols] per segment (as scores_f32_segment), box 64 x box_rows x 1
inline bool p_bf16_segment(CUtensorMap* m, const void* base, const Geom& g, int ncols, int seg, int box_rows = 32) {
    const int rows = seg == 0 ? g.T_txt : g.T_img;
    if (rows == 0) {
        memset(m, 0, sizeof(*m));
        return true;
    }
    const uint16_t* p = static_cast<const uint16_t*>(base) + (seg == 0 ? 0 : (size_t)g.T_txt * ncols);
    const cuuint64_t dims[3] = {(cuuint64_t)ncols, (cuuint64_t)rows, (cuuint64_t)g.B * g.H};
    const cuuint64_t strides[2] = {(cuuint64_t)ncols * 2, (cuuint64_t)g.S * ncols * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
    return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, p, dims, strides, box);
}

}  // namespace tmap
}  // namespace rlk

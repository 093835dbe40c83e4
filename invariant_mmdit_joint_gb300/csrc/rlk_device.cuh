// Device helpers shared by the kernels of librlk_joint_attn.so: bf16 packing,
// cp.async / ldmatrix / mma.sync wrappers (inline PTX) and the per-unit
// strict-math probe.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

namespace rlk {

// ------------------------------------------------------------ bf16
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// Round two floats to bf16 (nearest, ties to even) and pack lo | hi << 16.
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&p);
}

// ------------------------------------------------------------ exp2
// 2^x on the special-function unit (PTX ex2.approx.ftz.f32): relative error
// about 2^-22, results below 2^-126 flush to 0, 2^-inf = 0. Used only for
// softmax numerators, which are rounded to bf16 (2^-9 relative) before their
// products or summed into row sums of at least 1, so neither the error nor
// the flush is visible. A fixed hardware instruction: the same bits on every
// run and in every batch composition.
__device__ __forceinline__ float exp2_sfu(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ------------------------------------------------------------ shared memory
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte async copy global -> shared; when !valid the 16 bytes are zeroed.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
    int n = valid ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// D += A * B, m16n8k16, bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// A tile of rows x 128 bf16 in shared memory: a row is 256 bytes = 16 chunks
// of 16 bytes; chunk c of row r is stored at chunk position c ^ (r & 7), so
// that the 8 rows an ldmatrix phase reads hit 8 different bank groups.
__device__ __forceinline__ uint32_t tile_addr(uint32_t base, int row, int chunk) {
    return base + row * 256 + ((chunk ^ (row & 7)) << 4);
}

}  // namespace rlk

// ------------------------------------------------------------ strict-math probe
// Included once by every translation unit so that the probe is compiled with
// that unit's flags. Fast math (nvcc --use_fast_math) flushes subnormals,
// approximates division and square root and maps expf to an approximation
// whose error grows with |x|; each of these is detectable at run time.
#define RLK_DEFINE_STRICT_PROBE(FN_NAME)                                                     \
    namespace FN_NAME##_detail {                                                             \
    constexpr int kProbeN = 256;                                                             \
    __device__ float g_probe_in[3 * kProbeN + 2];                                            \
    __device__ float g_probe_out[3 * kProbeN + 1];                                           \
    __global__ void strict_probe_kernel() {                                                  \
        int i = threadIdx.x;                                                                 \
        float a = g_probe_in[i], b = g_probe_in[kProbeN + i];                                \
        g_probe_out[i] = a / b;                                                              \
        g_probe_out[kProbeN + i] = sqrtf(a);                                                 \
        g_probe_out[2 * kProbeN + i] = expf(g_probe_in[2 * kProbeN + i]);                    \
        if (i == 0) g_probe_out[3 * kProbeN] = g_probe_in[3 * kProbeN] * g_probe_in[3 * kProbeN + 1]; \
    }                                                                                        \
    }                                                                                        \
    namespace rlk {                                                                          \
    int FN_NAME(void) {                                                                      \
        using namespace ::FN_NAME##_detail;                                                  \
        float in[3 * kProbeN + 2], out[3 * kProbeN + 1];                                     \
        uint32_t st = 0x9e3779b9u;                                                           \
        for (int i = 0; i < 3 * kProbeN; ++i) {                                              \
            st = st * 1664525u + 1013904223u;                                                \
            float u = (float)(st >> 8) * (1.0f / 16777216.0f);                                \
            in[i] = i < 2 * kProbeN ? 1.0f + u * 1.0e6f : u * 160.0f - 80.0f;                \
        }                                                                                    \
        in[3 * kProbeN] = 1.0e-30f;                                                          \
        in[3 * kProbeN + 1] = 1.0e-10f;                                                      \
        if (cudaMemcpyToSymbol(g_probe_in, in, sizeof(in)) != cudaSuccess) return -1;        \
        strict_probe_kernel<<<1, kProbeN>>>();                                               \
        if (cudaGetLastError() != cudaSuccess) return -1;                                    \
        if (cudaMemcpyFromSymbol(out, g_probe_out, sizeof(out)) != cudaSuccess) return -1;   \
        for (int i = 0; i < kProbeN; ++i) {                                                  \
            double a = in[i], b = in[kProbeN + i];                                           \
            if (out[i] != (float)(a / b)) return 0;                                          \
            if (out[kProbeN + i] != (float)sqrt(a)) return 0;                                \
            double e = exp((double)in[2 * kProbeN + i]);                                     \
            double ulp = ldexp(1.0, ilogb(e) - 23);                                          \
            if (fabs((double)out[2 * kProbeN + i] - e) > 3.0 * ulp) return 0;                \
        }                                                                                    \
        if (!(out[3 * kProbeN] > 0.0f)) return 0;                                            \
        return 1;                                                                            \
    }                                                                                        \
    }

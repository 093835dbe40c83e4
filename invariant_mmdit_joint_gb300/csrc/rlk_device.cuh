// Device helpers shared by the kernels of librlk_joint_attn.so: bf16 packing,
// the softmax numerators' exp2, shared-memory addresses and the per-unit
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
// Softmax numerators 2^x use the CUDA math library's exp2f (maximum error
// 2 ulp, subnormal results kept, 2^-inf = 0), compiled without fast math:
// no approximate or flush-to-zero instruction is named here.
__device__ __forceinline__ float exp2_num(float x) { return exp2f(x); }

// ------------------------------------------------------------ shared memory
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
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

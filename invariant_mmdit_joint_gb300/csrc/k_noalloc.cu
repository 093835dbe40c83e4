// Allocation-free forward entry point.
//
// Some host programs cannot, or may not, allocate device memory on the call
// path: a plugin host that hands its plugins no workspace, a serving process
// whose memory pool already owns the device, or code that must not pay the
// implicit synchronisation a cudaMalloc / cudaFree can bring. For them this
// file provides rlk_joint_attn_fwd_noalloc(): the same forward kernels as
// rlk_joint_attn_fwd(), but with the forward context (normed and rotated q
// and k, the RMSNorm factors and the cos/sin table) placed in a fixed
// file-scope device array instead of a caller buffer. Nothing here calls
// cudaMalloc, cudaFree or any allocating library routine.
//
// The array is RLK_NOALLOC_SCRATCH_BYTES long and every GPU that loads the
// library holds it until the process exits. Each call first runs the regular
// forward's argument and device checks (same statuses, same order), then
// looks the array's device address up on the current device. The lookup is
// repeated on every call rather than cached: a cached address would go stale
// if the device's context were reset and the library's device code loaded
// again elsewhere. The first lookup on a device also loads this file's
// device code there, so make the first call on each device before any stream
// capture. All calls share the one array, so calls whose kernels overlap on
// the GPU (two streams, two host threads) race; serialise them. No byte of
// the array needs to start at zero: the forward writes every byte it reads
// before reading it.
#include <cuda_runtime.h>

#include "rlk_internal.h"

namespace {

constexpr size_t kScratchBytes = RLK_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_fwd_scratch[kScratchBytes];

rlk_status fwd_noalloc_impl(const rlk_ja_shape* shape, const void* q, const void* k, const void* v,
                            const float* g_q_txt, const float* g_k_txt, const float* g_q_img,
                            const float* g_k_img, const int32_t* txt_valid_len, void* out, float* lse,
                            void* stream) {
    rlk::Geom g;
    rlk::ValidLen vl;
    rlk_status st = rlk::fwd_validate(shape, q, k, v, g_q_txt, g_k_txt, g_q_img, g_k_img, txt_valid_len, out, lse,
                                      nullptr, false, &g, &vl);
    if (st != RLK_OK) return st;
    if (rlk::ctx_bytes_of(g) > kScratchBytes) return RLK_ERR_WORKSPACE;
    st = rlk::device_check(stream);
    if (st != RLK_OK) return st;
    // Host code cannot use the symbol's name as a device address: ask the
    // runtime for it on the current device.
    void* scratch = nullptr;
    if (cudaGetSymbolAddress(&scratch, g_fwd_scratch) != cudaSuccess || scratch == nullptr) return RLK_ERR_CUDA;
    return rlk::fwd_run(g, vl, q, k, v, g_q_txt, g_k_txt, g_q_img, g_k_img, out, lse, scratch, stream);
}

}  // namespace

// One operator-trace record per call (the nested regular forward adds its
// kernels to it).
extern "C" rlk_status rlk_joint_attn_fwd_noalloc(const rlk_ja_shape* shape, const void* q, const void* k,
                                                 const void* v, const float* g_q_txt, const float* g_k_txt,
                                                 const float* g_q_img, const float* g_k_img,
                                                 const int32_t* txt_valid_len, void* out, float* lse,
                                                 void* stream) {
    rlk::OpScope sc(rlk::kOpFwdNoalloc, shape);
    return sc.finish(fwd_noalloc_impl(shape, q, k, v, g_q_txt, g_k_txt, g_q_img, g_k_img, txt_valid_len, out, lse,
                                      stream));
}

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
// library holds it until the process exits. Its device address is looked up
// once per device, by the first call on that device, with that device
// current. All calls share the one array, so calls whose kernels overlap on
// the GPU (two streams, two host threads) race; serialise them. No byte of
// the array needs to start at zero: the forward writes every byte it reads
// before reading it.
#include <cuda_runtime.h>

#include <mutex>

#include "rlk_internal.h"

namespace {

constexpr size_t kScratchBytes = RLK_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_fwd_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices];

// Device address of g_fwd_scratch on the current device (set-up, once per
// device). Host code cannot use the symbol's name as a device address.
rlk_status scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return RLK_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_fwd_scratch) != cudaSuccess || p == nullptr) return RLK_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return RLK_OK;
}

rlk_status fwd_noalloc_impl(const rlk_ja_shape* shape, const void* q, const void* k, const void* v,
                            const float* g_q_txt, const float* g_k_txt, const float* g_q_img,
                            const float* g_k_img, const int32_t* txt_valid_len, void* out, float* lse,
                            void* stream) {
    const size_t need = rlk_joint_attn_ctx_bytes(shape);
    if (need == 0) {
        // an invalid shape: let the regular entry point report why, without
        // touching the device
        return rlk_joint_attn_fwd(shape, q, k, v, g_q_txt, g_k_txt, g_q_img, g_k_img, txt_valid_len, out, lse,
                                  nullptr, stream);
    }
    if (need > kScratchBytes) return RLK_ERR_WORKSPACE;
    void* scratch = nullptr;
    const rlk_status st = scratch_address(&scratch);
    if (st != RLK_OK) return st;
    return rlk_joint_attn_fwd(shape, q, k, v, g_q_txt, g_k_txt, g_q_img, g_k_img, txt_valid_len, out, lse, scratch,
                              stream);
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

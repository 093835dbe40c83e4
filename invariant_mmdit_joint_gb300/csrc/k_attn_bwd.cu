// Joint attention backward on the tcgen05 tensor cores (the "bwd" half of
// the WS1 attention rows of RFC #386 and of the "WS1 Single-GPU Kernel
// List"): two atomic-free kernels with the forward's warp roles.
//
//   dkdv: one CTA = (key tile of 128, head, sample). Walks every query tile
//         of 128 in one fixed ascending order (text tiles from token 0, then
//         image tiles from token T_txt). Per query tile i:
//           S^T  = K Q^T, dP^T = V dO^T            (tcgen05, A and B in smem)
//           P^T  = exp2(S^T * c - lse2), dS^T = P^T * (dP^T - Delta)
//                                                  (8 warps: key row = TMEM
//                                                   lane, 64 queries each;
//                                                   bf16 results into TMEM)
//           dV  += P^T dO,  dK += dS^T Q           (tcgen05, A from TMEM)
//         in two alternating TMEM regions, so tile i + 1's scores and dP^T
//         run while tile i's products finish; stores the bf16 dS^T tile in
//         the tensor cores' operand layout.
//   dq:   persistent; one unit = (query tile of 128, head, sample):
//         dQ += dS K over the key tiles in the forward's order, reading the
//         dS^T tiles back, so S and dP are computed once, not twice.
// Accumulators (dV, dK, dQ) stay in TMEM in FP32 for the whole unit and are
// written once. P and dS enter their products as bf16 (round to nearest
// even); dK and dQ use the same bf16 dS. lse2 = lse * log2(e) and Delta = rowsum(dO * O) come from the
// backward preprocess in a tile-padded layout (one 128-slot block per query
// tile; slots past a segment hold lse2 = +inf and Delta = 0, so their P is
// exactly 0). Every wait is bounded (RLK_ERR_DEVICE_TIMEOUT on give-up).
#include <atomic>

#include "rlk_device.cuh"
#include "rlk_internal.h"
#include "rlk_normrope_bwd.cuh"
#include "rlk_sm100.cuh"
#include "rlk_tmap.h"


RLK_DEFINE_STRICT_PROBE(probe_bwd_tu)

namespace rlk {
namespace {

using namespace sm100;

// dK/dV warps 0-7: elementwise (warp w owns TMEM lane quarter w % 4 and the
// column half w / 4 of each row); warp 8: TMA producer; warps 9 and 10: MMA
// issuers of chains X and Y (warp 9 owns the TMEM allocation).
constexpr int kEwWarps = 8;                       // elementwise warps
constexpr int kEwThreads = 32 * kEwWarps;
constexpr int kBoxBytes = 128 * 128;       // 128 rows x 64 bf16
constexpr int kTileBytes = 2 * kBoxBytes;  // 128 rows x 128 bf16
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr float kC = (float)(1.4426950408889634 * 0.08838834764831845);  // log2(e) / sqrt(128)
constexpr float kScale = 0.08838834764831845f;                          // 1 / sqrt(128)
constexpr uint32_t kIdescKK = idesc_bf16(128, 128, false, false);
constexpr uint32_t kIdescKM = idesc_bf16(128, 128, false, true);

__device__ int g_status_bwd;

struct BwdArgs {
    CUtensorMap map_q;    // qh [B*H*S, 128]
    CUtensorMap map_k;    // kh [B*H*S, 128]
    CUtensorMap map_v[2];   // v per segment (0 text, 1 image), 4-D (d, h, token, b)
    CUtensorMap map_do[2];  // dO per segment
    Geom g;
    ValidLen vl;
    const float* lse2_p;  // [B, H, nq_pad]
    const float* delta_p; // [B, H, nq_pad]
    SegBf16 dv;           // [B, S, H, 128] (text rows, image rows)
    uint8_t* ds_tiles;    // [n_pairs, nq, nq] images of 32 KB (query tile major)
    // the (sample, head) pairs of this launch: bh0 .. bh0 + n_pairs - 1 in
    // b * H + h order; the images are indexed from bh0
    int bh0, n_pairs;
    // output maps per segment (0 text, 1 image) so a tile's rows past its
    // segment are clipped: dV [B, S, H, 128] bf16, dk^ [B*H, S, 128] fp32
    CUtensorMap map_dv[2];
    CUtensorMap map_dk[2];
    float* dkh;  // dk^ = dK of the rotated, normalised keys / sqrt(128), fp32 [B, H, S, 128]
    // the RoPE / RMSNorm backward of the query rows in the dQ epilogue:
    // input q (bf16 [B, S, H, 128]), its RMSNorm factors rq [B, H, S], the
    // gains (q_txt, k_txt, q_img, k_img), the cos/sin table; outputs dQ and
    // the q gain-gradient partials of every (b, h, 128-token tile, 32-row
    // quarter) in dgt [B, H, 2 (q, k), n_tiles, 4, 128]
    SegBf16 q_in, dq_out;
    const float* rq;
    const float* gains[4];
    const float2* tab;
    float* dgt;
};

__device__ __forceinline__ void fail(volatile int* abort_flag) {
    *abort_flag = 1;
    atomicOr(&g_status_bwd, 1);
}

// K-major operand (rows x 128 bf16 as two 64-column boxes), k-step kk of 16
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t tile, int kk) {
    return sdesc_sw128(tile + (kk >> 2) * kBoxBytes + (kk & 3) * 32, 16, 1024);
}
// MN-major operand: the same tile read with its rows as the K dimension
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t tile, int kk) {
    return sdesc_sw128(tile + kk * 2048, kBoxBytes, 1024);
}

// 16-byte store of dS^T image data that skips L1 (the dQ kernel reads it
// back through L2).
__device__ __forceinline__ void st_image(uint8_t* p, uint4 v) {
    asm volatile("st.global.L1::no_allocate.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

// dS^T tile image (128 keys x 128 queries, bf16, 32 KB): the non-swizzled
// MN-major operand layout of the tensor cores. Query chunk C (8 queries) is
// a 2 KB block of 128 key rows of 16 bytes, so 8 consecutive keys of one
// chunk form one 128-byte core matrix; chunks along MN are 2 KB apart,
// 8-key groups along K 128 bytes apart.
constexpr int kDsChunkBytes = 2048;
__device__ __forceinline__ int ds_image_offset(int query, int key) {
    return (query >> 3) * kDsChunkBytes + key * 16 + (query & 7) * 2;
}
__device__ __forceinline__ uint64_t desc_ds_image(uint32_t tile, int kk) {
    return sdesc_noswizzle(tile + kk * 2 * 128, 128, kDsChunkBytes);
}

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, kWaitLimitNs));
}

// Query tile i (segment aligned): first token and end of its segment.
__device__ __forceinline__ void q_tile(const Geom& g, int i, int& q0, int& q_end) {
    if (i < g.ntq_txt) {
        q0 = i * 128;
        q_end = g.T_txt;
    } else {
        q0 = g.T_txt + (i - g.ntq_txt) * 128;
        q_end = g.S;
    }
}

// ====================================================================== dK, dV
// TMEM: dV [0, 128), dK [128, 256) and two 128-column regions R_0, R_1 at 256
// and 384, used by query tiles alternately (tile i in R_{i & 1}). In its
// region a tile's S^T lands first; once the elementwise warps have read it,
// dP^T is computed into the same columns; the warps then write the bf16 P^T
// and dS^T there (each warp into the columns its own dP^T came from), and
// dV and dK take them as their A operands. Two issuing threads on different
// SMSPs (so neither SMSP's elementwise warps carry all the issue work):
//   chain Y: S^T_0, S^T_1, dP^T_0; per tile i: dP^T_{i+1} (once the warps
//            have read S^T_{i+1}), then S^T_{i+2} into R_{i & 1} (once
//            chain X reports dV_i and dK_i complete there);
//   chain X: per tile i: dV_i once the warps have written P^T_i (before they
//            form dS^T_i), dK_i once dS^T_i is written, then a commit that
//            frees R_{i & 1}.
// So the next tile's scores are ready before its warps need them, and the
// warps form P^T_{i+1} while dV_i, dK_i and dP^T_{i+1} run.
// Shared memory: K, V, three Q slots (Q_i is still read by dK_i when
// S^T_{i+2} needs Q_{i+2}) and two dO slots, each with its tile's lse2 and
// Delta; no static shared memory (the barriers sit in the alignment slack
// or after the tiles). A slot frees on chain X's commit: every product
// reading it has been issued by then, the S^T and dP^T ones completed
// before the warps formed that tile's P^T and dS^T.
// Warps 0-7 (elementwise) and 8-11 (TMA producer, the two issuers, one idle
// warp) are three warpgroups launched at 168 registers a thread; the helper
// warpgroup drops to 56 and the elementwise ones rise to 224 (setmaxnreg), so
// the warps on the critical path run without spills (705 -> 660 us).
constexpr int kKvWarps = kEwWarps + 4;  // + TMA producer, two MMA issuers, one idle warp (a full warpgroup)
constexpr int kKvThreads = 32 * kKvWarps;
// registers per thread at launch, and after the split (helper warpgroup, elementwise warpgroups)
constexpr int kKvRegs = 168, kKvRegsHelper = 56, kKvRegsEw = 224;
constexpr int kKvWarpTma = kEwWarps, kKvWarpMma = kEwWarps + 1, kKvWarpMma2 = kEwWarps + 2;
constexpr int kKvQSlots = 3, kKvOSlots = 2;
constexpr int kKvSmemK = 0, kKvSmemV = kTileBytes, kKvSmemQ = 2 * kTileBytes;
constexpr int kKvSmemO = kKvSmemQ + kKvQSlots * kTileBytes;
constexpr int kKvSmemL = kKvSmemO + kKvOSlots * kTileBytes;   // lse2[128], delta[128] per dO slot
constexpr int kKvSmemBar = kKvSmemL + kKvOSlots * 1024;
constexpr int kKvBarBytes = 256;
constexpr uint32_t kProducerSleepNs = 512;
constexpr int kKvSmemBytes = kKvSmemBar + 1024;  // + alignment slack (holds the barriers when it can)
static_assert(kKvSmemBytes <= 232448, "dK/dV shared memory exceeds the per-block limit");
constexpr uint32_t kColDV = 0, kColDK = 128, kColR = 256;
constexpr int kEwCols = 128 / (kEwWarps / 4);  // query / output columns per elementwise warp
// bf16 A operand of k-step kk (queries 16 kk .. 16 kk + 15) in a region:
// warp group g = kk / 4 owns fp32 columns [64 g, 64 g + 64) and rewrites
// them as 32 packed P^T columns, then 32 packed dS^T columns
__device__ __forceinline__ uint32_t p_col(int kk) { return 64u * (kk >> 2) + 8u * (kk & 3); }
__device__ __forceinline__ uint32_t ds_col(int kk) { return 64u * (kk >> 2) + 32u + 8u * (kk & 3); }

__global__ void __launch_bounds__(kKvThreads, 1) attn_bwd_dkdv_tc_kernel(const __grid_constant__ BwdArgs a) {
    extern __shared__ uint8_t smem_raw[];

    const Geom& g = a.g;
    const int kt = blockIdx.x, pair = blockIdx.y;  // pair: within this launch's range
    const int h = (a.bh0 + pair) % g.H, b = (a.bh0 + pair) / g.H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool k_txt = kt < g.ntq_txt;
    const int k0 = k_txt ? kt * 128 : g.T_txt + (kt - g.ntq_txt) * 128;
    const int seg_end = k_txt ? g.T_txt : g.S;
    const int L = a.vl.L[b];
    const int kvalid_end = k_txt ? L : g.S;
    const size_t bh = (size_t)b * g.H + h;
    const int row_base = (int)(bh * g.S);
    const int nq = g.ntq_txt + g.ntq_img;

    float* dkh = a.dkh + bh * g.S * kHeadDim;

    if (k0 >= kvalid_end) {  // every key of the tile is masked: exact zeros
        const int rows = min(128, seg_end - k0);
        for (int i = tid; i < rows * 16; i += kKvThreads) {
            const int r = i >> 4, c = i & 15;
            *reinterpret_cast<uint4*>(seg_row(a.dv, g, b, k0 + r, h) + c * 8) = make_uint4(0, 0, 0, 0);
            float4* dst = reinterpret_cast<float4*>(dkh + (size_t)(k0 + r) * kHeadDim + c * 8);
            dst[0] = make_float4(0.f, 0.f, 0.f, 0.f);
            dst[1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        return;
    }

    const uint32_t sraw = smem_u32(smem_raw);
    const uint32_t sbase = (sraw + 1023u) & ~1023u;
    // barriers: in the slack below the tiles when it is large enough, else
    // after the lse2 / Delta slots (the request covers either case)
    const uint32_t sbar = (sbase - sraw >= (uint32_t)kKvBarBytes) ? sraw : sbase + kKvSmemBar;
    uint8_t* const bar_gen = smem_raw + (sbar - sraw);
    volatile int& abort_flag = *reinterpret_cast<volatile int*>(bar_gen + 240);
    uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(bar_gen + 244);
    const uint32_t sK = sbase + kKvSmemK, sV = sbase + kKvSmemV;
    auto slot_q = [&](int i) { return sbase + kKvSmemQ + (uint32_t)(i % kKvQSlots) * kTileBytes; };
    auto slot_o = [&](int i) { return sbase + kKvSmemO + (uint32_t)(i & 1) * kTileBytes; };
    auto slot_l = [&](int i) { return sbase + kKvSmemL + (uint32_t)(i & 1) * 1024u; };
    const uint32_t bar_kv = sbar;
    const uint32_t bar_qf = sbar + 8;        // [3] Q slot landed
    const uint32_t bar_qe = sbar + 32;       // [3] Q slot read by every product
    const uint32_t bar_of = sbar + 56;       // [2] dO slot (+ lse2, Delta) landed
    const uint32_t bar_oe = sbar + 72;       // [2] dO slot free
    const uint32_t bar_st = sbar + 88;       // [2] S^T of the region's tile computed
    const uint32_t bar_sr = sbar + 104;      // [2] S^T read by the warps (kEwThreads arrivals)
    const uint32_t bar_dp = sbar + 120;      // [2] dP^T computed
    const uint32_t bar_pds = sbar + 136;     // [2] P^T and dS^T written (kEwThreads arrivals)
    const uint32_t bar_done = sbar + 152;
    const uint32_t bar_drain = sbar + 160;   // [2]
    const uint32_t bar_rf = sbar + 176;      // [2] region consumed by dV and dK
    const uint32_t bar_pt = sbar + 192;      // [2] P^T written (kEwThreads arrivals)

    if (tid == 0) {
        abort_flag = 0;
        mbar_init(bar_kv, 1);
        for (int j = 0; j < kKvQSlots; ++j) {
            mbar_init(bar_qf + 8 * j, 1);
            mbar_init(bar_qe + 8 * j, 1);
        }
        for (int j = 0; j < 2; ++j) {
            mbar_init(bar_of + 8 * j, 1);
            mbar_init(bar_oe + 8 * j, 1);
            mbar_init(bar_st + 8 * j, 1);
            mbar_init(bar_sr + 8 * j, kEwThreads);
            mbar_init(bar_dp + 8 * j, 1);
            mbar_init(bar_pds + 8 * j, kEwThreads);
            mbar_init(bar_pt + 8 * j, kEwThreads);
        }
        mbar_init(bar_done, 1);
        mbar_init(bar_drain, 1);
        mbar_init(bar_drain + 8, 1);
        mbar_init(bar_rf, 1);
        mbar_init(bar_rf + 8, 1);
        fence_barrier_init();
    }
    if (warp == kKvWarpMma) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // Register split: the helper warpgroup gives registers up and the two
    // elementwise warpgroups take them, from the launch's own allotment
    // (the host launches only when the kernel was built at kKvRegs).
    static_assert(32 * (kKvWarps - kEwWarps) * kKvRegsHelper + 32 * kEwWarps * kKvRegsEw == kKvThreads * kKvRegs,
                  "register split must equal the launch allotment");
    if (warp >= kEwWarps) {
        setmaxnreg_dec<kKvRegsHelper>();
        if (warp == kKvWarpTma) {
            // ------------------------------------------------ TMA producer
            // In order: K, V; then per query tile i its Q slot (free once dK_{i-3}
            // has run) and its dO slot with lse2 and Delta (free once dV_{i-2}
            // has run, which follows the warps' last read of that tile).
            if (lane == 0) {
                prefetch_tensormap(&a.map_q);
                prefetch_tensormap(&a.map_k);
                prefetch_tensormap(&a.map_v[0]);
                prefetch_tensormap(&a.map_v[1]);
                prefetch_tensormap(&a.map_do[0]);
                prefetch_tensormap(&a.map_do[1]);
                mbar_expect_tx(bar_kv, 2 * kTileBytes);
                tma_load_2d(sK, &a.map_k, bar_kv, 0, row_base + k0);
                tma_load_2d(sK + kBoxBytes, &a.map_k, bar_kv, 64, row_base + k0);
                // tiles never straddle the streams: rows counted from the segment start
                const int vseg = k_txt ? 0 : 1, vrow = k_txt ? k0 : k0 - g.T_txt;
                tma_load_4d(sV, &a.map_v[vseg], bar_kv, 0, h, vrow, b);
                tma_load_4d(sV + kBoxBytes, &a.map_v[vseg], bar_kv, 64, h, vrow, b);
                int issued = 0;
                for (int i = 0; i < nq && !abort_flag; ++i) {
                    const int jq = i % kKvQSlots, jo = i & 1;
                    int q0, q_end;
                    q_tile(g, i, q0, q_end);
                    // the copies run ahead of the products: their waits back off
                    // (512 ns per failed poll) to leave SMSP 0's issue slots to
                    // the elementwise warps there (708.5 against 711 us)
                    if (i >= kKvQSlots && !mbar_wait_backoff(bar_qe + 8 * jq, ((i / kKvQSlots) + 1) & 1, &abort_flag,
                                                             kWaitLimitNs, kProducerSleepNs)) {
                        fail(&abort_flag);
                        break;
                    }
                    const uint32_t bq = bar_qf + 8 * jq;
                    mbar_expect_tx(bq, kTileBytes);
                    tma_load_2d(slot_q(i), &a.map_q, bq, 0, row_base + q0);
                    tma_load_2d(slot_q(i) + kBoxBytes, &a.map_q, bq, 64, row_base + q0);
                    if (i >= 2 && !mbar_wait_backoff(bar_oe + 8 * jo, ((i >> 1) + 1) & 1, &abort_flag, kWaitLimitNs,
                                                     kProducerSleepNs)) {
                        fail(&abort_flag);
                        break;
                    }
                    const uint32_t bo = bar_of + 8 * jo;
                    mbar_expect_tx(bo, kTileBytes + 1024);
                    const int oseg = i < g.ntq_txt ? 0 : 1, orow = oseg ? q0 - g.T_txt : q0;
                    tma_load_4d(slot_o(i), &a.map_do[oseg], bo, 0, h, orow, b);
                    tma_load_4d(slot_o(i) + kBoxBytes, &a.map_do[oseg], bo, 64, h, orow, b);
                    const size_t slot = bh * g.nq_pad + (size_t)i * 128;
                    bulk_load(slot_l(i), a.lse2_p + slot, 512, bo);
                    bulk_load(slot_l(i) + 512, a.delta_p + slot, 512, bo);
                    issued = i + 1;
                }
                // leave no copy in flight
                const volatile int no_abort = 0;
                mbar_wait(bar_kv, 0, &no_abort, kWaitLimitNs);
                for (int i = issued - kKvQSlots < 0 ? 0 : issued - kKvQSlots; i < issued; ++i)
                    mbar_wait(bar_qf + 8 * (i % kKvQSlots), (i / kKvQSlots) & 1, &no_abort, kWaitLimitNs);
                for (int i = issued - 2 < 0 ? 0 : issued - 2; i < issued; ++i)
                    mbar_wait(bar_of + 8 * (i & 1), (i >> 1) & 1, &no_abort, kWaitLimitNs);
            }
        } else if (warp == kKvWarpMma || warp == kKvWarpMma2) {
            // ------------------------------------------------ MMA issuers (chains X, Y)
            if (lane == 0) {
                const bool chain_y = warp == kKvWarpMma2;
                auto issue_scores = [&](int i, bool dp) {
                    const uint32_t at = dp ? sV : sK, bt = dp ? slot_o(i) : slot_q(i);
                    const uint32_t d = tmem + kColR + 128u * (uint32_t)(i & 1);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_ss(d, desc_kmajor(at, kk), desc_kmajor(bt, kk), kIdescKK, kk > 0);
                    mma_commit((dp ? bar_dp : bar_st) + 8 * (i & 1));
                };
                bool ok = mbar_wait(bar_kv, 0, &abort_flag, kWaitLimitNs);
                if (chain_y) {
                    ok = ok && mbar_wait(bar_qf, 0, &abort_flag, kWaitLimitNs);
                    if (ok) {
                        tc_fence_after();
                        issue_scores(0, false);
                    }
                    if (ok && nq > 1) {
                        ok = mbar_wait(bar_qf + 8, 0, &abort_flag, kWaitLimitNs);
                        if (ok) {
                            tc_fence_after();
                            issue_scores(1, false);
                        }
                    }
                    ok = ok && mbar_wait(bar_sr, 0, &abort_flag, kWaitLimitNs) &&
                         mbar_wait(bar_of, 0, &abort_flag, kWaitLimitNs);
                    if (ok) {
                        tc_fence_after();
                        issue_scores(0, true);
                    }
                    for (int i = 0; ok && i < nq; ++i) {
                        const int r = i & 1;
                        if (i + 1 < nq) {
                            if (!mbar_wait(bar_sr + 8 * (r ^ 1), ((i + 1) >> 1) & 1, &abort_flag, kWaitLimitNs) ||
                                !mbar_wait(bar_of + 8 * ((i + 1) & 1), ((i + 1) >> 1) & 1, &abort_flag, kWaitLimitNs)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            issue_scores(i + 1, true);
                        }
                        if (i + 2 < nq) {
                            if (!mbar_wait(bar_rf + 8 * r, (i >> 1) & 1, &abort_flag, kWaitLimitNs) ||
                                !mbar_wait(bar_qf + 8 * ((i + 2) % kKvQSlots), ((i + 2) / kKvQSlots) & 1, &abort_flag,
                                           kWaitLimitNs)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            issue_scores(i + 2, false);
                        }
                    }
                } else {
                    for (int i = 0; ok && i < nq; ++i) {
                        const int r = i & 1;
                        const uint32_t reg = tmem + kColR + 128u * (uint32_t)r;
                        // dV_i once P^T_i is written, dK_i once dS^T_i is
                        if (!mbar_wait(bar_pt + 8 * r, (i >> 1) & 1, &abort_flag, kWaitLimitNs)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            mma_ts(tmem + kColDV, reg + p_col(kk), desc_mnmajor(slot_o(i), kk), kIdescKM,
                                   (i > 0 || kk > 0) ? 1u : 0u);
                        mma_commit(bar_oe + 8 * (i & 1));
                        if (!mbar_wait(bar_pds + 8 * r, (i >> 1) & 1, &abort_flag, kWaitLimitNs)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            mma_ts(tmem + kColDK, reg + ds_col(kk), desc_mnmajor(slot_q(i), kk), kIdescKM,
                                   (i > 0 || kk > 0) ? 1u : 0u);
                        mma_commit(bar_qe + 8 * (i % kKvQSlots));
                        mma_commit(bar_rf + 8 * r);
                    }
                    if (ok) mma_commit(bar_done);
                }
                if (!ok) fail(&abort_flag);
                const uint32_t my_drain = bar_drain + (chain_y ? 8 : 0);
                mma_commit(my_drain);
                mbar_wait_drain(my_drain, 0, kWaitLimitNs);
            }
        }
    } else {
        setmaxnreg_inc<kKvRegsEw>();
        // ------------------------------------------------ elementwise warps
        // warp w: key rows 32 * (w % 4) + lane, query columns
        // [kEwCols * grp, kEwCols * (grp + 1)), grp = w / 4. No row
        // reduction: every element of P^T and dS^T is the thread's own.
        const int lq = warp & 3, grp = warp >> 2;
        const uint32_t lane_addr = (uint32_t)(lq * 32) << 16;
        const int kr = lq * 32 + lane;
        const int c0 = kEwCols * grp;
        const bool kvalid = k0 + kr < kvalid_end;
        bool ok = true;
        uint32_t pkd[kEwCols / 2];  // dS^T of the previous tile, packed, for its image
        uint8_t* ds_prev = nullptr;
        for (int i = 0; i < nq; ++i) {
            const int r = i & 1;
            const uint32_t reg = tmem + lane_addr + kColR + 128u * (uint32_t)r + c0;
            if (!warp_wait(bar_st + 8 * r, (i >> 1) & 1, &abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t rs[kEwCols];
#pragma unroll
            for (int c = 0; c < kEwCols; c += 32)
                tmem_ld32(reg + c, *reinterpret_cast<uint32_t(*)[32]>(&rs[c]));
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive(bar_sr + 8 * r);
            if (!warp_wait(bar_of + 8 * (i & 1), (i >> 1) & 1, &abort_flag)) {
                ok = false;
                break;
            }
            const float4* l2v = reinterpret_cast<const float4*>(smem_raw + (slot_l(i) - sraw)) + c0 / 4;
            const float4* dlv = l2v + 32;
            // P^T = exp2(S^T * c - lse2[query]) (masked keys: 0), kept in fp32 for dS
            float pf[kEwCols];
            if (kvalid) {  // the row's key is valid for the whole CTA: no per-element select
#pragma unroll
                for (int e4 = 0; e4 < kEwCols / 4; ++e4) {
                    const float4 l4 = l2v[e4];
                    const float lq4[4] = {l4.x, l4.y, l4.z, l4.w};
                    float x[4];
                    f2_unpack(fma_f2(f2_pack(__uint_as_float(rs[4 * e4]), __uint_as_float(rs[4 * e4 + 1])),
                                     f2_pack(kC, kC), f2_pack(-lq4[0], -lq4[1])), x[0], x[1]);
                    f2_unpack(fma_f2(f2_pack(__uint_as_float(rs[4 * e4 + 2]), __uint_as_float(rs[4 * e4 + 3])),
                                     f2_pack(kC, kC), f2_pack(-lq4[2], -lq4[3])), x[2], x[3]);
#pragma unroll
                    for (int u = 0; u < 4; ++u) pf[4 * e4 + u] = exp2_num(x[u]);
                }
            } else {  // a masked key: P = 0
#pragma unroll
                for (int e = 0; e < kEwCols; ++e) pf[e] = 0.0f;
            }
            // the previous tile's bf16 dS^T into its (query tile, key tile kt)
            // image for the dQ product (see ds_image_offset), while dP^T_i
            // computes: a warp's store of one query chunk covers 512
            // contiguous bytes
            if (ds_prev != nullptr) {
#pragma unroll
                for (int c = 0; c < kEwCols / 8; ++c)
                    st_image(ds_prev + c * kDsChunkBytes, make_uint4(pkd[4 * c], pkd[4 * c + 1], pkd[4 * c + 2], pkd[4 * c + 3]));
            }
            // dS^T = P^T * (dP^T - Delta[query])
            if (!warp_wait(bar_dp + 8 * r, (i >> 1) & 1, &abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // two chunks of 32 columns; once a chunk's dP^T is in registers its
            // columns take the packed P^T (chunk 0) or dS^T (chunk 1)
#pragma unroll
            for (int c = 0; c < kEwCols; c += 32) {
                uint32_t rd[32];
                tmem_ld32(reg + c, rd);
                tmem_ld_wait();
                if (c == 0) {
                    uint32_t pkp[kEwCols / 2];
#pragma unroll
                    for (int e = 0; e < kEwCols / 2; ++e) pkp[e] = pack_bf16(pf[2 * e], pf[2 * e + 1]);
                    tmem_st32(reg, *reinterpret_cast<const uint32_t(*)[32]>(&pkp[0]));
                    tmem_st_wait();
                    tc_fence_before();
                    mbar_arrive(bar_pt + 8 * r);
                }
#pragma unroll
                for (int e4 = 0; e4 < 8; ++e4) {
                    const float4 d4 = dlv[c / 4 + e4];
                    const float dq4[4] = {d4.x, d4.y, d4.z, d4.w};
                    float ds[4];
#pragma unroll
                    for (int u = 0; u < 4; u += 2)
                        f2_unpack(mul_f2(f2_pack(pf[c + 4 * e4 + u], pf[c + 4 * e4 + u + 1]),
                                         sub_f2(f2_pack(__uint_as_float(rd[4 * e4 + u]), __uint_as_float(rd[4 * e4 + u + 1])),
                                                f2_pack(dq4[u], dq4[u + 1]))),
                                  ds[u], ds[u + 1]);
                    pkd[c / 2 + 2 * e4] = pack_bf16(ds[0], ds[1]);
                    pkd[c / 2 + 2 * e4 + 1] = pack_bf16(ds[2], ds[3]);
                }
            }
            tmem_st32(reg + 32, *reinterpret_cast<const uint32_t(*)[32]>(&pkd[0]));
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bar_pds + 8 * r);
            ds_prev = a.ds_tiles + (((size_t)pair * nq + i) * nq + kt) * (size_t)kTileBytes + ds_image_offset(c0, kr);
        }
        if (ok && ds_prev != nullptr) {
#pragma unroll
            for (int c = 0; c < kEwCols / 8; ++c)
                st_image(ds_prev + c * kDsChunkBytes, make_uint4(pkd[4 * c], pkd[4 * c + 1], pkd[4 * c + 2], pkd[4 * c + 3]));
        }
        if (ok && warp_wait(bar_done, 0, &abort_flag)) {
            tc_fence_after();
            // Stage dV (bf16) and dK (fp32, times 1/sqrt(D)) in the K, V and
            // first Q slots (every product has finished) as six 128-row x
            // 128-byte boxes in the 128-byte-swizzled layout of the output
            // maps: dV boxes 0-1 (64 columns each), dK boxes 2-5 (32 columns
            // each). One thread then stores the tile with TMA; the segment
            // maps clip rows past the key's segment. Masked keys get zeros.
            uint8_t* stg = smem_raw + (sbase - sraw);
            const int sw = kr & 7;
#pragma unroll 1
            for (int c = 0; c < kEwCols; c += 32) {
                uint32_t rr[32];
                tmem_ld32(tmem + lane_addr + kColDV + c0 + c, rr);
                tmem_ld_wait();
                // dV box (c0 + c) / 64, 16-byte chunks from ((c0 + c) % 64) / 8
                uint8_t* dvrow = stg + ((c0 + c) >> 6) * kBoxBytes + kr * 128;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        w[e] = kvalid ? pack_bf16(__uint_as_float(rr[8 * q + 2 * e]), __uint_as_float(rr[8 * q + 2 * e + 1]))
                                      : 0u;
                    *reinterpret_cast<uint4*>(dvrow + (((((c0 + c) & 63) >> 3) + q) ^ sw) * 16) =
                        make_uint4(w[0], w[1], w[2], w[3]);
                }
                tmem_ld32(tmem + lane_addr + kColDK + c0 + c, rr);
                tmem_ld_wait();
                uint8_t* dkrow = stg + (2 + ((c0 + c) >> 5)) * kBoxBytes + kr * 128;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    float4 f;
                    f.x = kvalid ? __uint_as_float(rr[4 * q]) * kScale : 0.0f;
                    f.y = kvalid ? __uint_as_float(rr[4 * q + 1]) * kScale : 0.0f;
                    f.z = kvalid ? __uint_as_float(rr[4 * q + 2]) * kScale : 0.0f;
                    f.w = kvalid ? __uint_as_float(rr[4 * q + 3]) * kScale : 0.0f;
                    *reinterpret_cast<float4*>(dkrow + ((q ^ sw) << 4)) = f;
                }
            }
            fence_proxy_async_smem();
            named_barrier_sync(1, kEwThreads);
            if (tid == 0) {
                const int seg = k_txt ? 0 : 1;
                const int srow = k_txt ? k0 : k0 - g.T_txt;
                tma_store_4d(&a.map_dv[seg], sbase, 0, h, srow, b);
                tma_store_4d(&a.map_dv[seg], sbase + kBoxBytes, 64, h, srow, b);
#pragma unroll
                for (int q = 0; q < 4; ++q) tma_store_3d(&a.map_dk[seg], sbase + (2 + q) * kBoxBytes, 32 * q, srow, (int)bh);
                bulk_commit_group();
                bulk_wait_read_all();
            }
        } else {
            fail(&abort_flag);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kKvWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ====================================================================== dQ
// dQ_i = sum_j dS_ij K_j as a streaming tcgen05 GEMM over the bf16 dS^T
// images the dK/dV kernel wrote (one 32 KB image per (query tile, key tile)
// pair, query tile major, in the tensor cores' non-swizzled operand layout,
// so one bulk copy stages it and it enters the product as an MN-major A). Persistent: CTA c takes the units (query tile, head, sample)
// c, c + grid, ... in order; a unit sums its key tiles in the forward's
// order into one of two TMEM accumulators, so the epilogue of one unit
// overlaps the products of the next. No unit depends on which CTA runs it.
constexpr int kDqThreads = 192;  // warps 0-3 epilogue, 4 copies, 5 MMA
constexpr int kDqWarpTma = 4, kDqWarpMma = 5;
constexpr int kDqStages = 3;
constexpr int kDqStageBytes = 2 * kTileBytes;  // dS^T image, K tile
constexpr int kDqSmemBytes = kDqStages * kDqStageBytes + 1024;
constexpr uint32_t kDqTmemCols = 256;
constexpr uint32_t kIdescMM = idesc_bf16(128, 128, true, true);

struct DqUnit {
    int qt, h, b, pair;  // pair: within the launch's range (indexes the images)
};
// Units run from the last (sample, head) of the range down: the dK/dV
// kernel's last CTAs wrote those dS^T images, some still in L2 (317.0 ->
// 313.6 us measured).
__device__ __forceinline__ DqUnit dq_unit(const BwdArgs& a, int nq, int u) {
    DqUnit r;
    u = nq * a.n_pairs - 1 - u;
    r.qt = u % nq;
    r.pair = u / nq;
    r.h = (a.bh0 + r.pair) % a.g.H;
    r.b = (a.bh0 + r.pair) / a.g.H;
    return r;
}

__global__ void __launch_bounds__(kDqThreads, 1) attn_bwd_dq_tc_kernel(const __grid_constant__ BwdArgs a) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bars[2 * kDqStages + 5];
    __shared__ uint32_t tmem_slot;
    __shared__ volatile int abort_flag;

    const Geom& g = a.g;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nq = g.ntq_txt + g.ntq_img;
    const int n_units = nq * a.n_pairs;
    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    auto stage = [&](int s) { return sbase + s * kDqStageBytes; };
    const uint32_t bar_full = smem_u32(&bars[0]);                   // [3] stage loaded
    const uint32_t bar_empty = smem_u32(&bars[kDqStages]);          // [3] stage consumed
    const uint32_t bar_acc = smem_u32(&bars[2 * kDqStages]);        // [2] accumulator complete
    const uint32_t bar_free = smem_u32(&bars[2 * kDqStages + 2]);   // [2] accumulator read out
    const uint32_t bar_drain = smem_u32(&bars[2 * kDqStages + 4]);

    if (tid == 0) {
        abort_flag = 0;
        for (int s = 0; s < kDqStages; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar_acc + 8 * s, 1);
            mbar_init(bar_free + 8 * s, 128);
        }
        mbar_init(bar_drain, 1);
        fence_barrier_init();
    }
    if (warp == kDqWarpMma) {
        tmem_alloc(smem_u32(&tmem_slot), kDqTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    if (warp == kDqWarpTma) {
        // ------------------------------------------------ copies
        if (lane == 0) {
            prefetch_tensormap(&a.map_k);
            int t = 0;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < n_units && !abort_flag; u += gridDim.x) {
                const DqUnit w = dq_unit(a, nq, u);
                const int L = a.vl.L[w.b];
                const int nkt_txt = (L + 127) / 128;
                const int nkt = nkt_txt + g.ntq_img;
                const size_t bh = (size_t)w.b * g.H + w.h;
                const int row_base = (int)(bh * g.S);
                const uint8_t* tiles = a.ds_tiles + ((size_t)w.pair * nq + w.qt) * nq * (size_t)kTileBytes;
                for (int j = 0; j < nkt; ++j, ++t) {
                    const int s = t % kDqStages;
                    if (t >= kDqStages &&
                        !mbar_wait(bar_empty + 8 * s, ((t / kDqStages) + 1) & 1, &abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    const int kt = j < nkt_txt ? j : g.ntq_txt + (j - nkt_txt);
                    const int kk0 = j < nkt_txt ? j * 128 : g.T_txt + (j - nkt_txt) * 128;
                    const uint32_t bf = bar_full + 8 * s;
                    mbar_expect_tx(bf, kDqStageBytes);
                    bulk_load(stage(s), tiles + (size_t)kt * kTileBytes, kTileBytes, bf);
                    tma_load_2d(stage(s) + kTileBytes, &a.map_k, bf, 0, row_base + kk0);
                    tma_load_2d(stage(s) + kTileBytes + kBoxBytes, &a.map_k, bf, 64, row_base + kk0);
                }
            }
            if (!ok) fail(&abort_flag);
            const volatile int no_abort = 0;
            for (int tt = t - kDqStages < 0 ? 0 : t - kDqStages; tt < t; ++tt)
                mbar_wait(bar_full + 8 * (tt % kDqStages), (tt / kDqStages) & 1, &no_abort, kWaitLimitNs);
        }
    } else if (warp == kDqWarpMma) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            int t = 0, n = 0;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < n_units; u += gridDim.x, ++n) {
                const DqUnit w = dq_unit(a, nq, u);
                const int nkt = (a.vl.L[w.b] + 127) / 128 + g.ntq_img;
                const int buf = n & 1;
                if (n >= 2 && !mbar_wait(bar_free + 8 * buf, ((n >> 1) + 1) & 1, &abort_flag, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int j = 0; j < nkt; ++j, ++t) {
                    const int s = t % kDqStages;
                    if (!mbar_wait(bar_full + 8 * s, (t / kDqStages) & 1, &abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_ss(tmem + 128 * buf, desc_ds_image(stage(s), kk), desc_mnmajor(stage(s) + kTileBytes, kk),
                               kIdescMM, (j > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(bar_empty + 8 * s);
                }
                if (ok) mma_commit(bar_acc + 8 * buf);
            }
            if (!ok) fail(&abort_flag);
            mma_commit(bar_drain);
            const volatile int no_abort = 0;
            mbar_wait(bar_drain, 0, &no_abort, kWaitLimitNs);
        }
    } else {
        // ------------------------------------------------ epilogue warps 0-3: query row 32 w + lane
        // Per unit: the RoPE / RMSNorm backward of the tile's query rows
        // from dq^ = acc / sqrt(128) (TMEM): bf16 dQ rows and this warp's
        // partial of the tile's q gain gradient (its 32 rows summed by a
        // transposing butterfly), stored for the fold.
        const uint32_t lane_addr = (uint32_t)(warp * 32) << 16;
        const int r = warp * 32 + lane;
        int n = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++n) {
            const DqUnit w = dq_unit(a, nq, u);
            const int buf = n & 1;
            if (!warp_wait(bar_acc + 8 * buf, (n >> 1) & 1, &abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            int q0, q_end;
            q_tile(g, w.qt, q0, q_end);
            const bool row_ok = q0 + r < q_end;
            const int tok = row_ok ? q0 + r : q0;  // rows past the segment read a valid row, store nothing
            const size_t bh = (size_t)w.b * g.H + w.h;
            const uint32_t acc_addr = tmem + lane_addr + 128 * buf;
            auto dq_chunk = [&](int c, float (&dy)[32]) {
                uint32_t acc[32];
                tmem_ld32(acc_addr + 32 * c, acc);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) dy[i] = row_ok ? __uint_as_float(acc[i]) * kScale : 0.0f;
            };
            nrb_row(dq_chunk, row_ok, reinterpret_cast<const uint4*>(seg_row(a.q_in, g, w.b, tok, w.h)),
                    a.rq[bh * g.S + tok], w.qt < g.ntq_txt ? a.gains[0] : a.gains[2], tab_rows(a.tab, g, tok),
                    reinterpret_cast<uint4*>(seg_row(a.dq_out, g, w.b, tok, w.h)),
                    a.dgt + ((bh * 2 * nq + w.qt) * 4 + warp) * kHeadDim, lane);
            tc_fence_before();
            mbar_arrive(bar_free + 8 * buf);
        }
        if (!ok) fail(&abort_flag);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kDqWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, kDqTmemCols);
    }
}

// ---------------------------------------------------------------- tensor maps
bool make_args(BwdArgs* a, const Geom& g, const ValidLen& vl, const uint16_t* qh, const uint16_t* kh,
               const SegBf16& v, const SegBf16& dout, const float* lse2_p, const float* delta_p) {
    const uint64_t rows = (uint64_t)g.B * g.H * g.S;
    if (!tmap::rows_bf16(&a->map_q, qh, rows) || !tmap::rows_bf16(&a->map_k, kh, rows))
        return false;
    for (int seg = 0; seg < 2; ++seg)
        if (!tmap::seg_bf16(&a->map_v[seg], v, g, seg) || !tmap::seg_bf16(&a->map_do[seg], dout, g, seg))
            return false;
    a->g = g;
    a->vl = vl;
    a->lse2_p = lse2_p;
    a->delta_p = delta_p;
    a->dv = SegBf16{{nullptr, nullptr}, {0, 0}};
    a->dkh = nullptr;
    a->ds_tiles = nullptr;
    return true;
}

void set_norm_rope_io(BwdArgs* a, const NormRopeBwdIo& nr) {
    a->q_in = nr.q;
    a->dq_out = nr.dq;
    a->rq = nr.rq;
    for (int i = 0; i < 4; ++i) a->gains[i] = nr.gains[i];
    a->tab = nr.tab;
    a->dgt = nr.dgt;
}

}  // namespace

cudaError_t launch_attn_bwd_dkdv(const Geom& g, const ValidLen& vl, const uint16_t* qh, const uint16_t* kh,
                                 const SegBf16& v, const SegBf16& dout, const float* lse2_p, const float* delta_p,
                                 const SegBf16& dv, float* dkh, uint8_t* ds_tiles, int bh0, int n_pairs,
                                 cudaStream_t s) {
    BwdArgs args;
    if (!make_args(&args, g, vl, qh, kh, v, dout, lse2_p, delta_p)) return cudaErrorInvalidValue;
    if (bh0 < 0 || n_pairs < 1 || bh0 + n_pairs > g.B * g.H) return cudaErrorInvalidValue;
    args.bh0 = bh0;
    args.n_pairs = n_pairs;
    args.dv = dv;
    args.dkh = dkh;
    args.ds_tiles = ds_tiles;
    for (int seg = 0; seg < 2; ++seg)
        if (!tmap::seg_bf16(&args.map_dv[seg], dv, g, seg) || !tmap::bhsd_f32_segment(&args.map_dk[seg], dkh, g, seg))
            return cudaErrorInvalidValue;
    cudaError_t e =
        cudaFuncSetAttribute(attn_bwd_dkdv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kKvSmemBytes);
    if (e != cudaSuccess) return e;
    // the warpgroups' register split adds up to kKvRegs per launched thread:
    // a build at any other count would leave the elementwise warps waiting
    // for registers that are not there, so it is not launched
    // (a successful lookup is kept: every device runs the same build)
    static std::atomic<int> regs_at_launch{0};
    int regs = regs_at_launch.load(std::memory_order_relaxed);
    if (regs == 0) {
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, attn_bwd_dkdv_tc_kernel);
        if (e != cudaSuccess) return e;
        regs = fa.numRegs;
        regs_at_launch.store(regs, std::memory_order_relaxed);
    }
    if (regs != kKvRegs) return cudaErrorInvalidConfiguration;
    dim3 grid(g.ntq_txt + g.ntq_img, n_pairs);
    timing_begin(kKBwdDkDv, s);
    attn_bwd_dkdv_tc_kernel<<<grid, kKvThreads, kKvSmemBytes, s>>>(args);
    timing_end(kKBwdDkDv, s);
    return cudaGetLastError();
}

cudaError_t launch_attn_bwd_dq(const Geom& g, const ValidLen& vl, const uint16_t* kh, const uint8_t* ds_tiles,
                               const NormRopeBwdIo& nr, int bh0, int n_pairs, cudaStream_t s) {
    BwdArgs args;
    if (!tmap::rows_bf16(&args.map_k, kh, (uint64_t)g.B * g.H * g.S)) return cudaErrorInvalidValue;
    if (bh0 < 0 || n_pairs < 1 || bh0 + n_pairs > g.B * g.H) return cudaErrorInvalidValue;
    args.bh0 = bh0;
    args.n_pairs = n_pairs;
    args.g = g;
    args.vl = vl;
    args.ds_tiles = const_cast<uint8_t*>(ds_tiles);
    set_norm_rope_io(&args, nr);
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(attn_bwd_dq_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDqSmemBytes);
    if (e != cudaSuccess) return e;
    const int n_units = (g.ntq_txt + g.ntq_img) * n_pairs;
    const int grid = n_units < sms ? n_units : sms;
    timing_begin(kKBwdDq, s);
    attn_bwd_dq_tc_kernel<<<grid, kDqThreads, kDqSmemBytes, s>>>(args);
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

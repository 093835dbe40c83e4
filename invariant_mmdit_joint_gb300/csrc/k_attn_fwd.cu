// Joint attention forward on the 5th-generation tensor cores (tcgen05):
// rows joint_attn_qk_gemm, joint_attn_softmax and joint_attn_av_gemm of the
// RFC #386 WS1 table fused ("joint_attention_fused"), with an online
// softmax over key tiles.
//
// One CTA = two query tiles A and B of 128 rows (the same head, sample and
// stream segment) sharing every K/V tile; 18 warps:
//   warps 0-15 softmax, two threads per query row: warp w serves tile
//              (w >> 2) & 1, TMEM lane quarter w & 3 (rows 32 (w & 3) + lane)
//              and key half w >> 3 (S columns [64 (w >> 3), + 64)). Per key
//              tile a thread reads its half row of S from TMEM, the two
//              threads of a row trade their halves' maxima (and the previous
//              tile's half sums) through shared memory, keep a reference max
//              m and the sum l (FP32, log2 units), write P = exp2(s - m) as
//              bf16 back over S in two chunks (the half's first 32 keys,
//              then its last 32), each handed to the MMA once written, and
//              rescale their half of O in TMEM when m moves (only when the
//              row max has grown by more than 2^8) before the first chunk.
//              Epilogue: O / l, one bf16 cast, and lse.
//   warp 16    TMA producer: Q tiles once, then K and V tiles (two slots
//              each; a K slot frees when its S products are done, a V slot
//              when its PV products are done).
//   warp 17    MMA issuer (one thread) and TMEM owner, per key tile j:
//              PV_A(j) over key chunk 0 (k-steps 0, 1, 4, 5), then over key
//              chunk 1 (2, 3, 6, 7), S_A(j+1), and the same for tile B --
//              while one group runs its softmax the tensor core works for
//              the other.
// TMEM: S_A [0,128), O_A [128,256), S_B [256,384), O_B [384,512).
// A CTA runs tile A alone (group B idle) for a segment's odd last tile, and
// for the pairs past the grid's last full wave, which run as two single-tile
// CTAs so that the partial wave spreads over twice the SMs; a tile's bytes
// never depend on its partner.
// Query tiles are segment aligned (text from token 0, image from token
// T_txt); key tiles of 128 are visited in one fixed order (text tiles that
// hold a valid key, then image tiles), so a row's bytes never depend on B,
// its batch position, padding or the SM count. No split-KV, no atomics.
// Every wait is bounded; a wait that gives up records RLK_ERR_DEVICE_TIMEOUT
// in the status word and the CTA drains its copies and MMAs and exits.
#include <algorithm>
#include <atomic>

#include "rlk_device.cuh"
#include "rlk_internal.h"
#include "rlk_sm100.cuh"
#include "rlk_tmap.h"


RLK_DEFINE_STRICT_PROBE(probe_fwd_tu)

namespace rlk {

const int kFwdBlockQ = 128;
const int kFwdBlockKV = 128;

namespace {

using namespace sm100;

constexpr int kBM = 128, kBN = 128;
// warps 0-15 softmax (tile t = (w >> 2) & 1, key half (w >> 3), TMEM lane
// quarter w & 3: two threads per query row), 16 TMA, 17 MMA
constexpr int kSoftmaxWarps = 16;
constexpr int kThreads = 32 * (kSoftmaxWarps + 2);
constexpr int kWarpTma = kSoftmaxWarps, kWarpMma = kSoftmaxWarps + 1;
constexpr int kBoxBytes = 128 * 128;          // 128 rows x 64 bf16
constexpr int kTileBytes = 2 * kBoxBytes;     // 128 rows x 128 bf16
constexpr int kSmemQ = 0;                     // Q_A, Q_B
constexpr int kSmemK = 2 * kTileBytes;        // 2 slots
constexpr int kSmemV = 4 * kTileBytes;        // 2 slots
constexpr int kSmemBytes = 6 * kTileBytes + 1024;  // + alignment slack
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
// the producer's slot waits sleep this long per failed poll, leaving its
// SMSP's issue slots to the softmax warps (424.1 -> 422.7 us)
constexpr uint32_t kProducerSleepNs = 512;
constexpr float kC = (float)(1.4426950408889634 * 0.08838834764831845);  // log2(e) / sqrt(128)
constexpr float kLn2 = 0.6931471805599453f;

__device__ int g_status_fwd;

// Pairs split into single-tile CTAs beyond those of the partial last wave.
// At the 1024^2 CFG pair (816 pairs on 152 SMs) splitting the last wave's 56
// pairs gave 450 -> 442 us; 40 more changed nothing, 96 more cost 492 us.
constexpr int kFwdSplitExtra = 0;

// rlk_fwd_tile_schedule(): RLK_FWD_TILES_AUTO, _PAIRS or _SINGLE.
std::atomic<int> g_tile_policy{RLK_FWD_TILES_AUTO};

struct FwdArgs {
    CUtensorMap map_q;   // qh [B*H*S, 128] bf16, box 64 x 128
    CUtensorMap map_k;   // kh [B*H*S, 128]
    CUtensorMap map_v[2];  // v per segment (0 text, 1 image) as 4-D (d, h, token, b), box 64 x 1 x 128 x 1
    Geom g;
    ValidLen vl;
    float* lse;          // [B, H, S] or null
    CUtensorMap map_o[2];  // out per segment (0 text, 1 image): rows past a segment are clipped
    // key shard (kShard launches): column blocks [blk_begin, blk_end) of the
    // fused order, the online-softmax state handed in by the previous shard
    // (null for the first) and handed on to the next one (null for the
    // last, which writes out and lse instead). State per query row: m (log2
    // units) and l fp32 [B, H, S], O fp32 [B, H, S, 128] (not yet divided by l).
    int blk_begin, blk_end;
    // units of the 1-D grid: the pairs of query tiles, in the order pair,
    // head, sample; pairs below n_keep run as pairs, each later one as two
    // CTAs of one tile (filling what would be the last, partly empty wave)
    int npairs, n_keep;
    const float* st_in_m;
    const float* st_in_l;
    const float* st_in_o;
    float* st_out_m;
    float* st_out_l;
    float* st_out_o;
};

struct TileInfo {
    int k0, kend;
};
__device__ __forceinline__ TileInfo kv_tile(const Geom& g, int L, int nkt_txt, int j) {
    TileInfo t;
    if (j < nkt_txt) {
        t.k0 = j * kBN;
        t.kend = L;
    } else {
        t.k0 = g.T_txt + (j - nkt_txt) * kBN;
        t.kend = g.S;
    }
    return t;
}

__device__ __forceinline__ void fail(volatile int* abort_flag) {
    *abort_flag = 1;
    atomicOr(&g_status_fwd, 1);
}

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, kWaitLimitNs));
}

template <bool kShard>
__global__ void __launch_bounds__(kThreads, 1) attn_fwd_tc_kernel(const __grid_constant__ FwdArgs a) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bars[34];
    // the two threads of a query row trade their half's partial row max of
    // this key tile and their half's row sum of the previous one, through
    // slot j & 1 of (tile, half, row)
    __shared__ float2 xch[2][2][2][kBM];
    __shared__ uint32_t tmem_slot;
    __shared__ volatile int abort_flag;

    const Geom& g = a.g;
    const int u = blockIdx.x;
    const int pair = u < a.n_keep ? u : a.n_keep + ((u - a.n_keep) >> 1);
    const int part = u < a.n_keep ? -1 : ((u - a.n_keep) & 1);  // -1: both tiles, else tile 0 or 1 alone
    const int pt = pair % a.npairs, h = (pair / a.npairs) % g.H, b = pair / (a.npairs * g.H);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // the CTA's pair of query tiles (or one of them), inside one segment
    const int np_txt = (g.ntq_txt + 1) / 2;
    const bool q_txt = pt < np_txt;
    const int first = (q_txt ? 2 * pt : 2 * (pt - np_txt)) + (part == 1 ? 1 : 0);  // tile index inside the segment
    const int seg_tiles = q_txt ? g.ntq_txt : g.ntq_img;
    if (first >= seg_tiles) return;  // the second tile of a pair that has only one
    const bool has_b = part < 0 && first + 1 < seg_tiles;
    const int seg0 = q_txt ? 0 : g.T_txt;
    const int q_end = q_txt ? g.T_txt : g.S;
    // first rows of the two query tiles (scalars, selected by tile: an
    // array indexed at run time would live on the stack)
    const int q0a = seg0 + first * kBM, q0b = q0a + kBM;
    const int L = a.vl.L[b];
    const int nkt_txt = (L + kBN - 1) / kBN;
    const int nkt_all = nkt_txt + g.ntq_img;
    // tiles j0 .. j0 + nkt - 1 of the fused order run here; the loops below
    // count j locally (barrier phases, buffer slots) and name the tile j0 + j
    int j0 = 0, nkt = nkt_all;
    if (kShard) {
        auto fused_index = [&](int blk) { return blk < g.ntq_txt ? min(blk, nkt_txt) : nkt_txt + (blk - g.ntq_txt); };
        j0 = fused_index(a.blk_begin);
        nkt = fused_index(a.blk_end) - j0;
    }
    const bool last_shard = !kShard || j0 + nkt == nkt_all;
    const int row_base = (b * g.H + h) * g.S;  // first row of this (b, h) in qh / kh
    if (kShard && nkt == 0) {
        // no tile of this shard holds a valid key of this sample: the state
        // passes through unchanged (or starts empty)
        const size_t bh = (size_t)b * g.H + h;
        for (int i = threadIdx.x; i < 2 * kBM; i += kThreads) {
            const int n = ((i >> 7) ? q0b : q0a) + (i & 127);
            if (!(i < kBM || has_b) || n >= q_end) continue;
            const size_t rowi = bh * g.S + n;
            const bool have = a.st_in_m != nullptr && j0 > 0;
            a.st_out_m[rowi] = have ? a.st_in_m[rowi] : -INFINITY;
            a.st_out_l[rowi] = have ? a.st_in_l[rowi] : 0.0f;
            for (int d = 0; d < kHeadDim; ++d)
                a.st_out_o[rowi * kHeadDim + d] = have ? a.st_in_o[rowi * kHeadDim + d] : 0.0f;
        }
        return;
    }

    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const uint32_t sQ = sbase + kSmemQ, sK = sbase + kSmemK, sV = sbase + kSmemV;
    const uint32_t bar_q = smem_u32(&bars[0]);
    const uint32_t bar_kf = smem_u32(&bars[1]);   // [2] K slot loaded
    const uint32_t bar_vf = smem_u32(&bars[3]);   // [2] V slot loaded
    const uint32_t bar_ke = smem_u32(&bars[5]);   // [2] K slot free (S_A, S_B done)
    const uint32_t bar_ve = smem_u32(&bars[7]);   // [2] V slot free (PV_A, PV_B done)
    const uint32_t bar_s = smem_u32(&bars[9]);    // [2] per Q tile: S ready
    const uint32_t bar_p = smem_u32(&bars[11]);   // [2] per Q tile: P of key chunk 0 written
    const uint32_t bar_p1 = smem_u32(&bars[32]);  // [2] per Q tile: P of key chunk 1 written
    const uint32_t bar_o = smem_u32(&bars[13]);   // [2] per Q tile: PV done
    const uint32_t bar_drain = smem_u32(&bars[15]);
    const uint32_t bar_x = smem_u32(&bars[16]);   // [tile][quarter][slot]: both halves' values written

    if (tid == 0) {
        abort_flag = 0;
        mbar_init(bar_q, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar_kf + 8 * s, 1);
            mbar_init(bar_vf + 8 * s, 1);
            mbar_init(bar_ke + 8 * s, 1);
            mbar_init(bar_ve + 8 * s, 1);
            mbar_init(bar_s + 8 * s, 1);
            mbar_init(bar_p + 8 * s, 256);
            mbar_init(bar_p1 + 8 * s, 256);
            mbar_init(bar_o + 8 * s, 1);
        }
        mbar_init(bar_drain, 1);
        for (int x = 0; x < 16; ++x) mbar_init(bar_x + 8 * x, 64);
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
            prefetch_tensormap(&a.map_q);
            prefetch_tensormap(&a.map_k);
            prefetch_tensormap(&a.map_v[0]);
            prefetch_tensormap(&a.map_v[1]);
            mbar_expect_tx(bar_q, (has_b ? 2 : 1) * kTileBytes);
            tma_load_2d(sQ, &a.map_q, bar_q, 0, row_base + q0a);
            tma_load_2d(sQ + kBoxBytes, &a.map_q, bar_q, 64, row_base + q0a);
            if (has_b) {
                tma_load_2d(sQ + kTileBytes, &a.map_q, bar_q, 0, row_base + q0b);
                tma_load_2d(sQ + kTileBytes + kBoxBytes, &a.map_q, bar_q, 64, row_base + q0b);
            }
            int k_issued = 0, v_issued = 0;
            for (int j = 0; j < nkt && !abort_flag; ++j) {
                const int s = j & 1;
                if (j >= 2 &&
                    !mbar_wait_backoff(bar_ke + 8 * s, ((j >> 1) + 1) & 1, &abort_flag, kWaitLimitNs,
                                       kProducerSleepNs)) {
                    fail(&abort_flag);
                    break;
                }
                const TileInfo ti = kv_tile(g, L, nkt_txt, j0 + j);
                const uint32_t dk = sK + s * kTileBytes, dv = sV + s * kTileBytes;
                mbar_expect_tx(bar_kf + 8 * s, kTileBytes);
                tma_load_2d(dk, &a.map_k, bar_kf + 8 * s, 0, row_base + ti.k0);
                tma_load_2d(dk + kBoxBytes, &a.map_k, bar_kf + 8 * s, 64, row_base + ti.k0);
                k_issued = j + 1;
                if (j >= 2 &&
                    !mbar_wait_backoff(bar_ve + 8 * s, ((j >> 1) + 1) & 1, &abort_flag, kWaitLimitNs,
                                       kProducerSleepNs)) {
                    fail(&abort_flag);
                    break;
                }
                mbar_expect_tx(bar_vf + 8 * s, kTileBytes);
                // key tiles never straddle the streams: V comes from the
                // tile's own segment, rows counted from the segment start
                const int vseg = ti.k0 < g.T_txt ? 0 : 1;
                const int vrow = vseg ? ti.k0 - g.T_txt : ti.k0;
                tma_load_4d(dv, &a.map_v[vseg], bar_vf + 8 * s, 0, h, vrow, b);
                tma_load_4d(dv + kBoxBytes, &a.map_v[vseg], bar_vf + 8 * s, 64, h, vrow, b);
                v_issued = j + 1;
            }
            // drain: the copies of Q and of the last (up to) two K and V tiles have landed
            mbar_wait_drain(bar_q, 0, kWaitLimitNs);
            for (int j = k_issued - 2 < 0 ? 0 : k_issued - 2; j < k_issued; ++j)
                mbar_wait_drain(bar_kf + 8 * (j & 1), (j >> 1) & 1, kWaitLimitNs);
            for (int j = v_issued - 2 < 0 ? 0 : v_issued - 2; j < v_issued; ++j)
                mbar_wait_drain(bar_vf + 8 * (j & 1), (j >> 1) & 1, kWaitLimitNs);
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_bf16(128, 128, false, false);
            constexpr uint32_t idesc_o = idesc_bf16(128, 128, false, true);
            // S_t = Q_t K_j^T into TMEM [256 t, 256 t + 128)
            auto issue_s = [&](int t, int j) {
                const uint32_t dk = sK + (j & 1) * kTileBytes;
                const uint32_t qt = sQ + t * kTileBytes;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
                    mma_ss(tmem + 256 * t, sdesc_sw128(qt + off, 16, 1024), sdesc_sw128(dk + off, 16, 1024), idesc_s,
                           kk > 0);
                }
                mma_commit(bar_s + 8 * t);
            };
            // O_t += P_t V_j, P_t read from TMEM over S_t, in two parts: key
            // chunk 0 (k-steps 0, 1, 4, 5: keys 0-31 and 64-95, the first
            // P each softmax thread writes) once its P is written, then key
            // chunk 1 (k-steps 2, 3, 6, 7); that k-step order is the
            // accumulation order of O
            auto issue_pv = [&](int t, int j, int part) {
                const uint32_t dv = sV + (j & 1) * kTileBytes;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int kk = 2 * part + (i & 1) + 4 * (i >> 1);
                    mma_ts(tmem + 256 * t + 128, tmem + 256 * t + kk * 8, sdesc_sw128(dv + kk * 2048, kBoxBytes, 1024),
                           idesc_o, (j0 + j > 0 || kk > 0) ? 1u : 0u);
                }
                if (part == 1) mma_commit(bar_o + 8 * t);
            };
            auto wait_p = [&](uint32_t bar, int j) {
                return mbar_test(bar, j & 1) || mbar_wait(bar, j & 1, &abort_flag, kWaitLimitNs);
            };
            bool ok = mbar_wait(bar_q, 0, &abort_flag, kWaitLimitNs) &&
                      mbar_wait(bar_kf, 0, &abort_flag, kWaitLimitNs);
            if (ok) {
                tc_fence_after();
                issue_s(0, 0);
                if (has_b) issue_s(1, 0);
                mma_commit(bar_ke);
            }
            // Two wait points per key tile: a dependent barrier wait stalls
            // the issuing thread for ~100 cycles while the tensor pipe, which
            // buffers little, runs dry, so everything a pair of blocks needs
            // is checked at once (non-blocking tests, one branch), with
            // bounded blocking waits only when a check fails.
            for (int j = 0; ok && j < nkt; ++j) {
                const int s = j & 1, s1 = (j + 1) & 1;
                const bool more = j + 1 < nkt;
                // PV_A(j) needs P_A(j) and V(j); S_A(j+1) needs K(j+1)
                const uint32_t kf_bar = bar_kf + 8 * s1, kf_par = ((j + 1) >> 1) & 1;
                uint32_t r = mbar_test(bar_p, j & 1) & mbar_test(bar_vf + 8 * s, (j >> 1) & 1);
                if (more) r &= mbar_test(kf_bar, kf_par);
                if (!r && !(mbar_wait(bar_p, j & 1, &abort_flag, kWaitLimitNs) &&
                            mbar_wait(bar_vf + 8 * s, (j >> 1) & 1, &abort_flag, kWaitLimitNs) &&
                            (!more || mbar_wait(kf_bar, kf_par, &abort_flag, kWaitLimitNs)))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                issue_pv(0, j, 0);
                if (!wait_p(bar_p1, j)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                issue_pv(0, j, 1);
                if (more) issue_s(0, j + 1);
                if (has_b) {
                    // PV_B(j) needs P_B(j); S_B(j+1) reads the K(j+1) checked above
                    if (!wait_p(bar_p + 8, j)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issue_pv(1, j, 0);
                    if (!wait_p(bar_p1 + 8, j)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issue_pv(1, j, 1);
                }
                mma_commit(bar_ve + 8 * s);
                if (more) {
                    if (has_b) issue_s(1, j + 1);
                    mma_commit(bar_ke + 8 * s1);
                }
            }
            if (!ok) fail(&abort_flag);
            // drain every MMA this thread issued before TMEM is released
            mma_commit(bar_drain);
            mbar_wait_drain(bar_drain, 0, kWaitLimitNs);
        }
    } else if (warp < kSoftmaxWarps && (((warp >> 2) & 1) == 0 || has_b)) {
        // ------------------------------------------------ softmax warps
        // Tile t = (warp >> 2) & 1; this thread takes key columns
        // [64 hc, 64 hc + 64) of its query row and O columns [64 hc, + 64).
        // Barrier phases are consumed strictly in order (S_j, then PV_{j-1}
        // once per tile), so no waiter ever falls two phases behind.
        const int t = (warp >> 2) & 1, hc = warp >> 3, q4 = warp & 3;
        const int q0t = t ? q0b : q0a;
        const uint32_t lane_addr = (uint32_t)(q4 * 32) << 16;
        const uint32_t s_tmem = tmem + lane_addr + 256 * t;
        const uint32_t o_half = s_tmem + 128 + 64 * hc;
        const int row = q4 * 32 + lane;
        const uint32_t xbar = bar_x + 8 * (2 * (4 * t + q4));
        float m = -INFINITY, l = 0.0f;
        // this row's slot in a shard state (rows past the segment read a
        // valid row and write nothing)
        const size_t rowi = ((size_t)b * g.H + h) * g.S + min(q0t + row, q_end - 1);
        if (kShard && j0 > 0) {
            m = a.st_in_m[rowi];
            l = a.st_in_l[rowi];
        }
        // the row sum of tile j is (half 0's sum) + (half 1's sum), folded
        // into l as l = fmaf(l, alpha_j, rs_j) at the next exchange
        float rs_prev = 0.0f, alpha_prev = 1.0f;
        bool ok = true;
        auto exchange = [&](int j, float mine_max, float mine_sum, float2& other) {
            xch[j & 1][t][hc][row] = make_float2(mine_max, mine_sum);
            mbar_arrive(xbar + 8 * (j & 1));
            if (!mbar_wait(xbar + 8 * (j & 1), (j >> 1) & 1, &abort_flag, kWaitLimitNs)) return false;
            other = xch[j & 1][t][hc ^ 1][row];
            return true;
        };
        for (int j = 0; j < nkt; ++j) {
            if (!warp_wait(bar_s + 8 * t, j & 1, &abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const TileInfo ti = kv_tile(g, L, nkt_txt, j0 + j);
            const int nvalid = ti.kend - ti.k0 - 64 * hc;  // keys of this half with c < nvalid are valid
            // the half row's 64 scores; the packed P later reuses the first 32 entries
            uint32_t r[64];
            tmem_ld32(s_tmem + 64 * hc, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
            tmem_ld32(s_tmem + 64 * hc + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
            tmem_ld_wait();
            if (nvalid < 64) {
#pragma unroll
                for (int i = 0; i < 64; ++i) r[i] = i < nvalid ? r[i] : 0xff800000u;  // -inf
            }
            // max of the half row: eight interleaved partial maxima, then a
            // fixed tree; the row max is the larger of the two halves' (max
            // is exact in any order)
            float mp[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
                mp[e] = fmax3(__uint_as_float(r[e]), __uint_as_float(r[8 + e]), __uint_as_float(r[16 + e]));
#pragma unroll
            for (int e = 0; e < 8; ++e) mp[e] = fmax3(mp[e], __uint_as_float(r[24 + e]), __uint_as_float(r[32 + e]));
#pragma unroll
            for (int e = 0; e < 8; ++e) mp[e] = fmax3(mp[e], __uint_as_float(r[40 + e]), __uint_as_float(r[48 + e]));
#pragma unroll
            for (int e = 0; e < 8; ++e) mp[e] = fmaxf(mp[e], __uint_as_float(r[56 + e]));
            const float pm = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])),
                                   fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7])));
            float2 other;
            if (!exchange(j, pm, rs_prev, other)) {
                ok = false;
                break;
            }
            if (j > 0) l = fmaf(l, alpha_prev, rs_prev + other.y);  // (a + b == b + a exactly)
            const float mx = fmaxf(pm, other.x);
            // Lazy rescaling: a row moves its reference max m only when the
            // new max exceeds it by more than 8 (a factor 256), so rows
            // rarely touch O; until then p = exp2(s c - m) <= 256, exact in
            // the fp32 sums and within bf16 range. The decision depends only
            // on the row's own scores, and O / l is the same softmax.
            const float m_cand = fmaxf(m, mx * kC);  // log2 units
            const bool move = m_cand > m + 8.0f;      // always true on the first tile
            const float m_new = move ? m_cand : m;
            // (exp2f only in warps where some row moves: 423 -> 420 us)
            float alpha = 1.0f;
            if (__any_sync(0xffffffffu, move) && move) alpha = exp2f(m - m_new);
            // p = exp2(s * c - m), packed to bf16 into r[0..31] (pair i lands
            // on an entry already read); the half row's sum adds its column
            // i into partial i % 8, partials in a fixed tree (the argument
            // and the partial sums two lanes at a time: each lane rounds as
            // the scalar fmaf / add would)
            uint64_t sp2[4] = {0ull, 0ull, 0ull, 0ull};
            const uint64_t c2 = f2_pack(kC, kC), nm2 = f2_pack(-m_new, -m_new);
            auto numerators = [&](int i0) {
#pragma unroll
                for (int i = i0; i < i0 + 16; ++i) {
                    float x0, x1;
                    f2_unpack(fma_f2(f2_pack(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), c2, nm2), x0,
                              x1);
                    const float p0 = exp2_num(x0), p1 = exp2_num(x1);
                    sp2[i & 3] = add_f2(sp2[i & 3], f2_pack(p0, p1));
                    r[i] = pack_bf16(p0, p1);
                }
            };
            // key chunk 0 (this half's first 32 keys): P over S columns
            // [32 hc, + 16) (all halves have read their scores: the exchange
            // came after), then O rescaled, then the chunk handed to the MMA
            numerators(0);
            tmem_st16(s_tmem + 32 * hc, *reinterpret_cast<uint32_t(*)[16]>(&r[0]));
            if (j > 0) {
                // PV_{j-1} has finished writing O
                if (!warp_wait(bar_o + 8 * t, (j - 1) & 1, &abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // rescale this half of O in the rows that moved their max; the
                // decision is warp-wide and the other rows scale by exactly 1
                if (__any_sync(0xffffffffu, move)) {
                    uint32_t o32[32];
#pragma unroll 1
                    for (int c = 0; c < 2; ++c) {
                        tmem_ld32(o_half + 32 * c, o32);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o32[i] = __float_as_uint(__uint_as_float(o32[i]) * alpha);
                        tmem_st32(o_half + 32 * c, o32);
                    }
                }
            } else if (kShard && j0 > 0) {
                // first tile of a later shard: O is the previous shard's,
                // scaled by alpha as above (alpha is exactly 1 in rows whose
                // reference max stays, so those keep their bits)
                uint32_t o32[32];
                const float4* oin = reinterpret_cast<const float4*>(a.st_in_o + rowi * kHeadDim + 64 * hc);
#pragma unroll 1
                for (int c = 0; c < 2; ++c) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float4 x = oin[8 * c + i];
                        o32[4 * i] = __float_as_uint(x.x * alpha);
                        o32[4 * i + 1] = __float_as_uint(x.y * alpha);
                        o32[4 * i + 2] = __float_as_uint(x.z * alpha);
                        o32[4 * i + 3] = __float_as_uint(x.w * alpha);
                    }
                    tmem_st32(o_half + 32 * c, o32);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bar_p + 8 * t);
            // key chunk 1 (the half's last 32 keys): P over S columns [32 hc + 16, + 16)
            numerators(16);
            tmem_st16(s_tmem + 32 * hc + 16, *reinterpret_cast<uint32_t(*)[16]>(&r[16]));
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bar_p1 + 8 * t);
            float sp[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) f2_unpack(sp2[e], sp[2 * e], sp[2 * e + 1]);
            rs_prev = ((sp[0] + sp[1]) + (sp[2] + sp[3])) + ((sp[4] + sp[5]) + (sp[6] + sp[7]));
            alpha_prev = alpha;
            m = m_new;
        }
        // the last tile's row sum
        if (ok && nkt > 0) {
            float2 other;
            if (exchange(nkt, 0.0f, rs_prev, other))
                l = fmaf(l, alpha_prev, rs_prev + other.y);
            else
                ok = false;
        }
        if (ok && !last_shard && warp_wait(bar_o + 8 * t, (nkt - 1) & 1, &abort_flag)) {
            tc_fence_after();
            // hand the state on: m, l and O (not divided by l), fp32
            const bool mine = q0t + row < q_end;
            if (mine && hc == 0) {
                a.st_out_m[rowi] = m;
                a.st_out_l[rowi] = l;
            }
            float4* oout = reinterpret_cast<float4*>(a.st_out_o + rowi * kHeadDim + 64 * hc);
#pragma unroll 1
            for (int c = 0; c < 2; ++c) {
                uint32_t r[32];
                tmem_ld32(o_half + 32 * c, r);
                tmem_ld_wait();
                if (mine) {
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        oout[8 * c + i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                                      __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
                }
            }
        } else if (ok && last_shard && warp_wait(bar_o + 8 * t, (nkt - 1) & 1, &abort_flag)) {
            tc_fence_after();
            // O / l as bf16 into this tile's Q buffer (its last S product has
            // finished) as two 128-row x 128-byte boxes in the 128-byte
            // swizzle, box hc from this thread; one thread of the tile then
            // stores it with TMA, the segment map clipping rows past the
            // segment.
            const float inv = 1.0f / l;
            const int n = q0t + row;
            const uint32_t stg_u32 = sQ + t * kTileBytes;
            uint8_t* stg = smem_raw + (stg_u32 - smem_u32(smem_raw));
            const int sw = row & 7;
#pragma unroll 1
            for (int c = 0; c < 2; ++c) {
                uint32_t r[32];
                tmem_ld32(o_half + 32 * c, r);
                tmem_ld_wait();
                uint8_t* orow = stg + hc * kBoxBytes + row * 128;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        w[e] = pack_bf16(__uint_as_float(r[8 * q + 2 * e]) * inv, __uint_as_float(r[8 * q + 2 * e + 1]) * inv);
                    *reinterpret_cast<uint4*>(orow + (((c * 4 + q) ^ sw) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
            fence_proxy_async_smem();
            named_barrier_sync(1 + t, 256);
            if (warp == 4 * t && lane == 0) {
                const int seg = q_txt ? 0 : 1;
                const int srow = q0t - seg0;
                tma_store_4d(&a.map_o[seg], stg_u32, 0, h, srow, b);
                tma_store_4d(&a.map_o[seg], stg_u32 + kBoxBytes, 64, h, srow, b);
                bulk_commit_group();
                bulk_wait_read_all();
            }
            if (hc == 0 && n < q_end && a.lse != nullptr) a.lse[((size_t)b * g.H + h) * g.S + n] = (m + log2f(l)) * kLn2;
        } else {
            fail(&abort_flag);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

cudaError_t launch_attn_fwd(const Geom& g, const ValidLen& vl, const uint16_t* qh, const uint16_t* kh,
                            const SegBf16& v, const SegBf16& out, float* lse, cudaStream_t s) {
    FwdArgs local;
    const uint64_t rows = (uint64_t)g.B * g.H * g.S;
    if (!tmap::rows_bf16(&local.map_q, qh, rows) || !tmap::rows_bf16(&local.map_k, kh, rows) ||
        !tmap::seg_bf16(&local.map_v[0], v, g, 0) || !tmap::seg_bf16(&local.map_v[1], v, g, 1) ||
        !tmap::seg_bf16(&local.map_o[0], out, g, 0) || !tmap::seg_bf16(&local.map_o[1], out, g, 1))
        return cudaErrorInvalidValue;
    local.g = g;
    local.vl = vl;
    local.lse = lse;
    local.blk_begin = 0;
    local.blk_end = g.ntq_txt + g.ntq_img;
    local.st_in_m = local.st_in_l = local.st_in_o = nullptr;
    local.st_out_m = local.st_out_l = local.st_out_o = nullptr;
    cudaError_t e = cudaFuncSetAttribute(attn_fwd_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBytes);
    if (e != cudaSuccess) return e;
    local.npairs = (g.ntq_txt + 1) / 2 + (g.ntq_img + 1) / 2;
    const int total = local.npairs * g.H * g.B;
    // one CTA per SM: the pairs past the last full wave run as single tiles
    int dev = 0, sms = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int rem = total % sms;
    int split = rem == 0 ? 0 : std::min(total, rem + kFwdSplitExtra);
    const int policy = g_tile_policy.load();
    if (policy == RLK_FWD_TILES_PAIRS) split = 0;
    if (policy == RLK_FWD_TILES_SINGLE) split = total;
    local.n_keep = total - split;
    timing_begin(kKAttnFwd, s);
    attn_fwd_tc_kernel<false><<<(unsigned)(local.n_keep + 2 * split), kThreads, kSmemBytes, s>>>(local);
    timing_end(kKAttnFwd, s);
    return cudaGetLastError();
}

cudaError_t launch_attn_fwd_shard(const Geom& g, const ValidLen& vl, const uint16_t* qh, const uint16_t* kh,
                                  const SegBf16& v, int blk_begin, int blk_end, const float* state_in,
                                  float* state_out, const SegBf16* out, float* lse, cudaStream_t s) {
    FwdArgs local;
    const uint64_t rows = (uint64_t)g.B * g.H * g.S;
    if (!tmap::rows_bf16(&local.map_q, qh, rows) || !tmap::rows_bf16(&local.map_k, kh, rows) ||
        !tmap::seg_bf16(&local.map_v[0], v, g, 0) || !tmap::seg_bf16(&local.map_v[1], v, g, 1))
        return cudaErrorInvalidValue;
    // only the last shard writes out (its maps are unused elsewhere)
    if (out != nullptr) {
        if (!tmap::seg_bf16(&local.map_o[0], *out, g, 0) || !tmap::seg_bf16(&local.map_o[1], *out, g, 1))
            return cudaErrorInvalidValue;
    } else {
        memset(local.map_o, 0, sizeof(local.map_o));
    }
    local.g = g;
    local.vl = vl;
    local.lse = lse;
    local.blk_begin = blk_begin;
    local.blk_end = blk_end;
    // state layout: m [rows], l [rows], O [rows, 128]
    local.st_in_m = state_in;
    local.st_in_l = state_in != nullptr ? state_in + rows : nullptr;
    local.st_in_o = state_in != nullptr ? state_in + 2 * rows : nullptr;
    local.st_out_m = state_out;
    local.st_out_l = state_out != nullptr ? state_out + rows : nullptr;
    local.st_out_o = state_out != nullptr ? state_out + 2 * rows : nullptr;
    cudaError_t e = cudaFuncSetAttribute(attn_fwd_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBytes);
    if (e != cudaSuccess) return e;
    local.npairs = (g.ntq_txt + 1) / 2 + (g.ntq_img + 1) / 2;
    local.n_keep = local.npairs * g.H * g.B;  // every unit a pair
    timing_begin(kKAttnFwdShard, s);
    attn_fwd_tc_kernel<true><<<(unsigned)local.n_keep, kThreads, kSmemBytes, s>>>(local);
    timing_end(kKAttnFwdShard, s);
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

extern "C" int32_t rlk_fwd_tile_schedule(int32_t policy) {
    if (policy != RLK_FWD_TILES_AUTO && policy != RLK_FWD_TILES_PAIRS && policy != RLK_FWD_TILES_SINGLE) return -1;
    return rlk::g_tile_policy.exchange(policy);
}

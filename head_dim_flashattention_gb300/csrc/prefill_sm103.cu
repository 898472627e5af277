// Causal GQA/MQA FlashAttention forward for head dim 512 on sm_103a.
//
// The method: online softmax over key tiles -- running max m, running sum l,
// O rescaled when m moves -- so the [q x k] score matrix never reaches
// memory ("Writing a FlashAttention Prefill Kernel for Gemma 4", sections
// "The starting point" and "Head dim 512 breaks the textbook").
//
// Geometry of one work item (a cluster of two CTAs on two SMs):
//   * GQA row packing: the pair owns one 128-row tile of T = 128 / G query
//     tokens times the G query heads that share one KV head, so every K/V
//     tile serves all of them ("A custom attention kernel for Gemma 4 on the
//     RTX PRO 6000", "The kernel in three steps", step 1).  TMA gathers the
//     packed rows from q[seq, Hq, 512] with a 4-D box {64, G, 1, T}.
//   * Head-dim split across the pair: CTA h holds Q[:, 256h:256h+256] and
//     O[:, 256h:256h+256] in its tensor memory and reads only the matching
//     256 columns of K and V.  It computes the partial scores
//     S_h = Q_h K_h^T; the two CTAs swap S_h through distributed shared
//     memory and both run the same softmax on S_0 + S_1 (the head-dim split
//     of "Head dim 512 breaks the textbook" and of step 2 on the RTX PRO 6000
//     page, lifted from a warp pair to an SM pair).  A 128 x 512 fp32 O would
//     fill all 512 TMEM columns on its own; split this way each SM holds
//     O half (256 columns) + Q half (128 columns of bf16 pairs) + two S
//     buffers (2 x 64 columns).
//   * The swap moves 32 KiB per tile each way and the SM-to-SM network
//     carries about 20 B/clk per SM, so it is kept off the critical path: a
//     tile's partial scores are sent while the softmax of the previous tile
//     runs, S buffers are released as soon as they are read, and P goes to
//     shared memory, so S(j+2) = Q K(j+2)^T never waits behind O += P(j) V(j).
//   * Causal / sliding-window tile skipping: only key tiles that intersect
//     the visible band of the tile's rows are visited; only tiles that cross
//     the band's edge are masked element by element.
//
// Roles per CTA (256 threads): warp 0 lane 0 issues TMA loads, warp 1 lane 0
// issues tcgen05.mma (warp 1 also owns the TMEM allocation), warps 4-7 own
// TMEM lanes 0-127 (one packed row per thread) and run the score exchange,
// the softmax, the O correction and the epilogue.
//
// Shared memory: K half-tiles in a 3-deep ring, V half-tile single-buffered,
// two exchange buffers (also the Q staging area), two P buffers.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "fa512_device.cuh"
#include "fa512_internal.h"

namespace fa512 {
namespace prefill {

constexpr int D = 512;
constexpr int BM = 128;                 // packed rows per tile
constexpr int BN = 64;                  // keys per KV tile
constexpr int DH = 256;                 // head-dim columns per CTA
constexpr int NUM_THREADS = 256;
constexpr int K_STAGES = 3;
constexpr int HALF_CHUNK = BN * 128;    // one 64-column box of a K or V tile: 8 KiB
constexpr int HALF_TILE = 4 * HALF_CHUNK;   // 64 keys x 256 columns: 32 KiB
constexpr int X_BYTES = BM * BN * 4;        // one exchanged partial S: 32 KiB
constexpr int P_BYTES = BM * BN * 2;        // one P tile (bf16): 16 KiB

constexpr uint32_t TM_O = 0;            // 256 columns fp32
constexpr uint32_t TM_Q = 256;          // 128 columns (256 bf16 per row)
constexpr uint32_t TM_S = 384;          // 2 x 64 columns fp32

// Rescale O only when the row max grows by more than this (log2 units);
// until then the stale max stays the reference and p <= 2^8.
constexpr float RESCALE_THRESHOLD = 8.0f;

struct Smem {
    static constexpr int k = 0;                                  // K_STAGES x 32 KiB
    static constexpr int v = k + K_STAGES * HALF_TILE;           // 32 KiB
    static constexpr int x = v + HALF_TILE;                      // 2 x 32 KiB (Q staging first)
    static constexpr int pbuf = x + 2 * X_BYTES;                 // 2 x 16 KiB
    static constexpr int bars = pbuf + 2 * P_BYTES;
    enum {
        K_FULL = 0,
        K_EMPTY = K_FULL + K_STAGES,
        V_FULL = K_EMPTY + K_STAGES,
        V_EMPTY = V_FULL + 1,
        S_FULL = V_EMPTY + 1,            // 2: S(j) computed
        S_FREE = S_FULL + 2,             // 2: S(j) read into registers
        P_FULL = S_FREE + 2,             // 2: P(j) written to shared memory
        P_EMPTY = P_FULL + 2,            // 2: O += P(j) V(j) done with P(j)
        X_FULL = P_EMPTY + 2,            // 2: the peer's partial S has landed here
        X_EMPTY = X_FULL + 2,            // 2: the peer has consumed what we wrote there
        Q_FULL = X_EMPTY + 2,
        Q_READY = Q_FULL + 1,
        O_DONE = Q_READY + 1,
        DRAIN = O_DONE + 1,
        N_BARS = DRAIN + 1
    };
    static constexpr int tmem_addr = bars + N_BARS * 8;
    static constexpr int abort_flag = tmem_addr + 4;
    static constexpr int total = abort_flag + 4;
};
static_assert(Smem::total + 1024 <= 232448, "shared memory budget");

constexpr uint32_t IDESC_QK = make_idesc_bf16(BM, BN, 0);
constexpr uint32_t IDESC_PV = make_idesc_bf16(BM, DH, 1);

// Bounded wait that also gives up when another role of this CTA has aborted.
// `cluster_scope` uses acquire.cluster so that data a peer CTA released with
// its arrival is visible after the wait.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, unsigned* err,
                                              volatile int* abort, bool cluster_scope = false) {
    const uint32_t a = smem_u32(bar);
    auto try_once = [&]() {
        return cluster_scope ? mbar_try_wait_cluster(a, parity) : mbar_try_wait(a, parity);
    };
    if (try_once()) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (try_once()) return true;
        if ((i & 255u) == 0) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > kWaitLimitNs) {
                report_error(err, FA512_DEVICE_ERR_TIMEOUT);
                *abort = 1;
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool key_visible(int j, int qpos, const PrefillParams& p) {
    return j < p.seqlen_k && (!p.causal || j <= qpos) && (p.window <= 0 || j > qpos - p.window);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
prefill_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
               const __grid_constant__ CUtensorMap tmv, const PrefillParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Smem::bars);
    uint32_t* tmem_addr_smem = reinterpret_cast<uint32_t*>(smem + Smem::tmem_addr);
    volatile int* abort = reinterpret_cast<volatile int*>(smem + Smem::abort_flag);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const uint32_t half = cluster_ctarank();     // head-dim half of this CTA
    const uint32_t peer = half ^ 1u;

    // ---- work item: (q tile, KV head); heaviest (latest) q tiles first
    const int pair = blockIdx.x >> 1;
    const int kvh = pair % p.n_kv_heads;
    const int qt = p.num_q_tiles - 1 - pair / p.n_kv_heads;
    const int G = p.group;
    const int t0 = qt * p.tokens_per_tile;
    const int ntok = min(p.tokens_per_tile, p.seqlen_q - t0);
    const int p_first = p.q_offset + t0;
    const int p_last = p.q_offset + t0 + ntok - 1;
    int j_lo = 0, j_hi = p.seqlen_k;
    if (p.causal) j_hi = min(j_hi, p_last + 1);
    if (p.window > 0) j_lo = max(0, p_first - p.window + 1);
    if (j_hi < j_lo) j_hi = j_lo;
    const int kt_begin = j_lo / BN;
    const int n_kt = j_hi > j_lo ? (j_hi + BN - 1) / BN - kt_begin : 0;

    // this thread's packed row (warps 4-7)
    const int row = (warp & 3) * 32 + lane;
    const int tok = row / G;
    const int g = row - tok * G;
    const bool softmax_warp = warp >= 4;
    const bool valid_row = softmax_warp && row < p.rows_per_tile && tok < ntok;
    const int qpos = p.q_offset + t0 + tok;
    const int hq = kvh * G + g;

    if (n_kt == 0) {
        // no key is visible to any row of this tile: O = 0, LSE = -inf
        // (both CTAs of the pair take this branch together)
        if (valid_row) {
            uint4* dst = reinterpret_cast<uint4*>(
                p.out + (static_cast<size_t>(t0 + tok) * p.n_q_heads + hq) * D + half * DH);
            for (int i = 0; i < DH / 8; ++i) dst[i] = make_uint4(0u, 0u, 0u, 0u);
            if (half == 0 && p.lse) p.lse[static_cast<size_t>(hq) * p.seqlen_q + t0 + tok] = -INFINITY;
        }
        return;
    }

    if (warp == 0 && lane == 0) {
        for (int i = 0; i < Smem::N_BARS; ++i) {
            uint32_t count = 1;
            if (i == Smem::Q_READY || (i >= Smem::S_FREE && i < Smem::S_FREE + 2) ||
                (i >= Smem::P_FULL && i < Smem::P_FULL + 2))
                count = 128;                                           // every softmax thread
            if (i >= Smem::X_FULL && i < Smem::X_EMPTY + 2) count = 4;   // the peer's 4 softmax warps
            mbar_init(&bars[i], count);
        }
        // after any earlier timeout skip the work (both CTAs still meet at
        // the cluster barriers; a peer that did start gives up at its first
        // bounded wait)
        *abort = timed_out_before(p.err) ? 1 : 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmq);
        tma_prefetch_desc(&tmk);
        tma_prefetch_desc(&tmv);
    }
    if (warp == 1) {
        tmem_alloc(tmem_addr_smem, 512);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    // both CTAs' barriers exist before either side arrives remotely
    cluster_sync_all();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_addr_smem;

    const bool skip = *abort != 0;
    if (skip) {
        // nothing to do; fall through to the teardown
    } else if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------------ TMA producer
            mbar_arrive_expect_tx(&bars[Smem::Q_FULL], static_cast<uint32_t>(4 * 128 * p.rows_per_tile));
            for (int c = 0; c < 4; ++c)
                tma_load_4d(smem + Smem::x + c * (BM * 128), &tmq, &bars[Smem::Q_FULL],
                            static_cast<int>(half * 4 + c) * 64, 0, kvh, t0);
            auto load_k = [&](int j) -> bool {
                const int s = j % K_STAGES;
                if (!wait_or_abort(&bars[Smem::K_EMPTY + s], ((j / K_STAGES) & 1) ^ 1, p.err, abort))
                    return false;
                mbar_arrive_expect_tx(&bars[Smem::K_FULL + s], HALF_TILE);
                const int key0 = (kt_begin + j) * BN;
                for (int c = 0; c < 4; ++c)
                    tma_load_3d(smem + Smem::k + s * HALF_TILE + c * HALF_CHUNK, &tmk,
                                &bars[Smem::K_FULL + s], static_cast<int>(half * 4 + c) * 64, kvh, key0);
                return true;
            };
            auto load_v = [&](int j) -> bool {
                if (!wait_or_abort(&bars[Smem::V_EMPTY], (j & 1) ^ 1, p.err, abort)) return false;
                mbar_arrive_expect_tx(&bars[Smem::V_FULL], HALF_TILE);
                const int key0 = (kt_begin + j) * BN;
                for (int c = 0; c < 4; ++c)
                    tma_load_3d(smem + Smem::v + c * HALF_CHUNK, &tmv, &bars[Smem::V_FULL],
                                static_cast<int>(half * 4 + c) * 64, kvh, key0);
                return true;
            };
            // K runs up to three tiles ahead, V one: K(j+3) is free to load once
            // S(j) is computed, V(j+1) once O += P(j) V(j) is done
            bool ok = load_k(0) && load_v(0);
            for (int j = 1; ok && j < K_STAGES && j < n_kt; ++j) ok = load_k(j);
            for (int j = 0; ok && j < n_kt; ++j) {
                if (j + K_STAGES < n_kt) ok = load_k(j + K_STAGES);
                if (ok && j + 1 < n_kt) ok = load_v(j + 1);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------------------ MMA issue
            bool ok = wait_or_abort(&bars[Smem::Q_READY], 0, p.err, abort);
            tc_fence_after_sync();
            const uint32_t k_base = smem_u32(smem + Smem::k);
            const uint32_t v_base = smem_u32(smem + Smem::v);
            const uint32_t p_base = smem_u32(smem + Smem::pbuf);
            auto issue_qk = [&](int j) -> bool {
                const int s = j % K_STAGES;
                if (j >= 2 &&
                    !wait_or_abort(&bars[Smem::S_FREE + (j & 1)], ((j - 2) >> 1) & 1, p.err, abort))
                    return false;
                if (!wait_or_abort(&bars[Smem::K_FULL + s], (j / K_STAGES) & 1, p.err, abort)) return false;
                tc_fence_after_sync();
                const uint32_t sb = tmem + TM_S + static_cast<uint32_t>(j & 1) * BN;
                const uint32_t kb = k_base + s * HALF_TILE;
#pragma unroll
                for (int kk = 0; kk < DH / 16; ++kk) {
                    const uint64_t bd = make_sdesc_sw128(kb + (kk >> 2) * HALF_CHUNK + (kk & 3) * 32, 16, 1024);
                    tc_mma_ts(sb, tmem + TM_Q + kk * 8, bd, IDESC_QK, kk > 0 ? 1u : 0u);
                }
                tc_commit(&bars[Smem::S_FULL + (j & 1)]);
                tc_commit(&bars[Smem::K_EMPTY + s]);
                return true;
            };
            if (ok) ok = issue_qk(0);
            if (ok && n_kt > 1) ok = issue_qk(1);
            for (int j = 0; ok && j < n_kt; ++j) {
                // S(j+2) as soon as S(j) has been read, ahead of O += P(j) V(j)
                if (j + 2 < n_kt && !(ok = issue_qk(j + 2))) break;
                if (!(ok = wait_or_abort(&bars[Smem::P_FULL + (j & 1)], (j >> 1) & 1, p.err, abort))) break;
                if (!(ok = wait_or_abort(&bars[Smem::V_FULL], j & 1, p.err, abort))) break;
                tc_fence_after_sync();
                const uint32_t pb = p_base + static_cast<uint32_t>(j & 1) * P_BYTES;
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                    // P: K-major rows of 128 B; V: MN-major, 64-column boxes
                    // HALF_CHUNK apart, 8-key groups 1 KiB apart
                    const uint64_t ad = make_sdesc_sw128(pb + kk * 32, 16, 1024);
                    const uint64_t bd = make_sdesc_sw128(v_base + kk * 16 * 128, HALF_CHUNK, 1024);
                    tc_mma_ss(tmem + TM_O, ad, bd, IDESC_PV, (j > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(&bars[Smem::O_DONE]);
                tc_commit(&bars[Smem::P_EMPTY + (j & 1)]);
                tc_commit(&bars[Smem::V_EMPTY]);
            }
            // let every issued MMA finish before TMEM can be released
            tc_commit(&bars[Smem::DRAIN]);
            (void)mbar_wait(&bars[Smem::DRAIN], 0, p.err);
        }
    } else if (softmax_warp) {
        // ---------------------------------------------- exchange + softmax + epilogue
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t x_remote = map_to_cta(smem_u32(smem + Smem::x), peer);
        const uint32_t bar_remote = map_to_cta(smem_u32(bars), peer);
        float m_ref = -INFINITY;   // log2 units
        float l = 0.f;             // sum of the fp32 probabilities (for LSE)
        float l_b = 0.f;           // sum of the bf16-rounded probabilities (normalises O)
        bool ok = wait_or_abort(&bars[Smem::Q_FULL], 0, p.err, abort);
        if (ok) {
            // Q half of this row: shared memory (TMA swizzle) -> TMEM as bf16 pairs
            const uint8_t* qs = smem + Smem::x;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t w[32];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint4 v = *reinterpret_cast<const uint4*>(
                        qs + c * (BM * 128) + row * 128 + ((i ^ (row & 7)) << 4));
                    w[4 * i + 0] = v.x;
                    w[4 * i + 1] = v.y;
                    w[4 * i + 2] = v.z;
                    w[4 * i + 3] = v.w;
                }
                tmem_st32(tmem + lane_base + TM_Q + c * 32, w);
            }
            tmem_st_wait();
        }
        tc_fence_before_sync();
        mbar_arrive(&bars[Smem::Q_READY]);
        // the staging area is now free for the peer's partial scores; one
        // release-arrival per warp covers the reads of all its lanes
        __syncwarp();
        if (lane == 0) {
            mbar_arrive_remote(bar_remote + 8 * Smem::X_EMPTY);
            mbar_arrive_remote(bar_remote + 8 * (Smem::X_EMPTY + 1));
        }

        // Send this CTA's partial scores of tile j to the peer: read S(j) from
        // TMEM into `own`, release the S buffer, store into the peer's
        // exchange buffer j % 2 (layout [16-byte chunk][row], so each warp
        // store covers 512 contiguous bytes).  The arrival that publishes the
        // data is issued later, after the softmax of the previous tile.
        auto send_partial = [&](int j, float (&own)[64]) -> bool {
            const int b = j & 1;
            const uint32_t ph = static_cast<uint32_t>((j >> 1) & 1);
            if (!wait_or_abort(&bars[Smem::S_FULL + b], ph, p.err, abort)) return false;
            tc_fence_after_sync();
            uint32_t sr[2][32];
            const uint32_t s_col = TM_S + static_cast<uint32_t>(b) * BN;
            tmem_ld32(tmem + lane_base + s_col, sr[0]);
            tmem_ld32(tmem + lane_base + s_col + 32, sr[1]);
            tmem_ld_wait();
            tc_fence_before_sync();
            mbar_arrive(&bars[Smem::S_FREE + b]);
#pragma unroll
            for (int c = 0; c < 64; ++c) own[c] = __uint_as_float(sr[c >> 5][c & 31]);
            if (!wait_or_abort(&bars[Smem::X_EMPTY + b], ph, p.err, abort, true)) return false;
            const uint32_t xrow = static_cast<uint32_t>(b * X_BYTES + row * 16);
#pragma unroll
            for (int c = 0; c < 16; ++c)
                st_cluster_v4(x_remote + xrow + static_cast<uint32_t>(c) * (BM * 16), own[4 * c],
                              own[4 * c + 1], own[4 * c + 2], own[4 * c + 3]);
            return true;
        };
        auto publish_partial = [&](int j) {
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(bar_remote + 8 * (Smem::X_FULL + (j & 1)));
        };

        float own_cur[64], own_next[64];
        if (ok) ok = send_partial(0, own_cur);
        if (ok) publish_partial(0);
        for (int j = 0; ok && j < n_kt; ++j) {
            const int b = j & 1;
            const uint32_t ph = static_cast<uint32_t>((j >> 1) & 1);
            const bool more = j + 1 < n_kt;
            // the next tile's partial travels while this tile's softmax runs
            if (more && !(ok = send_partial(j + 1, own_next))) break;

            // S = S_0 + S_1: the peer's partial for tile j
            if (!(ok = wait_or_abort(&bars[Smem::X_FULL + b], ph, p.err, abort, true))) break;
            const uint8_t* xs = smem + Smem::x + b * X_BYTES + row * 16;
            float s[64];
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const float4 v = *reinterpret_cast<const float4*>(xs + c * (BM * 16));
                // fp32 addition is commutative, so both CTAs obtain bitwise-equal
                // S = S_0 + S_1 and hence identical P, m and l
                s[4 * c + 0] = own_cur[4 * c + 0] + v.x;
                s[4 * c + 1] = own_cur[4 * c + 1] + v.y;
                s[4 * c + 2] = own_cur[4 * c + 2] + v.z;
                s[4 * c + 3] = own_cur[4 * c + 3] + v.w;
            }

            const int key0 = (kt_begin + j) * BN;
            const bool tile_full = key0 + BN <= p.seqlen_k && (!p.causal || key0 + BN - 1 <= p_first) &&
                                   (p.window <= 0 || key0 > p_last - p.window);
            // scores stay unscaled until the exponent; a hidden key gets the
            // value that scales to -inf whatever the sign of the scale
            const bool neg_scale = p.scale_log2 < 0.f;
            if (!tile_full) {
                const float hidden = neg_scale ? INFINITY : -INFINITY;
#pragma unroll
                for (int c = 0; c < 64; ++c)
                    if (!key_visible(key0 + c, qpos, p)) s[c] = hidden;
            }
            float mx[16];
            if (!neg_scale) {
#pragma unroll
                for (int c = 0; c < 16; ++c)
                    mx[c] = fmaxf(fmaxf(s[4 * c], s[4 * c + 1]), fmaxf(s[4 * c + 2], s[4 * c + 3]));
#pragma unroll
                for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
                    for (int c = 0; c < w; ++c) mx[c] = fmaxf(mx[c], mx[c + w]);
            } else {
#pragma unroll
                for (int c = 0; c < 16; ++c)
                    mx[c] = fminf(fminf(s[4 * c], s[4 * c + 1]), fminf(s[4 * c + 2], s[4 * c + 3]));
#pragma unroll
                for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
                    for (int c = 0; c < w; ++c) mx[c] = fminf(mx[c], mx[c + w]);
            }
            const float tmax = mx[0] * p.scale_log2;   // row max in log2 units
            float m_use = m_ref, alpha = 1.f;
            if (tmax > m_ref + RESCALE_THRESHOLD) {
                m_use = tmax;
                alpha = fast_exp2(m_ref - m_use);   // 0 when m_ref = -inf
            }
            const float shift = m_use == -INFINITY ? 0.f : m_use;
            uint32_t pk[32];
            float2 ps[4], pb[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) ps[c] = pb[c] = make_float2(0.f, 0.f);
            const float2 sl2 = make_float2(p.scale_log2, p.scale_log2);
            const float2 nsh = make_float2(-shift, -shift);
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                // p = 2^(s * scale * log2(e) - shift), two lanes per instruction
                const float2 x = ffma2(make_float2(s[2 * c], s[2 * c + 1]), sl2, nsh);
                const float2 pr = make_float2(fast_exp2(x.x), fast_exp2(x.y));
                ps[c & 3] = fadd2(ps[c & 3], pr);
                pk[c] = pack_bf16x2(pr.x, pr.y);
                // the bf16 values the PV product actually uses
                pb[c & 3] = fadd2(pb[c & 3], make_float2(__uint_as_float(pk[c] << 16),
                                                         __uint_as_float(pk[c] & 0xffff0000u)));
            }
            const float2 ps01 = fadd2(fadd2(ps[0], ps[1]), fadd2(ps[2], ps[3]));
            const float2 pb01 = fadd2(fadd2(pb[0], pb[1]), fadd2(pb[2], pb[3]));
            l = l * alpha + (ps01.x + ps01.y);
            l_b = l_b * alpha + (pb01.x + pb01.y);
            m_ref = m_use;
            if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                // PV of the previous tile must be done before O is corrected
                if (!(ok = wait_or_abort(&bars[Smem::O_DONE], static_cast<uint32_t>((j - 1) & 1), p.err, abort)))
                    break;
                tc_fence_after_sync();
                for (int c = 0; c < DH / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(tmem + lane_base + TM_O + c * 32, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                    tmem_st32(tmem + lane_base + TM_O + c * 32, o);
                }
                tmem_st_wait();
            }
            // P(j) -> shared memory buffer b, K-major with the 128-byte swizzle
            // the MMA descriptor expects; buffer b last held P(j-2)
            if (j >= 2 && !(ok = wait_or_abort(&bars[Smem::P_EMPTY + b], ((j - 2) >> 1) & 1, p.err, abort)))
                break;
            {
                uint8_t* pdst = smem + Smem::pbuf + b * P_BYTES + row * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    *reinterpret_cast<uint4*>(pdst + ((c ^ (row & 7)) << 4)) =
                        make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
            }
            fence_proxy_async_smem();
            tc_fence_before_sync();
            mbar_arrive(&bars[Smem::P_FULL + b]);
            // publish the next tile's partial, then hand buffer b back to the peer
            if (more) publish_partial(j + 1);
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(bar_remote + 8 * (Smem::X_EMPTY + b));
#pragma unroll
            for (int c = 0; c < 64; ++c) own_cur[c] = own_next[c];
        }
        if (ok) ok = wait_or_abort(&bars[Smem::O_DONE], static_cast<uint32_t>((n_kt - 1) & 1), p.err, abort);
        if (ok) {
            tc_fence_after_sync();
            // O / sum(p~) with p~ the rounded weights PV used: O stays an exact
            // convex combination of V rows whatever the rounding of P
            const float inv_l = l_b > 0.f ? 1.f / l_b : 0.f;
            __nv_bfloat16* dst = p.out + (static_cast<size_t>(t0 + tok) * p.n_q_heads + hq) * D + half * DH;
            for (int c = 0; c < DH / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(tmem + lane_base + TM_O + c * 32, o);
                tmem_ld_wait();
                if (valid_row) {
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        pk[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l,
                                            __uint_as_float(o[2 * i + 1]) * inv_l);
                    uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        d4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                }
            }
            if (valid_row && half == 0 && p.lse)
                p.lse[static_cast<size_t>(hq) * p.seqlen_q + t0 + tok] =
                    l > 0.f ? (m_ref + log2f(l)) * 0.69314718055994530942f : -INFINITY;
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    // no CTA leaves while its peer may still write into its shared memory
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace prefill

int prefill_smem_bytes() { return prefill::Smem::total + 1024; }

cudaError_t launch_prefill(const CUtensorMap& tmq, const CUtensorMap& tmk, const CUtensorMap& tmv,
                           const PrefillParams& p, cudaStream_t stream) {
    const int smem = prefill_smem_bytes();
    cudaError_t e = cudaFuncSetAttribute(prefill::prefill_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int n_blocks = p.num_q_tiles * p.n_kv_heads * 2;   // one cluster of 2 per tile
    prefill::prefill_kernel<<<n_blocks, prefill::NUM_THREADS, smem, stream>>>(tmq, tmk, tmv, p);
    return cudaGetLastError();
}

}  // namespace fa512

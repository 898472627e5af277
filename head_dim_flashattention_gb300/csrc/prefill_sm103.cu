// Causal GQA/MQA FlashAttention forward for head dim 512 on sm_103a.
//
// The method: online softmax over key tiles -- running max m, running sum l,
// O rescaled when m moves -- so the [q x k] score matrix never reaches
// memory ("Writing a FlashAttention Prefill Kernel for Gemma 4", sections
// "The starting point" and "Head dim 512 breaks the textbook").
//
// Geometry of one work item (one CTA on one SM):
//   * GQA row packing: a 128-row tile holds T = 128 / G query tokens times
//     the G query heads that share one KV head, so every K/V tile serves all
//     of them ("A custom attention kernel for Gemma 4 on the RTX PRO 6000",
//     "The kernel in three steps", step 1).  TMA gathers the packed rows
//     from q[seq, Hq, 512] with a 4-D box {64, G, 1, T}.
//   * Output head-dim split: a 128 x 512 fp32 O would fill all 512 TMEM
//     columns on its own, so each q tile is served by two CTAs that each own
//     one 256-column half of O (the head-dim split of "Head dim 512 breaks
//     the textbook" and of step 2 on the RTX PRO 6000 page, lifted from
//     warps to SMs).  Both CTAs compute the same full S = Q K^T and the same
//     softmax, so no scores cross between SMs; the pair's only duplicated
//     work is S.  (Swapping half-width partial scores instead is bound by the
//     SM-to-SM network, about 20 B/clk per SM against 32 B/clk needed.)
//   * Operand placement: the tensor core reads shared-memory operands through
//     a 128 B/clk path, so as much as possible comes from TMEM.  TMEM holds O
//     half (256 columns), Q[:, 0:256] as bf16 pairs (128 columns) and two S
//     buffers (2 x 64 columns; P overwrites S in place).  Q[:, 256:512]
//     stays in shared memory.  S = Q_lo K_lo^T (A from TMEM) + Q_hi K_hi^T
//     (A from shared memory); O += P V_half with P from TMEM.
//   * Causal / sliding-window tile skipping: only key tiles that intersect
//     the visible band of the tile's rows are visited; only tiles that cross
//     the band's edge are masked element by element.
//
// Roles (256 threads): warp 0 lane 0 issues TMA loads, warp 1 lane 0 issues
// tcgen05.mma (warp 1 owns the TMEM allocation), warps 4-7 own TMEM lanes
// 0-127 (one packed row per thread) and run the softmax, the O correction
// and the epilogue.  S is double-buffered so S(j+1) is computed while the
// softmax works on tile j.
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
constexpr int DH = 256;                 // O columns per CTA
constexpr int NUM_THREADS = 256;
constexpr int K_STAGES = 2;
constexpr int Q_CHUNK = BM * 128;       // one 64-column box of Q: 16 KiB
constexpr int KV_CHUNK = BN * 128;      // one 64-column box of K or V: 8 KiB
constexpr int K_TILE = 8 * KV_CHUNK;    // 64 keys x 512 columns: 64 KiB
constexpr int V_TILE = 4 * KV_CHUNK;    // 64 keys x 256 columns: 32 KiB

constexpr uint32_t TM_O = 0;            // 256 columns fp32
constexpr uint32_t TM_Q = 256;          // 128 columns: Q[:, 0:256] as bf16 pairs
constexpr uint32_t TM_S = 384;          // 2 x 64 columns fp32; P (bf16) reuses the first 32

// Rescale O only when the row max grows by more than this (log2 units);
// until then the stale max stays the reference and p <= 2^8.
constexpr float RESCALE_THRESHOLD = 8.0f;

struct Smem {
    static constexpr int qhi = 0;                             // Q[:, 256:512]: 64 KiB
    static constexpr int k = qhi + 4 * Q_CHUNK;               // K_STAGES x 64 KiB
    static constexpr int v = k + K_STAGES * K_TILE;           // 32 KiB
    static constexpr int bars = v + V_TILE;
    enum {
        K_FULL = 0,
        K_EMPTY = K_FULL + K_STAGES,
        V_FULL = K_EMPTY + K_STAGES,
        V_EMPTY = V_FULL + 1,
        S_FULL = V_EMPTY + 1,            // 2
        P_FULL = S_FULL + 2,             // 2
        Q_FULL = P_FULL + 2,             // Q_hi and the Q_lo staging copy landed
        Q_READY = Q_FULL + 1,            // Q_lo is in TMEM, staging free
        O_DONE = Q_READY + 1,
        DRAIN = O_DONE + 1,
        N_BARS = DRAIN + 1
    };
    static constexpr int tmem_addr = bars + N_BARS * 8;
    static constexpr int abort_flag = tmem_addr + 4;
    static constexpr int total = abort_flag + 4;
    // Q[:, 0:256] is staged in K stage 1 before the first K tiles arrive
    static constexpr int qlo_staging = k + K_TILE;
};
static_assert(Smem::total + 1024 <= 232448, "shared memory budget");
static_assert(4 * Q_CHUNK <= K_TILE, "Q staging fits one K stage");

constexpr uint32_t IDESC_QK = make_idesc_bf16(BM, BN, 0);
constexpr uint32_t IDESC_PV = make_idesc_bf16(BM, DH, 1);

// Bounded wait that also gives up when another role of this CTA has aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, unsigned* err,
                                              volatile int* abort) {
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait(a, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(a, parity)) return true;
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

__global__ void __launch_bounds__(NUM_THREADS, 1)
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

    // ---- work item: (q tile, KV head, O half).  KV heads run one after the
    // other so that the CTAs resident at any time share one head's K and V
    // in L2; within a head the heaviest (latest) q tiles go first.
    const int half = blockIdx.x & 1;
    const int rest = blockIdx.x >> 1;
    const int kvh = rest / p.num_q_tiles;
    const int qt = p.num_q_tiles - 1 - rest % p.num_q_tiles;
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

    if (n_kt == 0 || timed_out_before(p.err)) {
        // no key is visible to any row of this tile: O = 0, LSE = -inf
        // (after an earlier pipeline timeout: skip the work)
        if (n_kt == 0 && valid_row) {
            uint4* dst = reinterpret_cast<uint4*>(
                p.out + (static_cast<size_t>(t0 + tok) * p.n_q_heads + hq) * D + half * DH);
            for (int i = 0; i < DH / 8; ++i) dst[i] = make_uint4(0u, 0u, 0u, 0u);
            if (half == 0 && p.lse) p.lse[static_cast<size_t>(hq) * p.seqlen_q + t0 + tok] = -INFINITY;
        }
        return;
    }

    if (warp == 0 && lane == 0) {
        for (int i = 0; i < Smem::N_BARS; ++i) {
            const bool per_thread = i == Smem::Q_READY || i == Smem::P_FULL || i == Smem::P_FULL + 1;
            mbar_init(&bars[i], per_thread ? 128 : 1);
        }
        *abort = 0;
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
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_addr_smem;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------------ TMA producer
            mbar_arrive_expect_tx(&bars[Smem::Q_FULL], static_cast<uint32_t>(8 * 128 * p.rows_per_tile));
            for (int c = 0; c < 4; ++c) {
                tma_load_4d(smem + Smem::qlo_staging + c * Q_CHUNK, &tmq, &bars[Smem::Q_FULL], c * 64, 0,
                            kvh, t0);
                tma_load_4d(smem + Smem::qhi + c * Q_CHUNK, &tmq, &bars[Smem::Q_FULL], (4 + c) * 64, 0, kvh,
                            t0);
            }
            auto load_k = [&](int j) -> bool {
                const int s = j % K_STAGES;
                if (!wait_or_abort(&bars[Smem::K_EMPTY + s], ((j / K_STAGES) & 1) ^ 1, p.err, abort))
                    return false;
                mbar_arrive_expect_tx(&bars[Smem::K_FULL + s], K_TILE);
                const int key0 = (kt_begin + j) * BN;
                for (int c = 0; c < 8; ++c)
                    tma_load_3d(smem + Smem::k + s * K_TILE + c * KV_CHUNK, &tmk, &bars[Smem::K_FULL + s],
                                c * 64, kvh, key0);
                return true;
            };
            auto load_v = [&](int j) -> bool {
                if (!wait_or_abort(&bars[Smem::V_EMPTY], (j & 1) ^ 1, p.err, abort)) return false;
                mbar_arrive_expect_tx(&bars[Smem::V_FULL], V_TILE);
                const int key0 = (kt_begin + j) * BN;
                for (int c = 0; c < 4; ++c)
                    tma_load_3d(smem + Smem::v + c * KV_CHUNK, &tmv, &bars[Smem::V_FULL], (half * 4 + c) * 64,
                                kvh, key0);
                return true;
            };
            bool ok = load_k(0) && load_v(0);
            // K stage 1 holds the Q staging copy until Q[:, 0:256] is in TMEM
            if (ok && n_kt > 1) ok = wait_or_abort(&bars[Smem::Q_READY], 0, p.err, abort) && load_k(1);
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
            const uint32_t qhi_base = smem_u32(smem + Smem::qhi);
            auto issue_qk = [&](int j) -> bool {
                const int s = j % K_STAGES;
                if (!wait_or_abort(&bars[Smem::K_FULL + s], (j / K_STAGES) & 1, p.err, abort)) return false;
                tc_fence_after_sync();
                const uint32_t sb = tmem + TM_S + static_cast<uint32_t>(j & 1) * BN;
                const uint32_t kb = k_base + s * K_TILE;
                // Alternate the two halves of the contraction: columns 0..255
                // take A = Q_lo from TMEM (2 KiB of shared-memory reads per
                // MMA), columns 256..511 A = Q_hi from shared memory (6 KiB),
                // which keeps the shared-memory read rate even and leaves room
                // for the TMA writes of the next tiles.
#pragma unroll
                for (int kk = 0; kk < 16; ++kk) {
                    const uint32_t off = (kk & 3) * 32;
                    const uint64_t bl = make_sdesc_sw128(kb + (kk >> 2) * KV_CHUNK + off, 16, 1024);
                    tc_mma_ts(sb, tmem + TM_Q + kk * 8, bl, IDESC_QK, kk > 0 ? 1u : 0u);
                    const uint64_t ad = make_sdesc_sw128(qhi_base + (kk >> 2) * Q_CHUNK + off, 16, 1024);
                    const uint64_t bh = make_sdesc_sw128(kb + (4 + (kk >> 2)) * KV_CHUNK + off, 16, 1024);
                    tc_mma_ss(sb, ad, bh, IDESC_QK, 1u);
                }
                tc_commit(&bars[Smem::S_FULL + (j & 1)]);
                tc_commit(&bars[Smem::K_EMPTY + s]);
                return true;
            };
            if (ok) ok = issue_qk(0);
            for (int j = 0; ok && j < n_kt; ++j) {
                // S(j+1) runs while the softmax works on tile j; its buffer last
                // held P(j-1), consumed by O += P(j-1) V(j-1) issued before it
                if (j + 1 < n_kt && !(ok = issue_qk(j + 1))) break;
                if (!(ok = wait_or_abort(&bars[Smem::P_FULL + (j & 1)], (j >> 1) & 1, p.err, abort))) break;
                if (!(ok = wait_or_abort(&bars[Smem::V_FULL], j & 1, p.err, abort))) break;
                tc_fence_after_sync();
                const uint32_t pb = tmem + TM_S + static_cast<uint32_t>(j & 1) * BN;
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                    // V is MN-major: 64-column boxes KV_CHUNK apart, 8-key groups 1 KiB apart
                    const uint64_t bd = make_sdesc_sw128(v_base + kk * 16 * 128, KV_CHUNK, 1024);
                    tc_mma_ts(tmem + TM_O, pb + kk * 8, bd, IDESC_PV, (j > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(&bars[Smem::O_DONE]);
                tc_commit(&bars[Smem::V_EMPTY]);
            }
            // let every issued MMA finish before TMEM can be released
            tc_commit(&bars[Smem::DRAIN]);
            (void)mbar_wait(&bars[Smem::DRAIN], 0, p.err);
        }
    } else if (softmax_warp) {
        // ---------------------------------------------- softmax + correction + epilogue
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        float m_ref = -INFINITY;   // log2 units
        float l = 0.f;             // sum of the fp32 probabilities (for LSE)
        float l_b = 0.f;           // sum of the bf16-rounded probabilities (normalises O)
        bool ok = wait_or_abort(&bars[Smem::Q_FULL], 0, p.err, abort);
        if (ok) {
            // Q[:, 0:256] of this row: staging copy (TMA swizzle) -> TMEM as bf16 pairs
            const uint8_t* qs = smem + Smem::qlo_staging;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t w[32];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint4 v = *reinterpret_cast<const uint4*>(
                        qs + c * Q_CHUNK + row * 128 + ((i ^ (row & 7)) << 4));
                    w[4 * i + 0] = v.x;
                    w[4 * i + 1] = v.y;
                    w[4 * i + 2] = v.z;
                    w[4 * i + 3] = v.w;
                }
                tmem_st32(tmem + lane_base + TM_Q + c * 32, w);
            }
            tmem_st_wait();
        }
        // the staging area becomes K stage 1: order these generic reads
        // before the TMA writes that follow the arrival
        fence_proxy_async_smem();
        tc_fence_before_sync();
        mbar_arrive(&bars[Smem::Q_READY]);

        for (int j = 0; ok && j < n_kt; ++j) {
            const int b = j & 1;
            const uint32_t ph = static_cast<uint32_t>((j >> 1) & 1);
            if (!(ok = wait_or_abort(&bars[Smem::S_FULL + b], ph, p.err, abort))) break;
            tc_fence_after_sync();
            uint32_t sr[2][32];
            const uint32_t s_col = TM_S + static_cast<uint32_t>(b) * BN;
            tmem_ld32(tmem + lane_base + s_col, sr[0]);
            tmem_ld32(tmem + lane_base + s_col + 32, sr[1]);
            tmem_ld_wait();
            float s[64];
#pragma unroll
            for (int c = 0; c < 64; ++c) s[c] = __uint_as_float(sr[c >> 5][c & 31]);

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
            }
            // P(j) overwrites the first 32 columns of S buffer b (already read)
            tmem_st32(tmem + lane_base + s_col, pk);
            tmem_st_wait();
            tc_fence_before_sync();
            mbar_arrive(&bars[Smem::P_FULL + b]);
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
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace prefill

int prefill_smem_bytes() { return prefill::Smem::total + 1024; }
int prefill_k_box_rows() { return prefill::BN; }
int prefill_v_box_rows() { return prefill::BN; }

cudaError_t launch_prefill(const CUtensorMap& tmq, const CUtensorMap& tmk, const CUtensorMap& tmv,
                           const PrefillParams& p, cudaStream_t stream) {
    const int smem = prefill_smem_bytes();
    cudaError_t e = cudaFuncSetAttribute(prefill::prefill_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int n_blocks = p.num_q_tiles * p.n_kv_heads * 2;   // two O halves per q tile
    prefill::prefill_kernel<<<n_blocks, prefill::NUM_THREADS, smem, stream>>>(tmq, tmk, tmv, p);
    return cudaGetLastError();
}

}  // namespace fa512

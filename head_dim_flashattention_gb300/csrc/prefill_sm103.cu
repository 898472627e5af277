// Causal GQA/MQA FlashAttention forward for head dim 512 on sm_103a.
//
// The method: online softmax over key tiles -- running max m, running sum l,
// O rescaled when m moves -- so the [q x k] score matrix never reaches
// memory ("Writing a FlashAttention Prefill Kernel for Gemma 4", sections
// "The starting point" and "Head dim 512 breaks the textbook").
//
// Geometry of one work item:
//   * GQA row packing: a 128-row tile holds T = 128 / G query tokens times
//     the G query heads that share one KV head, so every K/V tile serves all
//     of them ("A custom attention kernel for Gemma 4 on the RTX PRO 6000",
//     "The kernel in three steps", step 1).  TMA gathers the packed rows
//     from q[seq, Hq, 512] with a 4-D box {64, G, 1, T}.
//   * Output head-dim split: a 128 x 512 fp32 O would fill all 512 TMEM
//     columns on its own, so each q tile is served by two CTAs that each own
//     one 256-column half of O (the head-dim split of "Head dim 512 breaks
//     the textbook" and of step 2 on the RTX PRO 6000 page, lifted from
//     warps to SMs).  Both compute the same S = Q K^T and the same softmax,
//     so no scores cross between SMs.
//   * SM pairs: a cluster of two CTAs takes two consecutive q tiles with the
//     same O half and issues 2-SM MMAs (tcgen05 cta_group::2, M = 256): each
//     CTA keeps its own 128 rows of Q in shared memory and its own S, P and
//     O in TMEM, and holds one half of every K and V operand tile (K: half
//     of the keys, V: half of the output columns).  One MMA then does both
//     SMs' work from half the shared memory per SM, and the issuing thread --
//     whose barrier waits cost tensor-pipe time -- waits once per 16 (QK^T)
//     or 8 (PV) MMAs.
//   * 128-key tiles; S = Q K^T with M256 x N128 MMAs (both operands in
//     shared memory), O_half += P V_half with M256 x N256 MMAs (P from
//     TMEM).  TMEM: O half (256 columns) and two 128-column S buffers, P
//     (bf16 pairs) over S.  K and V stream through three 32 KiB slots per
//     CTA, each with one role: K head-dim columns 0-255, K columns 256-511
//     (this CTA's 64 keys each) and V (128 keys x this CTA's 128 output
//     columns).  The second K slot is released by the commit that marks S
//     ready and the V slot by the one that marks O done, and V's load is
//     counted on the barrier that marks P ready, so the issuing thread
//     waits three times and commits three times per tile.
//   * Causal / sliding-window tile skipping over the pair's visible band;
//     only the 64-key halves that cross a row's band edge are masked
//     element by element.
//
// Roles (320 threads per CTA): warp 0 lane 0 issues this CTA's TMA loads;
// warp 1 owns the TMEM allocation and, in the even CTA, lane 0 issues every
// MMA of the pair; warps 2-9 run the softmax, the O correction and the
// epilogue of this CTA's rows: TMEM lane quadrant (warp % 4) gives a warp its
// 32 rows, warps 2-5 take keys 0-63 of each tile and warps 6-9 keys 64-127,
// and the two warps of a quadrant swap row maxima through shared memory.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <algorithm>

#include "fa512_device.cuh"
#include "fa512_internal.h"
#include "fa512_pair.cuh"

namespace fa512 {
namespace prefill {
using namespace pair;

constexpr int D = 512;
constexpr int BM = 128;                 // packed rows per CTA tile
constexpr int BN = 128;                 // keys per KV tile
constexpr int BH = BN / 2;              // keys per softmax warp
constexpr int DH = 256;                 // O columns per CTA
constexpr int NUM_THREADS = 320;
constexpr int N_SOFTMAX_WARPS = 8;      // warps 2-9
constexpr int Q_CHUNK = BM * 128;       // one 64-column box of Q: 16 KiB
constexpr int SLOT = 32768;             // one slot (this CTA's half of the pair's operand tile)
constexpr int SLOT_KA = 0, SLOT_KB = 1, SLOT_V = 2;
constexpr int K_BOX_ROWS = BN / 2;      // K slot: four {64 columns, 64 keys} boxes
constexpr int K_BOX = K_BOX_ROWS * 128; // 8 KiB
constexpr int V_BOX_ROWS = BN;          // V slot: two {64 columns, 128 keys} boxes
constexpr int V_BOX = V_BOX_ROWS * 128; // 16 KiB

constexpr uint32_t TM_O = 0;            // 256 columns fp32
constexpr uint32_t TM_S = 256;          // 2 x 128 columns fp32; P (bf16) reuses them

// Rescale O only when the row max grows by more than this (log2 units);
// until then the stale max stays the reference and p <= 2^8.
constexpr float RESCALE_THRESHOLD = 8.0f;

struct Smem {
    static constexpr int q = 0;                               // 8 x 16 KiB
    static constexpr int ring = q + 8 * Q_CHUNK;              // 3 slots x 32 KiB
    static constexpr int xmax = ring + 3 * SLOT;              // [2 buffers][2 halves][128 rows] fp32
    static constexpr int bars = xmax + 2 * 2 * BM * 4;
    enum {
        FULL_KA = 0,                     // even CTA: both halves of K columns 0-255 landed
        FULL_KB = FULL_KA + 1,           // even CTA: ... columns 256-511
        EMPTY_KA = FULL_KB + 1,          // the first K slot may be refilled
        S_FULL = EMPTY_KA + 1,           // 2; also: the second K slot may be refilled
        P_FULL = S_FULL + 2,             // 2, even CTA: P of both CTAs in TMEM and V landed
        XCHG = P_FULL + 2,               // 2: row-max swap between the two softmax halves
        Q_FULL = XCHG + 2,               // even CTA: Q of both CTAs landed
        O_DONE = Q_FULL + 1,             // also: the V slot may be refilled
        L_XCHG = O_DONE + 1,             // final row-sum swap
        DRAIN = L_XCHG + 1,              // every issued MMA has completed
        V_TAIL = DRAIN + 1,              // paged: this CTA's V of the tile that holds the cache's end landed
        O_FINAL = V_TAIL + 1,            // the last O += P V has completed
        N_BARS = O_FINAL + 1
    };
    static constexpr int tmem_addr = bars + N_BARS * 8;
    static constexpr int abort_flag = tmem_addr + 4;
    static constexpr int skip_flag = abort_flag + 4;         // written by the even CTA into both
    static constexpr int total = skip_flag + 4;
};
// The dynamic shared-memory window starts 1 KiB aligned (checked at run
// time), which the 128-byte swizzle atoms need.
static_assert(Smem::total <= 232448, "shared memory budget");

constexpr uint32_t IDESC_QK = make_idesc_bf16(2 * BM, BN, 0);
constexpr uint32_t IDESC_PV = make_idesc_bf16(2 * BM, DH, 1);

__device__ __forceinline__ bool key_visible(int j, int qpos, int seqlen_k, const PrefillParams& p) {
    return j < seqlen_k && (!p.causal || j <= qpos) && (p.window <= 0 || j > qpos - p.window);
}

// PAGED: a batch of chunks (varlen rows through cu_seqlens_q) over a paged
// cache; K and V rows are found through the page table one 64-key half tile
// at a time (a page holds a whole number of half tiles).
template <bool PAGED>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
prefill_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
               const __grid_constant__ CUtensorMap tmv, const PrefillParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    // The alignment does not depend on the CTA, so both CTAs of a pair leave here together.
    if (smem_u32(smem) & 1023u) {
        if (threadIdx.x == 0) report_error(p.err, FA512_DEVICE_ERR_LAYOUT);
        return;
    }
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Smem::bars);
    uint32_t* tmem_addr_smem = reinterpret_cast<uint32_t*>(smem + Smem::tmem_addr);
    volatile int* abort = reinterpret_cast<volatile int*>(smem + Smem::abort_flag);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    // bound of every pipeline wait (the host may shorten it)
    const unsigned long long wait_ns = p.wait_limit_ns ? p.wait_limit_ns : kWaitLimitNs;

    // ---- work item: (q-tile pair, KV head, O half, rank in the pair), and in
    // varlen mode the sequence.  KV heads run one after the other so that
    // the CTAs resident at any time share one head's K and V in L2; within a
    // head the heaviest (latest) q tiles go first.
    const uint32_t rank = cluster_ctarank();            // == blockIdx.x & 1
    const int half = (blockIdx.x >> 1) & 1;
    const int rest = blockIdx.x >> 2;
    const int G = p.group;
    const int T = p.tokens_per_tile;
    int kvh, pair, seq = 0, q_start = 0;
    int seqlen_q = p.seqlen_q, seqlen_k = p.seqlen_k, q_offset = p.q_offset;
    if constexpr (PAGED) {
        // Work items are numbered sequence by sequence, KV head by KV head,
        // heaviest pair first, with no gaps: warp 0 finds this CTA's
        // sequence by a scan of the chunk lengths (one contiguous block of
        // sequences per lane), the others wait at the barrier below.
        int* found = reinterpret_cast<int*>(smem + Smem::xmax);   // idle until the pipeline starts
        const int two_t = 2 * T;
        // pairs of a chunk with rows [s0, s1) (0 for a malformed entry; block 0 records those)
        auto chunk_pairs = [&](int s0, int s1) -> int {
            int n = s1 - s0;
            if (s0 < 0 || n < 0 || s0 > p.total_q - n) {
                if (blockIdx.x == 0) report_error(p.err, FA512_DEVICE_ERR_INDEX);
                return 0;
            }
            if (n > p.max_seqlen_q) {
                if (blockIdx.x == 0) report_error(p.err, FA512_DEVICE_ERR_INDEX);
                n = p.max_seqlen_q;
            }
            return (n + two_t - 1) / two_t;
        };
        if (warp == 0) {
            const int item = rest;
            const int per = (p.batch + 31) >> 5;
            const int lo = min(p.batch, lane * per), hi = min(p.batch, lo + per);
            // up to 32 sequences: one sequence per lane, all loads in flight at once
            int s0 = 0, s1 = 0, kv = 0;
            if (per == 1 && lo < hi) {
                s0 = p.cu_seqlens_q[lo];
                s1 = p.cu_seqlens_q[lo + 1];
                kv = p.seqused_k[lo];
            }
            int cnt = 0;
            if (per == 1) {
                if (lo < hi) cnt = chunk_pairs(s0, s1) * p.n_kv_heads;
            } else {
                for (int b = lo; b < hi; ++b)
                    cnt += chunk_pairs(p.cu_seqlens_q[b], p.cu_seqlens_q[b + 1]) * p.n_kv_heads;
            }
            int incl = cnt;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int t = __shfl_up_sync(0xffffffffu, incl, d);
                if (lane >= d) incl += t;
            }
            const int excl = incl - cnt;
            const unsigned owner_mask = __ballot_sync(0xffffffffu, item >= excl && item < incl);
            if (owner_mask) {
                const int owner = __ffs(owner_mask) - 1;
                if (lane == owner) {
                    int f_seq = lo, acc = excl;
                    if (per > 1) {
                        for (int b = lo; b < hi; ++b) {
                            s0 = p.cu_seqlens_q[b];
                            s1 = p.cu_seqlens_q[b + 1];
                            const int c = chunk_pairs(s0, s1) * p.n_kv_heads;
                            if (item < acc + c) {
                                f_seq = b;
                                break;
                            }
                            acc += c;
                        }
                        kv = p.seqused_k[f_seq];
                    }
                    found[0] = f_seq;
                    found[1] = item - acc;
                    found[2] = s0;
                    found[3] = s1;
                    found[4] = kv;
                }
            } else if (lane == 0) {
                found[0] = -1;
            }
        }
        __syncthreads();
        seq = found[0];
        if (seq < 0) return;                            // past the last item: both CTAs of the pair
        const int off = found[1];
        q_start = found[2];
        seqlen_q = min(found[3] - q_start, p.max_seqlen_q);
        seqlen_k = found[4];
        const int n_pairs_seq = (seqlen_q + two_t - 1) / two_t;
        kvh = off / n_pairs_seq;
        const int order = off - kvh * n_pairs_seq;     // 0 = heaviest pair
        pair = n_pairs_seq - 1 - order;
        q_offset = seqlen_k - (found[3] - q_start);    // the chunk is its sequence's tail
        const int kv_cap = p.max_pages_per_seq << p.page_shift;
        if (seqlen_k < 0 || seqlen_k > kv_cap) {
            // recorded once per sequence; read up to the table's capacity
            if (tid == 0 && off == 0) report_error(p.err, FA512_DEVICE_ERR_INDEX);
            seqlen_k = seqlen_k < 0 ? 0 : kv_cap;
        }
    } else {
        const int n_pairs = (p.num_q_tiles + 1) / 2;
        kvh = rest / n_pairs;
        pair = n_pairs - 1 - rest % n_pairs;
    }
    const int qt = 2 * pair + static_cast<int>(rank);   // may be one past the last tile: no rows
    const int t0 = qt * T;
    const int ntok = min(T, seqlen_q - t0);              // <= 0 for a missing second tile
    const int p_first = q_offset + t0;
    const int p_last = q_offset + t0 + ntok - 1;
    // the pair's visible band (the same in both CTAs)
    const int pair_first = q_offset + 2 * pair * T;
    const int pair_last = q_offset + min(seqlen_q, (2 * pair + 2) * T) - 1;
    // paged: the tile that holds the cache's last key when that key does not
    // end a half tile (its V rows past the end are live pool memory)
    const int tail_tile = (PAGED && (seqlen_k & (K_BOX_ROWS - 1))) ? (seqlen_k - 1) / BN : -1;
    int j_lo = 0, j_hi = seqlen_k;
    if (p.causal) j_hi = min(j_hi, pair_last + 1);
    if (p.window > 0) j_lo = max(0, pair_first - p.window + 1);
    if (j_hi < j_lo) j_hi = j_lo;
    const int kt_begin = j_lo / BN;
    const int n_kt = j_hi > j_lo ? (j_hi + BN - 1) / BN - kt_begin : 0;

    // this thread's packed row and key half (warps 2-9)
    const bool softmax_warp = warp >= 2;
    const int row = (warp & 3) * 32 + lane;
    const int kh = warp >= 6 ? 1 : 0;
    const int tok = row / G;
    const int g = row - tok * G;
    const bool valid_row = softmax_warp && row < p.rows_per_tile && tok < ntok;
    const int qpos = q_offset + t0 + tok;
    const int hq = kvh * G + g;

    if (n_kt == 0) {
        // no key is visible to any row of the pair: O = 0, LSE = -inf
        if (valid_row) {
            uint4* dst = reinterpret_cast<uint4*>(
                p.out + (static_cast<size_t>(q_start + t0 + tok) * p.n_q_heads + hq) * D + half * DH + kh * 128);
            for (int i = 0; i < 128 / 8; ++i) dst[i] = make_uint4(0u, 0u, 0u, 0u);
            if (half == 0 && kh == 0 && p.lse)
                p.lse[static_cast<size_t>(hq) * p.total_q + q_start + t0 + tok] = -INFINITY;
        }
        return;
    }

    if (warp == 0 && lane == 0) {
        for (int i = 0; i < Smem::N_BARS; ++i) {
            uint32_t count = 1;
            if (i == Smem::XCHG || i == Smem::XCHG + 1 || i == Smem::L_XCHG) count = N_SOFTMAX_WARPS * 32;
            // one lane per softmax warp of both CTAs, plus the even CTA's V load
            if (i == Smem::P_FULL || i == Smem::P_FULL + 1) count = 2 * N_SOFTMAX_WARPS + 1;
            mbar_init(&bars[i], count);
        }
        *abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmq);
        tma_prefetch_desc(&tmk);
        tma_prefetch_desc(&tmv);
    }
    __syncthreads();
    cluster_sync_all();   // both CTAs running, barriers initialised
    // After an earlier pipeline timeout the pair skips its work; the even CTA
    // decides for both so that the two never part ways.
    if (rank == 0 && tid == 0) {
        const uint32_t skip = timed_out_before(p.err) ? 1u : 0u;
        st_cluster_u32(map_to_cta(smem_u32(smem + Smem::skip_flag), 0), skip);
        st_cluster_u32(map_to_cta(smem_u32(smem + Smem::skip_flag), 1), skip);
    }
    cluster_sync_all();
    if (*reinterpret_cast<volatile uint32_t*>(smem + Smem::skip_flag)) return;

    if (warp == 1) {
        tmem_alloc2(tmem_addr_smem, 512);
        tmem_relinquish2();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_addr_smem;
    // barriers of the even CTA, addressed from either CTA
    auto leader_bar = [&](int i) -> uint32_t { return map_to_cta(smem_u32(&bars[i]), 0); };

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------------ TMA producer
            const uint32_t q_bytes = static_cast<uint32_t>(8 * 128 * p.rows_per_tile);
            if (rank == 0) mbar_arrive_expect_tx(&bars[Smem::Q_FULL], 2 * q_bytes);
            for (int c = 0; c < 8; ++c)
                tma2_load_4d(smem + Smem::q + c * Q_CHUNK, &tmq, leader_bar(Smem::Q_FULL), c * 64, 0, kvh,
                             q_start + t0);
            // Row of the tensor map holding the first key of the 64-key half
            // tile that starts at logical key `key`: the key itself, or in
            // paged mode its slot in the pool.  Halves past the cache's end
            // (and pages outside the pool) read a row past the pool, which
            // the TMA unit fills with zeros.
            auto half_row = [&](int key) -> int {
                if constexpr (PAGED) {
                    if (key >= seqlen_k) return p.oob_row;
                    const int pg = p.page_table[static_cast<size_t>(seq) * p.max_pages_per_seq + (key >> p.page_shift)];
                    if (static_cast<unsigned>(pg) >= static_cast<unsigned>(p.num_pages)) {
                        report_error(p.err, FA512_DEVICE_ERR_INDEX);
                        return p.oob_row;
                    }
                    return (pg << p.page_shift) + (key & ((1 << p.page_shift) - 1));
                } else {
                    return key;
                }
            };
            // rows of the two half tiles of tile j (paged: looked up one tile ahead)
            int row_lo = half_row(kt_begin * BN), row_hi = half_row(kt_begin * BN + K_BOX_ROWS);
            int next_lo = 0, next_hi = 0;
            // K columns 0-255 of tile j (slot KA), columns 256-511 (slot KB): this CTA's half tile
            auto load_k = [&](int row, int slot, int c, uint32_t full) {
                for (int b = 0; b < 4; ++b)
                    tma2_load_3d(smem + Smem::ring + slot * SLOT + b * K_BOX, &tmk, full, (c * 4 + b) * 64, kvh,
                                 row);
            };

            if (rank == 0) {
                mbar_arrive_expect_tx(&bars[Smem::FULL_KA], 2 * SLOT);
                mbar_arrive_expect_tx(&bars[Smem::FULL_KB], 2 * SLOT);
            }
            // (test hook: the first pair's even CTA leaves out its first K
            // load, so that pair's waits run into their bound)
            if (!(p.test_skip_first_k_load && blockIdx.x == 0))
                load_k(rank ? row_hi : row_lo, SLOT_KA, 0, leader_bar(Smem::FULL_KA));
            load_k(rank ? row_hi : row_lo, SLOT_KB, 1, leader_bar(Smem::FULL_KB));
            bool ok = true;
            for (int j = 0; ok && j < n_kt; ++j) {
                const uint32_t ph = static_cast<uint32_t>(j & 1);
                if (j + 1 < n_kt) {
                    next_lo = half_row((kt_begin + j + 1) * BN);
                    next_hi = half_row((kt_begin + j + 1) * BN + K_BOX_ROWS);
                    // slot KA once the first half of S(j) is done, slot KB once S(j) is
                    if (!(ok = wait_or_abort(&bars[Smem::EMPTY_KA], ph, p.err, abort, wait_ns))) break;
                    if (rank == 0) mbar_arrive_expect_tx(&bars[Smem::FULL_KA], 2 * SLOT);
                    load_k(rank ? next_hi : next_lo, SLOT_KA, 0, leader_bar(Smem::FULL_KA));
                    if (!(ok = wait_or_abort(&bars[Smem::S_FULL + (j & 1)], (j >> 1) & 1, p.err, abort, wait_ns))) break;
                    if (rank == 0) mbar_arrive_expect_tx(&bars[Smem::FULL_KB], 2 * SLOT);
                    load_k(rank ? next_hi : next_lo, SLOT_KB, 1, leader_bar(Smem::FULL_KB));
                }
                // V(j) once O += P(j-1) V(j-1) is done; counted on P ready of tile j
                if (j > 0 && !(ok = wait_or_abort(&bars[Smem::O_DONE], (j - 1) & 1, p.err, abort, wait_ns))) break;
                if constexpr (PAGED) {
                    // Each V box is one half tile (one page or part of one).
                    // The tail tile's V lands on this CTA's own barrier: the
                    // softmax warps clear the rows past the cache's end before
                    // they mark P ready (a NaN there would survive a zero weight).
                    const bool tail = kt_begin + j == tail_tile;
                    uint32_t vbar;
                    if (tail) {
                        if (rank == 0) mbar_arrive(&bars[Smem::P_FULL + (j & 1)]);
                        mbar_arrive_expect_tx(&bars[Smem::V_TAIL], SLOT);
                        vbar = map_to_cta(smem_u32(&bars[Smem::V_TAIL]), rank);
                    } else {
                        if (rank == 0) mbar_arrive_expect_tx(&bars[Smem::P_FULL + (j & 1)], 2 * SLOT);
                        vbar = leader_bar(Smem::P_FULL + (j & 1));
                    }
                    for (int r = 0; r < 2; ++r)
                        for (int b = 0; b < 2; ++b)
                            tma2_load_3d(smem + Smem::ring + SLOT_V * SLOT + b * V_BOX + r * K_BOX, &tmv, vbar,
                                         (half * 4 + static_cast<int>(rank) * 2 + b) * 64, kvh, r ? row_hi : row_lo);
                } else {
                    if (rank == 0) mbar_arrive_expect_tx(&bars[Smem::P_FULL + (j & 1)], 2 * SLOT);
                    for (int b = 0; b < 2; ++b)
                        tma2_load_3d(smem + Smem::ring + SLOT_V * SLOT + b * V_BOX, &tmv,
                                     leader_bar(Smem::P_FULL + (j & 1)),
                                     (half * 4 + static_cast<int>(rank) * 2 + b) * 64, kvh, row_lo);
                }
                row_lo = next_lo;
                row_hi = next_hi;
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            // ------------------------------------------------------------ MMA issue (both SMs)
            bool ok = wait_or_abort(&bars[Smem::Q_FULL], 0, p.err, abort, wait_ns);
            const uint32_t ring_base = smem_u32(smem + Smem::ring);
            const uint32_t q_base = smem_u32(smem + Smem::q);
            auto issue_qk = [&](int j) -> bool {
                const uint32_t sb = tmem + TM_S + static_cast<uint32_t>(j & 1) * BN;
                for (int c = 0; c < 2; ++c) {
                    if (!wait_or_abort(&bars[c == 0 ? Smem::FULL_KA : Smem::FULL_KB], j & 1, p.err, abort, wait_ns))
                        return false;
                    tc_fence_after_sync();
                    const uint32_t kb = ring_base + (c == 0 ? SLOT_KA : SLOT_KB) * SLOT;
                    const uint32_t qa = q_base + c * 4 * Q_CHUNK;
                    const uint64_t ad0 = make_sdesc_sw128(qa, 16, 1024);
                    const uint64_t bd0 = make_sdesc_sw128(kb, 16, 1024);
#pragma unroll
                    for (int k16 = 0; k16 < 16; ++k16) {
                        // head-dim chunk 4c + (k16 >> 2), 16 columns at a time (start field in 16 B units)
                        const uint64_t off = static_cast<uint64_t>((k16 & 3) * 2);
                        mma2_ss(sb, ad0 + static_cast<uint64_t>((k16 >> 2) * (Q_CHUNK >> 4)) + off,
                                bd0 + static_cast<uint64_t>((k16 >> 2) * (K_BOX >> 4)) + off, IDESC_QK,
                                (c | k16) ? 1u : 0u);
                    }
                    commit2_both(&bars[c == 0 ? Smem::EMPTY_KA : Smem::S_FULL + (j & 1)]);
                }
                return true;
            };
            auto issue_pv = [&](int j) {
                const uint32_t pb = tmem + TM_S + static_cast<uint32_t>(j & 1) * BN;
                const uint32_t vb = ring_base + SLOT_V * SLOT;
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                    // V is MN-major: 64-column boxes V_BOX apart, 8-key groups 1 KiB apart;
                    // P of keys [64 h, 64 h + 64) sits at S columns [64 h, 64 h + 32)
                    const uint64_t bd = make_sdesc_sw128(vb, V_BOX, 1024) + static_cast<uint64_t>(kk * (16 * 128 >> 4));
                    mma2_ts(tmem + TM_O, pb + (kk >> 2) * BH + (kk & 3) * 8, bd, IDESC_PV,
                            (j > 0 || kk > 0) ? 1u : 0u);
                }
                commit2_both(&bars[Smem::O_DONE]);
            };
            if (ok) ok = issue_qk(0);
            for (int j = 0; ok && j < n_kt; ++j) {
                // S(j+1) runs while the softmax works on tile j; its buffer last
                // held P(j-1), consumed by O += P(j-1) V(j-1) issued before it
                if (j + 1 < n_kt && !(ok = issue_qk(j + 1))) break;
                // P(j) from both CTAs' softmax and V(j) in both CTAs' V slot
                if (!(ok = wait_or_abort(&bars[Smem::P_FULL + (j & 1)], (j >> 1) & 1, p.err, abort, wait_ns))) break;
                tc_fence_after_sync();
                issue_pv(j);
            }
            if (ok) commit2_both(&bars[Smem::O_FINAL]);
            // let every issued MMA finish before TMEM can be released
            commit2_local(&bars[Smem::DRAIN]);
            (void)mbar_wait(&bars[Smem::DRAIN], 0, p.err, wait_ns);
        }
    } else {
        // ---------------------------------------------- softmax + correction + epilogue
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        float* xmax = reinterpret_cast<float*>(smem + Smem::xmax);
        float m_ref = -INFINITY;   // log2 units, the same in both key halves
        float l = 0.f;             // this half's sum of the fp32 probabilities (for LSE)
        float l_b = 0.f;           // this half's sum of the bf16-rounded probabilities
        bool ok = true;
        const bool neg_scale = p.scale_log2 < 0.f;

        for (int j = 0; ok && j < n_kt; ++j) {
            const int b = j & 1;
            const uint32_t ph = static_cast<uint32_t>((j >> 1) & 1);
            // (every wait of a softmax warp is made warp-uniform: the warp
            // synchronises below and must leave the loop as one)
            if (!(ok = __all_sync(0xffffffffu, wait_or_abort(&bars[Smem::S_FULL + b], ph, p.err, abort, wait_ns)))) break;
            tc_fence_after_sync();
            uint32_t sr[2][32];
            const uint32_t s_col = TM_S + static_cast<uint32_t>(b) * BN + kh * BH;
            tmem_ld32(tmem + lane_base + s_col, sr[0]);
            tmem_ld32(tmem + lane_base + s_col + 32, sr[1]);
            tmem_ld_wait();
            float s[64];
#pragma unroll
            for (int c = 0; c < 64; ++c) s[c] = __uint_as_float(sr[c >> 5][c & 31]);

            const int key0 = (kt_begin + j) * BN + kh * BH;
            const bool half_full = ntok > 0 && key0 + BH <= seqlen_k &&
                                   (!p.causal || key0 + BH - 1 <= p_first) &&
                                   (p.window <= 0 || key0 > p_last - p.window);
            // scores stay unscaled until the exponent; a hidden key gets the
            // value that scales to -inf whatever the sign of the scale
            if (!half_full) {
                const float hidden = neg_scale ? INFINITY : -INFINITY;
#pragma unroll
                for (int c = 0; c < 64; ++c)
                    if (!key_visible(key0 + c, qpos, seqlen_k, p)) s[c] = hidden;
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
            // row max over the whole tile: swap the halves' maxima (log2 units).
            // Both halves then take the same decision on the same numbers.
            const float own_max = mx[0] * p.scale_log2;
            xmax[(b * 2 + kh) * BM + row] = own_max;
            mbar_arrive(&bars[Smem::XCHG + b]);
            if (!(ok = __all_sync(0xffffffffu, wait_or_abort(&bars[Smem::XCHG + b], ph, p.err, abort, wait_ns)))) break;
            const float tmax = fmaxf(own_max, xmax[(b * 2 + (kh ^ 1)) * BM + row]);

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
                // PV of the previous tile must be done before O is corrected;
                // each key half corrects its own 128 O columns
                if (!(ok = __all_sync(0xffffffffu, wait_or_abort(&bars[Smem::O_DONE],
                                                                 static_cast<uint32_t>((j - 1) & 1), p.err, abort, wait_ns))))
                    break;
                tc_fence_after_sync();
                for (int c = 0; c < 4; ++c) {
                    uint32_t o[32];
                    const uint32_t oc = TM_O + kh * 128 + c * 32;
                    tmem_ld32(tmem + lane_base + oc, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                    tmem_st32(tmem + lane_base + oc, o);
                }
            }
            // P of this key half overwrites the first 32 of its own 64 S columns
            tmem_st32(tmem + lane_base + s_col, pk);
            if constexpr (PAGED) {
                if (kt_begin + j == tail_tile) {
                    // the tile holding the cache's end: zero this CTA's V rows
                    // from the end to the end of its half tile, then hand them
                    // to the tensor core (async proxy)
                    if (!(ok = __all_sync(0xffffffffu, wait_or_abort(&bars[Smem::V_TAIL], 0, p.err, abort, wait_ns)))) break;
                    const int r0 = seqlen_k - tail_tile * BN;       // 1 .. 127, not 64
                    const int n16 = (((r0 + K_BOX_ROWS - 1) & ~(K_BOX_ROWS - 1)) - r0) * 8;   // 16-byte chunks per box
                    uint8_t* vs = smem + Smem::ring + SLOT_V * SLOT + r0 * 128;
                    for (int i = tid - 64; i < 2 * n16; i += N_SOFTMAX_WARPS * 32) {
                        const int b = i >= n16 ? 1 : 0;
                        *reinterpret_cast<uint4*>(vs + b * V_BOX + (i - b * n16) * 16) = make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_smem();
                }
            }
            tmem_st_wait();
            tc_fence_before_sync();
            __syncwarp();
            // one arrival per warp on the even CTA's barrier (a cluster-scope
            // release only where the barrier is the other CTA's)
            if (lane == 0) {
                if (rank == 0) mbar_arrive(&bars[Smem::P_FULL + b]);
                else mbar_arrive_remote(leader_bar(Smem::P_FULL + b));
            }
        }
        // O is final once PV(n_kt - 1) has completed: a barrier of its own,
        // committed once after the last PV, so no phase can be mistaken
        if (ok) ok = wait_or_abort(&bars[Smem::O_FINAL], 0, p.err, abort, wait_ns);
        // Swap the halves' row sums through the Q area, idle once every MMA
        // has completed.  Each thread arrives exactly once, so the wait ends.
        float* lsum = reinterpret_cast<float*>(smem + Smem::q);
        lsum[(kh * BM + row) * 2 + 0] = l;
        lsum[(kh * BM + row) * 2 + 1] = l_b;
        mbar_arrive(&bars[Smem::L_XCHG]);
        if (ok) ok = wait_or_abort(&bars[Smem::L_XCHG], 0, p.err, abort, wait_ns);
        if (ok) {
            tc_fence_after_sync();
            const float l_all = l + lsum[((kh ^ 1) * BM + row) * 2 + 0];
            const float lb_all = l_b + lsum[((kh ^ 1) * BM + row) * 2 + 1];
            // O / sum(p~) with p~ the rounded weights PV used: O stays an exact
            // convex combination of V rows whatever the rounding of P
            const float inv_l = lb_all > 0.f ? 1.f / lb_all : 0.f;
            __nv_bfloat16* dst =
                p.out + (static_cast<size_t>(q_start + t0 + tok) * p.n_q_heads + hq) * D + half * DH + kh * 128;
            for (int c = 0; c < 4; ++c) {
                uint32_t o[32];
                tmem_ld32(tmem + lane_base + TM_O + kh * 128 + c * 32, o);
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
            if (valid_row && half == 0 && kh == 0 && p.lse)
                p.lse[static_cast<size_t>(hq) * p.total_q + q_start + t0 + tok] =
                    l_all > 0.f ? (m_ref + log2f(l_all)) * 0.69314718055994530942f : -INFINITY;
        }
    }

    // Neither CTA leaves (or frees TMEM) while the pair's MMAs, loads or
    // remote arrivals may still touch it: every role above ends with bounded
    // waits, then both CTAs meet here.
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc2(tmem, 512);
    }
}

}  // namespace prefill

int prefill_smem_bytes() { return prefill::Smem::total; }
int prefill_k_box_rows() { return prefill::K_BOX_ROWS; }
int prefill_v_box_rows() { return prefill::V_BOX_ROWS; }
int prefill_paged_v_box_rows() { return prefill::K_BOX_ROWS; }

cudaError_t launch_prefill(const CUtensorMap& tmq, const CUtensorMap& tmk, const CUtensorMap& tmv,
                           const PrefillParams& p, cudaStream_t stream) {
    const int smem = prefill_smem_bytes();
    cudaError_t e = cudaFuncSetAttribute(prefill::prefill_kernel<false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // (q-tile pair, O half, rank) per KV head; clusters of two consecutive CTAs
    const int n_pairs = (p.num_q_tiles + 1) / 2;
    const int n_blocks = n_pairs * 4 * p.n_kv_heads;
    prefill::prefill_kernel<false><<<n_blocks, prefill::NUM_THREADS, smem, stream>>>(tmq, tmk, tmv, p);
    return cudaGetLastError();
}

cudaError_t launch_prefill_paged(const CUtensorMap& tmq, const CUtensorMap& tmk, const CUtensorMap& tmv,
                                 const PrefillParams& p, cudaStream_t stream) {
    const int smem = prefill_smem_bytes();
    cudaError_t e = cudaFuncSetAttribute(prefill::prefill_kernel<true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // (sequence, KV head, q-tile pair, O half, rank) numbered without gaps; the
    // chunks hold at most total_q / (2 T) + batch pairs
    const long long per_head = std::min(static_cast<long long>(p.batch) * p.max_pairs,
                                        (static_cast<long long>(p.total_q) + 2 * p.tokens_per_tile - 1) /
                                                (2 * p.tokens_per_tile) + p.batch);
    const long long n_blocks = per_head * p.n_kv_heads * 4;
    if (n_blocks == 0) return cudaSuccess;
    prefill::prefill_kernel<true><<<static_cast<unsigned>(n_blocks), prefill::NUM_THREADS, smem, stream>>>(
        tmq, tmk, tmv, p);
    return cudaGetLastError();
}

}  // namespace fa512

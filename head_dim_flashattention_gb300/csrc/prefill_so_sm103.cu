// Causal GQA/MQA FlashAttention forward for head dim 512 on sm_103a, with the
// score work and the output work on different SM pairs.
//
// The method: online softmax over key tiles -- running max m, running sum l,
// O rescaled when m moves -- so the [q x k] score matrix never reaches
// memory ("Writing a FlashAttention Prefill Kernel for Gemma 4", sections
// "The starting point" and "Head dim 512 breaks the textbook").
//
// A 128 x 512 fp32 O fills all 512 TMEM columns of an SM, so the SM that
// holds O has no room for S.  Here a cluster of four CTAs takes two
// consecutive GQA-packed q tiles of one KV head ("A custom attention kernel
// for Gemma 4 on the RTX PRO 6000", "The kernel in three steps", step 1):
//
//   * the score pair (cluster ranks 0, 1; one q tile each) keeps its Q tile
//     resident in shared memory, computes S = Q K^T with 2-SM MMAs
//     (tcgen05 cta_group::2, M256 x N128, each CTA holding 64 of a tile's
//     128 keys) into four S buffers in TMEM, and runs the online softmax;
//   * the output pair (ranks 2, 3) keeps the whole fp32 O of its q tile in
//     TMEM and computes O += P V with 2-SM MMAs (M256 x N256 per O half,
//     each CTA holding 128 of the half's 256 V columns), P read from its
//     shared memory.
//
// Every score CTA sends the bf16 P of each tile (and the per-row rescale
// factor alpha) to the output CTA with the same q tile through distributed
// shared memory (st.async with mbarrier completion), double-buffered.  S is
// computed once, so the tensor pipes execute the algorithmic FLOP only: the
// score pair 2 x 128 x 128 x 512 and the output pair 2 x 128 x 128 x 512
// multiply-adds per key tile.  (The pages split the head dimension across
// warps of one SM, "Head dim 512 breaks the textbook" and step 2 of the RTX
// PRO 6000 page; here the split is between the two products.)
//
// Score pair: K streams through three 32 KiB slots (a half tile: this CTA's
// 64 keys x 256 head-dim columns), each released by the commit after its 16
// MMAs; an S buffer is released when every softmax warp has read it, and the
// producer holds back a tile's first K half until its S buffer is free, so
// the MMA thread waits only for K.  Eight softmax warps: TMEM lane quadrant
// (warp % 4) gives a warp its 32 rows, warps 2-5 take keys 0-63 of each tile
// and warps 6-9 keys 64-127; the two warps of a quadrant swap row maxima
// through shared memory.  The row max is lazy: O is rescaled only when a
// row's max grows by more than 2^8.
//
// Output pair: V streams through four 32 KiB slots (two tiles x two O
// halves); the commit after a tile's 16 MMAs is multicast to all four CTAs
// and frees that tile's V slots, its P buffer, and lets O be corrected for
// the tile after it.  Eight correction warps apply alpha to O in TMEM
// (tcgen05.ld / st) when a row's max moved, then mark the tile ready; at the
// end they normalise O by the sum of the bf16 P values and write bf16 rows.
//
// Causal / sliding-window tile skipping over the pair's visible band; only
// the 64-key halves that cross a row's band edge are masked element by
// element.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "fa512_device.cuh"
#include "fa512_internal.h"
#include "fa512_pair.cuh"

namespace fa512 {
namespace prefill_so {
using namespace pair;

constexpr int D = 512;
constexpr int BM = 128;                  // packed rows per CTA tile
constexpr int BN = 128;                  // keys per KV tile
constexpr int BH = BN / 2;               // keys per softmax warp
constexpr int NUM_THREADS = 320;
constexpr int N_WORK_WARPS = 8;          // warps 2-9
constexpr int Q_CHUNK = BM * 128;        // one 64-column box of Q: 16 KiB
constexpr int SLOT = 32768;
constexpr int K_SLOTS = 3;               // score CTAs: K half tiles
constexpr int K_BOX_ROWS = BN / 2;       // {64 columns, 64 keys} boxes
constexpr int K_BOX = K_BOX_ROWS * 128;  // 8 KiB
constexpr int S_BUFS = 4;                // S buffers of 128 TMEM columns
constexpr int V_SLOTS = 4;               // output CTAs: 2 tiles x 2 O halves
constexpr int V_BOX_ROWS = BN;           // {64 columns, 128 keys} boxes
constexpr int V_BOX = V_BOX_ROWS * 128;  // 16 KiB
constexpr int P_CHUNK = BM * 128;        // P of 64 keys for 128 rows, bf16: 16 KiB
constexpr int P_BUF = 2 * P_CHUNK;       // one tile's P: 32 KiB
constexpr uint32_t P_TX = P_BUF + BM * 4;   // bytes landing per tile: P and alpha
constexpr uint32_t L_TX = BM * 4;           // the final row sums

// Rescale O only when the row max grows by more than this (log2 units);
// until then the stale max stays the reference and p <= 2^8.
constexpr float RESCALE_THRESHOLD = 8.0f;

constexpr uint16_t MASK_SCORE = 0x3, MASK_OUTPUT = 0xC, MASK_ALL = 0xF;

struct Smem {
    // score CTAs
    static constexpr int q = 0;                                 // 8 x 16 KiB
    static constexpr int kring = q + 8 * Q_CHUNK;               // 3 x 32 KiB
    static constexpr int role_end = kring + K_SLOTS * SLOT;     // 224 KiB
    // output CTAs
    static constexpr int vring = 0;                             // 4 x 32 KiB
    static constexpr int precv = vring + V_SLOTS * SLOT;        // 2 x 32 KiB
    static constexpr int alpha = precv + 2 * P_BUF;             // [2][128] f32
    static constexpr int lrecv = alpha + 2 * BM * 4;            // [128] f32
    // both
    static constexpr int xmax = role_end;                       // [2 buffers][2 halves][128] f32
    static constexpr int bars = xmax + 2 * 2 * BM * 4;
    enum {
        K_FULL = 0,                      // [3] score leader: both CTAs' half tile landed
        K_EMPTY = K_FULL + K_SLOTS,      // [3] score CTAs: the slot's MMAs completed
        S_FULL = K_EMPTY + K_SLOTS,      // [4] score CTAs: S of the tile is in TMEM
        S_FREE = S_FULL + S_BUFS,        // [4] score leader: both CTAs' softmax warps read S
        XCHG = S_FREE + S_BUFS,          // [2] score CTAs: row-max swap of the key halves
        Q_FULL = XCHG + 2,               // score leader: both Q tiles landed
        L_XCHG = Q_FULL + 1,             // score CTAs: row-sum swap
        PV_DONE = L_XCHG + 1,            // [2] all four: O += P V of the buffer's last tile completed
        PV_READY = PV_DONE + 2,          // [2] output leader: P landed and O corrected in both, V landed
        P_LANDED = PV_READY + 2,         // [2] output CTAs: P and alpha of the tile arrived
        O_FINAL = P_LANDED + 2,          // output CTAs: the last O += P V completed
        L_READY = O_FINAL + 1,           // output CTAs: the row sums arrived
        DRAIN = L_READY + 1,             // every MMA this CTA issued has completed
        N_BARS = DRAIN + 1
    };
    static constexpr int tmem_addr = bars + N_BARS * 8;
    static constexpr int abort_flag = tmem_addr + 4;
    static constexpr int skip_flag = abort_flag + 4;             // written by rank 0 into all four
    static constexpr int total = skip_flag + 4;
};
static_assert(Smem::lrecv + BM * 4 <= Smem::role_end, "output CTA layout");
// The dynamic shared-memory window starts 1 KiB aligned (checked at run
// time), which the 128-byte swizzle atoms need.
static_assert(Smem::total <= 232448, "shared memory budget");

constexpr uint32_t IDESC_QK = make_idesc_bf16(2 * BM, BN, 0);
constexpr uint32_t IDESC_PV = make_idesc_bf16(2 * BM, 256, 1);

__device__ __forceinline__ bool key_visible(int j, int qpos, const PrefillParams& p) {
    return j < p.seqlen_k && (!p.causal || j <= qpos) && (p.window <= 0 || j > qpos - p.window);
}

// Commit of every MMA issued so far by this thread, arriving on the barrier
// at this offset in each CTA of `mask` (cluster ranks).
__device__ __forceinline__ void commit2_mask(uint64_t* bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
        ::"r"(smem_u32(bar)), "h"(mask)
        : "memory");
}

// 16 bytes into another CTA's shared memory; the bytes complete_tx on that
// CTA's mbarrier (both addresses shared::cluster, in the same CTA).
__device__ __forceinline__ void st_async_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d,
                                            uint32_t bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];"
                 ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d), "r"(bar)
                 : "memory");
}
__device__ __forceinline__ void st_async_b32(uint32_t addr, uint32_t a, uint32_t bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];"
                 ::"r"(addr), "r"(a), "r"(bar)
                 : "memory");
}

// Bounded wait with cluster-scope acquire (for data another CTA delivered).
__device__ __forceinline__ bool wait_cluster_or_abort(uint64_t* bar, uint32_t parity, unsigned* err,
                                                      volatile int* abort, unsigned long long limit_ns) {
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait_cluster(a, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait_cluster(a, parity)) return true;
        if ((i & 255u) == 0) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > limit_ns) {
                report_error(err, FA512_DEVICE_ERR_TIMEOUT);
                *abort = 1;
                return false;
            }
        }
    }
}

__global__ void __cluster_dims__(4, 1, 1) __launch_bounds__(NUM_THREADS, 1)
prefill_so_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                  const __grid_constant__ CUtensorMap tmv, const PrefillParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    // The alignment does not depend on the CTA, so all four leave here together.
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
    const unsigned long long wait_ns = p.wait_limit_ns ? p.wait_limit_ns : kWaitLimitNs;

    // ---- work item: (q-tile pair, KV head); KV heads one after the other so
    // that resident clusters share one head's K and V in L2, the heaviest
    // (latest) q tiles of a head first.
    const uint32_t rank = cluster_ctarank();            // == blockIdx.x & 3
    const bool scorer = rank < 2;
    const uint32_t pr = rank & 1;                       // which q tile of the pair
    const int G = p.group;
    const int T = p.tokens_per_tile;
    const int n_pairs = (p.num_q_tiles + 1) / 2;
    const int item = blockIdx.x >> 2;
    const int kvh = item / n_pairs;
    const int pair = n_pairs - 1 - item % n_pairs;
    const int qt = 2 * pair + static_cast<int>(pr);    // may be one past the last tile: no rows
    const int t0 = qt * T;
    const int ntok = min(T, p.seqlen_q - t0);           // <= 0 for a missing second tile
    const int p_first = p.q_offset + t0;
    const int p_last = p.q_offset + t0 + ntok - 1;
    const int pair_first = p.q_offset + 2 * pair * T;
    const int pair_last = p.q_offset + min(p.seqlen_q, (2 * pair + 2) * T) - 1;
    int j_lo = 0, j_hi = p.seqlen_k;
    if (p.causal) j_hi = min(j_hi, pair_last + 1);
    if (p.window > 0) j_lo = max(0, pair_first - p.window + 1);
    if (j_hi < j_lo) j_hi = j_lo;
    const int kt_begin = j_lo / BN;
    const int n_kt = j_hi > j_lo ? (j_hi + BN - 1) / BN - kt_begin : 0;

    // this thread's packed row and half (warps 2-9): key half in the score
    // CTAs, O column half in the output CTAs
    const bool work_warp = warp >= 2;
    const int row = (warp & 3) * 32 + lane;
    const int kh = warp >= 6 ? 1 : 0;
    const int tok = row / G;
    const int g = row - tok * G;
    const bool valid_row = work_warp && row < p.rows_per_tile && tok < ntok;
    const int qpos = p.q_offset + t0 + tok;
    const int hq = kvh * G + g;

    if (n_kt == 0) {
        // no key is visible to any row of the pair: O = 0, LSE = -inf
        if (valid_row) {
            if (!scorer) {
                uint4* dst = reinterpret_cast<uint4*>(p.out + (static_cast<size_t>(t0 + tok) * p.n_q_heads + hq) * D +
                                                      kh * 256);
                for (int i = 0; i < 256 / 8; ++i) dst[i] = make_uint4(0u, 0u, 0u, 0u);
            } else if (kh == 0 && p.lse) {
                p.lse[static_cast<size_t>(hq) * p.total_q + t0 + tok] = -INFINITY;
            }
        }
        return;
    }

    if (warp == 0 && lane == 0) {
        for (int i = 0; i < Smem::N_BARS; ++i) {
            uint32_t count = 1;
            if (i == Smem::XCHG || i == Smem::XCHG + 1 || i == Smem::L_XCHG) count = N_WORK_WARPS * 32;
            if (i >= Smem::S_FREE && i < Smem::S_FREE + S_BUFS) count = 2 * N_WORK_WARPS;
            // one lane per correction warp of both output CTAs, plus the V load
            if (i == Smem::PV_READY || i == Smem::PV_READY + 1) count = 2 * N_WORK_WARPS + 1;
            mbar_init(&bars[i], count);
        }
        *abort = 0;
        fence_mbar_init();
        if (scorer) {
            tma_prefetch_desc(&tmq);
            tma_prefetch_desc(&tmk);
        } else {
            tma_prefetch_desc(&tmv);
        }
    }
    __syncthreads();
    cluster_sync_all();   // all four running, barriers initialised
    // After an earlier pipeline timeout the cluster skips its work; rank 0
    // decides for all four so that they never part ways.
    if (rank == 0 && tid == 0) {
        const uint32_t skip = timed_out_before(p.err) ? 1u : 0u;
        for (uint32_t r = 0; r < 4; ++r) st_cluster_u32(map_to_cta(smem_u32(smem + Smem::skip_flag), r), skip);
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
    // barrier i of cluster rank r
    auto bar_of = [&](int i, uint32_t r) -> uint32_t { return map_to_cta(smem_u32(&bars[i]), r); };
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;

    if (scorer) {
        if (warp == 0) {
            if (lane == 0) {
                // -------------------------------------------------- Q and K loads
                const uint32_t q_bytes = static_cast<uint32_t>(8 * 128 * p.rows_per_tile);
                if (rank == 0) mbar_arrive_expect_tx(&bars[Smem::Q_FULL], 2 * q_bytes);
                for (int c = 0; c < 8; ++c)
                    tma2_load_4d(smem + Smem::q + c * Q_CHUNK, &tmq, bar_of(Smem::Q_FULL, 0), c * 64, 0, kvh, t0);
                // half tile h: tile h / 2, head-dim columns 256 (h % 2) .. +256, this CTA's 64 keys
                for (int h = 0; h < 2 * n_kt; ++h) {
                    const int j = h >> 1, c = h & 1, s = h % K_SLOTS;
                    if (h >= K_SLOTS && !wait_or_abort(&bars[Smem::K_EMPTY + s], ((h / K_SLOTS) - 1) & 1, p.err,
                                                       abort, wait_ns))
                        break;
                    // the tile's S buffer must have been read before its QK^T may start
                    if (rank == 0 && c == 0 && j >= S_BUFS &&
                        !wait_or_abort(&bars[Smem::S_FREE + (j % S_BUFS)], ((j / S_BUFS) - 1) & 1, p.err, abort,
                                       wait_ns))
                        break;
                    if (rank == 0) mbar_arrive_expect_tx(&bars[Smem::K_FULL + s], 2 * SLOT);
                    // (test hook: the first cluster's rank 0 leaves out its first
                    // K half tile, so that cluster's waits run into their bound)
                    if (h == 0 && p.test_skip_first_k_load && blockIdx.x == 0) continue;
                    const int key = (kt_begin + j) * BN + static_cast<int>(pr) * K_BOX_ROWS;
                    for (int b = 0; b < 4; ++b)
                        tma2_load_3d(smem + Smem::kring + s * SLOT + b * K_BOX, &tmk, bar_of(Smem::K_FULL + s, 0),
                                     (c * 4 + b) * 64, kvh, key);
                }
            }
        } else if (warp == 1) {
            if (lane == 0 && rank == 0) {
                // -------------------------------------------------- S = Q K^T (both SMs)
                bool ok = wait_or_abort(&bars[Smem::Q_FULL], 0, p.err, abort, wait_ns);
                const uint64_t q_desc = make_sdesc_sw128(smem_u32(smem + Smem::q), 16, 1024);
                const uint64_t k_desc = make_sdesc_sw128(smem_u32(smem + Smem::kring), 16, 1024);
                for (int j = 0; ok && j < n_kt; ++j) {
                    const uint32_t sb = tmem + static_cast<uint32_t>(j % S_BUFS) * BN;
                    for (int c = 0; c < 2; ++c) {
                        const int h = 2 * j + c, s = h % K_SLOTS;
                        if (!(ok = wait_or_abort(&bars[Smem::K_FULL + s], (h / K_SLOTS) & 1, p.err, abort, wait_ns)))
                            break;
                        tc_fence_after_sync();
                        const uint64_t ad0 = q_desc + static_cast<uint64_t>(c * 4 * (Q_CHUNK >> 4));
                        const uint64_t bd0 = k_desc + static_cast<uint64_t>(s * (SLOT >> 4));
#pragma unroll
                        for (int k16 = 0; k16 < 16; ++k16) {
                            // head-dim chunk 4c + (k16 >> 2), 16 columns at a time (start field in 16 B units)
                            const uint64_t off = static_cast<uint64_t>((k16 & 3) * 2);
                            mma2_ss(sb, ad0 + static_cast<uint64_t>((k16 >> 2) * (Q_CHUNK >> 4)) + off,
                                    bd0 + static_cast<uint64_t>((k16 >> 2) * (K_BOX >> 4)) + off, IDESC_QK,
                                    (c | k16) ? 1u : 0u);
                        }
                        commit2_mask(&bars[Smem::K_EMPTY + s], MASK_SCORE);
                    }
                    if (ok) commit2_mask(&bars[Smem::S_FULL + (j % S_BUFS)], MASK_SCORE);
                }
                // let every issued MMA finish before TMEM can be released
                commit2_mask(&bars[Smem::DRAIN], static_cast<uint16_t>(1u << rank));
                (void)mbar_wait(&bars[Smem::DRAIN], 0, p.err, wait_ns);
            }
        } else {
            // ------------------------------------------------------ softmax
            float* xmax = reinterpret_cast<float*>(smem + Smem::xmax);
            float m_ref = -INFINITY;   // log2 units, the same in both key halves
            float l = 0.f;             // this half's sum of the fp32 probabilities (for LSE)
            float l_b = 0.f;           // this half's sum of the bf16-rounded probabilities
            bool ok = true;
            const bool neg_scale = p.scale_log2 < 0.f;
            const uint32_t out_rank = rank + 2;
            // this row's place in the output CTA's P buffers and alpha array
            const uint32_t p_dst = map_to_cta(smem_u32(smem + Smem::precv + kh * P_CHUNK + row * 128), out_rank);
            const uint32_t a_dst = map_to_cta(smem_u32(smem + Smem::alpha + row * 4), out_rank);

            for (int j = 0; ok && j < n_kt; ++j) {
                const int b4 = j % S_BUFS, b2 = j & 1;
                // (every wait of a softmax warp is made warp-uniform: the warp
                // synchronises below and must leave the loop as one)
                if (!(ok = __all_sync(0xffffffffu, wait_or_abort(&bars[Smem::S_FULL + b4], (j / S_BUFS) & 1, p.err,
                                                                 abort, wait_ns))))
                    break;
                tc_fence_after_sync();
                uint32_t sr[2][32];
                const uint32_t s_col = static_cast<uint32_t>(b4 * BN + kh * BH);
                tmem_ld32(tmem + lane_base + s_col, sr[0]);
                tmem_ld32(tmem + lane_base + s_col + 32, sr[1]);
                tmem_ld_wait();
                // the S buffer may take the QK^T four tiles on
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) {
                    if (rank == 0) mbar_arrive(&bars[Smem::S_FREE + b4]);
                    else mbar_arrive_remote(bar_of(Smem::S_FREE + b4, 0));
                }
                float s[64];
#pragma unroll
                for (int c = 0; c < 64; ++c) s[c] = __uint_as_float(sr[c >> 5][c & 31]);

                const int key0 = (kt_begin + j) * BN + kh * BH;
                const bool half_full = ntok > 0 && key0 + BH <= p.seqlen_k &&
                                       (!p.causal || key0 + BH - 1 <= p_first) &&
                                       (p.window <= 0 || key0 > p_last - p.window);
                // scores stay unscaled until the exponent; a hidden key gets the
                // value that scales to -inf whatever the sign of the scale
                if (!half_full) {
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
                // row max over the whole tile: swap the halves' maxima (log2
                // units); both halves then take the same decision on the same numbers
                const float own_max = mx[0] * p.scale_log2;
                xmax[(b2 * 2 + kh) * BM + row] = own_max;
                mbar_arrive(&bars[Smem::XCHG + b2]);
                if (!(ok = __all_sync(0xffffffffu, wait_or_abort(&bars[Smem::XCHG + b2], (j >> 1) & 1, p.err, abort,
                                                                 wait_ns))))
                    break;
                const float tmax = fmaxf(own_max, xmax[(b2 * 2 + (kh ^ 1)) * BM + row]);

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
                    const float2 pr2 = make_float2(fast_exp2(x.x), fast_exp2(x.y));
                    ps[c & 3] = fadd2(ps[c & 3], pr2);
                    pk[c] = pack_bf16x2(pr2.x, pr2.y);
                    // the bf16 values the PV product actually uses
                    pb[c & 3] = fadd2(pb[c & 3], make_float2(__uint_as_float(pk[c] << 16),
                                                             __uint_as_float(pk[c] & 0xffff0000u)));
                }
                const float2 ps01 = fadd2(fadd2(ps[0], ps[1]), fadd2(ps[2], ps[3]));
                const float2 pb01 = fadd2(fadd2(pb[0], pb[1]), fadd2(pb[2], pb[3]));
                l = l * alpha + (ps01.x + ps01.y);
                l_b = l_b * alpha + (pb01.x + pb01.y);
                m_ref = m_use;

                // the output CTA's P buffer b2 is free once O += P V of tile j - 2 completed
                if (j >= 2 && !(ok = __all_sync(0xffffffffu, wait_or_abort(&bars[Smem::PV_DONE + b2],
                                                                           ((j >> 1) - 1) & 1, p.err, abort,
                                                                           wait_ns))))
                    break;
                // P of this row's 64 keys: eight 16-byte pieces in the 128-byte
                // swizzle the MMA descriptor expects (piece c at c ^ (row % 8))
                const uint32_t dst = p_dst + static_cast<uint32_t>(b2 * P_BUF);
                const uint32_t xbar = bar_of(Smem::P_LANDED + b2, out_rank);
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8)
                    st_async_v4(dst + static_cast<uint32_t>(((c8 ^ (row & 7)) << 4)), pk[4 * c8], pk[4 * c8 + 1],
                                pk[4 * c8 + 2], pk[4 * c8 + 3], xbar);
                if (kh == 0) st_async_b32(a_dst + static_cast<uint32_t>(b2 * BM * 4), __float_as_uint(alpha), xbar);
            }
            // Swap the halves' row sums through the Q area, idle once every
            // QK^T has completed (the last S_FULL was seen).  Each thread
            // arrives exactly once, so the wait ends.
            float* lsum = reinterpret_cast<float*>(smem + Smem::q);
            lsum[(kh * BM + row) * 2 + 0] = l;
            lsum[(kh * BM + row) * 2 + 1] = l_b;
            mbar_arrive(&bars[Smem::L_XCHG]);
            if (ok) ok = wait_or_abort(&bars[Smem::L_XCHG], 0, p.err, abort, wait_ns);
            if (ok && kh == 0) {
                const float l_all = l + lsum[(BM + row) * 2 + 0];
                const float lb_all = l_b + lsum[(BM + row) * 2 + 1];
                // O / sum(p~) with p~ the rounded weights PV used: O stays an
                // exact convex combination of V rows whatever the rounding of P
                st_async_b32(map_to_cta(smem_u32(smem + Smem::lrecv + row * 4), out_rank), __float_as_uint(lb_all),
                             bar_of(Smem::L_READY, out_rank));
                if (valid_row && p.lse)
                    p.lse[static_cast<size_t>(hq) * p.total_q + t0 + tok] =
                        l_all > 0.f ? (m_ref + log2f(l_all)) * 0.69314718055994530942f : -INFINITY;
            }
        }
    } else {
        if (warp == 0) {
            if (lane == 0) {
                // -------------------------------------------------- V loads
                for (int j = 0; j < n_kt; ++j) {
                    const int b2 = j & 1;
                    // V slots of buffer b2 once O += P V of tile j - 2 completed
                    if (j >= 2 && !wait_or_abort(&bars[Smem::PV_DONE + b2], ((j >> 1) - 1) & 1, p.err, abort, wait_ns))
                        break;
                    if (rank == 2) mbar_arrive_expect_tx(&bars[Smem::PV_READY + b2], 2 * 2 * SLOT);
                    const int key = (kt_begin + j) * BN;
                    for (int hh = 0; hh < 2; ++hh)
                        for (int bx = 0; bx < 2; ++bx)
                            tma2_load_3d(smem + Smem::vring + (2 * b2 + hh) * SLOT + bx * V_BOX, &tmv,
                                         bar_of(Smem::PV_READY + b2, 2),
                                         (hh * 4 + static_cast<int>(pr) * 2 + bx) * 64, kvh, key);
                }
            }
        } else if (warp == 1) {
            if (lane == 0 && rank == 2) {
                // -------------------------------------------------- O += P V (both SMs)
                bool ok = true;
                const uint64_t p_desc = make_sdesc_sw128(smem_u32(smem + Smem::precv), 16, 1024);
                const uint64_t v_desc = make_sdesc_sw128(smem_u32(smem + Smem::vring), V_BOX, 1024);
                for (int j = 0; ok && j < n_kt; ++j) {
                    const int b2 = j & 1;
                    if (!(ok = wait_or_abort(&bars[Smem::PV_READY + b2], (j >> 1) & 1, p.err, abort, wait_ns)))
                        break;
                    tc_fence_after_sync();
                    const uint64_t ad0 = p_desc + static_cast<uint64_t>(b2 * (P_BUF >> 4));
                    const uint64_t bd0 = v_desc + static_cast<uint64_t>(2 * b2 * (SLOT >> 4));
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk) {
                        // P keys 16 kk .. 16 kk + 15: chunk kk / 4, 32 bytes per step within it;
                        // V is MN-major: 8-key groups 1 KiB apart
                        const uint64_t ad = ad0 + static_cast<uint64_t>((kk >> 2) * (P_CHUNK >> 4) + (kk & 3) * 2);
                        const uint64_t bd = bd0 + static_cast<uint64_t>(kk * (16 * 128 >> 4));
                        mma2_ss(tmem, ad, bd, IDESC_PV, (j > 0 || kk > 0) ? 1u : 0u);
                        mma2_ss(tmem + 256, ad, bd + static_cast<uint64_t>(SLOT >> 4), IDESC_PV,
                                (j > 0 || kk > 0) ? 1u : 0u);
                    }
                    // frees the tile's V slots and P buffer; O may be corrected for the next tile
                    commit2_mask(&bars[Smem::PV_DONE + b2], MASK_ALL);
                }
                if (ok) commit2_mask(&bars[Smem::O_FINAL], MASK_OUTPUT);
                commit2_mask(&bars[Smem::DRAIN], static_cast<uint16_t>(1u << rank));
                (void)mbar_wait(&bars[Smem::DRAIN], 0, p.err, wait_ns);
            }
        } else {
            // -------------------------------------------------- O correction + epilogue
            const float* alpha_s = reinterpret_cast<const float*>(smem + Smem::alpha);
            bool ok = true;
            if (warp == 2 && lane == 0) mbar_arrive_expect_tx(&bars[Smem::L_READY], L_TX);
            for (int j = 0; ok && j < n_kt; ++j) {
                const int b2 = j & 1;
                // P_LANDED[b2]'s phase for tile j - 2 completed before this point
                if (warp == 2 && lane == 0) mbar_arrive_expect_tx(&bars[Smem::P_LANDED + b2], P_TX);
                if (!(ok = __all_sync(0xffffffffu, wait_cluster_or_abort(&bars[Smem::P_LANDED + b2], (j >> 1) & 1,
                                                                         p.err, abort, wait_ns))))
                    break;
                // P arrived through the generic proxy; the MMA reads it through the async proxy
                fence_proxy_async_smem();
                const float a = alpha_s[b2 * BM + row];
                if (j > 0 && __any_sync(0xffffffffu, a != 1.f)) {
                    // O += P V of the previous tile must be done before O is corrected
                    if (!(ok = __all_sync(0xffffffffu, wait_or_abort(&bars[Smem::PV_DONE + ((j - 1) & 1)],
                                                                     ((j - 1) >> 1) & 1, p.err, abort, wait_ns))))
                        break;
                    tc_fence_after_sync();
                    for (int c = 0; c < 8; ++c) {
                        uint32_t o[32];
                        const uint32_t oc = static_cast<uint32_t>(kh * 256 + c * 32);
                        tmem_ld32(tmem + lane_base + oc, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * a);
                        tmem_st32(tmem + lane_base + oc, o);
                    }
                    tmem_st_wait();
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) {
                    if (rank == 2) mbar_arrive(&bars[Smem::PV_READY + b2]);
                    else mbar_arrive_remote(bar_of(Smem::PV_READY + b2, 2));
                }
            }
            if (ok) ok = __all_sync(0xffffffffu, wait_or_abort(&bars[Smem::O_FINAL], 0, p.err, abort, wait_ns));
            if (ok) ok = __all_sync(0xffffffffu, wait_cluster_or_abort(&bars[Smem::L_READY], 0, p.err, abort, wait_ns));
            if (ok) {
                tc_fence_after_sync();
                const float lb = reinterpret_cast<const float*>(smem + Smem::lrecv)[row];
                const float inv_l = lb > 0.f ? 1.f / lb : 0.f;
                __nv_bfloat16* dst = p.out + (static_cast<size_t>(t0 + tok) * p.n_q_heads + hq) * D + kh * 256;
                for (int c = 0; c < 8; ++c) {
                    uint32_t o[32];
                    tmem_ld32(tmem + lane_base + static_cast<uint32_t>(kh * 256 + c * 32), o);
                    tmem_ld_wait();
                    if (valid_row) {
                        uint32_t pk[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            pk[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
                        uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            d4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                    }
                }
            }
        }
    }

    // No CTA leaves (or frees TMEM) while the cluster's MMAs, loads, remote
    // stores or arrivals may still touch it: every role above ends with
    // bounded waits, then all four meet here.
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc2(tmem, 512);
    }
}

}  // namespace prefill_so

int prefill_so_smem_bytes() { return prefill_so::Smem::total; }

cudaError_t launch_prefill_so(const CUtensorMap& tmq, const CUtensorMap& tmk, const CUtensorMap& tmv,
                              const PrefillParams& p, cudaStream_t stream) {
    const int smem = prefill_so_smem_bytes();
    cudaError_t e = cudaFuncSetAttribute(prefill_so::prefill_so_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         smem);
    if (e != cudaSuccess) return e;
    // (rank in the cluster) per q-tile pair and KV head
    const int n_pairs = (p.num_q_tiles + 1) / 2;
    const long long n_blocks = static_cast<long long>(n_pairs) * 4 * p.n_kv_heads;
    prefill_so::prefill_so_kernel<<<static_cast<unsigned>(n_blocks), prefill_so::NUM_THREADS, smem, stream>>>(
        tmq, tmk, tmv, p);
    return cudaGetLastError();
}

}  // namespace fa512

// Sliding-window (or causal) GQA attention forward for head dim 256 on
// sm_103a: the local layers that sit between the head-dim-512 global layers.
//
// The local layers attend to the last 1,024 tokens with heads of 256
// dimensions ("A custom attention kernel for Gemma 4 on the RTX PRO 6000",
// "The deployment"; "Writing a FlashAttention Prefill Kernel for Gemma 4",
// the row-split kernel of the sliding layers).  The method is the same online
// softmax as the head-dim-512 kernel -- running max m, running sum l, O
// rescaled when m moves -- with the same GQA row packing (128-row tiles of
// 128 / G tokens times the G query heads of one KV head).
//
// What differs from the head-dim-512 kernel:
//   * A 128 x 256 fp32 O fits one CTA's TMEM next to two S buffers, so there
//     is no output split: a cluster of two CTAs takes two consecutive q tiles
//     (a pair) and issues 2-SM MMAs (cta_group::2, M = 256), each CTA holding
//     half of every K tile (64 keys x 256) and half of every V tile's output
//     columns (128 keys x 128).
//   * Under a 1,024-key window a pair sees only nine 128-key tiles,
//     so a per-launch setup (barriers, TMEM, the first loads) would cost
//     about as much as the work.  The kernel is persistent: one cluster per
//     SM pair walks a contiguous range of (KV head, pair) items, chosen on
//     the host so that every range carries about the same number of tiles.
//     Its pipeline runs on across items: Q is double-buffered (the next
//     item's Q lands while the current one is in use); an item's epilogue
//     runs after the next item's first softmax tile, so the tensor core is
//     not left waiting for it; and O leaves through TMA stores staged in the
//     item's Q buffer, which takes the Q of the item after next once the
//     store has read it.
//
// Roles (320 threads per CTA), as in the head-dim-512 kernel: warp 0 lane 0
// issues this CTA's TMA loads and stores; warp 1 owns TMEM and, in the even
// CTA, runs the MMA loop (one elected lane issues every MMA of the pair); warps 2-9 run the softmax, the O
// correction and the epilogue of this CTA's rows (TMEM lane quadrant
// warp % 4, keys 0-63 of a tile for warps 2-5 and 64-127 for warps 6-9).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <algorithm>
#include <vector>

#include "fa512_device.cuh"
#include "fa512_internal.h"
#include "fa512_pair.cuh"

namespace fa512 {
namespace local256 {
using namespace pair;

constexpr int D = 256;
constexpr int BM = 128;                 // packed rows per CTA tile
constexpr int BN = 128;                 // keys per KV tile
constexpr int BH = BN / 2;              // keys per softmax warp
constexpr int NUM_THREADS = 320;
constexpr int N_SOFTMAX_WARPS = 8;
constexpr int Q_CHUNK = BM * 128;       // one 64-column box of Q: 16 KiB
constexpr int Q_BUF = 4 * Q_CHUNK;      // a whole 128 x 256 Q tile: 64 KiB
constexpr int SLOT = 32768;             // one slot: this CTA's half of a K or V tile
constexpr int SLOT_K0 = 0, SLOT_V = 2;  // K slots 0 and 1 (by tile parity), then the V slot
constexpr int K_BOX_ROWS = BN / 2;      // K slot: four {64 columns, 64 keys} boxes
constexpr int K_BOX = K_BOX_ROWS * 128;
constexpr int V_BOX_ROWS = BN;          // V slot: two {64 columns, 128 keys} boxes
constexpr int V_BOX = V_BOX_ROWS * 128;
static_assert(4 * K_BOX == SLOT && 2 * V_BOX == SLOT, "slot size");
static_assert(K_BOX % 1024 == 0 && V_BOX % 1024 == 0, "boxes start on 128-byte swizzle atoms");

constexpr uint32_t TM_O = 0;            // 256 columns fp32
constexpr uint32_t TM_S = 256;          // 2 S buffers of 128 columns; P (bf16) reuses them
constexpr uint32_t S_STRIDE = 128;

constexpr float RESCALE_THRESHOLD = 8.0f;

struct Smem {
    static constexpr int q = 0;                               // 2 x 64 KiB
    static constexpr int ring = q + 2 * Q_BUF;                // K0, K1, V: 3 x 32 KiB
    static constexpr int xmax = ring + 3 * SLOT;              // [2 buffers][2 halves][128 rows] fp32
    static constexpr int bars = xmax + 2 * 2 * BM * 4;
    enum {
        FULL_K = 0,                      // 2, even CTA: both halves of K(g) landed in slot g & 1
        S_FULL = FULL_K + 2,             // 2: S(g) done; also: K slot g & 1 may be refilled
        P_FULL = S_FULL + 2,             // 2, even CTA: P of both CTAs in TMEM and V landed
        XCHG = P_FULL + 2,               // [2][4]: row-max swap between the two warps of a lane quadrant
        Q_FULL = XCHG + 8,               // 2, even CTA: Q of both CTAs landed in buffer i & 1
        O_DONE = Q_FULL + 2,             // O += P(g) V(g) done; also: the V slot may be refilled
        O_FINAL = O_DONE + 1,            // the last O += P V of an item has completed
        O_FREE = O_FINAL + 1,            // even CTA: both CTAs' softmax warps have read an item's O
        O_STAGED = O_FREE + 1,           // this CTA's O of an item is staged in its Q buffer
        DRAIN = O_STAGED + 1,            // every issued MMA has completed
        N_BARS = DRAIN + 1
    };
    static constexpr int tmem_addr = bars + N_BARS * 8;
    static constexpr int abort_flag = tmem_addr + 4;
    static constexpr int skip_flag = abort_flag + 4;
    static constexpr int total = skip_flag + 4;
};
static_assert(Smem::total <= 232448, "shared memory budget");

constexpr uint32_t IDESC_QK = make_idesc_bf16(2 * BM, BN, 0);
constexpr uint32_t IDESC_PV = make_idesc_bf16(2 * BM, D, 1);

// Geometry of work item idx (KV head major, pairs in order) for CTA `rank`.
struct Item {
    int kvh, pair;
    int t0, ntok;                // this CTA's first token and token count (<= 0: no rows)
    int p_first, p_last;         // positions of this CTA's first and last token
    int key_begin, n_kt;         // first key and 128-key tiles of the pair's visible band
};

__host__ __device__ inline Item item_geometry(int idx, const Prefill256Params& p, int rank) {
    Item it;
    it.kvh = idx / p.n_pairs;
    it.pair = idx - it.kvh * p.n_pairs;
    const int T = p.tokens_per_tile;
    it.t0 = (2 * it.pair + rank) * T;
    it.ntok = p.seqlen_q - it.t0 < T ? p.seqlen_q - it.t0 : T;
    it.p_first = p.q_offset + it.t0;
    it.p_last = p.q_offset + it.t0 + it.ntok - 1;
    const int pair_first = p.q_offset + 2 * it.pair * T;
    const int pair_end = (2 * it.pair + 2) * T < p.seqlen_q ? (2 * it.pair + 2) * T : p.seqlen_q;
    const int pair_last = p.q_offset + pair_end - 1;
    int j_lo = 0, j_hi = p.seqlen_k;
    if (p.causal && pair_last + 1 < j_hi) j_hi = pair_last + 1;
    if (p.window > 0 && pair_first - p.window + 1 > j_lo) j_lo = pair_first - p.window + 1;
    if (j_hi < j_lo) j_hi = j_lo;
    // the tiles start at the band's first key, not at a multiple of 128: a
    // window's band of 1,024 + 2T - 1 keys then takes 9 tiles at every
    // offset instead of 9 or 10 (the load's row coordinate has no alignment
    // rule; keys past the band are masked, rows past the keys read zeros)
    it.key_begin = j_lo;
    it.n_kt = j_hi > j_lo ? (j_hi - j_lo + BN - 1) / BN : 0;
    return it;
}

__device__ __forceinline__ bool key_visible(int j, int qpos, const Prefill256Params& p) {
    return j < p.seqlen_k && (!p.causal || j <= qpos) && (p.window <= 0 || j > qpos - p.window);
}

// Walks the key tiles of a range of items in order, skipping items with no
// visible key; qi counts the items that have tiles.
struct TileCursor {
    int idx, end, stride, qi, j, g;
    Item it;
    bool valid;
    __device__ __forceinline__ void first(int begin, int end_, const Prefill256Params& p, int rank) {
        stride = p.item_stride;
        idx = begin - stride;
        end = end_;
        qi = -1;
        j = 0;
        g = 0;
        valid = true;
        next_item(p, rank);
    }
    __device__ __forceinline__ void next_item(const Prefill256Params& p, int rank) {
        for (;;) {
            idx += stride;
            if (idx >= end) {
                valid = false;
                return;
            }
            it = item_geometry(idx, p, rank);
            if (it.n_kt > 0) {
                ++qi;
                j = 0;
                return;
            }
        }
    }
    __device__ __forceinline__ void advance(const Prefill256Params& p, int rank) {
        ++g;
        if (++j >= it.n_kt) next_item(p, rank);
    }
    __device__ __forceinline__ bool last_of_item() const { return j + 1 == it.n_kt; }
};

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
prefill256_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                  const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmo,
                  const __grid_constant__ Prefill256Params p) {
    extern __shared__ __align__(1024) uint8_t smem[];
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
    const uint32_t rank = cluster_ctarank();
    const int irank = static_cast<int>(rank);
    const int cluster = blockIdx.x >> 1;
    const int begin = p.range_start[cluster];
    const int end = p.item_stride == 1 ? p.range_start[cluster + 1] : p.n_items;
    if (begin >= end) return;   // both CTAs of the pair

    if (warp == 0 && lane == 0) {
        for (int i = 0; i < Smem::N_BARS; ++i) {
            uint32_t count = 1;
            if (i >= Smem::XCHG && i < Smem::XCHG + 8) count = 2;   // the two warps sharing the rows
            // one lane per softmax warp of both CTAs (plus the even CTA's V load)
            if (i == Smem::P_FULL || i == Smem::P_FULL + 1) count = 2 * N_SOFTMAX_WARPS + 1;
            if (i == Smem::O_FREE) count = 2 * N_SOFTMAX_WARPS;
            if (i == Smem::O_STAGED) count = N_SOFTMAX_WARPS;
            mbar_init(&bars[i], count);
        }
        *abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmq);
        tma_prefetch_desc(&tmk);
        tma_prefetch_desc(&tmv);
        tma_prefetch_desc(&tmo);
    }
    __syncthreads();
    cluster_sync_all();
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
    auto leader_bar = [&](int i) -> uint32_t { return map_to_cta(smem_u32(&bars[i]), 0); };

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------------ TMA producer
            // Also stores each item's O: the softmax warps stage it in the
            // item's Q buffer (free once its last S is done); that buffer
            // takes the Q of the item two ahead once the store has read it.
            const uint32_t q_bytes = static_cast<uint32_t>(4 * 128 * p.rows_per_tile);
            auto load_q = [&](const Item& it, int qi) {
                const int b = qi & 1;
                if (rank == 0) mbar_arrive_expect_tx(&bars[Smem::Q_FULL + b], 2 * q_bytes);
                for (int c = 0; c < 4; ++c)
                    tma2_load_4d(smem + Smem::q + b * Q_BUF + c * Q_CHUNK, &tmq, leader_bar(Smem::Q_FULL + b),
                                 c * 64, 0, it.kvh, it.t0);
            };
            auto load_k = [&](const TileCursor& t) {
                const int b = t.g & 1;
                if (rank == 0) mbar_arrive_expect_tx(&bars[Smem::FULL_K + b], 2 * SLOT);
                const int key0 = t.it.key_begin + t.j * BN + irank * K_BOX_ROWS;
                for (int c = 0; c < 4; ++c)
                    tma2_load_3d(smem + Smem::ring + (SLOT_K0 + b) * SLOT + c * K_BOX, &tmk,
                                 leader_bar(Smem::FULL_K + b), c * 64, t.it.kvh, key0);
            };
            // One thread runs four streams, each issued as soon as its own
            // condition holds (polled, so that no stream waits behind another):
            //   K(g) into slot g & 1 once S(g - 2) is done and the Q of its
            //        item is on its way;
            //   V(g) into the V slot once O += P(g-1) V(g-1) is done;
            //   O of an item once the softmax warps have staged it;
            //   Q of an item into the buffer of the item two before, once
            //        that item's O store has read it.
            // A condition polled for tile g cannot be confused with the one
            // for g + 2: that phase needs the very load that waits for it.
            TileCursor kc, vc, oc, qc;
            kc.first(begin, end, p, irank);
            vc = kc;
            oc = kc;
            qc = kc;
            for (int i = 0; i < 2 && qc.valid; ++i) {
                load_q(qc.it, qc.qi);
                qc.next_item(p, irank);
            }
            unsigned long long t_last = globaltimer_ns();
            uint32_t idle = 0;
            while (kc.valid || vc.valid || oc.valid) {
                bool progress = false;
                if (kc.valid && (!qc.valid || kc.qi < qc.qi) &&
                    (kc.g < 2 || mbar_test_wait(smem_u32(&bars[Smem::S_FULL + (kc.g & 1)]), ((kc.g - 2) >> 1) & 1))) {
                    load_k(kc);
                    kc.advance(p, irank);
                    progress = true;
                }
                if (vc.valid && (vc.g == 0 || mbar_test_wait(smem_u32(&bars[Smem::O_DONE]), (vc.g - 1) & 1))) {
                    const int g = vc.g;
                    if (rank == 0) mbar_arrive_expect_tx(&bars[Smem::P_FULL + (g & 1)], 2 * SLOT);
                    for (int b = 0; b < 2; ++b)
                        tma2_load_3d(smem + Smem::ring + SLOT_V * SLOT + b * V_BOX, &tmv,
                                     leader_bar(Smem::P_FULL + (g & 1)), (irank * 2 + b) * 64, vc.it.kvh,
                                     vc.it.key_begin + vc.j * BN);
                    vc.advance(p, irank);
                    progress = true;
                }
                if (oc.valid && mbar_test_wait(smem_u32(&bars[Smem::O_STAGED]), oc.qi & 1)) {
                    if (oc.it.ntok > 0)
                        for (int c = 0; c < 4; ++c)
                            tma_store_4d(&tmo, smem + Smem::q + (oc.qi & 1) * Q_BUF + c * Q_CHUNK, c * 64, 0,
                                         oc.it.kvh, oc.it.t0);
                    bulk_commit();
                    oc.next_item(p, irank);
                    progress = true;
                }
                if (qc.valid && !(oc.valid && oc.qi <= qc.qi - 2)) {
                    bulk_wait_read_all();
                    load_q(qc.it, qc.qi);
                    qc.next_item(p, irank);
                    progress = true;
                }
                if (progress) {
                    idle = 0;
                    continue;
                }
                __nanosleep(20);
                if ((++idle & 255u) == 1u) {
                    const unsigned long long now = globaltimer_ns();
                    if (idle == 1u) t_last = now;
                    if (*abort) break;
                    if (now - t_last > kWaitLimitNs) {
                        report_error(p.err, FA512_DEVICE_ERR_TIMEOUT);
                        *abort = 1;
                        break;
                    }
                }
            }
            bulk_wait_all();
        }
    } else if (warp == 1) {
        if (rank == 0) {
            // ------------------------------------------------------------ MMA issue (both SMs)
            // The whole warp walks the tiles and waits (warp-uniform, so the
            // MMA operands stay uniform); one elected lane issues and commits.
            const uint32_t ring_base = smem_u32(smem + Smem::ring);
            const uint32_t q_base = smem_u32(smem + Smem::q);
            bool ok = true;
            auto issue_qk = [&](const TileCursor& t) -> bool {
                const int b = t.g & 1;
                if (t.j == 0 && !__all_sync(0xffffffffu, wait_or_abort(&bars[Smem::Q_FULL + (t.qi & 1)],
                                                                       (t.qi >> 1) & 1, p.err, abort)))
                    return false;
                if (!__all_sync(0xffffffffu, wait_or_abort(&bars[Smem::FULL_K + b], (t.g >> 1) & 1, p.err, abort)))
                    return false;
                tc_fence_after_sync();
                const uint32_t sb = tmem + TM_S + static_cast<uint32_t>(b) * S_STRIDE;
                const uint64_t ad0 = make_sdesc_sw128(q_base + (t.qi & 1) * Q_BUF, 16, 1024);
                const uint64_t bd0 = make_sdesc_sw128(ring_base + (SLOT_K0 + b) * SLOT, 16, 1024);
                if (elect_one()) {
#pragma unroll
                    for (int k16 = 0; k16 < 16; ++k16) {
                        // head-dim chunk k16 >> 2, 16 columns at a time (start field in 16 B units)
                        const uint64_t off = static_cast<uint64_t>((k16 & 3) * 2);
                        mma2_ss(sb, ad0 + static_cast<uint64_t>((k16 >> 2) * (Q_CHUNK >> 4)) + off,
                                bd0 + static_cast<uint64_t>((k16 >> 2) * (K_BOX >> 4)) + off, IDESC_QK,
                                k16 ? 1u : 0u);
                    }
                    commit2_both(&bars[Smem::S_FULL + b]);
                }
                __syncwarp();
                return true;
            };
            auto issue_pv = [&](const TileCursor& t) -> bool {
                // an item's first PV overwrites O: the softmax warps must have
                // read the previous item's O out of TMEM
                if (t.j == 0 && t.qi >= 1) {
                    if (!__all_sync(0xffffffffu, wait_or_abort(&bars[Smem::O_FREE], (t.qi - 1) & 1, p.err, abort)))
                        return false;
                    tc_fence_after_sync();
                }
                const uint32_t pb = tmem + TM_S + static_cast<uint32_t>(t.g & 1) * S_STRIDE;
                const uint32_t vb = ring_base + SLOT_V * SLOT;
                const uint64_t bd0 = make_sdesc_sw128(vb, V_BOX, 1024);
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk) {
                        // V is MN-major: 64-column boxes V_BOX apart, 8-key groups 1 KiB apart;
                        // P of keys [64 h, 64 h + 64) sits at S columns [64 h, 64 h + 32)
                        const uint64_t bd = bd0 + static_cast<uint64_t>(kk * (16 * 128 >> 4));
                        mma2_ts(tmem + TM_O, pb + (kk >> 2) * BH + (kk & 3) * 8, bd, IDESC_PV,
                                (t.j > 0 || kk > 0) ? 1u : 0u);
                    }
                    commit2_both(&bars[Smem::O_DONE]);
                    if (t.last_of_item()) commit2_both(&bars[Smem::O_FINAL]);
                }
                __syncwarp();
                return true;
            };
            TileCursor cur, nxt;
            cur.first(begin, end, p, 0);
            if (cur.valid) ok = issue_qk(cur);
            while (ok && cur.valid) {
                nxt = cur;
                nxt.advance(p, 0);
                // S of the next tile (of this item or the next) runs while the
                // softmax works on this one; its buffer last held P(g-1)
                if (nxt.valid && !(ok = issue_qk(nxt))) break;
                if (!(ok = __all_sync(0xffffffffu, wait_or_abort(&bars[Smem::P_FULL + (cur.g & 1)], (cur.g >> 1) & 1,
                                                                 p.err, abort))))
                    break;
                tc_fence_after_sync();
                if (!(ok = issue_pv(cur))) break;
                cur = nxt;
            }
            if (elect_one()) commit2_local(&bars[Smem::DRAIN]);
            __syncwarp();
            (void)mbar_wait(&bars[Smem::DRAIN], 0, p.err);
        }
    } else {
        // ---------------------------------------------- softmax + correction + epilogue
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        float* xmax = reinterpret_cast<float*>(smem + Smem::xmax);
        const int row = (warp & 3) * 32 + lane;
        const int kh = warp >= 6 ? 1 : 0;
        const int G = p.group;
        const int tok = row / G;
        const int g_in = row - tok * G;
        const int pair_bar = 1 + (warp & 3);   // named barrier of the two warps of this quadrant
        const bool neg_scale = p.scale_log2 < 0.f;
        bool ok = true;

        // items with no visible key: O = 0, LSE = -inf
        for (int idx = begin; idx < end; idx += p.item_stride) {
            const Item it = item_geometry(idx, p, irank);
            if (it.n_kt != 0 || row >= p.rows_per_tile || tok >= it.ntok) continue;
            const int hq = it.kvh * G + g_in;
            uint4* d4 = reinterpret_cast<uint4*>(p.out + (static_cast<size_t>(it.t0 + tok) * p.n_q_heads + hq) * D +
                                                 kh * 128);
            for (int i = 0; i < 128 / 8; ++i) d4[i] = make_uint4(0u, 0u, 0u, 0u);
            if (kh == 0 && p.lse) p.lse[static_cast<size_t>(hq) * p.seqlen_q + it.t0 + tok] = -INFINITY;
        }

        // Epilogue of an item: wait for its last PV, read O out of TMEM (then
        // the next item's first PV may overwrite it), divide by the row sum
        // and stage it as bf16 in the item's Q buffer in the layout of the
        // output tensor map's box, for the producer's TMA store.  Returns
        // false, in both warps of the quadrant, once either cannot go on.
        auto epilogue = [&](const Item& e, int eqi, float em, float el, float elb) -> bool {
            bool eok = ok;
            if (eok) eok = __all_sync(0xffffffffu, wait_or_abort(&bars[Smem::O_FINAL], eqi & 1, p.err, abort));
            float o_c0 = 0.f, o_c1 = 0.f;   // the two O columns that carry the row sums
            if (eok) {
                tc_fence_after_sync();
                tmem_ld2(tmem + lane_base + TM_O + kh * 128, o_c0, o_c1);
                tmem_ld_wait();
                tmem_st2(tmem + lane_base + TM_O + kh * 128, el, elb);
                tmem_st_wait();
                tc_fence_before_sync();
            }
            // the two warps of the quadrant meet once per item
            if (!bar_and(pair_bar, 64, eok && !*abort)) return false;
            tc_fence_after_sync();
            float l_other, lb_other;
            tmem_ld2(tmem + lane_base + TM_O + (kh ^ 1) * 128, l_other, lb_other);
            tmem_ld_wait();
            const float l_all = el + l_other;
            const float lb_all = elb + lb_other;
            // O / sum(p~) with p~ the rounded weights PV used
            const float inv_l = lb_all > 0.f ? 1.f / lb_all : 0.f;
            uint8_t* stage = smem + Smem::q + (eqi & 1) * Q_BUF + row * 128;
            for (int c = 0; c < 4; ++c) {
                uint32_t o[32];
                tmem_ld32(tmem + lane_base + TM_O + kh * 128 + c * 32, o);
                tmem_ld_wait();
                if (c == 0) {
                    o[0] = __float_as_uint(o_c0);
                    o[1] = __float_as_uint(o_c1);
                }
                if (c == 3) {
                    // every O read of this warp is done
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) {
                        // (relaxed: O was read into registers, nothing to publish)
                        if (rank == 0) mbar_arrive(&bars[Smem::O_FREE]);
                        else mbar_arrive_remote_relaxed(leader_bar(Smem::O_FREE));
                    }
                }
                // 64 bytes of this row: 16-byte units (c & 1) * 4 .. + 3 of
                // column chunk 2 kh + (c >> 1), 128-byte swizzled
                uint8_t* chunk = stage + (kh * 2 + (c >> 1)) * Q_CHUNK;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int unit = ((c & 1) * 4 + u) ^ (row & 7);
                    *reinterpret_cast<uint4*>(chunk + unit * 16) = make_uint4(
                        pack_bf16x2(__uint_as_float(o[8 * u + 0]) * inv_l, __uint_as_float(o[8 * u + 1]) * inv_l),
                        pack_bf16x2(__uint_as_float(o[8 * u + 2]) * inv_l, __uint_as_float(o[8 * u + 3]) * inv_l),
                        pack_bf16x2(__uint_as_float(o[8 * u + 4]) * inv_l, __uint_as_float(o[8 * u + 5]) * inv_l),
                        pack_bf16x2(__uint_as_float(o[8 * u + 6]) * inv_l, __uint_as_float(o[8 * u + 7]) * inv_l));
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[Smem::O_STAGED]);
            if (kh == 0 && p.lse && row < p.rows_per_tile && tok < e.ntok)
                p.lse[static_cast<size_t>(e.kvh * G + g_in) * p.seqlen_q + e.t0 + tok] =
                    l_all > 0.f ? (em + log2f(l_all)) * 0.69314718055994530942f : -INFINITY;
            return true;
        };

        TileCursor cur;
        cur.first(begin, end, p, irank);
        float m_ref = -INFINITY, l = 0.f, l_b = 0.f;
        // the item whose epilogue waits for the next item's first tile
        bool pend = false;
        Item pit;
        int pqi = 0;
        float pm = 0.f, pl = 0.f, plb = 0.f;
        // A failed wait leaves ok false; the warp then skips the remaining
        // work but keeps meeting its partner at each epilogue, where both leave.
        bool met = true;   // the last meeting let both warps go on
        while (cur.valid) {
            const Item& it = cur.it;
            const int g = cur.g;
            const int j = cur.j;
            if (j == 0) {
                m_ref = -INFINITY;
                l = 0.f;
                l_b = 0.f;
            }
            const int b = g & 1;
            const uint32_t ph = static_cast<uint32_t>((g >> 1) & 1);
            if (ok) ok = __all_sync(0xffffffffu, wait_or_abort(&bars[Smem::S_FULL + b], ph, p.err, abort));
            if (ok) {
                tc_fence_after_sync();
                uint32_t sr[2][32];
                const uint32_t s_col = TM_S + static_cast<uint32_t>(b) * S_STRIDE + kh * BH;
                tmem_ld32(tmem + lane_base + s_col, sr[0]);
                tmem_ld32(tmem + lane_base + s_col + 32, sr[1]);
                tmem_ld_wait();
                float s[BH];
#pragma unroll
                for (int c = 0; c < BH; ++c) s[c] = __uint_as_float(sr[c >> 5][c & 31]);

                const int qpos = it.p_first + tok;
                const int key0 = it.key_begin + j * BN + kh * BH;
                const bool half_full = it.ntok > 0 && key0 + BH <= p.seqlen_k &&
                                       (!p.causal || key0 + BH - 1 <= it.p_first) &&
                                       (p.window <= 0 || key0 > it.p_last - p.window);
                if (!half_full) {
                    const float hidden = neg_scale ? INFINITY : -INFINITY;
#pragma unroll
                    for (int c = 0; c < BH; ++c)
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
                const float own_max = mx[0] * p.scale_log2;
                xmax[(b * 2 + kh) * BM + row] = own_max;
                __syncwarp();
                const int xb = Smem::XCHG + b * 4 + (warp & 3);      // one arrival per warp
                if (lane == 0) mbar_arrive(&bars[xb]);
                ok = __all_sync(0xffffffffu, wait_or_abort(&bars[xb], ph, p.err, abort));
                if (ok) {
                    const float tmax = fmaxf(own_max, xmax[(b * 2 + (kh ^ 1)) * BM + row]);
                    float m_use = m_ref, alpha = 1.f;
                    if (tmax > m_ref + RESCALE_THRESHOLD) {
                        m_use = tmax;
                        alpha = fast_exp2(m_ref - m_use);
                    }
                    const float shift = m_use == -INFINITY ? 0.f : m_use;
                    uint32_t pk[BH / 2];
                    float2 ps[4], pbs[4];
#pragma unroll
                    for (int c = 0; c < 4; ++c) ps[c] = pbs[c] = make_float2(0.f, 0.f);
                    const float2 sl2 = make_float2(p.scale_log2, p.scale_log2);
                    const float2 nsh = make_float2(-shift, -shift);
#pragma unroll
                    for (int c = 0; c < BH / 2; ++c) {
                        const float2 x = ffma2(make_float2(s[2 * c], s[2 * c + 1]), sl2, nsh);
                        const float2 pr = make_float2(fast_exp2(x.x), fast_exp2(x.y));
                        ps[c & 3] = fadd2(ps[c & 3], pr);
                        pk[c] = pack_bf16x2(pr.x, pr.y);
                        pbs[c & 3] = fadd2(pbs[c & 3], make_float2(__uint_as_float(pk[c] << 16),
                                                                   __uint_as_float(pk[c] & 0xffff0000u)));
                    }
                    const float2 ps01 = fadd2(fadd2(ps[0], ps[1]), fadd2(ps[2], ps[3]));
                    const float2 pb01 = fadd2(fadd2(pbs[0], pbs[1]), fadd2(pbs[2], pbs[3]));
                    l = l * alpha + (ps01.x + ps01.y);
                    l_b = l_b * alpha + (pb01.x + pb01.y);
                    m_ref = m_use;
                    if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                        // PV of the previous tile must be done before O is corrected
                        ok = __all_sync(0xffffffffu, wait_or_abort(&bars[Smem::O_DONE],
                                                                   static_cast<uint32_t>((g - 1) & 1), p.err, abort));
                        if (ok) {
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
                    }
                    if (ok) {
                        // P of this key half overwrites the first 32 of its own 64 S columns
                        tmem_st32(tmem + lane_base + s_col, pk);
                        tmem_st_wait();
                        tc_fence_before_sync();
                        __syncwarp();
                        if (lane == 0) {
                            // (relaxed: P went to TMEM by completed tensor-core
                            // stores, nothing to publish; a release here would
                            // hold the warp about a microsecond every tile)
                            if (rank == 0) mbar_arrive(&bars[Smem::P_FULL + b]);
                            else mbar_arrive_remote_relaxed(leader_bar(Smem::P_FULL + b));
                        }
                    }
                }
            }
            // the previous item's epilogue, now that this item's first P is on its way
            if (j == 0 && pend) {
                pend = false;
                if (!(met = epilogue(pit, pqi, pm, pl, plb))) break;
            }
            if (cur.last_of_item()) {
                pend = true;
                pit = it;
                pqi = cur.qi;
                pm = m_ref;
                pl = l;
                plb = l_b;
            }
            cur.advance(p, irank);
        }
        if (pend && met) (void)epilogue(pit, pqi, pm, pl, plb);
    }

    tc_fence_before_sync();
    __syncthreads();
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc2(tmem, 512);
    }
}

}  // namespace local256

int prefill256_smem_bytes() { return local256::Smem::total; }
int prefill256_k_box_rows() { return local256::K_BOX_ROWS; }
int prefill256_v_box_rows() { return local256::V_BOX_ROWS; }

// Deals the items (KV head major, pairs in order) round-robin to at most
// kMaxPersistentClusters clusters: cluster c takes items c, c + n, c + 2n, ...
// At any time the clusters then work on neighbouring q-tile pairs of one KV
// head, whose key window the L2 holds once for all of them (a contiguous
// range per cluster spread the clusters over every part of the sequence, and
// their windows did not fit).  Items cost about the same (a window of
// tiles), so the deal also balances the work.
void plan_prefill256(Prefill256Params& p, int n_sm) {
    const int max_clusters = std::min(kMaxPersistentClusters, std::max(1, n_sm / 2));
    const int n_clusters = std::max(1, std::min(max_clusters, p.n_items));
    p.n_clusters = n_clusters;
    p.item_stride = n_clusters;
    for (int c = 0; c < n_clusters; ++c) p.range_start[c] = c;
    p.range_start[n_clusters] = p.n_items;
}

cudaError_t launch_prefill256(const CUtensorMap& tmq, const CUtensorMap& tmk, const CUtensorMap& tmv,
                              const CUtensorMap& tmo, const Prefill256Params& p, cudaStream_t stream) {
    const int smem = prefill256_smem_bytes();
    cudaError_t e = cudaFuncSetAttribute(local256::prefill256_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    local256::prefill256_kernel<<<2 * p.n_clusters, local256::NUM_THREADS, smem, stream>>>(tmq, tmk, tmv, tmo, p);
    return cudaGetLastError();
}

}  // namespace fa512

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
//     resident, computes S = Q K^T with 2-SM MMAs (tcgen05 cta_group::2,
//     M256 x N128, each CTA holding 64 of a tile's 128 keys) into S buffers
//     in TMEM, and runs the online softmax;
//   * the output pair (ranks 2, 3) keeps the whole fp32 O of its q tile in
//     TMEM and computes O += P V with 2-SM MMAs (M256 x N256 per O half,
//     each CTA holding 128 of the half's 256 V columns), P read from its
//     shared memory.
//
// Every score CTA sends the bf16 P of each tile (and the per-row rescale
// factor alpha) to the output CTA with the same q tile through distributed
// shared memory.  S is computed once, so the tensor pipes execute the
// algorithmic FLOP only: the score pair 2 x 128 x 128 x 512 and the output
// pair 2 x 128 x 128 x 512 multiply-adds per key tile.  (The pages split the
// head dimension across warps of one SM, "Head dim 512 breaks the textbook"
// and step 2 of the RTX PRO 6000 page; here the split is between the two
// products.)
//
// Score pair (per CTA: the whole 128 x 512 bf16 Q tile in TMEM, 256
// columns, as the A operand of every QK^T, so that each MMA reads only K from
// shared memory; two S buffers in the other 256 columns): K streams through
// five 32 KiB slots (a half tile: this CTA's 64 keys x 256 head-dim columns),
// each released by the commit after its 16 MMAs; the MMA thread holds back a
// tile's QK^T until its S buffer has been read (the K loads run ahead).  Q lands in the last
// two K slots and the P staging area, and the MMA thread copies it into TMEM
// (tcgen05.cp, ahead of its first MMA) before either is needed.  Eight softmax warps: TMEM lane quadrant (warp % 4) gives a warp
// its 32 rows, warps 2-5 take keys 0-63 of each tile and warps 6-9 keys
// 64-127; they swap row maxima through shared memory.  The row max is lazy: O is rescaled only
// when a row's max grows by more than 2^16.  P goes to one of two staging
// buffers; a copy warp moves each staged tile with one bulk copy (the copy
// engine) into the output CTA, where it completes on that CTA's mbarrier;
// alpha follows by remote stores on the same barrier.
//
// Output pair (per CTA: the whole 128 x 512 fp32 O in TMEM): V streams
// through four 32 KiB slots (two tiles x two O halves), P lands in three
// buffers; the commit after a tile's 16 MMAs (M256 x N256 per O half, P and
// V from shared memory) is multicast to all four CTAs and frees that tile's
// V slots and P buffer and lets O be corrected for the next tile.  Eight
// correction warps apply alpha to O in TMEM (tcgen05.ld / st) when a row's
// max moved, then mark the tile ready; at the end they normalise O by the
// sum of the bf16 P values and write bf16 rows.
//
// A cluster-scope mbarrier arrival with release semantics stalls the thread
// that makes it for about a microsecond.  The per-tile signals to another CTA
// ("S read", "alpha read", "tile ready") publish no memory writes -- the
// values were loaded into registers, or the tensor-core stores completed --
// so the warps make them as relaxed arrivals, which cost no such stall; only
// a paged tail tile, whose cleared V rows the MMA must see, takes a release.
//
// Causal / sliding-window tile skipping over the pair's visible band; only
// the key parts that cross a row's band edge are masked element by
// element.
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
namespace prefill_so {
using namespace pair;

constexpr int D = 512;
constexpr int BM = 128;                  // packed rows per CTA tile
constexpr int BN = 128;                  // keys per KV tile
constexpr int N_WORK_WARPS = 8;          // warps 2-9
constexpr int COPY_WARP = 2 + N_WORK_WARPS;   // score CTAs: moves each staged P tile to the output CTA
constexpr int NUM_THREADS = (3 + N_WORK_WARPS) * 32;
constexpr int PARTS = N_WORK_WARPS / 4;  // warps per TMEM lane quadrant
constexpr int KP = BN / PARTS;           // score CTAs: keys of a tile per softmax warp (32)
constexpr int OP = D / PARTS;            // output CTAs: O columns per correction warp (128)
constexpr int Q_CHUNK = BM * 128;        // one 64-column box of Q: 16 KiB
constexpr int SLOT = 32768;
constexpr int K_SLOTS = 5;               // score CTAs: K half tiles
constexpr int K_BOX_ROWS = BN / 2;       // {64 columns, 64 keys} boxes
constexpr int K_BOX = K_BOX_ROWS * 128;  // 8 KiB
constexpr int S_BUFS = 2;                // S buffers of 128 TMEM columns
constexpr uint32_t TM_Q = S_BUFS * BN;   // the Q tile: head-dim column d in TMEM column TM_Q + d / 2
constexpr int Q_PARK_SLOT = K_SLOTS - 2; // Q chunks 0-3 land in K slots 3-4, chunks 4-7 in the staging area
constexpr int V_SLOTS = 4;               // output CTAs: 2 tiles x 2 O halves
constexpr int V_BOX_ROWS = BN;           // {64 columns, 128 keys} boxes
constexpr int V_BOX = V_BOX_ROWS * 128;  // 16 KiB
constexpr int P_CHUNK = BM * 128;        // P of 64 keys for 128 rows, bf16: 16 KiB
constexpr int P_BUF = 2 * P_CHUNK;       // one tile's P: 32 KiB
constexpr int P_BUFS = 3;                // output CTAs: P buffers
constexpr int STAGES = 2;                // score CTAs: P staging buffers
constexpr uint32_t P_TX = P_BUF + BM * 4;   // bytes landing per tile: P and alpha
constexpr uint32_t L_TX = BM * 4;           // the final row sums
static_assert((PARTS == 2 || PARTS == 4) && KP % 32 == 0, "two or four work warps per lane quadrant");

// Rescale O only when the row max grows by more than this (log2 units);
// until then the stale max stays the reference and p <= 2^16 (bf16 and the
// fp32 sums hold that range).  A rescale makes the output pair wait for the
// previous tile's O += P V, so rows that keep finding larger maxima (the
// stress rows) pay for each one: 2^16 measured faster than 2^8, 2^12 and 2^20.
constexpr float RESCALE_THRESHOLD = 16.0f;

constexpr uint16_t MASK_SCORE = 0x3, MASK_OUTPUT = 0xC, MASK_ALL = 0xF;

struct Smem {
    // score CTAs: the Q tile lands in the last two K slots and the staging
    // area and moves to TMEM before either is used for K or P
    static constexpr int kring = 0;                             // 5 x 32 KiB
    static constexpr int stage = kring + K_SLOTS * SLOT;        // 2 x 32 KiB
    static constexpr int xmax = stage + STAGES * P_BUF;         // [2 buffers][PARTS][128] f32
    // output CTAs
    static constexpr int vring = 0;                             // 4 x 32 KiB
    static constexpr int precv = vring + V_SLOTS * SLOT;        // 3 x 32 KiB
    static constexpr int alpha = precv + P_BUFS * P_BUF;        // [3][128] f32
    static constexpr int lrecv = alpha + P_BUFS * BM * 4;       // [128] f32
    // both
    // (2 KiB after the staging / P buffers: the score CTAs' row-max swap, the
    // output CTAs' alpha and row sums)
    static constexpr int bars = xmax + 2048;
    enum {
        K_FULL = 0,                      // [5] score leader: both CTAs' half tile landed
        K_EMPTY = K_FULL + K_SLOTS,      // [5] score CTAs: the slot's MMAs completed
        S_FULL = K_EMPTY + K_SLOTS,      // [2] score CTAs: S of the tile is in TMEM
        S_FREE = S_FULL + S_BUFS,        // [2] score leader: both CTAs' softmax warps read S
        XCHG = S_FREE + S_BUFS,          // [2][4] score CTAs: row-max swap of one lane quadrant's key parts
        Q_FULL = XCHG + 8,               // score leader: both CTAs' Q tiles landed (K slots 3-4, staging area)
        Q_COPIED = Q_FULL + 1,           // score CTAs: the Q tile was copied into TMEM (commit of the copies)
        P_STAGED = Q_COPIED + 1,         // [2] score CTAs: all softmax warps staged the tile's P
        STAGE_FREE = P_STAGED + STAGES,  // [2] score CTAs: the buffer's last copy landed, its alpha read
        S_READ = STAGE_FREE + STAGES,    // [2] score CTA 1: its softmax warps read S (forwarded to S_FREE)
        L_XCHG = S_READ + S_BUFS,        // score CTAs: row-sum swap
        PV_DONE = L_XCHG + 1,            // [3] all four: O += P V of the P buffer's last tile completed
        PV_READY = PV_DONE + P_BUFS,     // [3] output leader: P landed and O corrected in both, V landed
        P_LANDED = PV_READY + P_BUFS,    // [3] output CTAs: P and alpha of the tile arrived
        O_FINAL = P_LANDED + P_BUFS,     // output CTAs: the last O += P V completed
        L_READY = O_FINAL + 1,           // output CTAs: the row sums arrived
        V_TAIL = L_READY + 1,            // paged, output CTAs: this CTA's V of the tile holding the cache's end landed
        DRAIN = V_TAIL + 1,              // every MMA this CTA issued has completed
        N_BARS = DRAIN + 1
    };
    static constexpr int tmem_addr = bars + N_BARS * 8;
    static constexpr int abort_flag = tmem_addr + 4;
    static constexpr int skip_flag = abort_flag + 4;             // written by rank 0 into all four
    static constexpr int total = skip_flag + 4;
};
static_assert(Smem::lrecv + BM * 4 <= Smem::bars && Smem::xmax + 2 * PARTS * BM * 4 <= Smem::bars, "layout");
static_assert(Smem::kring % 1024 == 0 && Smem::precv % 1024 == 0, "swizzled buffers on 1 KiB");
// The dynamic shared-memory window starts 1 KiB aligned (checked at run
// time), which the 128-byte swizzle atoms need.
static_assert(Smem::total <= 232448, "shared memory budget");

constexpr uint32_t IDESC_QK = make_idesc_bf16(2 * BM, BN, 0);
constexpr uint32_t IDESC_PV = make_idesc_bf16(2 * BM, 256, 1);

__device__ __forceinline__ bool key_visible(int j, int qpos, int seqlen_k, const PrefillParams& p) {
    return j < seqlen_k && (!p.causal || j <= qpos) && (p.window <= 0 || j > qpos - p.window);
}

// Commit of every MMA issued so far by this thread, arriving on the barrier
// at this offset in each CTA of `mask` (cluster ranks).
__device__ __forceinline__ void commit2_mask(uint64_t* bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
        ::"r"(smem_u32(bar)), "h"(mask)
        : "memory");
}

// 4 bytes into another CTA's shared memory; the bytes complete_tx on that
// CTA's mbarrier (both addresses shared::cluster, in the same CTA).
__device__ __forceinline__ void st_async_b32(uint32_t addr, uint32_t a, uint32_t bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];"
                 ::"r"(addr), "r"(a), "r"(bar)
                 : "memory");
}

// Bulk copy of `bytes` from this CTA's shared memory to another CTA's (copy
// engine); the bytes complete_tx on the destination CTA's mbarrier.
__device__ __forceinline__ void bulk_copy_to_cluster(uint32_t dst_cluster, uint32_t src_cta, uint32_t bytes,
                                                     uint32_t bar_cluster) {
    asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst_cluster), "r"(src_cta), "r"(bytes), "r"(bar_cluster)
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

// PAGED: a batch of chunks (varlen rows through cu_seqlens_q) over a paged
// cache; K and V rows are found through the page table one 64-key half tile
// at a time (a page holds a whole number of half tiles).
template <bool PAGED>
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
    const int item = blockIdx.x >> 2;
    int kvh, pair, seq = 0, q_start = 0;
    int seqlen_q = p.seqlen_q, seqlen_k = p.seqlen_k, q_offset = p.q_offset;
    if constexpr (PAGED) {
        // Work items are numbered sequence by sequence, KV head by KV head,
        // heaviest pair first, with no gaps: warp 0 finds this cluster's
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
        if (seq < 0) return;                            // past the last item: all four CTAs
        const int off = found[1];
        q_start = found[2];
        seqlen_q = min(found[3] - q_start, p.max_seqlen_q);
        seqlen_k = found[4];
        const int n_pairs_seq = (seqlen_q + two_t - 1) / two_t;
        kvh = off / n_pairs_seq;
        pair = n_pairs_seq - 1 - (off - kvh * n_pairs_seq);   // 0 = heaviest pair first
        q_offset = seqlen_k - (found[3] - q_start);    // the chunk is its sequence's tail
        const int kv_cap = p.max_pages_per_seq << p.page_shift;
        if (seqlen_k < 0 || seqlen_k > kv_cap) {
            // recorded once per sequence; read up to the table's capacity
            if (tid == 0 && off == 0) report_error(p.err, FA512_DEVICE_ERR_INDEX);
            seqlen_k = seqlen_k < 0 ? 0 : kv_cap;
        }
        __syncthreads();                                // the scratch is reused below
    } else {
        const int n_pairs = (p.num_q_tiles + 1) / 2;
        kvh = item / n_pairs;
        pair = n_pairs - 1 - item % n_pairs;
    }
    const int qt = 2 * pair + static_cast<int>(pr);    // may be one past the last tile: no rows
    const int t0 = qt * T;
    const int ntok = min(T, seqlen_q - t0);             // <= 0 for a missing second tile
    const int p_first = q_offset + t0;
    const int p_last = q_offset + t0 + ntok - 1;
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
    // Row of the tensor map holding the first key of the 64-key half tile
    // that starts at logical key `key`: the key itself, or in paged mode its
    // slot in the pool.  Halves past the cache's end (and pages outside the
    // pool) read a row past the pool, which the TMA unit fills with zeros.
    // Paged: the producers load a half tile's page-table entry (page_entry)
    // several tiles before they need its row (half_row), so the dependent
    // load is off their critical path.
    auto page_entry = [&](int key) -> int {
        if constexpr (PAGED) {
            return key < seqlen_k
                       ? p.page_table[static_cast<size_t>(seq) * p.max_pages_per_seq + (key >> p.page_shift)]
                       : 0;
        } else {
            return 0;
        }
    };
    auto half_row = [&](int key, int pg) -> int {
        if constexpr (PAGED) {
            if (key >= seqlen_k) return p.oob_row;
            if (static_cast<unsigned>(pg) >= static_cast<unsigned>(p.num_pages)) {
                report_error(p.err, FA512_DEVICE_ERR_INDEX);
                return p.oob_row;
            }
            return (pg << p.page_shift) + (key & ((1 << p.page_shift) - 1));
        } else {
            return key;
        }
    };
    constexpr int PF = 4;   // paged: tiles whose page-table entries a producer holds ahead

    // this thread's packed row and part (warps 2-17): TMEM lane quadrant
    // warp % 4; part = 32 keys of a tile in the score CTAs, 128 O columns in
    // the output CTAs
    const bool work_warp = warp >= 2 && warp < COPY_WARP;
    const int row = (warp & 3) * 32 + lane;
    const int part = (warp - 2) >> 2;
    const int tok = row / G;
    const int g = row - tok * G;
    const bool valid_row = work_warp && row < p.rows_per_tile && tok < ntok;
    const int qpos = q_offset + t0 + tok;
    const int hq = kvh * G + g;

    if (n_kt == 0) {
        // no key is visible to any row of the pair: O = 0, LSE = -inf
        if (valid_row) {
            if (!scorer) {
                uint4* dst = reinterpret_cast<uint4*>(
                    p.out + (static_cast<size_t>(q_start + t0 + tok) * p.n_q_heads + hq) * D + part * OP);
                for (int i = 0; i < OP / 8; ++i) dst[i] = make_uint4(0u, 0u, 0u, 0u);
            } else if (part == 0 && p.lse) {
                p.lse[static_cast<size_t>(hq) * p.total_q + q_start + t0 + tok] = -INFINITY;
            }
        }
        return;
    }

    if (warp == 0 && lane == 0) {
        for (int i = 0; i < Smem::N_BARS; ++i) {
            uint32_t count = 1;
            if (i == Smem::L_XCHG) count = N_WORK_WARPS;
            if (i >= Smem::XCHG && i < Smem::XCHG + 8) count = PARTS;   // the warps sharing a lane quadrant
            // the leader's softmax warps, plus one forwarded arrival for the other CTA's
            if (i >= Smem::S_FREE && i < Smem::S_FREE + S_BUFS) count = N_WORK_WARPS + 1;
            // this CTA's softmax warps; the output CTA's correction warps
            if ((i >= Smem::P_STAGED && i < Smem::P_STAGED + STAGES) ||
                (i >= Smem::STAGE_FREE && i < Smem::STAGE_FREE + STAGES) ||
                (i >= Smem::S_READ && i < Smem::S_READ + S_BUFS))
                count = N_WORK_WARPS;
            // the correction warps of both output CTAs, plus the V load
            if (i >= Smem::PV_READY && i < Smem::PV_READY + P_BUFS) count = 2 * N_WORK_WARPS + 1;
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
                // Q is read once; K and V are read by every pair of the KV head
                const uint64_t pol_q = l2_policy_stream(), pol_kv = l2_policy_keep();
                const uint32_t q_bytes = static_cast<uint32_t>(8 * 128 * p.rows_per_tile);   // 8 boxes
                if (rank == 0) mbar_arrive_expect_tx(&bars[Smem::Q_FULL], 2 * q_bytes);
                for (int c = 0; c < 8; ++c)
                    tma2_load_4d_hint(smem + (c < 4 ? Smem::kring + Q_PARK_SLOT * SLOT + c * Q_CHUNK
                                                    : Smem::stage + (c - 4) * Q_CHUNK),
                                      &tmq, bar_of(Smem::Q_FULL, 0), c * 64, 0, kvh, q_start + t0, pol_q);
                // half tile h: tile h / 2, head-dim columns 256 (h % 2) .. +256, this CTA's 64 keys
                auto k_key = [&](int j) { return (kt_begin + j) * BN + static_cast<int>(pr) * K_BOX_ROWS; };
                int pf[PF];
#pragma unroll
                for (int i = 0; i < PF; ++i) pf[i] = i < n_kt ? page_entry(k_key(i)) : 0;
                int krow = 0;
                for (int h = 0; h < 2 * n_kt; ++h) {
                    const int j = h >> 1, c = h & 1, s = h % K_SLOTS;
                    if (h >= K_SLOTS && !wait_or_abort(&bars[Smem::K_EMPTY + s], ((h / K_SLOTS) - 1) & 1, p.err,
                                                       abort, wait_ns))
                        break;
                    // the slots that held Q: once Q has been copied into TMEM
                    if (h == Q_PARK_SLOT && !wait_or_abort(&bars[Smem::Q_COPIED], 0, p.err, abort, wait_ns)) break;
                    if (rank == 0) mbar_arrive_expect_tx(&bars[Smem::K_FULL + s], 2 * SLOT);
                    if (c == 0) {
                        // both head-dim halves of tile j read the same keys
                        krow = half_row(k_key(j), pf[0]);
#pragma unroll
                        for (int i = 0; i < PF - 1; ++i) pf[i] = pf[i + 1];
                        pf[PF - 1] = j + PF < n_kt ? page_entry(k_key(j + PF)) : 0;
                    }
                    // (test hook: the first cluster's rank 0 leaves out its first
                    // K half tile, so that cluster's waits run into their bound)
                    if (h == 0 && p.test_skip_first_k_load && blockIdx.x == 0) continue;
                    for (int b = 0; b < 4; ++b)
                        tma2_load_3d_hint(smem + Smem::kring + s * SLOT + b * K_BOX, &tmk,
                                          bar_of(Smem::K_FULL + s, 0), (c * 4 + b) * 64, kvh, krow, pol_kv);
                }
            }
        } else if (warp == 1 && rank == 1) {
            if (lane == 0) {
                // -------------------------------------------------- forward "S read" to the leader
                // (the softmax warps arrive locally: a remote arrival, even a
                // relaxed one, measured slower on their critical path)
                for (int j = 0; j < n_kt; ++j) {
                    if (!wait_or_abort(&bars[Smem::S_READ + (j % S_BUFS)], (j / S_BUFS) & 1, p.err, abort, wait_ns))
                        break;
                    mbar_arrive_remote_relaxed(bar_of(Smem::S_FREE + (j % S_BUFS), 0));
                }
            }
        } else if (warp == 1) {
            if (rank == 0) {
                // -------------------------------------------------- S = Q K^T (both SMs)
                // The whole warp runs the loop and its waits (warp-uniform, so
                // the MMA operands stay uniform); one elected lane issues.
                // Q of both CTAs into TMEM (the A operand of every QK^T): 32
                // copies of a 16-column slice, in the tensor-core pipeline
                // ahead of the first MMA; their commit frees the parking slots
                bool ok = __all_sync(0xffffffffu, wait_or_abort(&bars[Smem::Q_FULL], 0, p.err, abort, wait_ns));
                if (ok) {
                    tc_fence_after_sync();
                    if (elect_one()) {
#pragma unroll
                        for (int c8 = 0; c8 < 8; ++c8) {
                            const uint64_t qd = make_sdesc_sw128(
                                smem_u32(smem + (c8 < 4 ? Smem::kring + Q_PARK_SLOT * SLOT + c8 * Q_CHUNK
                                                        : Smem::stage + (c8 - 4) * Q_CHUNK)),
                                16, 1024);
#pragma unroll
                            for (int piece = 0; piece < 4; ++piece)
                                tmem_cp2_128x256b(tmem + TM_Q + static_cast<uint32_t>(c8 * 32 + piece * 8),
                                                  qd + static_cast<uint64_t>(piece * 2));
                        }
                        commit2_mask(&bars[Smem::Q_COPIED], MASK_SCORE);
                    }
                    __syncwarp();
                }
                const uint64_t k_desc = make_sdesc_sw128(smem_u32(smem + Smem::kring), 16, 1024);
                for (int j = 0; ok && j < n_kt; ++j) {
                    const uint32_t sb = tmem + static_cast<uint32_t>(j % S_BUFS) * BN;
                    // the tile's S buffer must have been read before its QK^T may start
                    if (j >= S_BUFS && !(ok = __all_sync(0xffffffffu, wait_or_abort(&bars[Smem::S_FREE + (j % S_BUFS)],
                                                                                    ((j / S_BUFS) - 1) & 1, p.err,
                                                                                    abort, wait_ns))))
                        break;
                    for (int c = 0; c < 2; ++c) {
                        const int h = 2 * j + c, s = h % K_SLOTS;
                        if (!(ok = __all_sync(0xffffffffu, wait_or_abort(&bars[Smem::K_FULL + s], (h / K_SLOTS) & 1,
                                                                         p.err, abort, wait_ns))))
                            break;
                        tc_fence_after_sync();
                        const uint64_t bd0 = k_desc + static_cast<uint64_t>(s * (SLOT >> 4));
                        if (elect_one()) {
#pragma unroll
                            for (int k16 = 0; k16 < 16; ++k16) {
                                // head-dim columns 256 c + 16 k16 .. +16: Q from TMEM (two bf16 a
                                // column), K from its box k16 / 4 (start field in 16 B units)
                                const uint64_t off = static_cast<uint64_t>((k16 & 3) * 2);
                                mma2_ts(sb, tmem + TM_Q + static_cast<uint32_t>(c * 128 + k16 * 8),
                                        bd0 + static_cast<uint64_t>((k16 >> 2) * (K_BOX >> 4)) + off, IDESC_QK,
                                        (c | k16) ? 1u : 0u);
                            }
                            commit2_mask(&bars[Smem::K_EMPTY + s], MASK_SCORE);
                            if (c == 1) commit2_mask(&bars[Smem::S_FULL + (j % S_BUFS)], MASK_SCORE);
                        }
                        __syncwarp();
                    }
                }
                // let every issued MMA finish before TMEM can be released
                if (elect_one()) commit2_mask(&bars[Smem::DRAIN], static_cast<uint16_t>(1u << rank));
                __syncwarp();
                (void)mbar_wait(&bars[Smem::DRAIN], 0, p.err, wait_ns);
            }
        } else if (warp == COPY_WARP) {
            if (lane == 0) {
                // -------------------------------------------------- P tiles to the output CTA
                const uint32_t out_rank = rank + 2;
                for (int j = 0; j < n_kt; ++j) {
                    const int b2 = j & 1, pb = j % P_BUFS;
                    // all softmax warps staged tile j, and the output CTA's P
                    // buffer pb is free (O += P V of tile j - 3 completed)
                    if (!wait_or_abort(&bars[Smem::P_STAGED + b2], (j >> 1) & 1, p.err, abort, wait_ns)) break;
                    if (j >= P_BUFS &&
                        !wait_or_abort(&bars[Smem::PV_DONE + pb], ((j / P_BUFS) - 1) & 1, p.err, abort, wait_ns))
                        break;
                    bulk_copy_to_cluster(map_to_cta(smem_u32(smem + Smem::precv + pb * P_BUF), out_rank),
                                         smem_u32(smem + Smem::stage + b2 * P_BUF), P_BUF,
                                         bar_of(Smem::P_LANDED + pb, out_rank));
                }
            }
        } else {
            // ------------------------------------------------------ softmax
            float* xmax = reinterpret_cast<float*>(smem + Smem::xmax);
            float m_ref = -INFINITY;   // log2 units, the same in all four parts
            float l = 0.f;             // this part's sum of the fp32 probabilities (for LSE)
            float l_b = 0.f;           // this part's sum of the bf16-rounded probabilities
            bool ok = true;
            const bool neg_scale = p.scale_log2 < 0.f;
            const uint32_t out_rank = rank + 2;
            const uint32_t a_dst = map_to_cta(smem_u32(smem + Smem::alpha + row * 4), out_rank);

            for (int j = 0; ok && j < n_kt; ++j) {
                const int b3 = j % S_BUFS, b2 = j & 1, pb = j % P_BUFS;
                // (every wait of a softmax warp is made warp-uniform: the warp
                // synchronises below and must leave the loop as one)
                if (!(ok = __all_sync(0xffffffffu, wait_or_abort(&bars[Smem::S_FULL + b3], (j / S_BUFS) & 1, p.err,
                                                                 abort, wait_ns))))
                    break;
                tc_fence_after_sync();
                uint32_t sr[KP];
#pragma unroll
                for (int c = 0; c < KP / 32; ++c)
                    tmem_ld32(tmem + lane_base + static_cast<uint32_t>(b3 * BN + part * KP + 32 * c),
                              *reinterpret_cast<uint32_t(*)[32]>(sr + 32 * c));
                tmem_ld_wait();
                // the S buffer may take the QK^T three tiles on
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[rank == 0 ? Smem::S_FREE + b3 : Smem::S_READ + b3]);
                float s[KP];
#pragma unroll
                for (int c = 0; c < KP; ++c) s[c] = __uint_as_float(sr[c]);

                const int key0 = (kt_begin + j) * BN + part * KP;
                const bool part_full = ntok > 0 && key0 + KP <= seqlen_k &&
                                       (!p.causal || key0 + KP - 1 <= p_first) &&
                                       (p.window <= 0 || key0 > p_last - p.window);
                // scores stay unscaled until the exponent; a hidden key gets the
                // value that scales to -inf whatever the sign of the scale
                if (!part_full) {
                    const float hidden = neg_scale ? INFINITY : -INFINITY;
#pragma unroll
                    for (int c = 0; c < KP; ++c)
                        if (!key_visible(key0 + c, qpos, seqlen_k, p)) s[c] = hidden;
                }
                float mx[KP / 4];
                if (!neg_scale) {
#pragma unroll
                    for (int c = 0; c < KP / 4; ++c)
                        mx[c] = fmaxf(fmaxf(s[4 * c], s[4 * c + 1]), fmaxf(s[4 * c + 2], s[4 * c + 3]));
#pragma unroll
                    for (int w = KP / 8; w >= 1; w >>= 1)
#pragma unroll
                        for (int c = 0; c < w; ++c) mx[c] = fmaxf(mx[c], mx[c + w]);
                } else {
#pragma unroll
                    for (int c = 0; c < KP / 4; ++c)
                        mx[c] = fminf(fminf(s[4 * c], s[4 * c + 1]), fminf(s[4 * c + 2], s[4 * c + 3]));
#pragma unroll
                    for (int w = KP / 8; w >= 1; w >>= 1)
#pragma unroll
                        for (int c = 0; c < w; ++c) mx[c] = fminf(mx[c], mx[c + w]);
                }
                // row max over the whole tile: the parts swap their maxima (log2
                // units); all then take the same decision on the same numbers
                const float own_max = mx[0] * p.scale_log2;
                xmax[(b2 * PARTS + part) * BM + row] = own_max;
                // one arrival per warp, after the warp's stores; only the PARTS
                // warps of this lane quadrant hold parts of these rows
                __syncwarp();
                const int xb = Smem::XCHG + b2 * 4 + (warp & 3);
                if (lane == 0) mbar_arrive(&bars[xb]);
                if (!(ok = __all_sync(0xffffffffu, wait_or_abort(&bars[xb], (j >> 1) & 1, p.err, abort,
                                                                 wait_ns))))
                    break;
                float tmax = own_max;
#pragma unroll
                for (int q4 = 1; q4 < PARTS; ++q4)
                    tmax = fmaxf(tmax, xmax[(b2 * PARTS + ((part + q4) % PARTS)) * BM + row]);

                float m_use = m_ref, alpha = 1.f;
                if (tmax > m_ref + RESCALE_THRESHOLD) {
                    m_use = tmax;
                    alpha = fast_exp2(m_ref - m_use);   // 0 when m_ref = -inf
                }
                const float shift = m_use == -INFINITY ? 0.f : m_use;
                uint32_t pk[KP / 2];
                float2 ps[4], pbs[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) ps[c] = pbs[c] = make_float2(0.f, 0.f);
                const float2 sl2 = make_float2(p.scale_log2, p.scale_log2);
                const float2 nsh = make_float2(-shift, -shift);
#pragma unroll
                for (int c = 0; c < KP / 2; ++c) {
                    // p = 2^(s * scale * log2(e) - shift), two lanes per instruction
                    const float2 x = ffma2(make_float2(s[2 * c], s[2 * c + 1]), sl2, nsh);
                    const float2 pr2 = make_float2(fast_exp2(x.x), fast_exp2(x.y));
                    ps[c & 3] = fadd2(ps[c & 3], pr2);
                    pk[c] = pack_bf16x2(pr2.x, pr2.y);
                    // the bf16 values the PV product actually uses
                    pbs[c & 3] = fadd2(pbs[c & 3], make_float2(__uint_as_float(pk[c] << 16),
                                                               __uint_as_float(pk[c] & 0xffff0000u)));
                }
                const float2 ps01 = fadd2(fadd2(ps[0], ps[1]), fadd2(ps[2], ps[3]));
                const float2 pb01 = fadd2(fadd2(pbs[0], pbs[1]), fadd2(pbs[2], pbs[3]));
                l = l * alpha + (ps01.x + ps01.y);
                l_b = l_b * alpha + (pb01.x + pb01.y);
                m_ref = m_use;

                // staging buffer b2: its copy of tile j - 2 has landed and the
                // output CTA has read that tile's alpha (which also means its
                // barrier phase for tile j - 3 has completed)
                if (j >= STAGES && !(ok = __all_sync(0xffffffffu, wait_or_abort(&bars[Smem::STAGE_FREE + b2],
                                                                               ((j >> 1) - 1) & 1, p.err, abort,
                                                                               wait_ns))))
                    break;
                // P of this row's KP keys: KP / 8 16-byte pieces of the row's
                // 128-byte line in its 64-key chunk, in the 128-byte swizzle the
                // MMA descriptor expects (piece c at c ^ (row % 8))
                uint8_t* stg = smem + Smem::stage + b2 * P_BUF + ((part * KP) >> 6) * P_CHUNK + row * 128;
#pragma unroll
                for (int c4 = 0; c4 < KP / 8; ++c4) {
                    const int pc = ((part * KP) & 63) / 8 + c4;
                    *reinterpret_cast<uint4*>(stg + ((pc ^ (row & 7)) << 4)) =
                        make_uint4(pk[4 * c4], pk[4 * c4 + 1], pk[4 * c4 + 2], pk[4 * c4 + 3]);
                }
                const uint32_t xbar = bar_of(Smem::P_LANDED + pb, out_rank);
                if (part == 0) st_async_b32(a_dst + static_cast<uint32_t>(pb * BM * 4), __float_as_uint(alpha), xbar);
                // the copy engine reads the staged tile: order these writes
                // before it; the copy warp moves the whole tile once all
                // softmax warps have staged
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[Smem::P_STAGED + b2]);
            }
            // Sum the parts' row sums through the K ring, idle once every QK^T
            // has completed (the last S_FULL was seen).  Each warp arrives
            // exactly once (its loop exits warp-uniformly), so the wait ends.
            float* lsum = reinterpret_cast<float*>(smem + Smem::kring);
            lsum[(part * BM + row) * 2 + 0] = l;
            lsum[(part * BM + row) * 2 + 1] = l_b;
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[Smem::L_XCHG]);
            if (ok) ok = wait_or_abort(&bars[Smem::L_XCHG], 0, p.err, abort, wait_ns);
            if (ok && part == 0) {
                float l_all = 0.f, lb_all = 0.f;
#pragma unroll
                for (int q4 = 0; q4 < PARTS; ++q4) {
                    l_all += lsum[(q4 * BM + row) * 2 + 0];
                    lb_all += lsum[(q4 * BM + row) * 2 + 1];
                }
                // O / sum(p~) with p~ the rounded weights PV used: O stays an
                // exact convex combination of V rows whatever the rounding of P
                st_async_b32(map_to_cta(smem_u32(smem + Smem::lrecv + row * 4), out_rank), __float_as_uint(lb_all),
                             bar_of(Smem::L_READY, out_rank));
                if (valid_row && p.lse)
                    p.lse[static_cast<size_t>(hq) * p.total_q + q_start + t0 + tok] =
                        l_all > 0.f ? (m_ref + log2f(l_all)) * 0.69314718055994530942f : -INFINITY;
            }
        }
    } else {
        if (warp == 0) {
            if (lane == 0) {
                // -------------------------------------------------- V loads
                const uint64_t pol_kv = l2_policy_keep();   // read by every pair of the KV head
                int pf[PF][2];
#pragma unroll
                for (int i = 0; i < PF; ++i)
#pragma unroll
                    for (int r = 0; r < 2; ++r)
                        pf[i][r] = i < n_kt ? page_entry((kt_begin + i) * BN + r * K_BOX_ROWS) : 0;
                for (int j = 0; j < n_kt; ++j) {
                    const int vb = j & 1;
                    // V buffer vb once O += P V of tile j - 2 completed
                    if (j >= 2 && !wait_or_abort(&bars[Smem::PV_DONE + (j - 2) % P_BUFS], ((j - 2) / P_BUFS) & 1,
                                                 p.err, abort, wait_ns))
                        break;
                    // (the tile's ready barrier goes with its P buffer: the
                    // correction warps may run three tiles ahead of the MMAs)
                    const int rb = j % P_BUFS;
                    const int key = (kt_begin + j) * BN;
                    if constexpr (PAGED) {
                        // Each V box is one half tile (one page or part of one).
                        // The tail tile's V lands on this CTA's own barrier: the
                        // correction warps clear the rows past the cache's end
                        // before they mark the tile ready (a NaN there would
                        // survive a zero weight).
                        const bool tail = kt_begin + j == tail_tile;
                        uint32_t vbar;
                        if (tail) {
                            if (rank == 2) mbar_arrive(&bars[Smem::PV_READY + rb]);
                            mbar_arrive_expect_tx(&bars[Smem::V_TAIL], 2 * SLOT);
                            vbar = bar_of(Smem::V_TAIL, rank);
                        } else {
                            if (rank == 2) mbar_arrive_expect_tx(&bars[Smem::PV_READY + rb], 2 * 2 * SLOT);
                            vbar = bar_of(Smem::PV_READY + rb, 2);
                        }
                        const int rows[2] = {half_row(key, pf[0][0]), half_row(key + K_BOX_ROWS, pf[0][1])};
#pragma unroll
                        for (int i = 0; i < PF - 1; ++i) {
                            pf[i][0] = pf[i + 1][0];
                            pf[i][1] = pf[i + 1][1];
                        }
#pragma unroll
                        for (int r = 0; r < 2; ++r)
                            pf[PF - 1][r] = j + PF < n_kt ? page_entry((kt_begin + j + PF) * BN + r * K_BOX_ROWS) : 0;
                        for (int hh = 0; hh < 2; ++hh)
                            for (int bx = 0; bx < 2; ++bx)
                                for (int r = 0; r < 2; ++r)
                                    tma2_load_3d_hint(smem + Smem::vring + (2 * vb + hh) * SLOT + bx * V_BOX +
                                                          r * K_BOX,
                                                      &tmv, vbar, (hh * 4 + static_cast<int>(pr) * 2 + bx) * 64, kvh,
                                                      rows[r], pol_kv);
                    } else {
                        if (rank == 2) mbar_arrive_expect_tx(&bars[Smem::PV_READY + rb], 2 * 2 * SLOT);
                        for (int hh = 0; hh < 2; ++hh)
                            for (int bx = 0; bx < 2; ++bx)
                                tma2_load_3d_hint(smem + Smem::vring + (2 * vb + hh) * SLOT + bx * V_BOX, &tmv,
                                                  bar_of(Smem::PV_READY + rb, 2),
                                                  (hh * 4 + static_cast<int>(pr) * 2 + bx) * 64, kvh, key, pol_kv);
                    }
                }
            }
        } else if (warp == 1) {
            if (rank == 2) {
                // -------------------------------------------------- O += P V (both SMs)
                // (the whole warp runs the loop, one elected lane issues)
                bool ok = true;
                const uint64_t p_desc = make_sdesc_sw128(smem_u32(smem + Smem::precv), 16, 1024);
                const uint64_t v_desc = make_sdesc_sw128(smem_u32(smem + Smem::vring), V_BOX, 1024);
                for (int j = 0; ok && j < n_kt; ++j) {
                    const int vb = j & 1, pb = j % P_BUFS;
                    if (!(ok = __all_sync(0xffffffffu, wait_or_abort(&bars[Smem::PV_READY + pb], (j / P_BUFS) & 1,
                                                                     p.err, abort, wait_ns))))
                        break;
                    tc_fence_after_sync();
                    const uint64_t ad0 = p_desc + static_cast<uint64_t>(pb * (P_BUF >> 4));
                    const uint64_t bd0 = v_desc + static_cast<uint64_t>(2 * vb * (SLOT >> 4));
                    if (elect_one()) {
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
                        commit2_mask(&bars[Smem::PV_DONE + pb], MASK_ALL);
                        if (j == n_kt - 1) commit2_mask(&bars[Smem::O_FINAL], MASK_OUTPUT);
                    }
                    __syncwarp();
                }
                if (elect_one()) commit2_mask(&bars[Smem::DRAIN], static_cast<uint16_t>(1u << rank));
                __syncwarp();
                (void)mbar_wait(&bars[Smem::DRAIN], 0, p.err, wait_ns);
            }
        } else if (work_warp) {
            // -------------------------------------------------- O correction + epilogue
            const float* alpha_s = reinterpret_cast<const float*>(smem + Smem::alpha);
            const uint32_t o_col = static_cast<uint32_t>(part * OP);
            bool ok = true;
            if (warp == 2 && lane == 0) mbar_arrive_expect_tx(&bars[Smem::L_READY], L_TX);
            for (int j = 0; ok && j < n_kt; ++j) {
                const int pb = j % P_BUFS;
                // P_LANDED[pb]'s phase for tile j - 3 completed before this point
                if (warp == 2 && lane == 0) mbar_arrive_expect_tx(&bars[Smem::P_LANDED + pb], P_TX);
                if (!(ok = __all_sync(0xffffffffu, wait_cluster_or_abort(&bars[Smem::P_LANDED + pb],
                                                                         (j / P_BUFS) & 1, p.err, abort, wait_ns))))
                    break;
                // P arrived through the copy engine and alpha through remote
                // stores; the MMA reads P through the async proxy
                fence_proxy_async_smem();
                const float a = alpha_s[pb * BM + row];
                const bool rescale = j > 0 && __any_sync(0xffffffffu, a != 1.f);
                // this tile's copy landed and its alpha was read: the score CTA's
                // staging buffer may take the tile after next (relaxed: nothing
                // to publish)
                if (lane == 0) mbar_arrive_remote_relaxed(bar_of(Smem::STAGE_FREE + (j & 1), rank - 2));
                if (rescale) {
                    // O += P V of the previous tile must be done before O is corrected
                    if (!(ok = __all_sync(0xffffffffu, wait_or_abort(&bars[Smem::PV_DONE + (j - 1) % P_BUFS],
                                                                     ((j - 1) / P_BUFS) & 1, p.err, abort, wait_ns))))
                        break;
                    tc_fence_after_sync();
                    for (int c = 0; c < OP / 32; ++c) {
                        uint32_t o[32];
                        const uint32_t oc = o_col + static_cast<uint32_t>(c * 32);
                        tmem_ld32(tmem + lane_base + oc, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * a);
                        tmem_st32(tmem + lane_base + oc, o);
                    }
                    tmem_st_wait();
                }
                if constexpr (PAGED) {
                    if (kt_begin + j == tail_tile) {
                        // the tile holding the cache's end: zero this CTA's V rows
                        // from the end to the end of its half tile, in both O
                        // halves' slots, then hand them to the tensor core (async proxy)
                        if (!(ok = __all_sync(0xffffffffu, wait_or_abort(&bars[Smem::V_TAIL], 0, p.err, abort,
                                                                         wait_ns))))
                            break;
                        const int r0 = seqlen_k - tail_tile * BN;       // 1 .. 127, not 64
                        const int n16 = (((r0 + K_BOX_ROWS - 1) & ~(K_BOX_ROWS - 1)) - r0) * 8;   // per box
                        uint8_t* vs = smem + Smem::vring + (2 * (j & 1)) * SLOT + r0 * 128;
                        for (int i = tid - 64; i < 4 * n16; i += N_WORK_WARPS * 32) {
                            const int bx = i / n16;                   // (O half, 64-column box)
                            *reinterpret_cast<uint4*>(vs + (bx >> 1) * SLOT + (bx & 1) * V_BOX + (i - bx * n16) * 16) =
                                make_uint4(0u, 0u, 0u, 0u);
                        }
                        fence_proxy_async_smem();
                    }
                }
                tc_fence_before_sync();
                __syncwarp();
                // O corrected (tcgen05.st completed) and P landed: relaxed, except
                // where a paged tail tile's cleared V rows must be published
                if (lane == 0) {
                    if (rank == 2) mbar_arrive(&bars[Smem::PV_READY + pb]);
                    else if (PAGED && kt_begin + j == tail_tile) mbar_arrive_remote(bar_of(Smem::PV_READY + pb, 2));
                    else mbar_arrive_remote_relaxed(bar_of(Smem::PV_READY + pb, 2));
                }
            }
            if (ok) ok = __all_sync(0xffffffffu, wait_or_abort(&bars[Smem::O_FINAL], 0, p.err, abort, wait_ns));
            if (ok) ok = __all_sync(0xffffffffu, wait_cluster_or_abort(&bars[Smem::L_READY], 0, p.err, abort, wait_ns));
            if (ok) {
                tc_fence_after_sync();
                const float lb = reinterpret_cast<const float*>(smem + Smem::lrecv)[row];
                const float inv_l = lb > 0.f ? 1.f / lb : 0.f;
                __nv_bfloat16* dst =
                    p.out + (static_cast<size_t>(q_start + t0 + tok) * p.n_q_heads + hq) * D + o_col;
                for (int c = 0; c < OP / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(tmem + lane_base + o_col + static_cast<uint32_t>(c * 32), o);
                    tmem_ld_wait();
                    if (valid_row) {
                        uint32_t pk[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            pk[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
                        // O is written once: streaming stores (evicted first from L2).
                        // Measured on one GB300: +1.2 % on the contiguous configs,
                        // -1.8 % on the paged ones, which keep plain stores.
                        uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const uint4 v = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                            if constexpr (PAGED) d4[i] = v;
                            else __stcs(d4 + i, v);
                        }
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

int prefill_smem_bytes() { return prefill_so::Smem::total; }
int prefill_k_box_rows() { return prefill_so::K_BOX_ROWS; }
int prefill_v_box_rows() { return prefill_so::V_BOX_ROWS; }
int prefill_paged_v_box_rows() { return prefill_so::K_BOX_ROWS; }

cudaError_t launch_prefill(const CUtensorMap& tmq, const CUtensorMap& tmk, const CUtensorMap& tmv,
                           const PrefillParams& p, cudaStream_t stream) {
    const int smem = prefill_smem_bytes();
    cudaError_t e = cudaFuncSetAttribute(prefill_so::prefill_so_kernel<false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // four CTAs (cluster ranks) per q-tile pair and KV head
    const int n_pairs = (p.num_q_tiles + 1) / 2;
    const long long n_blocks = static_cast<long long>(n_pairs) * 4 * p.n_kv_heads;
    prefill_so::prefill_so_kernel<false><<<static_cast<unsigned>(n_blocks), prefill_so::NUM_THREADS, smem, stream>>>(
        tmq, tmk, tmv, p);
    return cudaGetLastError();
}

cudaError_t launch_prefill_paged(const CUtensorMap& tmq, const CUtensorMap& tmk, const CUtensorMap& tmv,
                                 const PrefillParams& p, cudaStream_t stream) {
    const int smem = prefill_smem_bytes();
    cudaError_t e = cudaFuncSetAttribute(prefill_so::prefill_so_kernel<true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // (sequence, KV head, q-tile pair) numbered without gaps, four CTAs each;
    // the chunks hold at most total_q / (2 T) + batch pairs
    const long long per_head = std::min(static_cast<long long>(p.batch) * p.max_pairs,
                                        (static_cast<long long>(p.total_q) + 2 * p.tokens_per_tile - 1) /
                                                (2 * p.tokens_per_tile) + p.batch);
    const long long n_blocks = per_head * p.n_kv_heads * 4;
    if (n_blocks == 0) return cudaSuccess;
    prefill_so::prefill_so_kernel<true><<<static_cast<unsigned>(n_blocks), prefill_so::NUM_THREADS, smem, stream>>>(
        tmq, tmk, tmv, p);
    return cudaGetLastError();
}

}  // namespace fa512

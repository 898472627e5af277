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
// shared memory; two S buffers in the other 256 columns): a ring of five 32
// KiB slots carries, per item, four entries of Q (two 64-column boxes each;
// the MMA thread copies them into TMEM with tcgen05.cp once the previous
// item's QK^T has completed) and then the item's K half tiles (this CTA's 64
// keys x 256 head-dim columns), each slot released by the commit after its
// copies or its 16 MMAs; the MMA thread holds back a tile's QK^T until its S
// buffer has been read (the loads run ahead).  Eight softmax warps: TMEM lane
// quadrant (warp % 4) gives a warp its 32 rows, warps 2-5 take keys 0-63 of
// each tile and warps 6-9 keys 64-127; the two warps of a quadrant swap row
// maxima through shared memory.  The row max is lazy: O is rescaled only when
// a row's max grows by more than 2^16.  P goes to one of two staging buffers;
// a copy warp moves each staged tile with one bulk copy (the copy engine) into
// the output CTA, where it completes on that CTA's mbarrier; alpha follows by
// remote stores on the same barrier.  At the end of an item the two parts of a
// row add up their row sums and the sums go to the output CTA.
//
// Output pair (per CTA: the whole 128 x 512 fp32 O in TMEM): V streams
// through four 32 KiB slots (two tiles x two O halves), P lands in three
// buffers; the commit after a tile's 16 MMAs (M256 x N256 per O half, P and
// V from shared memory) is multicast to all four CTAs and frees that tile's
// V slots and P buffer and lets O be corrected for the next tile.  Eight
// correction warps apply alpha to O in TMEM (tcgen05.ld / st) when a row's
// max moved, then mark the tile ready; at the end they normalise O by the
// sum of the bf16 P values and write bf16 rows.  The next item's first
// O += P V, which overwrites O, waits for their tile-ready arrival after O
// has been read out.
//
// The kernel is persistent: as many clusters as can be resident take the
// work items round-robin, and every role walks the same item sequence with
// running counters, so the next item's loads and products overlap the end of
// the current one.
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
#include <atomic>
#include <string.h>

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
constexpr int V_SLOTS = 4;               // output CTAs: 2 tiles x 2 O halves
constexpr int V_BOX_ROWS = BN;           // {64 columns, 128 keys} boxes
constexpr int V_BOX = V_BOX_ROWS * 128;  // 16 KiB
constexpr int P_CHUNK = BM * 128;        // P of 64 keys for 128 rows, bf16: 16 KiB
constexpr int P_BUF = 2 * P_CHUNK;       // one tile's P: 32 KiB
constexpr int P_BUFS = 3;                // output CTAs: P buffers
constexpr int STAGES = 2;                // score CTAs: P staging buffers
constexpr uint32_t P_TX = P_BUF + BM * 4;   // bytes landing per tile: P and alpha
constexpr uint32_t L_TX = BM * 4;           // the final row sums
static_assert(PARTS == 2 && KP % 32 == 0, "two work warps per lane quadrant");

// Rescale O only when the row max grows by more than this (log2 units);
// until then the stale max stays the reference and p <= 2^16 (bf16 and the
// fp32 sums hold that range).  A rescale makes the output pair wait for the
// previous tile's O += P V, so rows that keep finding larger maxima (the
// stress rows) pay for each one: 2^16 measured faster than 2^8, 2^12 and 2^20.
constexpr float RESCALE_THRESHOLD = 16.0f;

constexpr uint16_t MASK_SCORE = 0x3, MASK_OUTPUT = 0xC, MASK_ALL = 0xF;

struct Smem {
    // score CTAs: Q and K entries of the ring (Q is copied on into TMEM)
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
        K_FULL = 0,                      // [5] score leader: both CTAs' ring entry (Q boxes or K half tile) landed
        K_EMPTY = K_FULL + K_SLOTS,      // [5] score CTAs: the entry's copies or MMAs completed
        S_FULL = K_EMPTY + K_SLOTS,      // [2] score CTAs: S of the tile is in TMEM
        S_FREE = S_FULL + S_BUFS,        // [2] score leader: both CTAs' softmax warps read S
        XCHG = S_FREE + S_BUFS,          // [2][4] score CTAs: row-max swap of one lane quadrant's key parts
        P_STAGED = XCHG + 8,             // [2] score CTAs: all softmax warps staged the tile's P
        STAGE_FREE = P_STAGED + STAGES,  // [2] score CTAs: the buffer's last copy landed, its alpha read
        S_READ = STAGE_FREE + STAGES,    // [2] score CTA 1: its softmax warps read S (forwarded to S_FREE)
        L_XCHG = S_READ + S_BUFS,        // score CTAs: part 1's row sums of the item are staged
        L_FREE = L_XCHG + 1,             // score CTAs: the output CTA read the item's row sums
        PV_DONE = L_FREE + 1,            // [3] all four: O += P V of the P buffer's last tile completed
        PV_READY = PV_DONE + P_BUFS,     // [3] output leader: P landed and O corrected in both, V landed
        P_LANDED = PV_READY + P_BUFS,    // [3] output CTAs: P and alpha of the tile arrived
        O_FINAL = P_LANDED + P_BUFS,     // output CTAs: the item's last O += P V completed
        L_READY = O_FINAL + 1,           // output CTAs: the item's row sums arrived
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

// 32 bytes (eight 32-bit words) to global memory in one store; STREAM: with
// the evict-first policy (data written once).  The address is 32-byte aligned.
template <bool STREAM>
__device__ __forceinline__ void st_global_v8(void* ptr, const uint32_t* v) {
    if constexpr (STREAM)
        asm volatile("st.global.cs.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(ptr), "r"(v[0]), "r"(v[1]),
                     "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                     : "memory");
    else
        asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(ptr), "r"(v[0]), "r"(v[1]),
                     "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
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

// Geometry of one work item (a q-tile pair of one KV head) for the cluster
// ranks with tile parity pr (which q tile of the pair).
struct Geo {
    bool valid;                  // the item exists
    int kvh, seq, q_start, seqlen_q, seqlen_k, q_offset;
    int t0, ntok, p_first, p_last;
    int kt_begin, n_kt, tail_tile;
};

// Work items are numbered KV head by KV head (contiguous), or sequence by
// sequence and KV head by KV head (paged), heaviest pair first, with no gaps.
// Called by a whole warp: in paged mode it finds the item's sequence by a
// scan of the chunk lengths (one contiguous block of sequences per lane).
template <bool PAGED>
__device__ Geo item_geometry(const PrefillParams& p, int item, uint32_t pr, int lane) {
    Geo g;
    g.valid = false;
    const int T = p.tokens_per_tile;
    int pair;
    g.seq = 0;
    g.q_start = 0;
    g.seqlen_q = p.seqlen_q;
    g.seqlen_k = p.seqlen_k;
    g.q_offset = p.q_offset;
    if constexpr (PAGED) {
        const int two_t = 2 * T;
        // pairs of a chunk with rows [s0, s1) (0 for a malformed entry, recorded)
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
            for (int b = lo; b < hi; ++b) cnt += chunk_pairs(p.cu_seqlens_q[b], p.cu_seqlens_q[b + 1]) * p.n_kv_heads;
        }
        int incl = cnt;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += t;
        }
        const int excl = incl - cnt;
        const unsigned owner_mask = __ballot_sync(0xffffffffu, item >= excl && item < incl);
        if (!owner_mask) return g;   // past the last item
        const int owner = __ffs(owner_mask) - 1;
        int f_seq = lo, acc = excl;
        if (lane == owner && per > 1) {
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
        f_seq = __shfl_sync(0xffffffffu, f_seq, owner);
        acc = __shfl_sync(0xffffffffu, acc, owner);
        s0 = __shfl_sync(0xffffffffu, s0, owner);
        s1 = __shfl_sync(0xffffffffu, s1, owner);
        kv = __shfl_sync(0xffffffffu, kv, owner);
        const int off = item - acc;
        g.seq = f_seq;
        g.q_start = s0;
        g.seqlen_q = min(s1 - s0, p.max_seqlen_q);
        g.seqlen_k = kv;
        const int n_pairs_seq = (g.seqlen_q + two_t - 1) / two_t;
        g.kvh = off / n_pairs_seq;
        pair = n_pairs_seq - 1 - (off - g.kvh * n_pairs_seq);   // 0 = heaviest pair first
        g.q_offset = g.seqlen_k - (s1 - s0);                    // the chunk is its sequence's tail
        const int kv_cap = p.max_pages_per_seq << p.page_shift;
        if (g.seqlen_k < 0 || g.seqlen_k > kv_cap) {
            // recorded (idempotently); read up to the table's capacity
            if (off == 0) report_error(p.err, FA512_DEVICE_ERR_INDEX);
            g.seqlen_k = g.seqlen_k < 0 ? 0 : kv_cap;
        }
    } else {
        const int n_pairs = (p.num_q_tiles + 1) / 2;
        if (item >= n_pairs * p.n_kv_heads) return g;
        g.kvh = item / n_pairs;
        pair = n_pairs - 1 - item % n_pairs;
    }
    g.valid = true;
    const int qt = 2 * pair + static_cast<int>(pr);    // may be one past the last tile: no rows
    g.t0 = qt * T;
    g.ntok = min(T, g.seqlen_q - g.t0);                 // <= 0 for a missing second tile
    g.p_first = g.q_offset + g.t0;
    g.p_last = g.q_offset + g.t0 + g.ntok - 1;
    const int pair_first = g.q_offset + 2 * pair * T;
    const int pair_last = g.q_offset + min(g.seqlen_q, (2 * pair + 2) * T) - 1;
    // paged: the tile that holds the cache's last key when that key does not
    // end a half tile (its V rows past the end are live pool memory)
    g.tail_tile = (PAGED && (g.seqlen_k & (K_BOX_ROWS - 1))) ? (g.seqlen_k - 1) / BN : -1;
    int j_lo = 0, j_hi = g.seqlen_k;
    if (p.causal) j_hi = min(j_hi, pair_last + 1);
    if (p.window > 0) j_lo = max(0, pair_first - p.window + 1);
    if (j_hi < j_lo) j_hi = j_lo;
    g.kt_begin = j_lo / BN;
    g.n_kt = j_hi > j_lo ? (j_hi + BN - 1) / BN - g.kt_begin : 0;
    return g;
}

// A persistent cluster of four takes the work items cluster, cluster + n,
// cluster + 2n, ... (n clusters): every role walks the same item sequence
// and keeps running counters (K-ring entries, tiles, items), so the barrier
// phases run on across items and the next item's Q loads, QK^T and P V
// overlap the end of the current one.  PAGED: a batch of chunks (varlen rows
// through cu_seqlens_q) over a paged cache; K and V rows are found through
// the page table one 64-key half tile at a time (a page holds a whole number
// of half tiles).
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

    const uint32_t rank = cluster_ctarank();            // == blockIdx.x & 3
    const bool scorer = rank < 2;
    const uint32_t pr = rank & 1;                       // which q tile of the pair
    const int G = p.group;
    const int cluster = blockIdx.x >> 2;
    const int n_clusters = gridDim.x >> 2;

    if (warp == 0 && lane == 0) {
        for (int i = 0; i < Smem::N_BARS; ++i) {
            uint32_t count = 1;
            if (i == Smem::L_XCHG) count = N_WORK_WARPS / PARTS;           // the part-1 softmax warps
            if (i >= Smem::XCHG && i < Smem::XCHG + 8) count = PARTS;   // the warps sharing a lane quadrant
            // the leader's softmax warps, plus one forwarded arrival for the other CTA's
            if (i >= Smem::S_FREE && i < Smem::S_FREE + S_BUFS) count = N_WORK_WARPS + 1;
            // this CTA's softmax warps; the output CTA's correction warps
            if ((i >= Smem::P_STAGED && i < Smem::P_STAGED + STAGES) ||
                (i >= Smem::STAGE_FREE && i < Smem::STAGE_FREE + STAGES) ||
                (i >= Smem::S_READ && i < Smem::S_READ + S_BUFS) || i == Smem::L_FREE)
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
    // a wait made by every lane of a warp, with a warp-uniform outcome
    auto wait_warp = [&](int i, uint32_t parity) -> bool {
        return __all_sync(0xffffffffu, wait_or_abort(&bars[i], parity, p.err, abort, wait_ns));
    };

    // Row of the tensor map holding the first key of the 64-key half tile
    // that starts at logical key `key`: the key itself, or in paged mode its
    // slot in the pool.  Halves past the cache's end (and pages outside the
    // pool) read a row past the pool, which the TMA unit fills with zeros.
    // Paged: the producers load a half tile's page-table entry (page_entry)
    // several tiles before they need its row (half_row), so the dependent
    // load is off their critical path.
    auto page_entry = [&](const Geo& gm, int key) -> int {
        if constexpr (PAGED) {
            return key < gm.seqlen_k
                       ? p.page_table[static_cast<size_t>(gm.seq) * p.max_pages_per_seq + (key >> p.page_shift)]
                       : 0;
        } else {
            return 0;
        }
    };
    auto half_row = [&](const Geo& gm, int key, int pg) -> int {
        if constexpr (PAGED) {
            if (key >= gm.seqlen_k) return p.oob_row;
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

    // this thread's packed row and part (warps 2-9): TMEM lane quadrant
    // warp % 4; part = 64 keys of a tile in the score CTAs, 256 O columns in
    // the output CTAs
    const bool work_warp = warp >= 2 && warp < COPY_WARP;
    const int row = (warp & 3) * 32 + lane;
    const int part = (warp - 2) >> 2;

    if (scorer) {
        if (warp == 0) {
            // ---------------------------------------------------- Q and K into the ring
            // Per item: four entries of Q (two 64-column boxes each; the MMA
            // thread copies them into TMEM), then the item's K half tiles
            // (tile h / 2, head-dim columns 256 (h % 2) .. +256, this CTA's
            // 64 keys).  Q is read once; K and V by every pair of the KV head.
            const uint64_t pol_q = l2_policy_stream(), pol_kv = l2_policy_keep();
            const uint32_t q_box_bytes = static_cast<uint32_t>(128 * p.rows_per_tile);
            int e = 0;   // ring entries so far
            bool ok = true, first_k = true;
            auto take_slot = [&](int& s) -> bool {
                s = e % K_SLOTS;
                return e < K_SLOTS || wait_warp(Smem::K_EMPTY + s, ((e / K_SLOTS) - 1) & 1);
            };
            for (int item = cluster; ok; item += n_clusters) {
                const Geo gm = item_geometry<PAGED>(p, item, pr, lane);
                if (!gm.valid) break;
                if (gm.n_kt == 0) continue;
                for (int qe = 0; qe < 4 && ok; ++qe) {
                    int s;
                    if (!(ok = take_slot(s))) break;
                    if (lane == 0) {
                        if (rank == 0) mbar_arrive_expect_tx(&bars[Smem::K_FULL + s], 2 * 2 * q_box_bytes);
                        for (int bx = 0; bx < 2; ++bx)
                            tma2_load_4d_hint(smem + Smem::kring + s * SLOT + bx * Q_CHUNK, &tmq,
                                              bar_of(Smem::K_FULL + s, 0), (2 * qe + bx) * 64, 0, gm.kvh,
                                              gm.q_start + gm.t0, pol_q);
                    }
                    ++e;
                }
                if (!ok) break;
                auto k_key = [&](int j) { return (gm.kt_begin + j) * BN + static_cast<int>(pr) * K_BOX_ROWS; };
                int pf[PF];
#pragma unroll
                for (int i = 0; i < PF; ++i) pf[i] = i < gm.n_kt ? page_entry(gm, k_key(i)) : 0;
                int krow = 0;
                for (int h = 0; h < 2 * gm.n_kt; ++h) {
                    const int j = h >> 1, c = h & 1;
                    int s;
                    if (!(ok = take_slot(s))) break;
                    if (c == 0) {
                        // both head-dim halves of tile j read the same keys
                        krow = half_row(gm, k_key(j), pf[0]);
#pragma unroll
                        for (int i = 0; i < PF - 1; ++i) pf[i] = pf[i + 1];
                        pf[PF - 1] = j + PF < gm.n_kt ? page_entry(gm, k_key(j + PF)) : 0;
                    }
                    // (test hook: the first cluster's rank 0 leaves out its first
                    // K half tile, so that cluster's waits run into their bound)
                    const bool skip = first_k && p.test_skip_first_k_load && blockIdx.x == 0;
                    first_k = false;
                    if (lane == 0) {
                        if (rank == 0) mbar_arrive_expect_tx(&bars[Smem::K_FULL + s], 2 * SLOT);
                        if (!skip)
                            for (int b = 0; b < 4; ++b)
                                tma2_load_3d_hint(smem + Smem::kring + s * SLOT + b * K_BOX, &tmk,
                                                  bar_of(Smem::K_FULL + s, 0), (c * 4 + b) * 64, gm.kvh, krow,
                                                  pol_kv);
                    }
                    ++e;
                }
            }
        } else if (warp == 1 && rank == 1) {
            // ---------------------------------------------------- forward "S read" to the leader
            // (the softmax warps arrive locally: a remote arrival, even a
            // relaxed one, measured slower on their critical path)
            int t = 0;
            bool ok = true;
            for (int item = cluster; ok; item += n_clusters) {
                const Geo gm = item_geometry<PAGED>(p, item, pr, lane);
                if (!gm.valid) break;
                for (int j = 0; j < gm.n_kt; ++j, ++t) {
                    if (!(ok = wait_warp(Smem::S_READ + (t % S_BUFS), (t / S_BUFS) & 1))) break;
                    if (lane == 0) mbar_arrive_remote_relaxed(bar_of(Smem::S_FREE + (t % S_BUFS), 0));
                }
            }
        } else if (warp == 1) {
            // ---------------------------------------------------- S = Q K^T (both SMs)
            // The whole warp runs the loop and its waits (warp-uniform, so the
            // MMA operands stay uniform); one elected lane issues.
            const uint64_t k_desc = make_sdesc_sw128(smem_u32(smem + Smem::kring), 16, 1024);
            int e = 0, t = 0;
            bool ok = true;
            for (int item = cluster; ok; item += n_clusters) {
                const Geo gm = item_geometry<PAGED>(p, item, pr, lane);
                if (!gm.valid) break;
                if (gm.n_kt == 0) continue;
                // The item's Q overwrites the TMEM the previous item's QK^T
                // read: wait for the commit of that item's last tile first.
                if (t > 0 && !(ok = wait_warp(Smem::S_FULL + ((t - 1) % S_BUFS), ((t - 1) / S_BUFS) & 1))) break;
                for (int qe = 0; qe < 4; ++qe, ++e) {
                    const int s = e % K_SLOTS;
                    if (!(ok = wait_warp(Smem::K_FULL + s, (e / K_SLOTS) & 1))) break;
                    tc_fence_after_sync();
                    if (elect_one()) {
                        // boxes 2 qe, 2 qe + 1 of both CTAs' Q into TMEM: four
                        // 16-column slices each, ahead of the MMAs that read them
#pragma unroll
                        for (int bx = 0; bx < 2; ++bx) {
                            const uint64_t qd = make_sdesc_sw128(smem_u32(smem + Smem::kring + s * SLOT + bx * Q_CHUNK),
                                                                 16, 1024);
#pragma unroll
                            for (int piece = 0; piece < 4; ++piece)
                                tmem_cp2_128x256b(tmem + TM_Q + static_cast<uint32_t>((2 * qe + bx) * 32 + piece * 8),
                                                  qd + static_cast<uint64_t>(piece * 2));
                        }
                        commit2_mask(&bars[Smem::K_EMPTY + s], MASK_SCORE);
                    }
                    __syncwarp();
                }
                for (int j = 0; ok && j < gm.n_kt; ++j, ++t) {
                    const uint32_t sb = tmem + static_cast<uint32_t>(t % S_BUFS) * BN;
                    // the tile's S buffer must have been read before its QK^T may start
                    if (t >= S_BUFS && !(ok = wait_warp(Smem::S_FREE + (t % S_BUFS), ((t / S_BUFS) - 1) & 1))) break;
                    for (int c = 0; c < 2; ++c, ++e) {
                        const int s = e % K_SLOTS;
                        if (!(ok = wait_warp(Smem::K_FULL + s, (e / K_SLOTS) & 1))) break;
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
                            if (c == 1) commit2_mask(&bars[Smem::S_FULL + (t % S_BUFS)], MASK_SCORE);
                        }
                        __syncwarp();
                    }
                }
            }
            // let every issued MMA finish before TMEM can be released
            if (elect_one()) commit2_mask(&bars[Smem::DRAIN], static_cast<uint16_t>(1u << rank));
            __syncwarp();
            (void)mbar_wait(&bars[Smem::DRAIN], 0, p.err, wait_ns);
        } else if (warp == COPY_WARP) {
            // ---------------------------------------------------- P tiles to the output CTA
            const uint32_t out_rank = rank + 2;
            int t = 0;
            bool ok = true;
            for (int item = cluster; ok; item += n_clusters) {
                const Geo gm = item_geometry<PAGED>(p, item, pr, lane);
                if (!gm.valid) break;
                for (int j = 0; j < gm.n_kt; ++j, ++t) {
                    const int b2 = t & 1, pb = t % P_BUFS;
                    // all softmax warps staged tile t, and the output CTA's P
                    // buffer pb is free (O += P V of tile t - 3 completed)
                    if (!(ok = wait_warp(Smem::P_STAGED + b2, (t >> 1) & 1))) break;
                    if (t >= P_BUFS && !(ok = wait_warp(Smem::PV_DONE + pb, ((t / P_BUFS) - 1) & 1))) break;
                    if (lane == 0)
                        bulk_copy_to_cluster(map_to_cta(smem_u32(smem + Smem::precv + pb * P_BUF), out_rank),
                                             smem_u32(smem + Smem::stage + b2 * P_BUF), P_BUF,
                                             bar_of(Smem::P_LANDED + pb, out_rank));
                }
            }
        } else {
            // ---------------------------------------------------- softmax
            float* xmax = reinterpret_cast<float*>(smem + Smem::xmax);
            const bool neg_scale = p.scale_log2 < 0.f;
            const uint32_t out_rank = rank + 2;
            const uint32_t a_dst = map_to_cta(smem_u32(smem + Smem::alpha + row * 4), out_rank);
            int t = 0, ic = 0;   // tiles, items with keys
            bool ok = true;
            for (int item = cluster; ok; item += n_clusters) {
                const Geo gm = item_geometry<PAGED>(p, item, pr, lane);
                if (!gm.valid) break;
                const int tok = row / G;
                const int g = row - tok * G;
                const bool valid_row = row < p.rows_per_tile && tok < gm.ntok;
                const int qpos = gm.q_offset + gm.t0 + tok;
                const int hq = gm.kvh * G + g;
                if (gm.n_kt == 0) {
                    // no key is visible to any row of the pair: LSE = -inf
                    if (valid_row && part == 0 && p.lse)
                        p.lse[static_cast<size_t>(hq) * p.total_q + gm.q_start + gm.t0 + tok] = -INFINITY;
                    continue;
                }
                float m_ref = -INFINITY;   // log2 units, the same in all parts
                float l = 0.f;             // this part's sum of the fp32 probabilities (for LSE)
                float l_b = 0.f;           // this part's sum of the bf16-rounded probabilities
                for (int j = 0; j < gm.n_kt; ++j, ++t) {
                    const int b3 = t % S_BUFS, b2 = t & 1, pb = t % P_BUFS;
                    // (every wait of a softmax warp is warp-uniform: the warp
                    // synchronises below and must leave the loop as one)
                    if (!(ok = wait_warp(Smem::S_FULL + b3, (t / S_BUFS) & 1))) break;
                    tc_fence_after_sync();
                    uint32_t sr[KP];
#pragma unroll
                    for (int c = 0; c < KP / 32; ++c)
                        tmem_ld32(tmem + lane_base + static_cast<uint32_t>(b3 * BN + part * KP + 32 * c),
                                  *reinterpret_cast<uint32_t(*)[32]>(sr + 32 * c));
                    tmem_ld_wait();
                    // the S buffer may take the QK^T two tiles on
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars[rank == 0 ? Smem::S_FREE + b3 : Smem::S_READ + b3]);
                    float s[KP];
#pragma unroll
                    for (int c = 0; c < KP; ++c) s[c] = __uint_as_float(sr[c]);

                    const int key0 = (gm.kt_begin + j) * BN + part * KP;
                    const bool part_full = gm.ntok > 0 && key0 + KP <= gm.seqlen_k &&
                                           (!p.causal || key0 + KP - 1 <= gm.p_first) &&
                                           (p.window <= 0 || key0 > gm.p_last - p.window);
                    // scores stay unscaled until the exponent; a hidden key gets the
                    // value that scales to -inf whatever the sign of the scale
                    if (!part_full) {
                        const float hidden = neg_scale ? INFINITY : -INFINITY;
#pragma unroll
                        for (int c = 0; c < KP; ++c)
                            if (!key_visible(key0 + c, qpos, gm.seqlen_k, p)) s[c] = hidden;
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
                    if (!(ok = wait_warp(xb, (t >> 1) & 1))) break;
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

                    // staging buffer b2: its copy of tile t - 2 has landed and the
                    // output CTA has read that tile's alpha (which also means its
                    // barrier phase for tile t - 3 has completed)
                    if (t >= STAGES && !(ok = wait_warp(Smem::STAGE_FREE + b2, ((t >> 1) - 1) & 1))) break;
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
                if (!ok) break;
                // The parts' row sums meet in the staging buffer the next tile
                // will use, once its last copy has landed: part 1 leaves them
                // in the first 8 bytes of its rows' lines of the first chunk,
                // which only this quadrant's part 0 writes next (after it has
                // read them), and part 0 adds them to its own.
                const int bn = t & 1;
                if (t >= STAGES && !(ok = wait_warp(Smem::STAGE_FREE + bn, ((t >> 1) - 1) & 1))) break;
                float2* lx = reinterpret_cast<float2*>(smem + Smem::stage + bn * P_BUF + row * 128);
                if (part == 1) {
                    *lx = make_float2(l, l_b);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars[Smem::L_XCHG]);
                } else {
                    if (!(ok = wait_warp(Smem::L_XCHG, ic & 1))) break;
                    const float2 other = *lx;
                    const float l_all = l + other.x, lb_all = l_b + other.y;
                    // the output CTA's row-sum slot is free once it has read
                    // the previous item's sums
                    if (ic >= 1 && !(ok = wait_warp(Smem::L_FREE, (ic - 1) & 1))) break;
                    // O / sum(p~) with p~ the rounded weights PV used: O stays an
                    // exact convex combination of V rows whatever the rounding of P
                    st_async_b32(map_to_cta(smem_u32(smem + Smem::lrecv + row * 4), out_rank), __float_as_uint(lb_all),
                                 bar_of(Smem::L_READY, out_rank));
                    if (valid_row && p.lse)
                        p.lse[static_cast<size_t>(hq) * p.total_q + gm.q_start + gm.t0 + tok] =
                            l_all > 0.f ? (m_ref + log2f(l_all)) * 0.69314718055994530942f : -INFINITY;
                }
                ++ic;
            }
        }
    } else {
        if (warp == 0) {
            // ---------------------------------------------------- V loads
            const uint64_t pol_kv = l2_policy_keep();   // read by every pair of the KV head
            int t = 0;
            bool ok = true;
            for (int item = cluster; ok; item += n_clusters) {
                const Geo gm = item_geometry<PAGED>(p, item, pr, lane);
                if (!gm.valid) break;
                if (gm.n_kt == 0) continue;
                int pf[PF][2];
#pragma unroll
                for (int i = 0; i < PF; ++i)
#pragma unroll
                    for (int r = 0; r < 2; ++r)
                        pf[i][r] = i < gm.n_kt ? page_entry(gm, (gm.kt_begin + i) * BN + r * K_BOX_ROWS) : 0;
                for (int j = 0; j < gm.n_kt; ++j, ++t) {
                    const int vb = t & 1;
                    // V buffer vb once O += P V of tile t - 2 completed
                    if (t >= 2 && !(ok = wait_warp(Smem::PV_DONE + (t - 2) % P_BUFS, ((t - 2) / P_BUFS) & 1))) break;
                    // (the tile's ready barrier goes with its P buffer: the
                    // correction warps may run three tiles ahead of the MMAs)
                    const int rb = t % P_BUFS;
                    const int key = (gm.kt_begin + j) * BN;
                    if constexpr (PAGED) {
                        // Each V box is one half tile (one page or part of one).
                        // The tail tile's V lands on this CTA's own barrier: the
                        // correction warps clear the rows past the cache's end
                        // before they mark the tile ready (a NaN there would
                        // survive a zero weight).
                        const bool tail = gm.kt_begin + j == gm.tail_tile;
                        const int rows[2] = {half_row(gm, key, pf[0][0]), half_row(gm, key + K_BOX_ROWS, pf[0][1])};
#pragma unroll
                        for (int i = 0; i < PF - 1; ++i) {
                            pf[i][0] = pf[i + 1][0];
                            pf[i][1] = pf[i + 1][1];
                        }
#pragma unroll
                        for (int r = 0; r < 2; ++r)
                            pf[PF - 1][r] = j + PF < gm.n_kt
                                                ? page_entry(gm, (gm.kt_begin + j + PF) * BN + r * K_BOX_ROWS)
                                                : 0;
                        if (lane == 0) {
                            uint32_t vbar;
                            if (tail) {
                                if (rank == 2) mbar_arrive(&bars[Smem::PV_READY + rb]);
                                mbar_arrive_expect_tx(&bars[Smem::V_TAIL], 2 * SLOT);
                                vbar = bar_of(Smem::V_TAIL, rank);
                            } else {
                                if (rank == 2) mbar_arrive_expect_tx(&bars[Smem::PV_READY + rb], 2 * 2 * SLOT);
                                vbar = bar_of(Smem::PV_READY + rb, 2);
                            }
                            for (int hh = 0; hh < 2; ++hh)
                                for (int bx = 0; bx < 2; ++bx)
                                    for (int r = 0; r < 2; ++r)
                                        tma2_load_3d_hint(smem + Smem::vring + (2 * vb + hh) * SLOT + bx * V_BOX +
                                                              r * K_BOX,
                                                          &tmv, vbar, (hh * 4 + static_cast<int>(pr) * 2 + bx) * 64,
                                                          gm.kvh, rows[r], pol_kv);
                        }
                    } else {
                        if (lane == 0) {
                            if (rank == 2) mbar_arrive_expect_tx(&bars[Smem::PV_READY + rb], 2 * 2 * SLOT);
                            for (int hh = 0; hh < 2; ++hh)
                                for (int bx = 0; bx < 2; ++bx)
                                    tma2_load_3d_hint(smem + Smem::vring + (2 * vb + hh) * SLOT + bx * V_BOX, &tmv,
                                                      bar_of(Smem::PV_READY + rb, 2),
                                                      (hh * 4 + static_cast<int>(pr) * 2 + bx) * 64, gm.kvh, key,
                                                      pol_kv);
                        }
                    }
                }
            }
        } else if (warp == 1) {
            if (rank == 2) {
                // -------------------------------------------------- O += P V (both SMs)
                // (the whole warp runs the loop, one elected lane issues)
                const uint64_t p_desc = make_sdesc_sw128(smem_u32(smem + Smem::precv), 16, 1024);
                const uint64_t v_desc = make_sdesc_sw128(smem_u32(smem + Smem::vring), V_BOX, 1024);
                int t = 0;
                bool ok = true;
                for (int item = cluster; ok; item += n_clusters) {
                    const Geo gm = item_geometry<PAGED>(p, item, pr, lane);
                    if (!gm.valid) break;
                    for (int j = 0; j < gm.n_kt; ++j, ++t) {
                        const int vb = t & 1, pb = t % P_BUFS;
                        // P landed and O corrected in both CTAs (for an item's
                        // first tile: the previous item's O read out), V landed
                        if (!(ok = wait_warp(Smem::PV_READY + pb, (t / P_BUFS) & 1))) break;
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
                            if (j == gm.n_kt - 1) commit2_mask(&bars[Smem::O_FINAL], MASK_OUTPUT);
                        }
                        __syncwarp();
                    }
                }
                if (elect_one()) commit2_mask(&bars[Smem::DRAIN], static_cast<uint16_t>(1u << rank));
                __syncwarp();
                (void)mbar_wait(&bars[Smem::DRAIN], 0, p.err, wait_ns);
            }
        } else if (work_warp) {
            // -------------------------------------------------- O correction + epilogue
            const float* alpha_s = reinterpret_cast<const float*>(smem + Smem::alpha);
            const uint32_t o_col = static_cast<uint32_t>(part * OP);
            // 32-byte stores need a 32-byte aligned O (rows are 1 KiB apart)
            const bool out32 = (reinterpret_cast<uintptr_t>(p.out) & 31u) == 0;
            int t = 0, ic = 0, tails = 0;   // tiles, items with keys, paged tail tiles
            bool ok = true;
            for (int item = cluster; ok; item += n_clusters) {
                const Geo gm = item_geometry<PAGED>(p, item, pr, lane);
                if (!gm.valid) break;
                const int tok = row / G;
                const int g = row - tok * G;
                const bool valid_row = row < p.rows_per_tile && tok < gm.ntok;
                const int hq = gm.kvh * G + g;
                __nv_bfloat16* dst = p.out + (static_cast<size_t>(gm.q_start + gm.t0 + tok) * p.n_q_heads + hq) * D + o_col;
                if (gm.n_kt == 0) {
                    // no key is visible to any row of the pair: O = 0
                    if (valid_row) {
                        uint4* d4 = reinterpret_cast<uint4*>(dst);
                        for (int i = 0; i < OP / 8; ++i) d4[i] = make_uint4(0u, 0u, 0u, 0u);
                    }
                    continue;
                }
                if (warp == 2 && lane == 0) mbar_arrive_expect_tx(&bars[Smem::L_READY], L_TX);
                for (int j = 0; j < gm.n_kt; ++j, ++t) {
                    const int pb = t % P_BUFS;
                    // P_LANDED[pb]'s phase for tile t - 3 completed before this point
                    if (warp == 2 && lane == 0) mbar_arrive_expect_tx(&bars[Smem::P_LANDED + pb], P_TX);
                    if (!(ok = __all_sync(0xffffffffu, wait_cluster_or_abort(&bars[Smem::P_LANDED + pb],
                                                                             (t / P_BUFS) & 1, p.err, abort, wait_ns))))
                        break;
                    // P arrived through the copy engine and alpha through remote
                    // stores; the MMA reads P through the async proxy
                    fence_proxy_async_smem();
                    const float a = alpha_s[pb * BM + row];
                    const bool rescale = j > 0 && __any_sync(0xffffffffu, a != 1.f);
                    // this tile's copy landed and its alpha was read: the score CTA's
                    // staging buffer may take the tile after next (relaxed: nothing
                    // to publish)
                    if (lane == 0) mbar_arrive_remote_relaxed(bar_of(Smem::STAGE_FREE + (t & 1), rank - 2));
                    if (rescale) {
                        // O += P V of the previous tile must be done before O is corrected
                        if (!(ok = wait_warp(Smem::PV_DONE + (t - 1) % P_BUFS, ((t - 1) / P_BUFS) & 1))) break;
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
                    bool tail = false;
                    if constexpr (PAGED) {
                        if (gm.kt_begin + j == gm.tail_tile) {
                            // the tile holding the cache's end: zero this CTA's V rows
                            // from the end to the end of its half tile, in both O
                            // halves' slots, then hand them to the tensor core (async proxy)
                            tail = true;
                            if (!(ok = wait_warp(Smem::V_TAIL, tails & 1))) break;
                            ++tails;
                            const int r0 = gm.seqlen_k - gm.tail_tile * BN;   // 1 .. 127, not 64
                            const int n16 = (((r0 + K_BOX_ROWS - 1) & ~(K_BOX_ROWS - 1)) - r0) * 8;   // per box
                            uint8_t* vs = smem + Smem::vring + (2 * (t & 1)) * SLOT + r0 * 128;
                            for (int i = tid - 64; i < 4 * n16; i += N_WORK_WARPS * 32) {
                                const int bx = i / n16;                   // (O half, 64-column box)
                                *reinterpret_cast<uint4*>(vs + (bx >> 1) * SLOT + (bx & 1) * V_BOX + (i - bx * n16) * 16) =
                                    make_uint4(0u, 0u, 0u, 0u);
                            }
                            fence_proxy_async_smem();
                        }
                    }
                    // O corrected (tcgen05.st completed) and P landed: relaxed, except
                    // where a paged tail tile's cleared V rows must be published
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) {
                        if (rank == 2) mbar_arrive(&bars[Smem::PV_READY + pb]);
                        else if (tail) mbar_arrive_remote(bar_of(Smem::PV_READY + pb, 2));
                        else mbar_arrive_remote_relaxed(bar_of(Smem::PV_READY + pb, 2));
                    }
                }
                if (!ok) break;
                // ---- epilogue: O / sum(p~) as bf16 rows
                if (!(ok = wait_warp(Smem::O_FINAL, ic & 1))) break;
                if (!(ok = __all_sync(0xffffffffu, wait_cluster_or_abort(&bars[Smem::L_READY], ic & 1, p.err, abort,
                                                                         wait_ns))))
                    break;
                tc_fence_after_sync();
                const float lb = reinterpret_cast<const float*>(smem + Smem::lrecv)[row];
                const float inv_l = lb > 0.f ? 1.f / lb : 0.f;
                // the row-sum slot may take the next item's sums (relaxed: the
                // value is in a register)
                __syncwarp();
                if (lane == 0) mbar_arrive_remote_relaxed(bar_of(Smem::L_FREE, rank - 2));
                // O is read out of TMEM before the next item's first tile is
                // marked ready (its O += P V overwrites O), 64 columns at a
                // time; each row's 128 bytes leave as four 32-byte stores, so
                // every store writes whole sectors and the store queue holds
                // up the next TMEM load less (the stores drain while the next
                // item's first O += P V runs)
                for (int c = 0; c < OP / 64; ++c) {
                    uint32_t o[64];
                    tmem_ld32(tmem + lane_base + o_col + static_cast<uint32_t>(c * 64),
                              *reinterpret_cast<uint32_t(*)[32]>(o));
                    tmem_ld32(tmem + lane_base + o_col + static_cast<uint32_t>(c * 64 + 32),
                              *reinterpret_cast<uint32_t(*)[32]>(o + 32));
                    tmem_ld_wait();
                    if (valid_row) {
                        uint32_t pk[32];
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            pk[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
                        __nv_bfloat16* d = dst + c * 64;
                        if (out32) {
                            // O is written once: streaming stores (evicted first from
                            // L2) on the contiguous configs, plain ones when paged
#pragma unroll
                            for (int i = 0; i < 4; ++i) st_global_v8<!PAGED>(d + i * 16, pk + 8 * i);
                        } else {
                            uint4* d4 = reinterpret_cast<uint4*>(d);
#pragma unroll
                            for (int i = 0; i < 8; ++i) d4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                        }
                    }
                }
                ++ic;
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

// Persistent clusters: as many as can be resident at once (but no more than
// the items), each walking its share of the items.
template <bool PAGED>
static cudaError_t launch_persistent(const CUtensorMap& tmq, const CUtensorMap& tmk, const CUtensorMap& tmv,
                                     const PrefillParams& p, long long n_items, cudaStream_t stream) {
    if (n_items <= 0) return cudaSuccess;
    const int smem = prefill_smem_bytes();
    auto kern = prefill_so::prefill_so_kernel<PAGED>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // resident clusters of four on this device: queried once per device
    constexpr int kMaxDev = 64;
    static std::atomic<int> resident[2][kMaxDev];
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    int clusters = (dev >= 0 && dev < kMaxDev) ? resident[PAGED][dev].load(std::memory_order_relaxed) : 0;
    if (clusters < 1) {
        cudaLaunchConfig_t cfg;
        memset(&cfg, 0, sizeof cfg);
        cfg.gridDim = dim3(4 * 64);
        cfg.blockDim = dim3(prefill_so::NUM_THREADS);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess || clusters < 1) {
            (void)cudaGetLastError();
            int sms = 0;
            if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
            clusters = std::max(1, sms / 4);
        } else if (dev >= 0 && dev < kMaxDev) {
            resident[PAGED][dev].store(clusters, std::memory_order_relaxed);
        }
    }
    const long long n = std::min<long long>(clusters, n_items);
    prefill_so::prefill_so_kernel<PAGED><<<static_cast<unsigned>(4 * n), prefill_so::NUM_THREADS, smem, stream>>>(
        tmq, tmk, tmv, p);
    return cudaGetLastError();
}

cudaError_t launch_prefill(const CUtensorMap& tmq, const CUtensorMap& tmk, const CUtensorMap& tmv,
                           const PrefillParams& p, cudaStream_t stream) {
    // (q-tile pair, KV head) items
    const long long n_items = static_cast<long long>((p.num_q_tiles + 1) / 2) * p.n_kv_heads;
    return launch_persistent<false>(tmq, tmk, tmv, p, n_items, stream);
}

cudaError_t launch_prefill_paged(const CUtensorMap& tmq, const CUtensorMap& tmk, const CUtensorMap& tmv,
                                 const PrefillParams& p, cudaStream_t stream) {
    // (sequence, KV head, q-tile pair) items numbered without gaps; the
    // chunks hold at most total_q / (2 T) + batch pairs
    const long long per_head = std::min(static_cast<long long>(p.batch) * p.max_pairs,
                                        (static_cast<long long>(p.total_q) + 2 * p.tokens_per_tile - 1) /
                                                (2 * p.tokens_per_tile) + p.batch);
    return launch_persistent<true>(tmq, tmk, tmv, p, per_head * p.n_kv_heads, stream);
}

}  // namespace fa512

// Paged split-K decode for head dim 512 (Flash-Decoding), sm_103a.
//
// "Flash-Decoding for MQA in CUDA" (mila.toddt.me), section "One KV head
// breaks the textbook": the key sequence of each (sequence, KV head) is split
// across CTAs; each split writes an unnormalised (O, m, l) partial and a
// small fixup kernel applies the online-softmax merge.  The same section:
// walk absolute positions, read only the live band [max(0, len - window),
// len), keep K/V tiles double-buffered and rescale once per tile.
// vllm-project/flash-attention PR #199, "Performance": the cache is paged
// (page size 64), 8 query heads over 4 KV heads, q_len 1; "Summary": the
// cache may be stored in FP8 E4M3.
//
// Work item = (split, KV head, sequence); the rows of a work item are the
// (token, head) pairs of the KV head's query group, q_len * G <= 16, each
// masked at its own position (the last q_len positions of the cache).  Which
// kernel runs:
//   decode_stream_kernel<G>   one token, G <= 2, splits shorter than 1,024
//                             positions (bf16): FMA streaming warps;
//   decode_bf16_mma_kernel    up to 8 rows otherwise (bf16): streaming warps
//                             on mma.sync with the rows in N;
//   decode_fp8_mma_kernel     up to 8 rows over an FP8 cache: the same design
//                             with every byte widened exactly to f16, one
//                             split per 4-warp CTA, four CTAs per SM;
//   decode_split_kernel<FP8>  9 to 16 rows: a CTA's warps share TMA-loaded
//                             tiles of 32 positions (FP8 tiles converted
//                             exactly to bf16), S and PV on mma.sync;
//   decode_merge_kernel<CS>   combines the splits' (O, m, l) partials, each
//                             row in CS column slices.
// HBM traffic per position and KV head: 1 KiB of K + 1 KiB of V (bf16) or
// 512 + 512 bytes (FP8).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "fa512_device.cuh"
#include "fa512_internal.h"

namespace fa512 {
namespace decode {

// Programmatic dependent launch: a split kernel lets the merge kernel that
// follows it on the stream be scheduled while it still runs; the merge waits
// for the split kernel's completion (and its memory) before reading.
__device__ __forceinline__ void allow_merge_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void wait_for_splits() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

constexpr int D = 512;
constexpr int TILE_K = 32;                       // key positions per tile
constexpr int NUM_STAGES = 3;
constexpr int NUM_WARPS = 8;
constexpr int NUM_THREADS = NUM_WARPS * 32;
constexpr int CHUNK_BYTES = TILE_K * 128;        // one 64-column box column
constexpr int TILE_BYTES = 8 * CHUNK_BYTES;      // 32 x 512 bf16 = 32 KiB
constexpr int STAGE_BYTES = 2 * TILE_BYTES;      // K + V
constexpr int Q_BYTES = 16 * D * 2;              // 16 padded query rows
constexpr int P_STRIDE = 80;                     // bytes per P row (64 + pad)
constexpr int P_BYTES = 16 * P_STRIDE;

// FP8 E4M3 cache: a stage holds the tile's K and V bytes (32 positions x
// 512 bytes each) as two 256-byte boxes per row run, [half][position][256];
// after the stage lands every thread converts its share into one bf16 tile
// in the layout of a bf16 stage (e4m3 -> bf16 is exact), which the MMA code
// then reads unchanged.
constexpr int F8_BOX_BYTES = 256;                // head-dim bytes per FP8 box
constexpr int F8_TILE_BYTES = TILE_K * D;        // 32 x 512 e4m3 = 16 KiB
constexpr int F8_STAGE_BYTES = 2 * F8_TILE_BYTES;

template <bool FP8>
struct Smem {
    // Offsets inside the dynamic shared memory block (1024-byte aligned base).
    static constexpr int stages = 0;
    static constexpr int stage_bytes = FP8 ? F8_STAGE_BYTES : STAGE_BYTES;
    // FP8: the converted bf16 tile (K then V); bf16: each stage is read in place
    static constexpr int tile = NUM_STAGES * stage_bytes;
    static constexpr int q = tile + (FP8 ? STAGE_BYTES : 0);
    static constexpr int p = q + Q_BYTES;
    static constexpr int xs = p + P_BYTES;                    // 4 warps x 32 lanes x float4
    static constexpr int redm = xs + 4 * 32 * 16;            // [4][16] float
    static constexpr int redl = redm + 4 * 16 * 4;           // [4][16] float
    static constexpr int full_bar = redl + 4 * 16 * 4;       // NUM_STAGES x u64
    static constexpr int total = full_bar + NUM_STAGES * 8;
};

__device__ __forceinline__ uint32_t swz(int row, int chunk16) {
    // byte offset of 16-byte chunk `chunk16` (0..7) of 128-byte line `row`
    // under the TMA 128-byte swizzle
    return static_cast<uint32_t>(row * 128 + ((chunk16 ^ (row & 7)) << 4));
}

// Which positions of tile t (absolute positions [32t, 32t+32)) are loaded:
// a run of box_rows positions is loaded iff it overlaps [lo, hi) and its page
// index is valid.  Returns a 32-bit mask of loaded positions and the number
// of loaded runs.
struct TilePlan {
    uint32_t loaded;   // bit r: position 32t + r was loaded
    int runs;
};

__device__ __forceinline__ TilePlan plan_tile(const DecodeParams& p, int b, int t, int lo,
                                              int hi, bool record) {
    TilePlan plan{0u, 0};
    const int box_rows = p.box_rows;
    for (int r0 = 0; r0 < TILE_K; r0 += box_rows) {
        const int pos0 = t * TILE_K + r0;
        if (pos0 + box_rows <= lo || pos0 >= hi) continue;
        const int lp = pos0 / p.page_size;
        const int page = p.page_table[static_cast<size_t>(b) * p.max_pages_per_seq + lp];
        if (page < 0 || page >= p.num_pages) {
            if (record) report_error(p.err, FA512_DEVICE_ERR_INDEX);
            continue;
        }
        const uint32_t bits = (box_rows >= 32) ? 0xffffffffu : ((1u << box_rows) - 1u);
        plan.loaded |= bits << r0;
        plan.runs += 1;
    }
    return plan;
}

template <bool FP8>
__device__ __forceinline__ void issue_tile(const DecodeParams& p, const CUtensorMap* tmk,
                                           const CUtensorMap* tmv, uint8_t* stage,
                                           uint64_t* bar, int b, int kvh, int t, int lo, int hi) {
    const TilePlan plan = plan_tile(p, b, t, lo, hi, true);
    const int box_rows = p.box_rows;
    // K and V rows of every loaded run: 512 elements each
    const uint32_t row_bytes = FP8 ? static_cast<uint32_t>(D) : static_cast<uint32_t>(D) * 2u;
    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(plan.runs) * box_rows * row_bytes * 2u);
    for (int r0 = 0; r0 < TILE_K; r0 += box_rows) {
        if (!((plan.loaded >> r0) & 1u)) continue;
        const int pos0 = t * TILE_K + r0;
        const int lp = pos0 / p.page_size;
        const int page = p.page_table[static_cast<size_t>(b) * p.max_pages_per_seq + lp];
        const int row = page * p.page_size + (pos0 - lp * p.page_size);
        if constexpr (FP8) {
            for (int c = 0; c < D / F8_BOX_BYTES; ++c) {
                const int off = c * (TILE_K * F8_BOX_BYTES) + r0 * F8_BOX_BYTES;
                tma_load_3d(stage + off, tmk, bar, c * F8_BOX_BYTES, kvh, row);
                tma_load_3d(stage + F8_TILE_BYTES + off, tmv, bar, c * F8_BOX_BYTES, kvh, row);
            }
        } else {
            for (int c = 0; c < 8; ++c) {
                tma_load_3d(stage + c * CHUNK_BYTES + r0 * 128, tmk, bar, c * 64, kvh, row);
                tma_load_3d(stage + TILE_BYTES + c * CHUNK_BYTES + r0 * 128, tmv, bar, c * 64, kvh,
                            row);
            }
        }
    }
}

// Two e4m3 values (low byte first) -> two bf16 (low half first), exactly:
// the hardware e4m3x2 -> f16x2 conversion, widened through fp32.
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t two_bytes) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<unsigned short>(two_bytes)));
    float lo, hi;
    asm("cvt.f32.f16 %0, %1;" : "=f"(lo) : "h"(static_cast<unsigned short>(h2 & 0xffffu)));
    asm("cvt.f32.f16 %0, %1;" : "=f"(hi) : "h"(static_cast<unsigned short>(h2 >> 16)));
    return pack_bf16x2(lo, hi);
}

// FP8 stage -> bf16 tile in the bf16 stage layout (column group of 64
// elements at CHUNK_BYTES steps, 128-byte rows under the 128-byte swizzle).
// V rows of positions outside `valid` are written as zeros, so P = 0 never
// meets stale or poisoned values; K rows there are masked in the scores.
// Each thread converts 8-element units: a warp covers 256 contiguous bytes
// of one row (conflict-free reads) and writes all eight 16-byte chunks of
// four 128-byte lines (conflict-free writes).
__device__ __forceinline__ void convert_fp8_stage(const uint8_t* stage, uint8_t* tile,
                                                  uint32_t valid, int tid) {
#pragma unroll
    for (int kv = 0; kv < 2; ++kv) {
        const uint8_t* src = stage + kv * F8_TILE_BYTES;
        uint8_t* dst = tile + kv * TILE_BYTES;
#pragma unroll
        for (int k = 0; k < (TILE_K * D / 8) / NUM_THREADS; ++k) {
            const int u = k * NUM_THREADS + tid;     // unit: 8 elements
            const int r = u >> 6;                    // 64 units per position
            const int e0 = (u & 63) * 8;             // first element of the unit
            uint4 out = make_uint4(0u, 0u, 0u, 0u);
            if (kv == 0 || ((valid >> r) & 1u)) {
                const uint2 w = *reinterpret_cast<const uint2*>(
                    src + (e0 / F8_BOX_BYTES) * (TILE_K * F8_BOX_BYTES) + r * F8_BOX_BYTES +
                    (e0 % F8_BOX_BYTES));
                out.x = e4m3x2_to_bf16x2(w.x & 0xffffu);
                out.y = e4m3x2_to_bf16x2(w.x >> 16);
                out.z = e4m3x2_to_bf16x2(w.y & 0xffffu);
                out.w = e4m3x2_to_bf16x2(w.y >> 16);
            }
            *reinterpret_cast<uint4*>(dst + (e0 >> 6) * CHUNK_BYTES + swz(r, (e0 & 63) >> 3)) = out;
        }
    }
}

// One CTA streams its split's key tiles of TILE_K = 32 positions through a
// NUM_STAGES-deep ring in shared memory filled by TMA (one box per page run),
// computes S = Q K^T and O += P V for its rows with bf16 mma.sync (rows padded
// to 16), and keeps the softmax state in the log2 domain.
template <bool FP8>
__global__ void __launch_bounds__(NUM_THREADS, 1)
decode_split_kernel(const __grid_constant__ CUtensorMap tmk,
                    const __grid_constant__ CUtensorMap tmv, const DecodeParams p) {
    allow_merge_launch();
    using Smem = decode::Smem<FP8>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + Smem::full_bar);
    float* redm = reinterpret_cast<float*>(smem + Smem::redm);
    float* redl = reinterpret_cast<float*>(smem + Smem::redl);
    float4* xs = reinterpret_cast<float4*>(smem + Smem::xs);

    const int split = blockIdx.x;
    const int kvh = blockIdx.y;
    const int b = blockIdx.z;
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int G = p.group;
    const int R = p.q_len * G;      // query rows: (token t, head g) -> row t * G + g

    // ---- live band of this sequence
    int len = p.kv_lens[b];
    if (len < 0 || len > p.len_cap) {
        if (tid == 0 && split == 0 && kvh == 0) report_error(p.err, FA512_DEVICE_ERR_INDEX);
        len = len < 0 ? 0 : p.len_cap;
    }
    // union of the rows' bands: row t sees [pos_t - window + 1, pos_t] with
    // pos_t = len - q_len + t
    const int hi = len;
    const int w_lo = len - p.q_len + 1 - p.window;
    const int lo = (p.window > 0 && w_lo > 0) ? w_lo : 0;
    const int t_lo = lo / TILE_K;
    const int t_hi = (hi + TILE_K - 1) / TILE_K;
    const int t_begin = t_lo + split * p.tiles_per_split;
    int t_end = t_begin + p.tiles_per_split;
    if (t_end > t_hi) t_end = t_hi;
    const int n_tiles = t_end > t_begin ? t_end - t_begin : 0;

    if (tid == 0) {
        for (int s = 0; s < NUM_STAGES; ++s) mbar_init(&full_bar[s], 1);
        fence_mbar_init();
        tma_prefetch_desc(&tmk);
        tma_prefetch_desc(&tmv);
    }
    // ---- Q rows of the G heads of this KV head, zero-padded to 16, swizzled
    {
        uint8_t* qs = smem + Smem::q;
        for (int i = tid; i < 16 * 64; i += NUM_THREADS) {
            const int row = i >> 6, c = i & 63;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (row < R) {
                const size_t h = (static_cast<size_t>(b) * p.q_len + row / G) * p.n_q_heads + kvh * G + row % G;
                v = reinterpret_cast<const uint4*>(p.q + h * D)[c];
            }
            *reinterpret_cast<uint4*>(qs + row * 1024 + (((c & ~7) | ((c ^ row) & 7)) << 4)) = v;
        }
    }
    __syncthreads();

    // prologue loads
    if (tid == 0) {
        for (int s = 0; s < NUM_STAGES - 1 && s < n_tiles; ++s)
            issue_tile<FP8>(p, &tmk, &tmv, smem + s * Smem::stage_bytes, &full_bar[s], b, kvh,
                            t_begin + s, lo, hi);
    }

    // ---- Q fragments (A operand) for this warp's half of the head dim
    const int nt = warp & 3;       // QK: n-tile (8 positions) of the tile
    const int dh = warp >> 2;      // QK: half of the head dim
    uint32_t qa[16][4];
    {
        const uint32_t qbase = smem_u32(smem + Smem::q);
        const int mi = lane >> 3, rr = lane & 7;
        const int row = rr + 8 * (mi & 1);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int kk = dh * 16 + j;
            const int c = 2 * kk + (mi >> 1);
            ldmatrix_x4(qa[j][0], qa[j][1], qa[j][2], qa[j][3],
                        qbase + row * 1024 + (((c & ~7) | ((c ^ row) & 7)) << 4));
        }
    }

    float o[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    // positions of this thread's score rows lane/4 and lane/4 + 8 (-1: padding row, sees nothing)
    const int qpos0 = (lane >> 2) < R ? len - p.q_len + (lane >> 2) / G : -1;
    const int qpos1 = (lane >> 2) + 8 < R ? len - p.q_len + ((lane >> 2) + 8) / G : -1;
    float m_run0 = -INFINITY, m_run1 = -INFINITY;   // rows lane/4 and lane/4 + 8
    float l_run0 = 0.f, l_run1 = 0.f;               // partial over this thread's positions
    bool ok = true;
    int failed_it = n_tiles;

    for (int it = 0; it < n_tiles; ++it) {
        const int t = t_begin + it;
        const int st = it % NUM_STAGES;
        // the bf16 K/V tile the MMAs read: the stage itself, or the FP8
        // stage's converted copy
        uint8_t* stage = FP8 ? smem + Smem::tile : smem + st * Smem::stage_bytes;
        // refill the stage consumed in the previous iteration
        if (tid == 0 && it + NUM_STAGES - 1 < n_tiles) {
            const int nst = (it + NUM_STAGES - 1) % NUM_STAGES;
            issue_tile<FP8>(p, &tmk, &tmv, smem + nst * Smem::stage_bytes, &full_bar[nst], b,
                            kvh, t + NUM_STAGES - 1, lo, hi);
        }
        const TilePlan plan = plan_tile(p, b, t, lo, hi, false);
        // live positions of this tile: loaded and inside [lo, hi)
        uint32_t valid = plan.loaded;
        {
            const int pos0 = t * TILE_K;
            const int a = lo - pos0 > 0 ? lo - pos0 : 0;
            const int e = hi - pos0 < TILE_K ? hi - pos0 : TILE_K;
            const uint32_t upto = e >= 32 ? 0xffffffffu : ((1u << e) - 1u);
            const uint32_t from = a >= 32 ? 0u : ~((1u << a) - 1u);
            valid &= upto & from;
        }
        if (!mbar_wait(&full_bar[st], static_cast<uint32_t>((it / NUM_STAGES) & 1), p.err)) {
            ok = false;
        }
        // FP8: the previous tile's MMAs are past the barrier that ended the
        // last iteration, so the bf16 tile can be rewritten (after a failed
        // wait the converted bytes are never used)
        if constexpr (FP8) convert_fp8_stage(smem + st * Smem::stage_bytes, stage, valid, tid);
        if (__syncthreads_or(!ok)) {
            ok = false;
            failed_it = it;
            break;
        }

        // zero V rows that hold no live position (stale or poisoned data)
        if (!FP8 && valid != 0xffffffffu) {
            uint8_t* vt = stage + TILE_BYTES;
            for (int i = tid; i < TILE_K * 64; i += NUM_THREADS) {
                const int r = i & 31, cc = i >> 5;   // cc: 0..63 16-byte chunks of the row
                if (!((valid >> r) & 1u))
                    *reinterpret_cast<uint4*>(vt + (cc >> 3) * CHUNK_BYTES + r * 128 +
                                              ((cc & 7) << 4)) = make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
            __syncthreads();
        }

        // ---- S = Q K^T for n-tile nt over head-dim half dh
        float sc[4] = {0.f, 0.f, 0.f, 0.f};
        {
            const uint32_t kbase = smem_u32(stage);
            const int mi = lane >> 3;
            const int row = nt * 8 + (lane & 7);
#pragma unroll
            for (int j = 0; j < 16; j += 2) {
                const int kk = dh * 16 + j + (mi >> 1);
                const int sub = 2 * (kk & 3) + (mi & 1);
                uint32_t r0, r1, r2, r3;
                ldmatrix_x4(r0, r1, r2, r3, kbase + (kk >> 2) * CHUNK_BYTES + swz(row, sub));
                mma_bf16_16816(sc, qa[j], r0, r1);
                mma_bf16_16816(sc, qa[j + 1], r2, r3);
            }
        }
        if (dh == 1) xs[nt * 32 + lane] = make_float4(sc[0], sc[1], sc[2], sc[3]);
        __syncthreads();
        float pr[4];
        if (dh == 0) {
            const float4 x = xs[nt * 32 + lane];
            sc[0] += x.x;
            sc[1] += x.y;
            sc[2] += x.z;
            sc[3] += x.w;
            const int r = nt * 8 + 2 * (lane & 3);
            const bool v0 = (valid >> r) & 1u, v1 = (valid >> (r + 1)) & 1u;
            // each row sees the live keys up to its own position (and inside its window)
            const int pos = t * TILE_K + r;
            auto sees = [&](int kpos, int qp) {
                return kpos <= qp && (p.window <= 0 || kpos > qp - p.window);
            };
            sc[0] = v0 && sees(pos, qpos0) ? sc[0] * p.scale_log2 : -INFINITY;
            sc[1] = v1 && sees(pos + 1, qpos0) ? sc[1] * p.scale_log2 : -INFINITY;
            sc[2] = v0 && sees(pos, qpos1) ? sc[2] * p.scale_log2 : -INFINITY;
            sc[3] = v1 && sees(pos + 1, qpos1) ? sc[3] * p.scale_log2 : -INFINITY;
            float mx0 = fmaxf(sc[0], sc[1]), mx1 = fmaxf(sc[2], sc[3]);
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
            if ((lane & 3) == 0) {
                redm[nt * 16 + (lane >> 2)] = mx0;
                redm[nt * 16 + (lane >> 2) + 8] = mx1;
            }
        }
        __syncthreads();
        const int row0 = lane >> 2, row1 = row0 + 8;
        float tm0 = fmaxf(fmaxf(redm[row0], redm[16 + row0]), fmaxf(redm[32 + row0], redm[48 + row0]));
        float tm1 = fmaxf(fmaxf(redm[row1], redm[16 + row1]), fmaxf(redm[32 + row1], redm[48 + row1]));
        const float mn0 = fmaxf(m_run0, tm0), mn1 = fmaxf(m_run1, tm1);
        // a row that has seen no key yet keeps m = -inf; use 0 as its shift
        const float sh0 = mn0 == -INFINITY ? 0.f : mn0;
        const float sh1 = mn1 == -INFINITY ? 0.f : mn1;
        const float a0 = fast_exp2(m_run0 - sh0), a1 = fast_exp2(m_run1 - sh1);
        m_run0 = mn0;
        m_run1 = mn1;
        if (dh == 0) {
            pr[0] = fast_exp2(sc[0] - sh0);
            pr[1] = fast_exp2(sc[1] - sh0);
            pr[2] = fast_exp2(sc[2] - sh1);
            pr[3] = fast_exp2(sc[3] - sh1);
            l_run0 = l_run0 * a0 + pr[0] + pr[1];
            l_run1 = l_run1 * a1 + pr[2] + pr[3];
            uint8_t* ps = smem + Smem::p;
            const int col = nt * 8 + 2 * (lane & 3);
            *reinterpret_cast<uint32_t*>(ps + row0 * P_STRIDE + col * 2) = pack_bf16x2(pr[0], pr[1]);
            *reinterpret_cast<uint32_t*>(ps + row1 * P_STRIDE + col * 2) = pack_bf16x2(pr[2], pr[3]);
        }
        __syncthreads();

        // ---- O += P V for head-dim columns [64 warp, 64 warp + 64)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            o[j][0] *= a0;
            o[j][1] *= a0;
            o[j][2] *= a1;
            o[j][3] *= a1;
        }
        {
            const uint32_t pbase = smem_u32(smem + Smem::p);
            const uint32_t vbase = smem_u32(stage + TILE_BYTES + warp * CHUNK_BYTES);
            const int mi = lane >> 3;
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                uint32_t a[4];
                {
                    const int row = (lane & 7) + 8 * (mi & 1);
                    const int col = 16 * kk + 8 * (mi >> 1);
                    ldmatrix_x4(a[0], a[1], a[2], a[3], pbase + row * P_STRIDE + col * 2);
                }
                const int pos = 16 * kk + (lane & 7) + 8 * (mi & 1);
#pragma unroll
                for (int j = 0; j < 8; j += 2) {
                    uint32_t r0, r1, r2, r3;
                    ldmatrix_x4_trans(r0, r1, r2, r3, vbase + swz(pos, j + (mi >> 1)));
                    mma_bf16_16816(o[j], a, r0, r1);
                    mma_bf16_16816(o[j + 1], a, r2, r3);
                }
            }
        }
        __syncthreads();   // stage, P and the reduction buffers are free again
    }

    // Timeout path: before leaving, wait (bounded) for every tile load that
    // was issued but not consumed, so no copy lands in shared memory after
    // this CTA has exited.
    if (!ok && tid == 0) {
        for (int k = failed_it; k < n_tiles && k < failed_it + NUM_STAGES; ++k)
            if (!mbar_wait(&full_bar[k % NUM_STAGES], static_cast<uint32_t>((k / NUM_STAGES) & 1),
                           p.err))
                break;
    }

    // ---- l: sum over quad lanes and the 4 score warps
    if (warp < 4) {
        l_run0 += __shfl_xor_sync(0xffffffffu, l_run0, 1);
        l_run0 += __shfl_xor_sync(0xffffffffu, l_run0, 2);
        l_run1 += __shfl_xor_sync(0xffffffffu, l_run1, 1);
        l_run1 += __shfl_xor_sync(0xffffffffu, l_run1, 2);
        if ((lane & 3) == 0) {
            redl[warp * 16 + (lane >> 2)] = l_run0;
            redl[warp * 16 + (lane >> 2) + 8] = l_run1;
        }
    }
    __syncthreads();
    const size_t S = static_cast<size_t>(p.num_splits);
    const int row0 = lane >> 2, row1 = row0 + 8;
    // partial O (unnormalised), this warp's 64 columns
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int d = warp * 64 + 8 * j + 2 * (lane & 3);
        if (row0 < R) {
            const size_t h = (static_cast<size_t>(b) * p.q_len + row0 / G) * p.n_q_heads + kvh * G + row0 % G;
            *reinterpret_cast<float2*>(p.ws_o + (h * S + split) * D + d) =
                FP8 ? make_float2(ok ? o[j][0] * p.o_scale : 0.f, ok ? o[j][1] * p.o_scale : 0.f)
                    : make_float2(ok ? o[j][0] : 0.f, ok ? o[j][1] : 0.f);
        }
        if (row1 < R) {
            const size_t h = (static_cast<size_t>(b) * p.q_len + row1 / G) * p.n_q_heads + kvh * G + row1 % G;
            *reinterpret_cast<float2*>(p.ws_o + (h * S + split) * D + d) =
                FP8 ? make_float2(ok ? o[j][2] * p.o_scale : 0.f, ok ? o[j][3] * p.o_scale : 0.f)
                    : make_float2(ok ? o[j][2] : 0.f, ok ? o[j][3] : 0.f);
        }
    }
    // every thread holds the running max of rows lane/4 and lane/4 + 8;
    // warp 0 publishes them for the partial record
    if (warp == 0 && (lane & 3) == 0) {
        redm[lane >> 2] = m_run0;
        redm[(lane >> 2) + 8] = m_run1;
    }
    __syncthreads();
    if (tid < R) {
        const size_t h = (static_cast<size_t>(b) * p.q_len + tid / G) * p.n_q_heads + kvh * G + tid % G;
        const float l = redl[tid] + redl[16 + tid] + redl[32 + tid] + redl[48 + tid];
        const float m = redm[tid];
        p.ws_ml[(h * S + split) * 2 + 0] = ok && n_tiles > 0 ? m : -INFINITY;
        p.ws_ml[(h * S + split) * 2 + 1] = ok && n_tiles > 0 ? l : 0.f;
    }
}


// ---------------------------------------------------------------------------
// Streaming variant for small query groups (G <= 2 query heads per KV head).
//
// With two query heads per KV head the split is a pure stream of 2 KiB per
// position (K row + V row) and about 2 FLOP per byte, so it runs on the FP32
// units without any CTA-wide synchronisation: each warp owns every 8th chunk
// of 4 positions of the split, copies its lanes' 32-byte slices of the K and
// V rows into a private shared-memory ring with cp.async (positions outside
// the live band are zero-filled, never read), and keeps its own online
// softmax state with one (m, l) rescale per chunk ("Flash-Decoding for MQA in
// CUDA", "One KV head breaks the textbook": tile-granular rescale).  The 8
// warps' (m, l, O) are merged once at the end into the split's partial.
namespace stream {

constexpr int POS = 4;                   // positions per chunk
constexpr int STAGES = 3;                // chunks in flight per warp
constexpr int WARPS = 8;
constexpr int CHUNK_BYTES = 2 * POS * D * 2;          // K and V rows: 8 KiB
constexpr int RING_BYTES = WARPS * STAGES * CHUNK_BYTES;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
    // src-size 0 fills the 16 bytes with zeros without touching global memory
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void unpack8(const uint4 a, const uint4 b, float (&f)[16]) {
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

template <int G>
__global__ void __launch_bounds__(WARPS * 32, 1)
decode_stream_kernel(const DecodeParams p) {
    allow_merge_launch();
    extern __shared__ __align__(16) uint8_t smem[];
    const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    int len = p.kv_lens[b];
    if (len < 0 || len > p.len_cap) {
        if (threadIdx.x == 0 && split == 0 && kvh == 0) report_error(p.err, FA512_DEVICE_ERR_INDEX);
        len = len < 0 ? 0 : p.len_cap;
    }
    const int hi = len;
    const int lo = (p.window > 0 && len - p.window > 0) ? len - p.window : 0;
    // the split covers tiles of TILE_K positions, as in the tiled variant
    const int t_begin = lo / TILE_K + split * p.tiles_per_split;
    const int pb = max(lo, t_begin * TILE_K);
    const int pe = min(hi, (t_begin + p.tiles_per_split) * TILE_K);
    const int n_chunks = pe > pb ? (pe - pb + POS - 1) / POS : 0;

    // this lane's 16 head-dim columns of the G query rows, in fp32
    float q[G][16];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const uint4* src = reinterpret_cast<const uint4*>(
            p.q + (static_cast<size_t>(b) * p.n_q_heads + kvh * G + g) * D + lane * 16);
        unpack8(src[0], src[1], q[g]);
    }
    float m[G], l[G], o[G][16];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        m[g] = -INFINITY;
        l[g] = 0.f;
#pragma unroll
        for (int d = 0; d < 16; ++d) o[g][d] = 0.f;
    }

    const uint32_t ring = smem_u32(smem) + warp * STAGES * CHUNK_BYTES;
    // chunk k of this warp covers positions pb + (warp + 8k) * POS ...
    const int my_chunks = n_chunks > warp ? (n_chunks - warp + WARPS - 1) / WARPS : 0;
    // Page of position pos0 + (lane % POS) of chunk k.  Each chunk's pages are
    // loaded one chunk before its copies are issued, so the copies never wait
    // on a page-table load.
    auto page_of = [&](int k) -> int {
        const int pos = pb + (warp + WARPS * k) * POS + (lane & (POS - 1));
        return (k < my_chunks && pos < pe)
                   ? p.page_table[static_cast<size_t>(b) * p.max_pages_per_seq + pos / p.page_size]
                   : 0;
    };
    auto issue = [&](int k, int page_lane) {
        if (k < my_chunks) {
            const int pos0 = pb + (warp + WARPS * k) * POS;
            const uint32_t st = ring + (k % STAGES) * CHUNK_BYTES;
#pragma unroll
            for (int i = 0; i < POS; ++i) {
                const int pos = pos0 + i;
                const int page = __shfl_sync(0xffffffffu, page_lane, i);
                bool valid = pos < pe;
                size_t row = 0;
                if (valid) {
                    if (page < 0 || page >= p.num_pages) {
                        report_error(p.err, FA512_DEVICE_ERR_INDEX);
                        valid = false;
                    } else {
                        row = (static_cast<size_t>(page) * p.page_size + (pos & (p.page_size - 1))) * p.n_kv_heads + kvh;
                    }
                }
                const __nv_bfloat16* ks = p.k_pages + row * D + lane * 16;
                const __nv_bfloat16* vs = p.v_pages + row * D + lane * 16;
                const uint32_t kd = st + i * (D * 2) + lane * 32;
                const uint32_t vd = st + (POS + i) * (D * 2) + lane * 32;
                cp_async16(kd, ks, valid);
                cp_async16(kd + 16, ks + 8, valid);
                cp_async16(vd, vs, valid);
                cp_async16(vd + 16, vs + 8, valid);
            }
        }
        cp_async_commit();   // one group per chunk slot, empty past the end
    };
    int page_next = page_of(STAGES - 1);
#pragma unroll
    for (int k = 0; k < STAGES - 1; ++k) issue(k, page_of(k));

    for (int k = 0; k < my_chunks; ++k) {
        const int page_now = page_next;
        page_next = page_of(k + STAGES);
        issue(k + STAGES - 1, page_now);
        cp_async_wait<STAGES - 1>();   // this lane's copies of chunk k have landed
        const uint8_t* st = smem + (warp * STAGES + (k % STAGES)) * CHUNK_BYTES;
        const int pos0 = pb + (warp + WARPS * k) * POS;
        float s[POS][G];
#pragma unroll
        for (int i = 0; i < POS; ++i) {
            float kf[16];
            const uint4* kr = reinterpret_cast<const uint4*>(st + i * (D * 2) + lane * 32);
            unpack8(kr[0], kr[1], kf);
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float acc = 0.f;
#pragma unroll
                for (int d = 0; d < 16; ++d) acc = fmaf(q[g][d], kf[d], acc);
                s[i][g] = acc;
            }
        }
#pragma unroll
        for (int i = 0; i < POS; ++i)
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float v = s[i][g];
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
                s[i][g] = (pos0 + i < pe) ? v * p.scale_log2 : -INFINITY;
            }
        float pr[POS][G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float cm = s[0][g];
#pragma unroll
            for (int i = 1; i < POS; ++i) cm = fmaxf(cm, s[i][g]);
            const float mn = fmaxf(m[g], cm);
            const float sh = mn == -INFINITY ? 0.f : mn;   // no key seen yet
            const float a = fast_exp2(m[g] - sh);
            float ps = 0.f;
#pragma unroll
            for (int i = 0; i < POS; ++i) {
                pr[i][g] = fast_exp2(s[i][g] - sh);
                ps += pr[i][g];
            }
            l[g] = l[g] * a + ps;
            m[g] = mn;
#pragma unroll
            for (int d = 0; d < 16; ++d) o[g][d] *= a;
        }
#pragma unroll
        for (int i = 0; i < POS; ++i) {
            float vf[16];
            const uint4* vr = reinterpret_cast<const uint4*>(st + (POS + i) * (D * 2) + lane * 32);
            unpack8(vr[0], vr[1], vf);
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
                for (int d = 0; d < 16; ++d) o[g][d] = fmaf(pr[i][g], vf[d], o[g][d]);
        }
    }
    cp_async_wait<0>();
    __syncthreads();   // every warp is done with its ring: reuse it for the merge

    float* so = reinterpret_cast<float*>(smem);                 // [WARPS][G][512]
    float* sml = so + WARPS * G * D;                             // [WARPS][G][2]
#pragma unroll
    for (int g = 0; g < G; ++g) {
        float4* dst = reinterpret_cast<float4*>(so + (warp * G + g) * D + lane * 16);
#pragma unroll
        for (int d = 0; d < 4; ++d)
            dst[d] = make_float4(o[g][4 * d], o[g][4 * d + 1], o[g][4 * d + 2], o[g][4 * d + 3]);
        if (lane == 0) {
            sml[(warp * G + g) * 2] = m[g];
            sml[(warp * G + g) * 2 + 1] = l[g];
        }
    }
    __syncthreads();
    const size_t S = static_cast<size_t>(p.num_splits);
    for (int idx = threadIdx.x; idx < G * D; idx += WARPS * 32) {
        const int g = idx / D, d = idx - g * D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < WARPS; ++w) M = fmaxf(M, sml[(w * G + g) * 2]);
        float acc = 0.f, L = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < WARPS; ++w) {
                const float wt = fast_exp2(sml[(w * G + g) * 2] - M);   // 0 for a warp with no key
                acc += wt * so[(w * G + g) * D + d];
                L += wt * sml[(w * G + g) * 2 + 1];
            }
        }
        const size_t h = static_cast<size_t>(b) * p.n_q_heads + kvh * G + g;
        p.ws_o[(h * S + split) * D + d] = acc;
        if (d == 0) {
            p.ws_ml[(h * S + split) * 2 + 0] = M;
            p.ws_ml[(h * S + split) * 2 + 1] = M == -INFINITY ? 0.f : L;
        }
    }
}

}  // namespace stream

// ---------------------------------------------------------------------------
// FP8 E4M3 cache, up to 8 query rows (q_len * G <= 8): streaming warps on the
// tensor cores.
//
// Decoding every cache byte to fp32 for FMA dot products costs more issue
// slots per position than HBM takes to deliver it, so here the products run
// on mma.sync (f16 operands, fp32 accumulation) with the query rows in the N
// dimension: S^T = K Q^T (M = 16 positions, K = head dims) and O^T = V^T P^T
// (M = 16 head-dim columns, K = 16 positions).  E4M3 -> f16 is exact, through
// the hardware e4m3x2 -> f16x2 conversion: a K operand pair is two
// neighbouring bytes of one row, a V pair two positions' bytes of one column,
// gathered by one byte permute.
//
// A CTA is one split of the keys and four warps, one per head-dim slice of
// 128.  The four stream the split's chunks of 16 positions together: each
// copies its slice of the chunk's K and V rows (128 + 128 bytes a position)
// into a private cp.async ring, forms its slice of S^T, and the four swap
// their partial scores through shared memory at a CTA barrier, so all hold
// the same scores, softmax state and P; each then accumulates its own 128
// columns of O^T and, after the split's last chunk, writes them to the
// split's (O, m, l) partial straight from its registers.  Four such CTAs
// share an SM (16 warps): while one waits on its first page-table entries
// and copies, or writes its partial, the other three keep streaming, and a
// finished CTA's slot takes the next split at once.
//
// (The bf16 kernel below groups four such position groups in one CTA of 16
// warps and merges them in shared memory before writing one partial.)
namespace mma8 {

constexpr int GROUPS = 4;                        // position groups of the bf16 kernel's CTA
constexpr int SLICES = 4;                        // head-dim slices
constexpr int WARPS = GROUPS * SLICES;
constexpr int CPOS = 16;                         // positions per chunk
constexpr int SLICE = D / SLICES;                // head-dim bytes (elements) per warp: 128
constexpr int KSTEPS = SLICE / 16;               // k-steps of 16 per slice: 8
constexpr int MTILES = SLICE / 16;               // m-tiles of 16 columns per slice: 8
constexpr int STAGES = 3;
constexpr int CHUNK_BYTES = 2 * CPOS * SLICE;    // this warp's K and V slices: 4 KiB
constexpr int RING_BYTES = WARPS * STAGES * CHUNK_BYTES;
constexpr int XCH_BYTES = 2 * GROUPS * SLICES * 32 * 16;   // [parity][group][slice][lane] float4
constexpr int SMEM_BYTES = RING_BYTES + XCH_BYTES;
static_assert(WARPS * 8 * SLICE * 4 + WARPS * 8 * 2 * 4 <= RING_BYTES, "merge buffer fits the ring");

// the FP8 kernel's CTA: one position group
constexpr int F8_WARPS = SLICES;
constexpr int F8_CTAS_PER_SM = 4;
constexpr int F8_RING_BYTES = F8_WARPS * STAGES * CHUNK_BYTES;    // 48 KiB
constexpr int F8_XCH_BYTES = 2 * SLICES * 32 * 16;                // [parity][slice][lane] float4
constexpr int F8_SMEM_BYTES = F8_RING_BYTES + F8_XCH_BYTES;
static_assert(F8_CTAS_PER_SM * (F8_SMEM_BYTES + 1024) <= 228 * 1024, "four CTAs fit an SM's shared memory");

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// 16-byte piece c of row r (a chunk position, K or V) sits at piece
// (c + 4r + 2 (r / 2)) & 7 of the row: the async copies (lane pairs fill one
// row each), the K reads (lanes of a quarter warp read pieces t of rows g,
// g + 1) and the V reads (piece g of rows 2t, 2t + 1) then touch eight
// different bank groups per quarter warp.
__device__ __forceinline__ int swz(int r) { return 4 * r + 2 * (r >> 1); }

__device__ __forceinline__ void bar_group(int id) {
    asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory");
}

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two e4m3 values (low byte first) -> f16x2, exactly (hardware conversion).
__device__ __forceinline__ uint32_t e4m3x2_f16x2(uint32_t two) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<unsigned short>(two)));
    return h2;
}

// Byte k of word x and byte k of word y -> f16x2 {x_k, y_k}, exactly: one
// permute gathers the two bytes, the hardware conversion widens them.
template <int K>
__device__ __forceinline__ uint32_t e4m3_pair_f16x2(uint32_t x, uint32_t y) {
    constexpr uint32_t sel = K | ((4 + K) << 4);
    uint32_t t;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(t) : "r"(x), "r"(y), "n"(sel));
    return e4m3x2_f16x2(t & 0xffffu);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Transpose of an 8 x 8 matrix of 16-bit values held in the mma fragment
// layout (lane 4 i + j holds elements (i, 2j) and (i, 2j + 1)).
__device__ __forceinline__ uint32_t transpose8x8(uint32_t a) {
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}

__global__ void __launch_bounds__(F8_WARPS * 32, F8_CTAS_PER_SM)
decode_fp8_mma_kernel(const DecodeParams p) {
    allow_merge_launch();
    extern __shared__ __align__(16) uint8_t smem[];
    const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int sl = threadIdx.x >> 5, lane = threadIdx.x & 31;   // warp = head-dim slice
    const int g = lane >> 2, t = lane & 3;   // mma fragment coordinates
    const int G = p.group;
    const int R = p.q_len * G;               // query rows, <= 8

    int len = p.kv_lens[b];
    if (len < 0 || len > p.len_cap) {
        if (threadIdx.x == 0 && split == 0 && kvh == 0) report_error(p.err, FA512_DEVICE_ERR_INDEX);
        len = len < 0 ? 0 : p.len_cap;
    }
    // union of the rows' bands (the row of token t sees [pos - window + 1, pos])
    const int hi = len;
    const int w_lo = len - p.q_len + 1 - p.window;
    const int lo = (p.window > 0 && w_lo > 0) ? w_lo : 0;
    const int t_begin = lo / TILE_K + split * p.tiles_per_split;
    const int pb = max(lo, t_begin * TILE_K);
    const int pe = min(hi, (t_begin + p.tiles_per_split) * TILE_K);
    const int n_chunks = pe > pb ? (pe - pb + CPOS - 1) / CPOS : 0;

    // ---- Q^T fragments of this warp's slice: b0/b1 of k-step (j, s) hold
    // row g's elements 64 j + 16 t + 4 s + {0, 1} / {2, 3}, in f16 after a
    // power-of-two scale per row and slice that keeps the largest element
    // below 2^15 (exact; every partial score is unscaled before the swap)
    uint32_t qb[KSTEPS][2];
    float rs[2];                              // 1 / (this slice's scale) of rows 2t, 2t + 1
    {
        float qmax = 0.f;
        float qv[KSTEPS][4];
        const bool row_ok = g < R;
        const size_t qrow = (static_cast<size_t>(b) * p.q_len + (row_ok ? g / G : 0)) * p.n_q_heads +
                            kvh * G + (row_ok ? g % G : 0);
#pragma unroll
        for (int j = 0; j < KSTEPS / 4; ++j) {
            // 16 elements: 64 j + 16 t .. + 15 of this slice
            const uint4* src = reinterpret_cast<const uint4*>(p.q + qrow * D + sl * SLICE + 64 * j + 16 * t);
            const uint4 a = row_ok ? src[0] : make_uint4(0u, 0u, 0u, 0u);
            const uint4 c = row_ok ? src[1] : make_uint4(0u, 0u, 0u, 0u);
            const uint32_t w[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                qv[4 * j + s][0] = __uint_as_float(w[2 * s] << 16);
                qv[4 * j + s][1] = __uint_as_float(w[2 * s] & 0xffff0000u);
                qv[4 * j + s][2] = __uint_as_float(w[2 * s + 1] << 16);
                qv[4 * j + s][3] = __uint_as_float(w[2 * s + 1] & 0xffff0000u);
#pragma unroll
                for (int e = 0; e < 4; ++e) qmax = fmaxf(qmax, fabsf(qv[4 * j + s][e]));
            }
        }
        // the row's maximum over its four lanes (t) of this slice
        qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, 1));
        qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, 2));
        // qscale = 2^(14 - E), E = exponent of qmax (qmax = 0 or not finite: 1)
        const int E = (__float_as_uint(qmax) >> 23) & 0xff;
        const int biased = min(127 + 14 + 127 - E, 254);     // 2^(14 - (E - 127)), at most 2^127
        const float qscale = (qmax > 0.f && E < 255) ? __uint_as_float(static_cast<uint32_t>(biased) << 23) : 1.f;
#pragma unroll
        for (int k = 0; k < KSTEPS; ++k) {
            qb[k][0] = pack_f16x2(qv[k][0] * qscale, qv[k][1] * qscale);
            qb[k][1] = pack_f16x2(qv[k][2] * qscale, qv[k][3] * qscale);
        }
        // rows 2t, 2t + 1 are held by lanes with g = 2t, 2t + 1
        rs[0] = 1.f / __shfl_sync(0xffffffffu, qscale, 4 * (2 * t));
        rs[1] = 1.f / __shfl_sync(0xffffffffu, qscale, 4 * (2 * t + 1));
    }
    // positions of rows 2t and 2t + 1 (-1: padding row, sees nothing)
    int qpos[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int r = 2 * t + i;
        qpos[i] = r < R ? len - p.q_len + r / G : -1;
    }

    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    float o[MTILES][4];                       // O^T: m-tile i = columns 16 g + 2 i, 16 g + 2 i + 1
#pragma unroll
    for (int i = 0; i < MTILES; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

    const uint32_t ring = smem_u32(smem) + sl * STAGES * CHUNK_BYTES;
    float4* xch = reinterpret_cast<float4*>(smem + F8_RING_BYTES);

    // copy plan: lane l fetches position l / 2 of the chunk; at step s it
    // copies 16-byte piece (l & 1) + 2 (s % 4) of that position's K slice
    // (s < 4) or V slice (s >= 4), so every instruction covers whole 32-byte
    // sectors.
    // page of this lane's position in chunk k, loaded one chunk before the
    // chunk's copies are issued (the copies never wait on the page table)
    auto page_of = [&](int k) -> int {
        const int pos = pb + k * CPOS + (lane >> 1);
        return (k < n_chunks && pos < pe)
                   ? p.page_table[static_cast<size_t>(b) * p.max_pages_per_seq + pos / p.page_size]
                   : 0;
    };
    auto issue = [&](int k, int page) {
        if (k < n_chunks) {
            const int pos = pb + k * CPOS + (lane >> 1);
            bool valid = pos < pe;
            size_t row = 0;
            if (valid) {
                if (page < 0 || page >= p.num_pages) {
                    report_error(p.err, FA512_DEVICE_ERR_INDEX);
                    valid = false;
                } else {
                    row = (static_cast<size_t>(page) * p.page_size + (pos & (p.page_size - 1))) * p.n_kv_heads + kvh;
                }
            }
            const uint8_t* ksrc = p.k8 + row * D + sl * SLICE;
            const uint8_t* vsrc = p.v8 + row * D + sl * SLICE;
            const uint32_t st = ring + (k % STAGES) * CHUNK_BYTES;
            const int r = lane >> 1;
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const int c = (lane & 1) + 2 * (s & 3);
                const uint32_t dst = st + (s >> 2) * (CPOS * SLICE) + r * SLICE + (((c + swz(r)) & 7) << 4);
                cp_async16(dst, (s < 4 ? ksrc : vsrc) + c * 16, valid);
            }
        }
        cp_async_commit();
    };
    int page_next = page_of(STAGES - 1);
#pragma unroll
    for (int k = 0; k < STAGES - 1; ++k) issue(k, page_of(k));

    for (int k = 0; k < n_chunks; ++k) {
        const int page_now = page_next;
        page_next = page_of(k + STAGES);
        issue(k + STAGES - 1, page_now);
        cp_async_wait<STAGES - 1>();
        __syncwarp();                         // every lane's copies of chunk k are visible
        const uint8_t* kst = smem + (sl * STAGES + (k % STAGES)) * CHUNK_BYTES;
        const uint8_t* vst = kst + CPOS * SLICE;
        const int pos0 = pb + k * CPOS;

        // ---- S^T slice = K_slice Q_slice^T, one accumulator chain per 64
        // head-dim elements, summed at the end
        float sc[4];
        {
            float acc[KSTEPS / 4][4];
#pragma unroll
            for (int j = 0; j < KSTEPS / 4; ++j) {
                acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
                const uint4 ka = *reinterpret_cast<const uint4*>(kst + g * SLICE + (((4 * j + t + swz(g)) & 7) << 4));
                const uint4 kb = *reinterpret_cast<const uint4*>(kst + (g + 8) * SLICE + (((4 * j + t + swz(g + 8)) & 7) << 4));
                const uint32_t wa[4] = {ka.x, ka.y, ka.z, ka.w}, wb[4] = {kb.x, kb.y, kb.z, kb.w};
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_f16_16816(acc[j], e4m3x2_f16x2(wa[s] & 0xffffu), e4m3x2_f16x2(wb[s] & 0xffffu),
                                  e4m3x2_f16x2(wa[s] >> 16), e4m3x2_f16x2(wb[s] >> 16),
                                  qb[4 * j + s][0], qb[4 * j + s][1]);
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) sc[e] = (acc[0][e] + acc[1][e]) * (e & 1 ? rs[1] : rs[0]);
        }
        // ---- swap slices with the other three warps: S = (S_0 + S_1) + (S_2 + S_3),
        // each slice unscaled by its own row scale first (a power of two,
        // exact); the same sum, in the same order, in all four warps
        {
            float4* base = xch + (k & 1) * SLICES * 32 + lane;
            base[sl * 32] = make_float4(sc[0], sc[1], sc[2], sc[3]);
            __syncthreads();
            const float4 x0 = base[0], x1 = base[32], x2 = base[64], x3 = base[96];
            sc[0] = (x0.x + x1.x) + (x2.x + x3.x);
            sc[1] = (x0.y + x1.y) + (x2.y + x3.y);
            sc[2] = (x0.z + x1.z) + (x2.z + x3.z);
            sc[3] = (x0.w + x1.w) + (x2.w + x3.w);
        }
        // ---- online softmax: this thread holds positions g, g + 8 of rows
        // 2t, 2t + 1; both rows step together (independent shuffle chains)
        float pr[4], sv[2][2], cm[2], al[2], ps[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            auto sees = [&](int kp) {
                return kp < pe && kp <= qpos[i] && (p.window <= 0 || kp > qpos[i] - p.window);
            };
            sv[i][0] = sees(pos0 + g) ? sc[i] * p.scale_log2 : -INFINITY;
            sv[i][1] = sees(pos0 + g + 8) ? sc[2 + i] * p.scale_log2 : -INFINITY;
            cm[i] = fmaxf(sv[i][0], sv[i][1]);
        }
        // the chunk maxima of both rows in one packed bf16x2 reduction: the
        // running max is only the softmax's reference and needs to be the
        // same in every lane of a row, not exact (bf16 keeps fp32's range;
        // rounding moves it by < 0.4 %, so p stays below 2^(0.004 |s|))
        {
            uint32_t c2 = pack_bf16x2(cm[0], cm[1]);
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                const uint32_t x = __shfl_xor_sync(0xffffffffu, c2, off);
                asm("max.bf16x2 %0, %0, %1;" : "+r"(c2) : "r"(x));
            }
            cm[0] = __uint_as_float(c2 << 16);
            cm[1] = __uint_as_float(c2 & 0xffff0000u);
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const float mn = fmaxf(m[i], cm[i]);
            const float sh = mn == -INFINITY ? 0.f : mn;
            // a row that has still seen no key has nothing to rescale
            al[i] = mn == -INFINITY ? 1.f : fast_exp2(m[i] - sh);
            pr[i] = fast_exp2(sv[i][0] - sh);
            pr[2 + i] = fast_exp2(sv[i][1] - sh);
            ps[i] = pr[i] + pr[2 + i];
            m[i] = mn;
        }
        // l stays a per-lane partial (every lane of a row rescales by the
        // same alpha); the lanes are summed once, after the last chunk
        l[0] = l[0] * al[0] + ps[0];
        l[1] = l[1] * al[1] + ps[1];
        if (__any_sync(0xffffffffu, al[0] != 1.f || al[1] != 1.f)) {
#pragma unroll
            for (int c = 0; c < MTILES; ++c) {
                o[c][0] *= al[0];
                o[c][1] *= al[1];
                o[c][2] *= al[0];
                o[c][3] *= al[1];
            }
        }
        // ---- P^T fragments b0 = P[row g][pos 2t, 2t + 1], b1 = P[g][2t + 8, 2t + 9]:
        // this lane holds P[2t, 2t + 1][pos g] (and pos g + 8), i.e. element
        // (g, 2t) of the 8 x 8 matrix [pos][row] in fragment layout; its
        // transpose is the B fragment
        const uint32_t pb0 = transpose8x8(pack_f16x2(pr[0], pr[1]));
        const uint32_t pb1 = transpose8x8(pack_f16x2(pr[2], pr[3]));
        // ---- O^T slice += V_slice^T P^T: thread g's columns are bytes
        // 16 g .. 16 g + 15 of each row (column pair i at bytes 2i, 2i + 1);
        // rows 2t, 2t + 1, 2t + 8, 2t + 9
        uint32_t vw[4][4];
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) {
            const int r = 2 * t + (rr & 1) + 8 * (rr >> 1);
            const uint4 x = *reinterpret_cast<const uint4*>(vst + r * SLICE + (((g + swz(r)) & 7) << 4));
            vw[rr][0] = x.x;
            vw[rr][1] = x.y;
            vw[rr][2] = x.z;
            vw[rr][3] = x.w;
        }
#pragma unroll
        for (int i = 0; i < MTILES; ++i) {
            const int wi = i >> 1;
            uint32_t a0, a1, a2, a3;
            if (i & 1) {
                a0 = e4m3_pair_f16x2<2>(vw[0][wi], vw[1][wi]);
                a1 = e4m3_pair_f16x2<3>(vw[0][wi], vw[1][wi]);
                a2 = e4m3_pair_f16x2<2>(vw[2][wi], vw[3][wi]);
                a3 = e4m3_pair_f16x2<3>(vw[2][wi], vw[3][wi]);
            } else {
                a0 = e4m3_pair_f16x2<0>(vw[0][wi], vw[1][wi]);
                a1 = e4m3_pair_f16x2<1>(vw[0][wi], vw[1][wi]);
                a2 = e4m3_pair_f16x2<0>(vw[2][wi], vw[3][wi]);
                a3 = e4m3_pair_f16x2<1>(vw[2][wi], vw[3][wi]);
            }
            mma_f16_16816(o[i], a0, a1, a2, a3, pb0, pb1);
        }
        __syncwarp();                         // the stage may be refilled
    }
    cp_async_wait<0>();
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) l[i] += __shfl_xor_sync(0xffffffffu, l[i], off);

    // ---- this split's partial, unnormalised and times v_scale: row 2t + i
    // holds columns 16 g .. 16 g + 15 of this slice (m-tile j: columns
    // 16 g + 2 j in o[j][i], 16 g + 2 j + 1 in o[j][2 + i]); m and l are the
    // same in every slice warp, written by slice 0.  A split that saw no key
    // has m = -inf and O = 0.
    const size_t S = static_cast<size_t>(p.num_splits);
    const float osc = p.o_scale;              // v_scale of the FP8 cache
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int r = 2 * t + i;
        if (r < R) {
            const size_t hq = (static_cast<size_t>(b) * p.q_len + r / G) * p.n_q_heads + kvh * G + r % G;
            float4* dst = reinterpret_cast<float4*>(p.ws_o + (hq * S + split) * D + sl * SLICE + 16 * g);
#pragma unroll
            for (int j = 0; j < MTILES / 2; ++j)
                dst[j] = make_float4(o[2 * j][i] * osc, o[2 * j][2 + i] * osc, o[2 * j + 1][i] * osc,
                                     o[2 * j + 1][2 + i] * osc);
            if (sl == 0 && g == 0) {
                p.ws_ml[(hq * S + split) * 2 + 0] = m[i];
                p.ws_ml[(hq * S + split) * 2 + 1] = m[i] == -INFINITY ? 0.f : l[i];
            }
        }
    }
}

}  // namespace mma8

// ---------------------------------------------------------------------------
// bf16 cache, 3 to 8 query rows (several tokens, or 3-8 query heads per KV
// head): the streaming tensor-core design of the FP8 kernel above, for the
// rows the FMA streaming kernel cannot take, with four position groups of
// four slice warps in one CTA (16 warps) that stride over the split's
// chunks and merge their (O, m, l) in shared memory at the end.  A bf16
// position carries 2 KiB, so the design's per-position instruction cost fits
// twice the HBM time it has at FP8; its operands need no widening (K pairs are the A
// operand as stored; each V operand pair is one 16-bit permute of two
// positions' words).  Shared memory (16 warps x 3 stages) holds chunks of 8
// positions: S^T runs with M = 16 over 8 positions (the other 8 rows zero)
// and O^T = V^T P^T with K = 16 over them (the other 8 zero).
namespace mma16 {

using mma8::GROUPS;
using mma8::SLICES;
using mma8::WARPS;
constexpr int CPOS = 8;                          // positions per chunk
constexpr int SLICE = D / SLICES;                // head-dim elements per warp: 128
constexpr int ROW = SLICE * 2;                   // bytes of a row slice: 256
constexpr int KGROUPS = SLICE / 32;              // 16-byte loads per K row: 4 (2 k-steps each)
constexpr int MTILES = SLICE / 16;               // m-tiles of 16 columns: 8
constexpr int STAGES = 3;
constexpr int CHUNK_BYTES = 2 * CPOS * ROW;      // 4 KiB
constexpr int RING_BYTES = WARPS * STAGES * CHUNK_BYTES;
constexpr int XCH_BYTES = mma8::XCH_BYTES;
constexpr int SMEM_BYTES = RING_BYTES + XCH_BYTES;
static_assert(WARPS * 8 * SLICE * 4 + WARPS * 8 * 2 * 4 <= RING_BYTES, "merge buffer fits the ring");

// 16-byte piece c of a K row r sits at piece (c + 4r) & 15, of a V row at
// (c + 4r + r/2 + 2 (r/4)) & 15: the async copies (four lanes per row), the K
// reads (pieces 4j + t of row g) and the V reads (pieces 2g, 2g + 1 of rows
// 2t, 2t + 1) then touch eight different bank groups per quarter warp.
__device__ __forceinline__ int swz_k(int r) { return 4 * r; }
__device__ __forceinline__ int swz_v(int r) { return 4 * r + (r >> 1) + 2 * (r >> 2); }

__device__ __forceinline__ uint32_t prmt(uint32_t x, uint32_t y, uint32_t sel) {
    uint32_t t;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(t) : "r"(x), "r"(y), "r"(sel));
    return t;
}

__global__ void __launch_bounds__(WARPS * 32, 1)
decode_bf16_mma_kernel(const DecodeParams p) {
    allow_merge_launch();
    extern __shared__ __align__(16) uint8_t smem[];
    const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // a position group's four slice warps sit on the four different SM
    // sub-partitions (warp % 4), so that while they meet at their per-chunk
    // barrier each scheduler still has the other groups' warps to issue
    const int pg = warp / SLICES;            // position group
    const int sl = warp & (SLICES - 1);      // head-dim slice
    const int g = lane >> 2, t = lane & 3;   // mma fragment coordinates
    const int G = p.group;
    const int R = p.q_len * G;               // query rows, <= 8

    int len = p.kv_lens[b];
    if (len < 0 || len > p.len_cap) {
        if (threadIdx.x == 0 && split == 0 && kvh == 0) report_error(p.err, FA512_DEVICE_ERR_INDEX);
        len = len < 0 ? 0 : p.len_cap;
    }
    const int hi = len;
    const int w_lo = len - p.q_len + 1 - p.window;
    const int lo = (p.window > 0 && w_lo > 0) ? w_lo : 0;
    const int t_begin = lo / TILE_K + split * p.tiles_per_split;
    const int pb = max(lo, t_begin * TILE_K);
    const int pe = min(hi, (t_begin + p.tiles_per_split) * TILE_K);
    const int n_chunks = pe > pb ? (pe - pb + CPOS - 1) / CPOS : 0;
    const int my_chunks = n_chunks > pg ? (n_chunks - pg + GROUPS - 1) / GROUPS : 0;

    // ---- Q^T fragments (bf16, as stored): b0/b1 of k-step (j, s) hold row
    // g's elements 32 j + 8 t + 4 s + {0, 1} / {2, 3} of this slice
    uint32_t qb[2 * KGROUPS][2];
    {
        const bool row_ok = g < R;
        const size_t qrow = (static_cast<size_t>(b) * p.q_len + (row_ok ? g / G : 0)) * p.n_q_heads +
                            kvh * G + (row_ok ? g % G : 0);
#pragma unroll
        for (int j = 0; j < KGROUPS; ++j) {
            const uint4 a = row_ok ? *reinterpret_cast<const uint4*>(p.q + qrow * D + sl * SLICE + 32 * j + 8 * t)
                                   : make_uint4(0u, 0u, 0u, 0u);
            qb[2 * j][0] = a.x;
            qb[2 * j][1] = a.y;
            qb[2 * j + 1][0] = a.z;
            qb[2 * j + 1][1] = a.w;
        }
    }
    int qpos[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int r = 2 * t + i;
        qpos[i] = r < R ? len - p.q_len + r / G : -1;
    }

    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    float o[MTILES][4];                       // O^T: m-tile i = columns 16 g + 2 i, 16 g + 2 i + 1
#pragma unroll
    for (int i = 0; i < MTILES; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

    const uint32_t ring = smem_u32(smem) + warp * STAGES * CHUNK_BYTES;
    float4* xch = reinterpret_cast<float4*>(smem + RING_BYTES);

    // copy plan: lane l fetches position l / 4 of the chunk; at step s it
    // copies piece (l & 3) + 4 (s % 4) of that position's K slice (s < 4) or
    // V slice (s >= 4): four lanes cover 64 contiguous bytes of a row
    // page of this lane's position in chunk k, loaded one chunk before the
    // chunk's copies are issued (the copies never wait on the page table)
    auto page_of = [&](int k) -> int {
        const int pos = pb + (pg + GROUPS * k) * CPOS + (lane >> 2);
        return (k < my_chunks && pos < pe)
                   ? p.page_table[static_cast<size_t>(b) * p.max_pages_per_seq + pos / p.page_size]
                   : 0;
    };
    auto issue = [&](int k, int page) {
        if (k < my_chunks) {
            const int pos = pb + (pg + GROUPS * k) * CPOS + (lane >> 2);
            bool valid = pos < pe;
            size_t row = 0;
            if (valid) {
                if (page < 0 || page >= p.num_pages) {
                    report_error(p.err, FA512_DEVICE_ERR_INDEX);
                    valid = false;
                } else {
                    row = (static_cast<size_t>(page) * p.page_size + (pos & (p.page_size - 1))) * p.n_kv_heads + kvh;
                }
            }
            const uint8_t* ksrc = reinterpret_cast<const uint8_t*>(p.k_pages + row * D + sl * SLICE);
            const uint8_t* vsrc = reinterpret_cast<const uint8_t*>(p.v_pages + row * D + sl * SLICE);
            const uint32_t st = ring + (k % STAGES) * CHUNK_BYTES;
            const int r = lane >> 2;
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const int c = (lane & 3) + 4 * (s & 3);
                const int f = s < 4 ? swz_k(r) : swz_v(r);
                const uint32_t dst = st + (s >> 2) * (CPOS * ROW) + r * ROW + (((c + f) & 15) << 4);
                mma8::cp_async16(dst, (s < 4 ? ksrc : vsrc) + c * 16, valid);
            }
        }
        mma8::cp_async_commit();
    };
    int page_next = page_of(STAGES - 1);
#pragma unroll
    for (int k = 0; k < STAGES - 1; ++k) issue(k, page_of(k));

    for (int k = 0; k < my_chunks; ++k) {
        const int page_now = page_next;
        page_next = page_of(k + STAGES);
        issue(k + STAGES - 1, page_now);
        mma8::cp_async_wait<STAGES - 1>();
        __syncwarp();                         // every lane's copies of chunk k are visible
        const uint8_t* kst = smem + (warp * STAGES + (k % STAGES)) * CHUNK_BYTES;
        const uint8_t* vst = kst + CPOS * ROW;
        const int pos0 = pb + (pg + GROUPS * k) * CPOS;

        // ---- S^T slice = K_slice Q_slice^T over positions g (rows g + 8 are zero);
        // one accumulator chain per 32 head-dim elements, summed at the end
        float sc[2];
        {
            float acc[KGROUPS][4];
#pragma unroll
            for (int j = 0; j < KGROUPS; ++j) {
                acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
                const uint4 ka = *reinterpret_cast<const uint4*>(kst + g * ROW + (((4 * j + t + swz_k(g)) & 15) << 4));
                mma_bf16_16816(acc[j], {ka.x, 0u, ka.y, 0u}, qb[2 * j][0], qb[2 * j][1]);
                mma_bf16_16816(acc[j], {ka.z, 0u, ka.w, 0u}, qb[2 * j + 1][0], qb[2 * j + 1][1]);
            }
            sc[0] = (acc[0][0] + acc[1][0]) + (acc[2][0] + acc[3][0]);
            sc[1] = (acc[0][1] + acc[1][1]) + (acc[2][1] + acc[3][1]);
        }
        // ---- swap slices with the group's other warps: S = (S_0 + S_1) + (S_2 + S_3)
        {
            float2* base = reinterpret_cast<float2*>(xch) + ((k & 1) * GROUPS + pg) * SLICES * 32 + lane;
            base[sl * 32] = make_float2(sc[0], sc[1]);
            mma8::bar_group(1 + pg);
            const float2 x0 = base[0], x1 = base[32], x2 = base[64], x3 = base[96];
            sc[0] = (x0.x + x1.x) + (x2.x + x3.x);
            sc[1] = (x0.y + x1.y) + (x2.y + x3.y);
        }
        // ---- online softmax: this thread holds position g of rows 2t, 2t + 1
        float pr[2], cm[2], al[2], ps[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int kp = pos0 + g;
            const bool sees = kp < pe && kp <= qpos[i] && (p.window <= 0 || kp > qpos[i] - p.window);
            pr[i] = sees ? sc[i] * p.scale_log2 : -INFINITY;
            cm[i] = pr[i];
        }
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            const float x0 = __shfl_xor_sync(0xffffffffu, cm[0], off);
            const float x1 = __shfl_xor_sync(0xffffffffu, cm[1], off);
            cm[0] = fmaxf(cm[0], x0);
            cm[1] = fmaxf(cm[1], x1);
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const float mn = fmaxf(m[i], cm[i]);
            const float sh = mn == -INFINITY ? 0.f : mn;
            al[i] = mn == -INFINITY ? 1.f : fast_exp2(m[i] - sh);
            pr[i] = fast_exp2(pr[i] - sh);
            ps[i] = pr[i];
            m[i] = mn;
        }
        // l stays a per-lane partial (every lane of a row rescales by the
        // same alpha); the lanes are summed once, after the last chunk
        l[0] = l[0] * al[0] + ps[0];
        l[1] = l[1] * al[1] + ps[1];
        if (__any_sync(0xffffffffu, al[0] != 1.f || al[1] != 1.f)) {
#pragma unroll
            for (int c = 0; c < MTILES; ++c) {
                o[c][0] *= al[0];
                o[c][1] *= al[1];
                o[c][2] *= al[0];
                o[c][3] *= al[1];
            }
        }
        // ---- P^T fragment b0 = P[row g][pos 2t, 2t + 1] (bf16; b1, positions
        // 2t + 8 and 2t + 9, is zero); P[r][q] sits in lane 4 q + r / 2,
        // register r & 1.  (Shuffles here: a movmatrix transpose, faster in the
        // FP8 kernel, measured 2 % slower in this one.)
        uint32_t pb0;
        {
            const int src0 = 4 * (2 * t) + (g >> 1), src1 = 4 * (2 * t + 1) + (g >> 1);
            const float e00 = __shfl_sync(0xffffffffu, pr[0], src0), e01 = __shfl_sync(0xffffffffu, pr[1], src0);
            const float e10 = __shfl_sync(0xffffffffu, pr[0], src1), e11 = __shfl_sync(0xffffffffu, pr[1], src1);
            const bool odd = g & 1;
            pb0 = pack_bf16x2(odd ? e01 : e00, odd ? e11 : e10);
        }
        // ---- O^T slice += V_slice^T P^T: thread g's columns are elements
        // 16 g .. 16 g + 15 (bytes 32 g .. 32 g + 31) of rows 2t, 2t + 1;
        // M rows g / g + 8 of m-tile i are columns 16 g + 2 i / + 1
        uint32_t v0[8], v1[8];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            const uint4 x = *reinterpret_cast<const uint4*>(vst + (2 * t) * ROW + (((2 * g + h2 + swz_v(2 * t)) & 15) << 4));
            const uint4 y = *reinterpret_cast<const uint4*>(vst + (2 * t + 1) * ROW + (((2 * g + h2 + swz_v(2 * t + 1)) & 15) << 4));
            v0[4 * h2 + 0] = x.x; v0[4 * h2 + 1] = x.y; v0[4 * h2 + 2] = x.z; v0[4 * h2 + 3] = x.w;
            v1[4 * h2 + 0] = y.x; v1[4 * h2 + 1] = y.y; v1[4 * h2 + 2] = y.z; v1[4 * h2 + 3] = y.w;
        }
#pragma unroll
        for (int i = 0; i < MTILES; ++i) {
            // a0 = {V[2t][col 16g + 2i], V[2t + 1][same]}, a1 = the next column
            const uint32_t a0 = prmt(v0[i], v1[i], 0x5410u);
            const uint32_t a1 = prmt(v0[i], v1[i], 0x7632u);
            mma_bf16_16816(o[i], {a0, a1, 0u, 0u}, pb0, 0u);
        }
        __syncwarp();                         // the stage may be refilled
    }
    mma8::cp_async_wait<0>();
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) l[i] += __shfl_xor_sync(0xffffffffu, l[i], off);
    __syncthreads();   // every warp is done with its ring: reuse it for the merge

    float* so = reinterpret_cast<float*>(smem);
    float* sml = so + WARPS * 8 * SLICE;
#pragma unroll
    for (int i = 0; i < MTILES; ++i) {
        const int c0 = 16 * g + 2 * i, c1 = c0 + 1;
        so[(warp * 8 + 2 * t) * SLICE + c0] = o[i][0];
        so[(warp * 8 + 2 * t + 1) * SLICE + c0] = o[i][1];
        so[(warp * 8 + 2 * t) * SLICE + c1] = o[i][2];
        so[(warp * 8 + 2 * t + 1) * SLICE + c1] = o[i][3];
    }
    if (g == 0) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            sml[(warp * 8 + 2 * t + i) * 2] = m[i];
            sml[(warp * 8 + 2 * t + i) * 2 + 1] = l[i];
        }
    }
    __syncthreads();
    const size_t S = static_cast<size_t>(p.num_splits);
    for (int idx = threadIdx.x; idx < R * D; idx += WARPS * 32) {
        const int r = idx / D, d = idx - r * D;
        const int h = d / SLICE, c = d - h * SLICE;
        float M = -INFINITY;
#pragma unroll
        for (int q = 0; q < GROUPS; ++q) M = fmaxf(M, sml[((q * SLICES + h) * 8 + r) * 2]);
        float acc = 0.f, L = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int q = 0; q < GROUPS; ++q) {
                const int w = q * SLICES + h;   // the warp of group q, slice h
                const float wt = fast_exp2(sml[(w * 8 + r) * 2] - M);
                acc += wt * so[(w * 8 + r) * SLICE + c];
                L += wt * sml[(w * 8 + r) * 2 + 1];
            }
        }
        const size_t hq = (static_cast<size_t>(b) * p.q_len + r / G) * p.n_q_heads + kvh * G + r % G;
        p.ws_o[(hq * S + split) * D + d] = acc;
        if (d == 0) {
            p.ws_ml[(hq * S + split) * 2 + 0] = M;
            p.ws_ml[(hq * S + split) * 2 + 1] = M == -INFINITY ? 0.f : L;
        }
    }
}

}  // namespace mma16



// One block per (sequence, query token, query head) and slice of CS column
// slices: merges the splits' (O, m, l) -- M = max m_s, w_s = 2^(m_s - M),
// O = sum w_s O_s / sum w_s l_s ("Flash-Decoding for MQA in CUDA", "One KV
// head breaks the textbook").  256 threads: the slice's column quads x
// groups of splits (CS = 1: 128 quads x 2 groups; CS = 4: 32 quads x 8
// groups, four blocks per row, for batches whose rows alone leave most SMs
// idle).  Every thread issues the loads of its splits' O columns first, then
// the block finds the weights from the (m, l) pairs, so the merge costs about
// one memory round trip; the groups' sums meet in shared memory.
constexpr int MERGE_THREADS = 256;
constexpr int MERGE_UNROLL = 16;         // splits a thread loads up front
constexpr int MAX_SPLITS = 1024;

template <int CS>
__global__ void __launch_bounds__(MERGE_THREADS)
decode_merge_kernel(const DecodeParams p) {
    constexpr int QB = D / 4 / CS;                  // column quads of the slice
    constexpr int NG = MERGE_THREADS / QB;          // groups of splits
    static_assert(QB * NG == MERGE_THREADS, "threads = quads x groups");
    __shared__ float sw[MAX_SPLITS];      // w_s
    __shared__ float4 sacc[NG - 1][QB];
    __shared__ float smax[MERGE_THREADS / 32], ssum[MERGE_THREADS / 32];
    wait_for_splits();
    const int h = blockIdx.x;
    const int bt = blockIdx.y;      // sequence * q_len + token
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cq = tid % QB, grp = tid / QB;
    const int col = blockIdx.z * (D / CS) + cq * 4;
    const size_t bh = static_cast<size_t>(bt) * p.n_q_heads + h;
    const int S = p.num_splits;
    const float* ob = p.ws_o + bh * S * D + col;
    float4 x[MERGE_UNROLL];
#pragma unroll
    for (int i = 0; i < MERGE_UNROLL; ++i) {
        const int sp = grp + i * NG;
        x[i] = sp < S ? *reinterpret_cast<const float4*>(ob + static_cast<size_t>(sp) * D)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const float2* ml = reinterpret_cast<const float2*>(p.ws_ml + bh * S * 2);
    float2 mine = make_float2(-INFINITY, 0.f);
    if (tid < S) mine = ml[tid];
    float mloc = mine.x;
    for (int sp = tid + MERGE_THREADS; sp < S; sp += MERGE_THREADS) mloc = fmaxf(mloc, ml[sp].x);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, off));
    if (lane == 0) smax[warp] = mloc;
    __syncthreads();
    float M = smax[0];
#pragma unroll
    for (int w = 1; w < MERGE_THREADS / 32; ++w) M = fmaxf(M, smax[w]);
    float lloc = 0.f;
    for (int sp = tid; sp < S; sp += MERGE_THREADS) {
        const float2 v = sp == tid ? mine : ml[sp];
        // 0 for an empty split (m = -inf), and for every split when all are empty
        const float w = M == -INFINITY ? 0.f : fast_exp2(v.x - M);
        sw[sp] = w;
        lloc += w * v.y;
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) lloc += __shfl_xor_sync(0xffffffffu, lloc, off);
    if (lane == 0) ssum[warp] = lloc;
    __syncthreads();
    float L = 0.f;
#pragma unroll
    for (int w = 0; w < MERGE_THREADS / 32; ++w) L += ssum[w];
    __nv_bfloat16* out = p.out + bh * D + col;
    const bool lse_here = p.lse && tid == 0 && blockIdx.z == 0;
    if (M == -INFINITY) {
        if (grp == 0) *reinterpret_cast<uint2*>(out) = make_uint2(0u, 0u);
        if (lse_here) p.lse[bh] = -INFINITY;
        return;
    }
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    auto add = [&](float w, const float4& v) {
        // a split whose weight underflowed contributes nothing, whatever it holds
        if (w != 0.f) {
            acc.x = fmaf(w, v.x, acc.x);
            acc.y = fmaf(w, v.y, acc.y);
            acc.z = fmaf(w, v.z, acc.z);
            acc.w = fmaf(w, v.w, acc.w);
        }
    };
#pragma unroll
    for (int i = 0; i < MERGE_UNROLL; ++i) {
        const int sp = grp + i * NG;
        if (sp < S) add(sw[sp], x[i]);
    }
#pragma unroll 4
    for (int sp = grp + MERGE_UNROLL * NG; sp < S; sp += NG)
        add(sw[sp], *reinterpret_cast<const float4*>(ob + static_cast<size_t>(sp) * D));
    if (grp > 0) sacc[grp - 1][cq] = acc;
    __syncthreads();
    if (grp == 0) {
#pragma unroll
        for (int g = 0; g < NG - 1; ++g) {
            const float4 a = sacc[g][cq];
            acc.x += a.x;
            acc.y += a.y;
            acc.z += a.z;
            acc.w += a.w;
        }
        const float inv = 1.f / L;
        uint2 packed;
        packed.x = pack_bf16x2(acc.x * inv, acc.y * inv);
        packed.y = pack_bf16x2(acc.z * inv, acc.w * inv);
        *reinterpret_cast<uint2*>(out) = packed;
        if (lse_here) p.lse[bh] = (M + log2f(L)) * 0.69314718055994530942f;
    }
}

}  // namespace decode

int decode_smem_bytes() { return decode::Smem<false>::total + 1024; }

int decode_fp8_box_bytes() { return decode::F8_BOX_BYTES; }

int decode_fp8_mma_rows() { return 8; }

bool decode_merge_sliced(long long rows) { return rows * 4 <= 152; }

int decode_fp8_ctas_per_sm() { return decode::mma8::F8_CTAS_PER_SM; }

int decode_tile_positions() { return decode::TILE_K; }

constexpr int TILE_POSITIONS = decode::TILE_K;

template <int G>
static cudaError_t launch_stream(const DecodeParams& p, cudaStream_t stream) {
    const int smem = decode::stream::RING_BYTES;
    cudaError_t e = cudaFuncSetAttribute(decode::stream::decode_stream_kernel<G>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    dim3 grid(p.num_splits, p.n_kv_heads, p.batch);
    decode::stream::decode_stream_kernel<G><<<grid, decode::stream::WARPS * 32, smem, stream>>>(p);
    return cudaGetLastError();
}

static cudaError_t launch_bf16_mma(const DecodeParams& p, cudaStream_t stream) {
    const int smem = decode::mma16::SMEM_BYTES;
    cudaError_t e = cudaFuncSetAttribute(decode::mma16::decode_bf16_mma_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    dim3 grid(p.num_splits, p.n_kv_heads, p.batch);
    decode::mma16::decode_bf16_mma_kernel<<<grid, decode::mma8::WARPS * 32, smem, stream>>>(p);
    return cudaGetLastError();
}

static cudaError_t launch_fp8_mma(const DecodeParams& p, cudaStream_t stream) {
    const int smem = decode::mma8::F8_SMEM_BYTES;
    cudaError_t e = cudaFuncSetAttribute(decode::mma8::decode_fp8_mma_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    dim3 grid(p.num_splits, p.n_kv_heads, p.batch);
    decode::mma8::decode_fp8_mma_kernel<<<grid, decode::mma8::F8_WARPS * 32, smem, stream>>>(p);
    return cudaGetLastError();
}

template <bool FP8>
static cudaError_t launch_split_and_merge(const CUtensorMap& tmk, const CUtensorMap& tmv,
                                          const DecodeParams& p, cudaStream_t stream) {
    cudaError_t e;
    if (FP8 && p.q_len * p.group <= decode_fp8_mma_rows()) {
        e = launch_fp8_mma(p, stream);
    } else if (!FP8 && p.q_len == 1 && p.group <= 2 && p.tiles_per_split * TILE_POSITIONS < 1024) {
        // short splits (small batches): the FMA streaming kernel's lighter
        // set-up wins; from 1024 positions a split on, the tensor-core one
        e = p.group == 1 ? launch_stream<1>(p, stream) : launch_stream<2>(p, stream);
    } else if (!FP8 && p.q_len * p.group <= 8) {
        e = launch_bf16_mma(p, stream);
    } else {
        // larger query groups or several tokens: S and PV on the tensor cores
        // (q_len * G rows padded to 16)
        const int smem = decode::Smem<FP8>::total + 1024;
        e = cudaFuncSetAttribute(decode::decode_split_kernel<FP8>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        dim3 grid(p.num_splits, p.n_kv_heads, p.batch);
        decode::decode_split_kernel<FP8><<<grid, decode::NUM_THREADS, smem, stream>>>(tmk, tmv, p);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) return e;
    // the merge may be scheduled while the split kernel runs (it waits for
    // it); rows too few to spread over the SMs are merged in four column
    // slices each
    const bool sliced = decode_merge_sliced(static_cast<long long>(p.n_q_heads) * p.batch * p.q_len);
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3(p.n_q_heads, p.batch * p.q_len, sliced ? 4 : 1);
    cfg.blockDim = dim3(decode::MERGE_THREADS);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return sliced ? cudaLaunchKernelEx(&cfg, decode::decode_merge_kernel<4>, p)
                  : cudaLaunchKernelEx(&cfg, decode::decode_merge_kernel<1>, p);
}

cudaError_t launch_decode(const CUtensorMap& tmk, const CUtensorMap& tmv, const DecodeParams& p,
                          cudaStream_t stream) {
    return launch_split_and_merge<false>(tmk, tmv, p, stream);
}

cudaError_t launch_decode_fp8(const CUtensorMap& tmk, const CUtensorMap& tmv,
                              const DecodeParams& p, cudaStream_t stream) {
    return launch_split_and_merge<true>(tmk, tmv, p, stream);
}

}  // namespace fa512

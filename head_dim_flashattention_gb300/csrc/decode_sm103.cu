// Paged split-K decode for head dim 512 (Flash-Decoding), sm_103a.
//
// "Flash-Decoding for MQA in CUDA" (mila.toddt.me), section "One KV head
// breaks the textbook": the key sequence of each (sequence, KV head) is split
// across CTAs; each split writes an unnormalised (O, m, l) partial and a
// small fixup kernel applies the online-softmax merge.  The same section:
// walk absolute positions, read only the live band [max(0, len - window),
// len), keep K/V tiles double-buffered and rescale once per tile.
// vllm-project/flash-attention PR #199, "Performance": the cache is paged
// (page size 64), 8 query heads over 4 KV heads, q_len 1.
//
// Work item = (split, KV head, sequence).  One CTA streams its split's key
// tiles of TILE_K = 32 positions through a NUM_STAGES-deep ring in shared
// memory filled by TMA (one 64-column box per page run), computes
// S = Q K^T and O += P V for the G query heads of its KV head with bf16
// mma.sync (rows padded to 16), and keeps the softmax state in the log2
// domain.  HBM traffic per position and KV head: 1 KiB of K + 1 KiB of V.
// With q_len query tokens per sequence (the last q_len positions of its
// cache) the rows are (token, head) pairs, q_len * G <= 16, each masked at
// its own position.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "fa512_device.cuh"
#include "fa512_internal.h"

namespace fa512 {
namespace decode {

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

template <bool FP8>
__global__ void __launch_bounds__(NUM_THREADS, 1)
decode_split_kernel(const __grid_constant__ CUtensorMap tmk,
                    const __grid_constant__ CUtensorMap tmv, const DecodeParams p) {
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

constexpr int STAGES = 3;                // chunks in flight per warp
constexpr int WARPS = 8;
// A chunk is 8 KiB of K and V rows: 4 positions of a bf16 cache, 8 of an
// FP8 E4M3 cache.  A lane owns 16 head-dim columns of every row: 32 bytes of
// a bf16 row, 16 bytes of an FP8 row.
template <bool FP8>
struct Cfg {
    static constexpr int POS = FP8 ? 8 : 4;              // positions per chunk
    static constexpr int ROW_BYTES = FP8 ? D : D * 2;
    static constexpr int LANE_BYTES = ROW_BYTES / 32;
};
constexpr int CHUNK_BYTES = 8192;
static_assert(2 * Cfg<false>::POS * Cfg<false>::ROW_BYTES == CHUNK_BYTES, "chunk size");
static_assert(2 * Cfg<true>::POS * Cfg<true>::ROW_BYTES == CHUNK_BYTES, "chunk size");
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

// 16 e4m3 values -> fp32 times 2^-120, exactly, with integer operations
// only (the conversion units would bound the kernel below the HBM rate).
// An E4M3 byte s.eeee.mmm placed as fp32 bits s at 31 and eeee.mmm at 26..20
// is the fp32 number 2^(e-127) (1 + m/8) for e >= 1 and the subnormal
// (m/8) 2^-126 for e = 0 (zero included), i.e. the E4M3 value (bias 7,
// subnormals (m/8) 2^-6) times 2^-120.  An arithmetic right shift by 4 of
// the byte placed at bits 31..24 puts it there; the mask clears the copies
// of the sign.  (The E4M3 NaN code would read as 480: codes are read only
// inside the live band, where a cache holds finite values.)
__device__ __forceinline__ void unpack16_e4m3_scaled(const uint4 a, float (&f)[16]) {
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
    constexpr uint32_t M = 0x87f00000u;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[4 * i + 0] = __uint_as_float(static_cast<uint32_t>(static_cast<int32_t>(w[i] << 24) >> 4) & M);
        f[4 * i + 1] = __uint_as_float(static_cast<uint32_t>(static_cast<int32_t>(w[i] << 16) >> 4) & M);
        f[4 * i + 2] = __uint_as_float(static_cast<uint32_t>(static_cast<int32_t>(w[i] << 8) >> 4) & M);
        f[4 * i + 3] = __uint_as_float(static_cast<uint32_t>(static_cast<int32_t>(w[i]) >> 4) & M);
    }
}

// One chunk of FP8 positions for the G query rows of this lane's warp.
//
// Scores: each lane forms its 16-column partial q.k' (k' = k 2^-120) with
// f32x2 FMAs; the POS x G partials are summed over the 32 lanes by a
// transposing butterfly (each step halves the values a lane carries), so
// that lanes 32/NV apart ... end up holding one total each: value j = i G + g
// sits in lanes with (lane / (32 / NV)) == j.  The chunk max and sum per row
// are then reduced over those lanes, each lane evaluates one exp2, and the
// probabilities are broadcast back for O += p v' (p pre-multiplied by 2^120,
// so the product is p v in the normal range).
template <int G>
__device__ __forceinline__ void fp8_chunk(const uint8_t* st, int lane, int pos0, int pe,
                                          float sl_hi, const float2 (&qq)[16], float (&m)[G],
                                          float (&l)[G], float2 (&o)[G][8]) {
    constexpr int POS = Cfg<true>::POS;
    constexpr int ROW = Cfg<true>::ROW_BYTES;
    constexpr int NV = POS * G;                    // 8 or 16 partial scores
    constexpr int LPV = 32 / NV;                   // lanes that end up holding one value
    float v[NV];
#pragma unroll
    for (int i = 0; i < POS; ++i) {
        float kf[16];
        unpack16_e4m3_scaled(*reinterpret_cast<const uint4*>(st + i * ROW + lane * 16), kf);
        if constexpr (G == 2) {
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int d = 0; d < 16; ++d) acc = ffma2(qq[d], make_float2(kf[d], kf[d]), acc);
            v[i * 2] = acc.x;
            v[i * 2 + 1] = acc.y;
        } else {
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int d = 0; d < 8; ++d) acc = ffma2(qq[d], make_float2(kf[2 * d], kf[2 * d + 1]), acc);
            v[i] = acc.x + acc.y;
        }
    }
    // transposing butterfly: after the step at offset `off` a lane keeps the
    // upper half of its values when (lane & off) != 0, the lower half otherwise
#pragma unroll
    for (int off = 16, cnt = NV; cnt > 1; off >>= 1, cnt >>= 1) {
        const bool up = (lane & off) != 0;
#pragma unroll
        for (int t = 0; t < cnt / 2; ++t) {
            const float send = up ? v[t] : v[t + cnt / 2];
            const float keep = up ? v[t + cnt / 2] : v[t];
            v[t] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
#pragma unroll
    for (int off = LPV / 2; off >= 1; off >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);

    const int j = lane / LPV;                      // the value this lane holds
    const int i = j / G, g = j - i * G;
    // score in log2 units: v 2^120 scale log2(e), in two steps that cannot overflow
    const float s = (pos0 + i < pe) ? (v[0] * 0x1p64f) * sl_hi : -INFINITY;
    // chunk max of row g: over the lanes holding values j' = i' G + g
    float cm = s;
#pragma unroll
    for (int off = LPV * G; off < 32; off <<= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, off));
    float mg[G], ag[G];
#pragma unroll
    for (int gg = 0; gg < G; ++gg) {
        // every lane learns both rows' chunk maxima (lane gg * LPV holds row gg's)
        const float c = __shfl_sync(0xffffffffu, cm, gg * LPV);
        const float mn = fmaxf(m[gg], c);
        mg[gg] = mn == -INFINITY ? 0.f : mn;      // a row with no key yet shifts by 0
        ag[gg] = fast_exp2(m[gg] - mg[gg]);
        m[gg] = mn;
    }
    const float pj = fast_exp2(s - (G == 2 && g == 1 ? mg[G - 1] : mg[0]));
    float ps = pj;
#pragma unroll
    for (int off = LPV * G; off < 32; off <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
#pragma unroll
    for (int gg = 0; gg < G; ++gg) {
        l[gg] = l[gg] * ag[gg] + __shfl_sync(0xffffffffu, ps, gg * LPV);
        if (ag[gg] != 1.f) {                       // the same in every lane
#pragma unroll
            for (int d = 0; d < 8; ++d) o[gg][d] = ffma2(o[gg][d], make_float2(ag[gg], ag[gg]),
                                                         make_float2(0.f, 0.f));
        }
    }
    const float pjs = pj * 0x1p120f;
#pragma unroll
    for (int ii = 0; ii < POS; ++ii) {
        float vf[16];
        unpack16_e4m3_scaled(*reinterpret_cast<const uint4*>(st + (POS + ii) * ROW + lane * 16), vf);
#pragma unroll
        for (int gg = 0; gg < G; ++gg) {
            const float pv = __shfl_sync(0xffffffffu, pjs, (ii * G + gg) * LPV);
            const float2 pp = make_float2(pv, pv);
#pragma unroll
            for (int d = 0; d < 8; ++d)
                o[gg][d] = ffma2(pp, make_float2(vf[2 * d], vf[2 * d + 1]), o[gg][d]);
        }
    }
}

template <int G, bool FP8>
__global__ void __launch_bounds__(WARPS * 32, 1)
decode_stream_kernel(const DecodeParams p) {
    constexpr int POS = Cfg<FP8>::POS;
    constexpr int ROW = Cfg<FP8>::ROW_BYTES;
    constexpr int LB = Cfg<FP8>::LANE_BYTES;
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
    // FP8: q as f32x2 operands (G = 2: the two rows' column d; G = 1: columns
    // 2e, 2e + 1), O as column pairs, and the score scale times 2^56 (the
    // decoded keys carry 2^-120: 2^64 is applied to the dot product first)
    float2 qq[16], o2[G][8];
    const float sl_hi = p.scale_log2 * 0x1p56f;
    if constexpr (FP8) {
#pragma unroll
        for (int d = 0; d < 16; ++d)
            qq[d] = G == 2 ? make_float2(q[0][d], q[G - 1][d])
                           : make_float2(q[0][(2 * d) & 15], q[0][(2 * d + 1) & 15]);
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int d = 0; d < 8; ++d) o2[g][d] = make_float2(0.f, 0.f);
    }

    const uint32_t ring = smem_u32(smem) + warp * STAGES * CHUNK_BYTES;
    // chunk k of this warp covers positions pb + (warp + 8k) * POS ...
    const int my_chunks = n_chunks > warp ? (n_chunks - warp + WARPS - 1) / WARPS : 0;
    auto issue = [&](int k) {
        if (k < my_chunks) {
            const int pos0 = pb + (warp + WARPS * k) * POS;
            const uint32_t st = ring + (k % STAGES) * CHUNK_BYTES;
#pragma unroll
            for (int i = 0; i < POS; ++i) {
                const int pos = pos0 + i;
                bool valid = pos < pe;
                size_t row = 0;
                if (valid) {
                    const int page = p.page_table[static_cast<size_t>(b) * p.max_pages_per_seq + pos / p.page_size];
                    if (page < 0 || page >= p.num_pages) {
                        report_error(p.err, FA512_DEVICE_ERR_INDEX);
                        valid = false;
                    } else {
                        row = (static_cast<size_t>(page) * p.page_size + (pos & (p.page_size - 1))) * p.n_kv_heads + kvh;
                    }
                }
                const uint32_t kd = st + i * ROW + lane * LB;
                const uint32_t vd = st + (POS + i) * ROW + lane * LB;
                if constexpr (FP8) {
                    cp_async16(kd, p.k8 + row * D + lane * 16, valid);
                    cp_async16(vd, p.v8 + row * D + lane * 16, valid);
                } else {
                    const __nv_bfloat16* ks = p.k_pages + row * D + lane * 16;
                    const __nv_bfloat16* vs = p.v_pages + row * D + lane * 16;
                    cp_async16(kd, ks, valid);
                    cp_async16(kd + 16, ks + 8, valid);
                    cp_async16(vd, vs, valid);
                    cp_async16(vd + 16, vs + 8, valid);
                }
            }
        }
        cp_async_commit();   // one group per chunk slot, empty past the end
    };
#pragma unroll
    for (int k = 0; k < STAGES - 1; ++k) issue(k);

    for (int k = 0; k < my_chunks; ++k) {
        issue(k + STAGES - 1);
        cp_async_wait<STAGES - 1>();   // this lane's copies of chunk k have landed
        const uint8_t* st = smem + (warp * STAGES + (k % STAGES)) * CHUNK_BYTES;
        const int pos0 = pb + (warp + WARPS * k) * POS;
        if constexpr (FP8) {
            fp8_chunk<G>(st, lane, pos0, pe, sl_hi, qq, m, l, o2);
        } else {
            float s[POS][G];
    #pragma unroll
            for (int i = 0; i < POS; ++i) {
                float kf[16];
                const uint4* kr = reinterpret_cast<const uint4*>(st + i * ROW + lane * LB);
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
                const uint4* vr = reinterpret_cast<const uint4*>(st + (POS + i) * ROW + lane * LB);
                unpack8(vr[0], vr[1], vf);
    #pragma unroll
                for (int g = 0; g < G; ++g)
    #pragma unroll
                    for (int d = 0; d < 16; ++d) o[g][d] = fmaf(pr[i][g], vf[d], o[g][d]);
            }
        }
    }
    cp_async_wait<0>();
    __syncthreads();   // every warp is done with its ring: reuse it for the merge
    if constexpr (FP8) {
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int d = 0; d < 8; ++d) {
                o[g][2 * d] = o2[g][d].x;
                o[g][2 * d + 1] = o2[g][d].y;
            }
    }

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
        p.ws_o[(h * S + split) * D + d] = FP8 ? acc * p.o_scale : acc;
        if (d == 0) {
            p.ws_ml[(h * S + split) * 2 + 0] = M;
            p.ws_ml[(h * S + split) * 2 + 1] = M == -INFINITY ? 0.f : L;
        }
    }
}

}  // namespace stream

// One block per (sequence, query token, query head): merges the splits' (O, m, l).
__global__ void __launch_bounds__(128)
decode_merge_kernel(const DecodeParams p) {
    const int h = blockIdx.x;
    const int bt = blockIdx.y;      // sequence * q_len + token
    const size_t bh = static_cast<size_t>(bt) * p.n_q_heads + h;
    const int S = p.num_splits;
    const float* ml = p.ws_ml + bh * S * 2;
    float M = -INFINITY;
    for (int s = 0; s < S; ++s) M = fmaxf(M, ml[2 * s]);
    const int d = threadIdx.x * 4;
    __nv_bfloat16* out = p.out + bh * D + d;
    if (M == -INFINITY) {
        *reinterpret_cast<uint2*>(out) = make_uint2(0u, 0u);
        if (p.lse && threadIdx.x == 0) p.lse[bh] = -INFINITY;
        return;
    }
    float L = 0.f, acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
    const float* ob = p.ws_o + bh * S * D + d;
    for (int s = 0; s < S; ++s) {
        const float w = fast_exp2(ml[2 * s] - M);   // 0 for an empty split (m = -inf)
        L += w * ml[2 * s + 1];
        if (w != 0.f) {
            const float4 x = *reinterpret_cast<const float4*>(ob + static_cast<size_t>(s) * D);
            acc0 += w * x.x;
            acc1 += w * x.y;
            acc2 += w * x.z;
            acc3 += w * x.w;
        }
    }
    const float inv = 1.f / L;
    uint2 packed;
    packed.x = pack_bf16x2(acc0 * inv, acc1 * inv);
    packed.y = pack_bf16x2(acc2 * inv, acc3 * inv);
    *reinterpret_cast<uint2*>(out) = packed;
    if (p.lse && threadIdx.x == 0) p.lse[bh] = (M + log2f(L)) * 0.69314718055994530942f;
}

}  // namespace decode

int decode_smem_bytes() { return decode::Smem<false>::total + 1024; }

int decode_fp8_box_bytes() { return decode::F8_BOX_BYTES; }

int decode_tile_positions() { return decode::TILE_K; }

template <int G, bool FP8>
static cudaError_t launch_stream(const DecodeParams& p, cudaStream_t stream) {
    const int smem = decode::stream::RING_BYTES;
    cudaError_t e = cudaFuncSetAttribute(decode::stream::decode_stream_kernel<G, FP8>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    dim3 grid(p.num_splits, p.n_kv_heads, p.batch);
    decode::stream::decode_stream_kernel<G, FP8><<<grid, decode::stream::WARPS * 32, smem, stream>>>(p);
    return cudaGetLastError();
}

template <bool FP8>
static cudaError_t launch_split_and_merge(const CUtensorMap& tmk, const CUtensorMap& tmv,
                                          const DecodeParams& p, cudaStream_t stream) {
    cudaError_t e;
    if (p.q_len == 1 && p.group == 1) {
        e = launch_stream<1, FP8>(p, stream);
    } else if (p.q_len == 1 && p.group == 2) {
        e = launch_stream<2, FP8>(p, stream);
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
    dim3 mgrid(p.n_q_heads, p.batch * p.q_len);
    decode::decode_merge_kernel<<<mgrid, 128, 0, stream>>>(p);
    return cudaGetLastError();
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

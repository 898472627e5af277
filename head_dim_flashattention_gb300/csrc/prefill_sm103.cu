// Causal GQA/MQA FlashAttention forward for head dim 512 on sm_103a.
//
// The method: online softmax over key tiles -- running max m, running sum l,
// O rescaled when m moves -- so the [q x k] score matrix never reaches
// memory ("Writing a FlashAttention Prefill Kernel for Gemma 4", sections
// "The starting point" and "Head dim 512 breaks the textbook").
//
// Tile geometry:
//   * GQA row packing: a 128-row tile holds T = 128 / G query tokens times
//     the G query heads that share one KV head, so every K/V tile serves all
//     of them ("A custom attention kernel for Gemma 4 on the RTX PRO 6000",
//     "The kernel in three steps", step 1).  TMA gathers the packed rows
//     directly from q[seq, Hq, 512] with a 4-D box {64, G, 1, T}.
//   * Head-dim split: a 128 x 512 fp32 O would fill all 512 TMEM columns, so
//     each CTA owns one 256-column half of O (same page, step 2, and the
//     head-dim split of the Mila kernel, "Head dim 512 breaks the
//     textbook").  This version computes the full S = Q K^T in both halves.
//   * Causal / sliding-window tile skipping: only key tiles that intersect
//     the visible band of the tile's rows are visited; only tiles that cross
//     the band's edge are masked element by element.
//
// Roles: warps 0-3 own TMEM lanes 0-127 (one packed row per thread) and run
// the softmax, the O correction and the epilogue; lane 0 of warp 4 issues
// the TMA loads and the tcgen05.mma instructions.
//
// TMEM columns: O half [0, 256) fp32, S [256, 320) fp32, P [320, 352) bf16x2.
// Shared memory: Q 128 KiB (8 column boxes of 64), K 64 KiB, V half 32 KiB,
// all in the TMA 128-byte swizzle that the MMA descriptors read.
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
constexpr int NUM_THREADS = 160;
constexpr int Q_CHUNK = BM * 128;       // one 64-column box of Q: 16 KiB
constexpr int KV_CHUNK = BN * 128;      // one 64-column box of K or V: 8 KiB

constexpr uint32_t TM_O = 0;
constexpr uint32_t TM_S = 256;
constexpr uint32_t TM_P = 320;

// Rescale O only when the row max grows by more than this (log2 units);
// until then the stale max stays the reference and p <= 2^8.
constexpr float RESCALE_THRESHOLD = 8.0f;

struct Smem {
    static constexpr int q = 0;
    static constexpr int k = q + 8 * Q_CHUNK;
    static constexpr int v = k + 8 * KV_CHUNK;
    static constexpr int bars = v + 4 * KV_CHUNK;
    // barriers: q_full, k_full, v_full, s_full, p_full, o_done, drain
    static constexpr int n_bars = 7;
    static constexpr int tmem_addr = bars + n_bars * 8;
    static constexpr int abort_flag = tmem_addr + 4;
    static constexpr int total = abort_flag + 4;
};
enum { B_Q = 0, B_K, B_V, B_S, B_P, B_O, B_DRAIN };

constexpr uint32_t IDESC_QK = make_idesc_bf16(BM, BN, 0);
constexpr uint32_t IDESC_PV = make_idesc_bf16(BM, DH, 1);

// Bounded wait that also gives up when another role has aborted.
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

    // ---- work item: (q tile, KV head, D half); heaviest (latest) q tiles first
    const int half = blockIdx.x & 1;
    const int rest = blockIdx.x >> 1;
    const int kvh = rest % p.n_kv_heads;
    const int qt = p.num_q_tiles - 1 - rest / p.n_kv_heads;
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

    // this thread's packed row (warps 0-3)
    const int row = warp * 32 + lane;
    const int tok = row / G;
    const int g = row - tok * G;
    const bool valid_row = warp < 4 && row < p.rows_per_tile && tok < ntok;
    const int qpos = p.q_offset + t0 + tok;
    const int hq = kvh * G + g;

    if (n_kt == 0) {
        // no key is visible to any row of this tile: O = 0, LSE = -inf
        if (valid_row) {
            uint4* dst = reinterpret_cast<uint4*>(
                p.out + (static_cast<size_t>(t0 + tok) * p.n_q_heads + hq) * D + half * DH);
            for (int i = 0; i < DH / 8; ++i) dst[i] = make_uint4(0u, 0u, 0u, 0u);
            if (half == 0 && p.lse) p.lse[static_cast<size_t>(hq) * p.seqlen_q + t0 + tok] = -INFINITY;
        }
        return;
    }

    if (warp == 4) {
        if (lane == 0) {
            for (int i = 0; i < Smem::n_bars; ++i) mbar_init(&bars[i], i == B_P ? 128 : 1);
            *abort = 0;
            fence_mbar_init();
            tma_prefetch_desc(&tmq);
            tma_prefetch_desc(&tmk);
            tma_prefetch_desc(&tmv);
        }
        __syncwarp();
        tmem_alloc(tmem_addr_smem, 512);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_addr_smem;

    if (warp == 4) {
        if (lane == 0) {
            // ------------------------------------------------ producer + MMA issue
            const uint32_t q_bytes = static_cast<uint32_t>(8 * 128 * p.rows_per_tile);
            mbar_arrive_expect_tx(&bars[B_Q], q_bytes);
            for (int c = 0; c < 8; ++c)
                tma_load_4d(smem + Smem::q + c * Q_CHUNK, &tmq, &bars[B_Q], c * 64, 0, kvh, t0);
            auto load_k = [&](int j) {
                mbar_arrive_expect_tx(&bars[B_K], 8 * KV_CHUNK);
                const int key0 = (kt_begin + j) * BN;
                for (int c = 0; c < 8; ++c)
                    tma_load_3d(smem + Smem::k + c * KV_CHUNK, &tmk, &bars[B_K], c * 64, kvh, key0);
            };
            auto load_v = [&](int j) {
                mbar_arrive_expect_tx(&bars[B_V], 4 * KV_CHUNK);
                const int key0 = (kt_begin + j) * BN;
                for (int c = 0; c < 4; ++c)
                    tma_load_3d(smem + Smem::v + c * KV_CHUNK, &tmv, &bars[B_V],
                                (half * 4 + c) * 64, kvh, key0);
            };
            load_k(0);
            load_v(0);
            int k_out = 1, v_out = 1;   // loads in flight (for the abort drain)
            bool ok = wait_or_abort(&bars[B_Q], 0, p.err, abort);
            const uint32_t q_base = smem_u32(smem + Smem::q);
            const uint32_t k_base = smem_u32(smem + Smem::k);
            const uint32_t v_base = smem_u32(smem + Smem::v);
            for (int j = 0; ok && j < n_kt; ++j) {
                const uint32_t ph = static_cast<uint32_t>(j & 1);
                if (!(ok = wait_or_abort(&bars[B_K], ph, p.err, abort))) break;
                k_out = 0;
                tc_fence_after_sync();
                // S = Q K^T: 32 k-steps of 16 over the full head dim
#pragma unroll 4
                for (int kk = 0; kk < 32; ++kk) {
                    const uint32_t off = static_cast<uint32_t>((kk & 3) * 32);
                    const uint64_t ad = make_sdesc_sw128(q_base + (kk >> 2) * Q_CHUNK + off, 16, 1024);
                    const uint64_t bd = make_sdesc_sw128(k_base + (kk >> 2) * KV_CHUNK + off, 16, 1024);
                    tc_mma_ss(tmem + TM_S, ad, bd, IDESC_QK, kk > 0 ? 1u : 0u);
                }
                tc_commit(&bars[B_S]);
                // the K buffer is free once S is complete
                if (!(ok = wait_or_abort(&bars[B_S], ph, p.err, abort))) break;
                if (j + 1 < n_kt) {
                    load_k(j + 1);
                    k_out = 1;
                }
                // O += P V once the softmax has written P (and corrected O)
                if (!(ok = wait_or_abort(&bars[B_P], ph, p.err, abort))) break;
                if (!(ok = wait_or_abort(&bars[B_V], ph, p.err, abort))) break;
                v_out = 0;
                tc_fence_after_sync();
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                    // V is MN-major: 64-column blocks KV_CHUNK apart, 8-key groups 1 KiB apart
                    const uint64_t bd = make_sdesc_sw128(v_base + kk * 16 * 128, KV_CHUNK, 1024);
                    tc_mma_ts(tmem + TM_O, tmem + TM_P + kk * 8, bd, IDESC_PV,
                              (j > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(&bars[B_O]);
                if (!(ok = wait_or_abort(&bars[B_O], ph, p.err, abort))) break;
                if (j + 1 < n_kt) {
                    load_v(j + 1);
                    v_out = 1;
                }
            }
            if (!ok) {
                // drain: let issued MMAs and copies finish before TMEM and
                // shared memory are released
                tc_commit(&bars[B_DRAIN]);
                (void)mbar_wait(&bars[B_DRAIN], 0, p.err);
                (void)k_out;
                (void)v_out;
            }
        }
    } else {
        // ------------------------------------------------ softmax + epilogue
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        float m_ref = -INFINITY;   // log2 units
        float l = 0.f;      // sum of the fp32 probabilities (for LSE)
        float l_b = 0.f;    // sum of the bf16-rounded probabilities (normalises O)
        bool ok = true;
        for (int j = 0; j < n_kt; ++j) {
            const uint32_t ph = static_cast<uint32_t>(j & 1);
            if (!(ok = wait_or_abort(&bars[B_S], ph, p.err, abort))) break;
            tc_fence_after_sync();
            uint32_t sr[2][32];
            tmem_ld32(tmem + lane_base + TM_S, sr[0]);
            tmem_ld32(tmem + lane_base + TM_S + 32, sr[1]);
            tmem_ld_wait();
            const int key0 = (kt_begin + j) * BN;
            const bool tile_full = key0 + BN <= p.seqlen_k && (!p.causal || key0 + BN - 1 <= p_first) &&
                                   (p.window <= 0 || key0 > p_last - p.window);
            float s[64];
            float tmax = -INFINITY;
#pragma unroll
            for (int c = 0; c < 64; ++c) {
                float x = __uint_as_float(sr[c >> 5][c & 31]) * p.scale_log2;
                if (!tile_full && !key_visible(key0 + c, qpos, p)) x = -INFINITY;
                s[c] = x;
                tmax = fmaxf(tmax, x);
            }
            float m_use = m_ref, alpha = 1.f;
            if (tmax > m_ref + RESCALE_THRESHOLD) {
                m_use = tmax;
                alpha = fast_exp2(m_ref - m_use);   // 0 when m_ref = -inf
            }
            const float shift = m_use == -INFINITY ? 0.f : m_use;
            uint32_t pk[32];
            float rs = 0.f, rs_b = 0.f;
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const float p0 = fast_exp2(s[2 * c] - shift);
                const float p1 = fast_exp2(s[2 * c + 1] - shift);
                rs += p0 + p1;
                pk[c] = pack_bf16x2(p0, p1);
                // the bf16 values the PV product actually uses
                rs_b += __uint_as_float(pk[c] << 16) + __uint_as_float(pk[c] & 0xffff0000u);
            }
            l = l * alpha + rs;
            l_b = l_b * alpha + rs_b;
            m_ref = m_use;
            if (j > 0) {
                // PV of the previous tile must be done before P and O are touched
                if (!(ok = wait_or_abort(&bars[B_O], ph ^ 1u, p.err, abort))) break;
                tc_fence_after_sync();
                if (__any_sync(0xffffffffu, alpha != 1.f)) {
                    for (int c = 0; c < DH / 32; ++c) {
                        uint32_t o[32];
                        tmem_ld32(tmem + lane_base + TM_O + c * 32, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tmem_st32(tmem + lane_base + TM_O + c * 32, o);
                    }
                }
            }
            tmem_st32(tmem + lane_base + TM_P, pk);
            tmem_st_wait();
            tc_fence_before_sync();
            mbar_arrive(&bars[B_P]);
        }
        if (ok) ok = wait_or_abort(&bars[B_O], static_cast<uint32_t>((n_kt - 1) & 1), p.err, abort);
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
    if (warp == 4) {
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
    const int n_blocks = p.num_q_tiles * p.n_kv_heads * 2;
    prefill::prefill_kernel<<<n_blocks, prefill::NUM_THREADS, smem, stream>>>(tmq, tmk, tmv, p);
    return cudaGetLastError();
}

}  // namespace fa512

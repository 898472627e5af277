// Internal interface between the C ABI (api.cu) and the kernel translation
// units.  Not installed; the public interface is include/fa512.h.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fa512 {

struct DecodeParams {
    const __nv_bfloat16* q;        // [batch, q_len, n_q_heads, 512]
    const __nv_bfloat16* k_pages;  // [num_pages, page_size, n_kv_heads, 512]
    const __nv_bfloat16* v_pages;
    // FP8 E4M3 cache (same layout, one byte per element; null for a bf16
    // cache): a key element is k_scale * e4m3, a value element v_scale * e4m3.
    // k_scale is folded into scale_log2, v_scale into o_scale.
    const uint8_t* k8;
    const uint8_t* v8;
    float o_scale;                 // multiplies the split partials O (FP8 cache: v_scale)
    const int32_t* page_table;     // [batch, max_pages_per_seq]
    const int32_t* kv_lens;        // [batch]
    float* ws_o;                   // [batch, q_len, n_q_heads, num_splits, 512] unnormalised O
    float* ws_ml;                  // [batch, q_len, n_q_heads, num_splits, 2] (m in log2 units, l)
    __nv_bfloat16* out;            // [batch, q_len, n_q_heads, 512]
    float* lse;                    // [batch, q_len, n_q_heads] or null
    int batch, n_q_heads, n_kv_heads, group;
    int q_len;                     // query tokens per sequence: its last q_len positions
    int page_size, box_rows, num_pages, max_pages_per_seq;
    int len_cap;                   // min(max_kv_len, max_pages_per_seq * page_size)
    int window;
    int tiles_per_split, num_splits;
    float scale_log2;              // scale * log2(e)
    unsigned* err;                 // device error word
};

int decode_smem_bytes();
int decode_tile_positions();
cudaError_t launch_decode(const CUtensorMap& tmk, const CUtensorMap& tmv, const DecodeParams& p,
                          cudaStream_t stream);
// FP8 cache: tmk / tmv map the e4m3 pages as bytes, boxes of
// decode_fp8_box_bytes() head-dim bytes x box_rows positions, no swizzle.
int decode_fp8_box_bytes();
// FP8 cache with q_len * G <= decode_fp8_mma_rows(): the split kernel runs
// decode_fp8_ctas_per_sm() CTAs per SM, one split each.
int decode_fp8_mma_rows();
int decode_fp8_ctas_per_sm();
// The merge kernel takes `rows` (sequence, token, query head) rows in four
// column slices each (128 splits loaded up front) when this is true, else
// whole (32 splits up front).
bool decode_merge_sliced(long long rows);
cudaError_t launch_decode_fp8(const CUtensorMap& tmk, const CUtensorMap& tmv,
                              const DecodeParams& p, cudaStream_t stream);

struct PrefillParams {
    __nv_bfloat16* out;            // [total_q, n_q_heads, 512]
    float* lse;                    // [n_q_heads, total_q] or null
    int seqlen_q, seqlen_k, q_offset, n_q_heads, n_kv_heads, group;
    int tokens_per_tile;           // query tokens packed per 128-row tile
    int rows_per_tile;             // tokens_per_tile * group (<= 128)
    int num_q_tiles;               // per KV head (contiguous mode)
    int causal, window;
    float scale_log2;              // scale * log2(e)
    unsigned* err;
    int total_q;                   // rows of q / out (contiguous mode: seqlen_q)
    // varlen mode over a paged cache (the contiguous kernel ignores these)
    const int32_t* page_table;     // [batch, max_pages_per_seq]
    const int32_t* cu_seqlens_q;   // [batch + 1]
    const int32_t* seqused_k;      // [batch]
    int batch, max_seqlen_q, max_pairs;
    int page_shift, num_pages, max_pages_per_seq;
    int oob_row;                   // num_pages * page_size: a row past the pool (TMA fills zeros)
    unsigned long long wait_limit_ns;  // bound of each pipeline wait (0: the default, 2 s)
    int test_skip_first_k_load;    // test hook: CTA 0 does not issue its first K load
};

int prefill_smem_bytes();
int prefill_k_box_rows();   // keys per K box (one head-dim chunk of a key tile)
int prefill_v_box_rows();   // keys per V box (one key slice)

// Head dim 256 (the sliding-window local layers): a persistent kernel, one
// cluster of two CTAs per SM pair, each walking a contiguous range of
// (KV head, q-tile pair) items.
constexpr int kMaxPersistentClusters = 128;

struct Prefill256Params {
    __nv_bfloat16* out;            // [seqlen_q, n_q_heads, 256]
    float* lse;                    // [n_q_heads, seqlen_q] or null
    int seqlen_q, seqlen_k, q_offset, n_q_heads, n_kv_heads, group;
    int tokens_per_tile, rows_per_tile, num_q_tiles, n_pairs, n_items;
    int causal, window;
    float scale_log2;
    unsigned* err;
    int n_clusters;
    // items of cluster c: range_start[c], + item_stride, ... below range_start[c + 1]
    int item_stride;
    int range_start[kMaxPersistentClusters + 1];
};

int prefill256_smem_bytes();
int prefill256_k_box_rows();
int prefill256_v_box_rows();
void plan_prefill256(Prefill256Params& p, int n_sm);
cudaError_t launch_prefill256(const CUtensorMap& tmq, const CUtensorMap& tmk, const CUtensorMap& tmv,
                              const CUtensorMap& tmo, const Prefill256Params& p, cudaStream_t stream);

// Sets the text fa512_last_error_message() returns on this thread.
void set_last_error_message(const char* msg);
cudaError_t launch_prefill(const CUtensorMap& tmq, const CUtensorMap& tmk, const CUtensorMap& tmv,
                           const PrefillParams& p, cudaStream_t stream);
int prefill_paged_v_box_rows();   // keys per V box over a paged cache (one page-aligned half tile)
cudaError_t launch_prefill_paged(const CUtensorMap& tmq, const CUtensorMap& tmk, const CUtensorMap& tmv,
                                 const PrefillParams& p, cudaStream_t stream);

}  // namespace fa512

// C ABI of the fa512 library: argument validation, TMA tensor-map encoding,
// split-count choice, workspace sizing and kernel launch on the caller's
// stream.  See include/fa512.h for the contract of every entry point.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "fa512.h"
#include "fa512_internal.h"

// Device error word: bit 0 = a pipeline wait ran past its bound, bit 1 = a
// page index or kv length outside the declared ranges.  One per device.
__device__ unsigned fa512_device_error_word;

namespace {

constexpr int kHeadDim = FA512_HEAD_DIM;
constexpr unsigned long long kDefaultWaitLimitNs = 2000000000ull;   // the kernels' own default
thread_local char g_last_error[512];

fa512_status fail(fa512_status st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));

fa512_status fail(fa512_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return st;
}

fa512_status cuda_fail(cudaError_t e, const char* what) {
    return fail(FA512_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---- per-device state: address of the device error word
std::mutex g_mu;
constexpr int kMaxDevices = 64;
unsigned* g_err_ptr[kMaxDevices];

cudaError_t device_error_ptr(unsigned** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_err_ptr[dev]) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, fa512_device_error_word);
        if (e != cudaSuccess) return e;
        g_err_ptr[dev] = static_cast<unsigned*>(ptr);
    }
    *out = g_err_ptr[dev];
    return cudaSuccess;
}

// ---- tensor maps through the driver entry point (no link-time libcuda)
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

fa512_status get_encoder(EncodeTiledFn* fn) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_encode) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                                         cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !f)
            return fail(FA512_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
        g_encode = reinterpret_cast<EncodeTiledFn>(f);
    }
    *fn = g_encode;
    return FA512_OK;
}

// Tensor map; dims/strides innermost first, strides in bytes for dims
// 1..rank-1.
fa512_status encode_map(CUtensorMap* m, CUtensorMapDataType dtype, CUtensorMapSwizzle swizzle,
                        const void* base, int rank, const uint64_t* dims,
                        const uint64_t* strides_bytes, const uint32_t* box) {
    EncodeTiledFn enc;
    fa512_status st = get_encoder(&enc);
    if (st != FA512_OK) return st;
    cuuint64_t gd[5], gs[4];
    cuuint32_t bx[5], es[5];
    for (int i = 0; i < rank; ++i) {
        gd[i] = dims[i];
        bx[i] = box[i];
        es[i] = 1;
    }
    for (int i = 0; i < rank - 1; ++i) gs[i] = strides_bytes[i];
    CUresult r = enc(m, dtype, static_cast<cuuint32_t>(rank),
                     const_cast<void*>(base), gd, gs, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(FA512_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return FA512_OK;
}

// bf16 tensor map with 128-byte swizzle.
fa512_status encode_bf16(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                         const uint64_t* strides_bytes, const uint32_t* box) {
    return encode_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, CU_TENSOR_MAP_SWIZZLE_128B, base, rank,
                      dims, strides_bytes, box);
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 152;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        return 152;
    }
    return n;
}

bool pow2_page(int ps) { return ps == 16 || ps == 32 || ps == 64 || ps == 128 || ps == 256; }

// Tiles of the decode band (upper bound over sequences) for a host-side bound
// on the kv length.  A window can straddle one extra tile boundary.
long long band_tiles(int max_kv_len, int window) {
    const int tk = fa512::decode_tile_positions();
    long long band = max_kv_len;
    if (window > 0 && window < band) band = window;
    long long t = (band + tk - 1) / tk;
    if (window > 0 && window < max_kv_len) t += 1;
    return t;
}

// Split count for `items` (sequence, KV head) pairs of `tiles` key tiles,
// one 16-warp split CTA per SM.
int choose_splits(long long items, long long tiles, int n_sm) {
    if (items <= 0 || tiles <= 1) return 1;
    long long best_s = 1;
    double best = 1e300;
    const long long s_max = tiles < 1024 ? tiles : 1024;
    for (long long s = 1; s <= s_max; ++s) {
        const long long waves = (items * s + n_sm - 1) / n_sm;
        const long long per = (tiles + s - 1) / s;
        // time model: waves x (tiles per split + fixed cost of ~2 tiles)
        const double cost = static_cast<double>(waves) * static_cast<double>(per + 2);
        if (cost < best) {
            best = cost;
            best_s = s;
        }
    }
    return static_cast<int>(best_s);
}

// Split count for the FP8 kernel, four CTAs per SM, one split each, `rows`
// (sequence, token, query head) rows to merge.  Times in tile times of one
// CTA.  Large batches (the merge takes whole rows): a finished CTA's slot
// takes the next split at once, so the work spreads over the slots in
// fractions of a round rather than whole waves:
//   max(1, items x s / slots) x (tiles per split + 2)   streaming + start
//   + 0.75 x tiles per split                             the ragged end
//   + 0.2 x max(0, s - 32)                               merge loads past the
//                                                        merge kernel's first 32
// Small batches (every CTA resident at once, the merge in column slices):
// an SM's time is its CTAs x tiles per split, and one CTA alone runs no
// faster than two sharing the SM (it is latency-bound), so
//   max(2, CTAs on the busiest SM) x tiles per split.
// Both fitted to times of batch 1/16/64 x KV 4096/16384/28672, 4 KV heads,
// over 8 split counts each: within 0.5 % of the best count per shape.
int choose_splits_fp8(long long items, long long tiles, int n_sm, long long rows) {
    if (items <= 0 || tiles <= 1) return 1;
    const bool small = fa512::decode_merge_sliced(rows);
    const double slots = static_cast<double>(fa512::decode_fp8_ctas_per_sm()) * n_sm;
    long long best_s = 1;
    double best = 1e300;
    const long long s_max = tiles < 128 ? tiles : 128;
    for (long long s = 1; s <= s_max; ++s) {
        const double per = static_cast<double>((tiles + s - 1) / s);
        double cost;
        if (small) {
            const long long busiest = (items * s + n_sm - 1) / n_sm;
            cost = static_cast<double>(busiest > 2 ? busiest : 2) * per;
        } else {
            const double x = static_cast<double>(items * s) / slots;
            cost = (x > 1.0 ? x : 1.0) * (per + 2.0) + 0.75 * per +
                   0.2 * static_cast<double>(s > 32 ? s - 32 : 0);
        }
        if (cost < best) {
            best = cost;
            best_s = s;
        }
    }
    return static_cast<int>(best_s);
}

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

size_t workspace_for(int batch, int n_q_heads, int splits) {
    const size_t rows = static_cast<size_t>(batch) * n_q_heads * splits;
    return round256(rows * kHeadDim * sizeof(float)) + round256(rows * 2 * sizeof(float));
}

}  // namespace

void fa512::set_last_error_message(const char* msg) {
    snprintf(g_last_error, sizeof g_last_error, "%s", msg ? msg : "");
}

extern "C" {

const char* fa512_status_string(fa512_status s) {
    switch (s) {
        case FA512_OK: return "FA512_OK";
        case FA512_ERR_INVALID_ARG: return "FA512_ERR_INVALID_ARG";
        case FA512_ERR_UNSUPPORTED: return "FA512_ERR_UNSUPPORTED";
        case FA512_ERR_CUDA: return "FA512_ERR_CUDA";
        case FA512_ERR_TIMEOUT: return "FA512_ERR_TIMEOUT";
        case FA512_ERR_WORKSPACE: return "FA512_ERR_WORKSPACE";
        case FA512_ERR_DEVICE_INDEX: return "FA512_ERR_DEVICE_INDEX";
    }
    return "FA512_UNKNOWN_STATUS";
}

const char* fa512_last_error_message(void) { return g_last_error; }

}  // extern "C"

namespace {

// Body of fa512_prefill; the test hook below reaches it with a short wait
// bound and one K load left out.
fa512_status prefill_call(const void* q, const void* k, const void* v, void* out, float* lse,
                          int seqlen_q, int seqlen_k, int q_offset, int n_q_heads, int n_kv_heads,
                          float scale, int causal, int window, fa512_stream_t stream,
                          unsigned long long wait_limit_ns, int skip_first_k_load) {
    g_last_error[0] = 0;
    if (seqlen_q < 0 || seqlen_k < 0 || q_offset < 0)
        return fail(FA512_ERR_INVALID_ARG, "negative length or offset");
    if (n_kv_heads < 1 || n_q_heads < 1 || n_q_heads % n_kv_heads != 0)
        return fail(FA512_ERR_INVALID_ARG, "n_q_heads (%d) must be a positive multiple of n_kv_heads (%d)",
                    n_q_heads, n_kv_heads);
    const int G = n_q_heads / n_kv_heads;
    if (G > 128) return fail(FA512_ERR_UNSUPPORTED, "more than 128 query heads per KV head");
    if (!(scale == scale) || isinf(scale)) return fail(FA512_ERR_INVALID_ARG, "scale is not finite");
    if (static_cast<long long>(q_offset) + seqlen_q > 0x7fffffffLL)
        return fail(FA512_ERR_INVALID_ARG, "q_offset + seqlen_q overflows int32 positions");
    if (seqlen_q == 0) return FA512_OK;
    if (!q || !out || (seqlen_k > 0 && (!k || !v)))
        return fail(FA512_ERR_INVALID_ARG, "null tensor pointer");
    if (!aligned16(q) || !aligned16(out) || (seqlen_k > 0 && (!aligned16(k) || !aligned16(v))))
        return fail(FA512_ERR_INVALID_ARG, "q, k, v and out must be 16-byte aligned");
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u))
        return fail(FA512_ERR_INVALID_ARG, "lse must be 4-byte aligned");

    unsigned* err = nullptr;
    cudaError_t e = device_error_ptr(&err);
    if (e != cudaSuccess) return cuda_fail(e, "device error word");

    fa512::PrefillParams p;
    memset(&p, 0, sizeof p);
    p.out = static_cast<__nv_bfloat16*>(out);
    p.lse = lse;
    p.seqlen_q = seqlen_q;
    p.total_q = seqlen_q;
    p.seqlen_k = seqlen_k;
    p.q_offset = q_offset;
    p.n_q_heads = n_q_heads;
    p.n_kv_heads = n_kv_heads;
    p.group = G;
    p.tokens_per_tile = 128 / G;
    p.rows_per_tile = p.tokens_per_tile * G;
    p.num_q_tiles = (seqlen_q + p.tokens_per_tile - 1) / p.tokens_per_tile;
    p.causal = causal ? 1 : 0;
    p.window = window > 0 ? window : 0;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.err = err;
    p.wait_limit_ns = wait_limit_ns;
    p.test_skip_first_k_load = skip_first_k_load;
    if (static_cast<long long>(p.num_q_tiles) * n_kv_heads * 2 > 0x7fffffffLL)
        return fail(FA512_ERR_UNSUPPORTED, "grid too large");

    CUtensorMap tmq, tmk, tmv;
    memset(&tmk, 0, sizeof tmk);
    memset(&tmv, 0, sizeof tmv);
    {
        const uint64_t dims[4] = {static_cast<uint64_t>(kHeadDim), static_cast<uint64_t>(G),
                                  static_cast<uint64_t>(n_kv_heads), static_cast<uint64_t>(seqlen_q)};
        const uint64_t strides[3] = {kHeadDim * 2ull, static_cast<uint64_t>(G) * kHeadDim * 2ull,
                                     static_cast<uint64_t>(n_q_heads) * kHeadDim * 2ull};
        const uint32_t box[4] = {64u, static_cast<uint32_t>(G), 1u,
                                 static_cast<uint32_t>(p.tokens_per_tile)};
        fa512_status st = encode_bf16(&tmq, q, 4, dims, strides, box);
        if (st != FA512_OK) return st;
    }
    if (seqlen_k > 0) {
        const uint64_t dims[3] = {static_cast<uint64_t>(kHeadDim), static_cast<uint64_t>(n_kv_heads),
                                  static_cast<uint64_t>(seqlen_k)};
        const uint64_t strides[2] = {kHeadDim * 2ull, static_cast<uint64_t>(n_kv_heads) * kHeadDim * 2ull};
        // the kernel streams K in head-dim chunks of a whole key tile and V
        // in key slices; it states the box height of each
        const uint32_t kbox[3] = {64u, 1u, static_cast<uint32_t>(fa512::prefill_k_box_rows())};
        const uint32_t vbox[3] = {64u, 1u, static_cast<uint32_t>(fa512::prefill_v_box_rows())};
        fa512_status st = encode_bf16(&tmk, k, 3, dims, strides, kbox);
        if (st != FA512_OK) return st;
        st = encode_bf16(&tmv, v, 3, dims, strides, vbox);
        if (st != FA512_OK) return st;
    }
    e = fa512::launch_prefill(tmq, tmk, tmv, p, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
    return FA512_OK;
}

}  // namespace

extern "C" {

fa512_status fa512_prefill(const void* q, const void* k, const void* v, void* out, float* lse,
                           int seqlen_q, int seqlen_k, int q_offset, int n_q_heads,
                           int n_kv_heads, float scale, int causal, int window,
                           fa512_stream_t stream) {
    return prefill_call(q, k, v, out, lse, seqlen_q, seqlen_k, q_offset, n_q_heads, n_kv_heads,
                        scale, causal, window, stream, kDefaultWaitLimitNs, 0);
}

fa512_status fa512_test_prefill_missing_load(const void* q, const void* k, const void* v, void* out,
                                             float* lse, int seqlen_q, int seqlen_k, int q_offset,
                                             int n_q_heads, int n_kv_heads, float scale, int causal,
                                             int window, uint64_t wait_limit_ns,
                                             fa512_stream_t stream) {
    if (wait_limit_ns < 1000000ull || wait_limit_ns > kDefaultWaitLimitNs)
        return fail(FA512_ERR_INVALID_ARG, "wait_limit_ns must lie in [1 ms, 2 s]");
    if (seqlen_k < 1) return fail(FA512_ERR_INVALID_ARG, "the hook needs at least one key");
    return prefill_call(q, k, v, out, lse, seqlen_q, seqlen_k, q_offset, n_q_heads, n_kv_heads,
                        scale, causal, window, stream, wait_limit_ns, 1);
}

fa512_status fa512_prefill_d256(const void* q, const void* k, const void* v, void* out, float* lse,
                                int seqlen_q, int seqlen_k, int q_offset, int n_q_heads,
                                int n_kv_heads, float scale, int causal, int window,
                                fa512_stream_t stream) {
    g_last_error[0] = 0;
    constexpr int kD = 256;
    if (seqlen_q < 0 || seqlen_k < 0 || q_offset < 0)
        return fail(FA512_ERR_INVALID_ARG, "negative length or offset");
    if (n_kv_heads < 1 || n_q_heads < 1 || n_q_heads % n_kv_heads != 0)
        return fail(FA512_ERR_INVALID_ARG, "n_q_heads (%d) must be a positive multiple of n_kv_heads (%d)",
                    n_q_heads, n_kv_heads);
    const int G = n_q_heads / n_kv_heads;
    if (G > 128) return fail(FA512_ERR_UNSUPPORTED, "more than 128 query heads per KV head");
    if (!(scale == scale) || isinf(scale)) return fail(FA512_ERR_INVALID_ARG, "scale is not finite");
    if (static_cast<long long>(q_offset) + seqlen_q > 0x7fffffffLL)
        return fail(FA512_ERR_INVALID_ARG, "q_offset + seqlen_q overflows int32 positions");
    if (seqlen_q == 0) return FA512_OK;
    if (!q || !out || (seqlen_k > 0 && (!k || !v)))
        return fail(FA512_ERR_INVALID_ARG, "null tensor pointer");
    if (!aligned16(q) || !aligned16(out) || (seqlen_k > 0 && (!aligned16(k) || !aligned16(v))))
        return fail(FA512_ERR_INVALID_ARG, "q, k, v and out must be 16-byte aligned");
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u))
        return fail(FA512_ERR_INVALID_ARG, "lse must be 4-byte aligned");

    unsigned* err = nullptr;
    cudaError_t e = device_error_ptr(&err);
    if (e != cudaSuccess) return cuda_fail(e, "device error word");

    fa512::Prefill256Params p;
    memset(&p, 0, sizeof p);
    p.out = static_cast<__nv_bfloat16*>(out);
    p.lse = lse;
    p.seqlen_q = seqlen_q;
    p.seqlen_k = seqlen_k;
    p.q_offset = q_offset;
    p.n_q_heads = n_q_heads;
    p.n_kv_heads = n_kv_heads;
    p.group = G;
    p.tokens_per_tile = 128 / G;
    p.rows_per_tile = p.tokens_per_tile * G;
    p.num_q_tiles = (seqlen_q + p.tokens_per_tile - 1) / p.tokens_per_tile;
    p.n_pairs = (p.num_q_tiles + 1) / 2;
    if (static_cast<long long>(p.n_pairs) * n_kv_heads > 0x7fffffffLL)
        return fail(FA512_ERR_UNSUPPORTED, "too many work items");
    p.n_items = p.n_pairs * n_kv_heads;
    p.causal = causal ? 1 : 0;
    p.window = window > 0 ? window : 0;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.err = err;
    fa512::plan_prefill256(p, sm_count());

    CUtensorMap tmq, tmk, tmv, tmo;
    memset(&tmk, 0, sizeof tmk);
    memset(&tmv, 0, sizeof tmv);
    {
        const uint64_t dims[4] = {static_cast<uint64_t>(kD), static_cast<uint64_t>(G),
                                  static_cast<uint64_t>(n_kv_heads), static_cast<uint64_t>(seqlen_q)};
        const uint64_t strides[3] = {kD * 2ull, static_cast<uint64_t>(G) * kD * 2ull,
                                     static_cast<uint64_t>(n_q_heads) * kD * 2ull};
        const uint32_t box[4] = {64u, static_cast<uint32_t>(G), 1u,
                                 static_cast<uint32_t>(p.tokens_per_tile)};
        fa512_status st = encode_bf16(&tmq, q, 4, dims, strides, box);
        if (st != FA512_OK) return st;
        // O leaves through the same box shape (a staged tile per TMA store)
        st = encode_bf16(&tmo, out, 4, dims, strides, box);
        if (st != FA512_OK) return st;
    }
    if (seqlen_k > 0) {
        const uint64_t dims[3] = {static_cast<uint64_t>(kD), static_cast<uint64_t>(n_kv_heads),
                                  static_cast<uint64_t>(seqlen_k)};
        const uint64_t strides[2] = {kD * 2ull, static_cast<uint64_t>(n_kv_heads) * kD * 2ull};
        // K in {64 columns, 48 keys} boxes (each CTA of a pair holds half a
        // 96-key tile), V in {64 columns, 96 keys} boxes
        const uint32_t kbox[3] = {64u, 1u, static_cast<uint32_t>(fa512::prefill256_k_box_rows())};
        const uint32_t vbox[3] = {64u, 1u, static_cast<uint32_t>(fa512::prefill256_v_box_rows())};
        fa512_status st = encode_bf16(&tmk, k, 3, dims, strides, kbox);
        if (st != FA512_OK) return st;
        st = encode_bf16(&tmv, v, 3, dims, strides, vbox);
        if (st != FA512_OK) return st;
    }
    e = fa512::launch_prefill256(tmq, tmk, tmv, tmo, p, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "head-dim-256 prefill launch");
    return FA512_OK;
}

fa512_status fa512_prefill_paged(const void* q, const void* k_pages, const void* v_pages,
                                 const int32_t* page_table, const int32_t* cu_seqlens_q,
                                 const int32_t* seqused_k, void* out, float* lse, int batch,
                                 int total_q, int max_seqlen_q, int n_q_heads, int n_kv_heads,
                                 int page_size, int num_pages, int max_pages_per_seq, float scale,
                                 int causal, int window, fa512_stream_t stream) {
    g_last_error[0] = 0;
    if (batch < 0 || total_q < 0 || max_seqlen_q < 0)
        return fail(FA512_ERR_INVALID_ARG, "negative batch, total_q or max_seqlen_q");
    if (n_kv_heads < 1 || n_q_heads < 1 || n_q_heads % n_kv_heads != 0)
        return fail(FA512_ERR_INVALID_ARG, "n_q_heads (%d) must be a positive multiple of n_kv_heads (%d)",
                    n_q_heads, n_kv_heads);
    const int G = n_q_heads / n_kv_heads;
    if (G > 128) return fail(FA512_ERR_UNSUPPORTED, "more than 128 query heads per KV head");
    if (page_size != 64 && page_size != 128 && page_size != 256)
        return fail(FA512_ERR_UNSUPPORTED, "prefill over a paged cache needs page_size 64, 128 or 256");
    if (num_pages < 1 || max_pages_per_seq < 1)
        return fail(FA512_ERR_INVALID_ARG, "num_pages and max_pages_per_seq must be >= 1");
    if (static_cast<long long>(num_pages) * page_size > 0x7fffffffLL - 256 ||
        static_cast<long long>(max_pages_per_seq) * page_size > 0x7fffffffLL - 256)
        return fail(FA512_ERR_UNSUPPORTED, "page pool or page table too large for int32 key rows");
    if (!(scale == scale) || isinf(scale)) return fail(FA512_ERR_INVALID_ARG, "scale is not finite");
    if (batch == 0 || total_q == 0 || max_seqlen_q == 0) return FA512_OK;
    if (!q || !out || !k_pages || !v_pages || !page_table || !cu_seqlens_q || !seqused_k)
        return fail(FA512_ERR_INVALID_ARG, "null pointer");
    if (!aligned16(q) || !aligned16(out) || !aligned16(k_pages) || !aligned16(v_pages))
        return fail(FA512_ERR_INVALID_ARG, "q, k_pages, v_pages and out must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(page_table) | reinterpret_cast<uintptr_t>(cu_seqlens_q) |
         reinterpret_cast<uintptr_t>(seqused_k)) & 3u)
        return fail(FA512_ERR_INVALID_ARG, "int32 arrays must be 4-byte aligned");
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u))
        return fail(FA512_ERR_INVALID_ARG, "lse must be 4-byte aligned");

    unsigned* err = nullptr;
    cudaError_t e = device_error_ptr(&err);
    if (e != cudaSuccess) return cuda_fail(e, "device error word");

    fa512::PrefillParams p;
    memset(&p, 0, sizeof p);
    p.out = static_cast<__nv_bfloat16*>(out);
    p.lse = lse;
    p.total_q = total_q;
    p.n_q_heads = n_q_heads;
    p.n_kv_heads = n_kv_heads;
    p.group = G;
    p.tokens_per_tile = 128 / G;
    p.rows_per_tile = p.tokens_per_tile * G;
    p.causal = causal ? 1 : 0;
    p.window = window > 0 ? window : 0;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.err = err;
    p.page_table = page_table;
    p.cu_seqlens_q = cu_seqlens_q;
    p.seqused_k = seqused_k;
    p.batch = batch;
    p.max_seqlen_q = max_seqlen_q;
    const long long tiles = (static_cast<long long>(max_seqlen_q) + p.tokens_per_tile - 1) / p.tokens_per_tile;
    p.max_pairs = static_cast<int>((tiles + 1) / 2);
    int shift = 0;
    while ((1 << shift) < page_size) ++shift;
    p.page_shift = shift;
    p.num_pages = num_pages;
    p.max_pages_per_seq = max_pages_per_seq;
    p.oob_row = num_pages * page_size;
    if (static_cast<long long>(batch) * n_kv_heads * p.max_pairs * 4 > 0x7fffffffLL)
        return fail(FA512_ERR_UNSUPPORTED, "grid too large");

    CUtensorMap tmq, tmk, tmv;
    {
        const uint64_t dims[4] = {static_cast<uint64_t>(kHeadDim), static_cast<uint64_t>(G),
                                  static_cast<uint64_t>(n_kv_heads), static_cast<uint64_t>(total_q)};
        const uint64_t strides[3] = {kHeadDim * 2ull, static_cast<uint64_t>(G) * kHeadDim * 2ull,
                                     static_cast<uint64_t>(n_q_heads) * kHeadDim * 2ull};
        const uint32_t box[4] = {64u, static_cast<uint32_t>(G), 1u,
                                 static_cast<uint32_t>(p.tokens_per_tile)};
        fa512_status st = encode_bf16(&tmq, q, 4, dims, strides, box);
        if (st != FA512_OK) return st;
    }
    {
        // the pool as rows of keys: [num_pages * page_size, n_kv_heads, 512]
        const uint64_t dims[3] = {static_cast<uint64_t>(kHeadDim), static_cast<uint64_t>(n_kv_heads),
                                  static_cast<uint64_t>(num_pages) * page_size};
        const uint64_t strides[2] = {kHeadDim * 2ull, static_cast<uint64_t>(n_kv_heads) * kHeadDim * 2ull};
        const uint32_t kbox[3] = {64u, 1u, static_cast<uint32_t>(fa512::prefill_k_box_rows())};
        const uint32_t vbox[3] = {64u, 1u, static_cast<uint32_t>(fa512::prefill_paged_v_box_rows())};
        fa512_status st = encode_bf16(&tmk, k_pages, 3, dims, strides, kbox);
        if (st != FA512_OK) return st;
        st = encode_bf16(&tmv, v_pages, 3, dims, strides, vbox);
        if (st != FA512_OK) return st;
    }
    e = fa512::launch_prefill_paged(tmq, tmk, tmv, p, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "paged prefill launch");
    return FA512_OK;
}

int fa512_decode_auto_splits(int batch, int n_kv_heads, int page_size, int max_kv_len) {
    (void)page_size;
    if (batch <= 0 || n_kv_heads <= 0 || max_kv_len <= 0) return 1;
    return choose_splits(static_cast<long long>(batch) * n_kv_heads, band_tiles(max_kv_len, 0),
                         sm_count());
}

int fa512_decode_auto_splits_fp8(int batch, int q_len, int n_q_heads, int n_kv_heads,
                                 int page_size, int max_kv_len) {
    if (batch <= 0 || q_len < 1 || n_kv_heads <= 0 || n_q_heads <= 0 || max_kv_len <= 0) return 1;
    if (q_len * (n_q_heads / n_kv_heads) > fa512::decode_fp8_mma_rows())
        return fa512_decode_auto_splits(batch, n_kv_heads, page_size, max_kv_len);
    return choose_splits_fp8(static_cast<long long>(batch) * n_kv_heads, band_tiles(max_kv_len, 0),
                             sm_count(), static_cast<long long>(batch) * q_len * n_q_heads);
}

size_t fa512_decode_workspace_bytes_fp8(int batch, int q_len, int n_q_heads, int n_kv_heads,
                                        int page_size, int max_kv_len, int num_splits) {
    if (batch < 0 || q_len < 1 || n_q_heads <= 0 || n_kv_heads <= 0 || max_kv_len < 0 ||
        num_splits < 0 || num_splits > 1024)
        return 0;
    const int s = num_splits > 0 ? num_splits
                                 : fa512_decode_auto_splits_fp8(batch, q_len, n_q_heads, n_kv_heads,
                                                                page_size, max_kv_len);
    return workspace_for(batch * q_len, n_q_heads, s);
}

size_t fa512_decode_workspace_bytes_q(int batch, int q_len, int n_q_heads, int n_kv_heads,
                                      int page_size, int max_kv_len, int num_splits) {
    if (batch < 0 || q_len < 1 || n_q_heads <= 0 || n_kv_heads <= 0 || max_kv_len < 0 ||
        num_splits < 0 || num_splits > 1024)
        return 0;
    const int s = num_splits > 0 ? num_splits
                                 : fa512_decode_auto_splits(batch, n_kv_heads, page_size, max_kv_len);
    return workspace_for(batch * q_len, n_q_heads, s);
}

size_t fa512_decode_workspace_bytes(int batch, int n_q_heads, int n_kv_heads, int page_size,
                                    int max_kv_len, int num_splits) {
    return fa512_decode_workspace_bytes_q(batch, 1, n_q_heads, n_kv_heads, page_size, max_kv_len,
                                          num_splits);
}

}  // extern "C"

namespace {

// Body of the decode entry points.  fp8: k_pages / v_pages hold e4m3 bytes
// and a key (value) element is k_scale (v_scale) times its e4m3 value.
fa512_status decode_call(const void* q, const void* k_pages, const void* v_pages,
                         const int32_t* page_table, const int32_t* kv_lens, void* out, float* lse,
                         int batch, int q_len, int n_q_heads, int n_kv_heads, int page_size,
                         int num_pages, int max_pages_per_seq, int max_kv_len, float scale,
                         int window, int num_splits, void* workspace, size_t workspace_bytes,
                         bool fp8, float k_scale, float v_scale, fa512_stream_t stream) {
    g_last_error[0] = 0;
    if (batch < 0) return fail(FA512_ERR_INVALID_ARG, "negative batch");
    if (q_len < 1) return fail(FA512_ERR_INVALID_ARG, "q_len must be >= 1");
    if (n_kv_heads < 1 || n_q_heads < 1 || n_q_heads % n_kv_heads != 0)
        return fail(FA512_ERR_INVALID_ARG, "n_q_heads (%d) must be a positive multiple of n_kv_heads (%d)",
                    n_q_heads, n_kv_heads);
    const int G = n_q_heads / n_kv_heads;
    if (G > 16) return fail(FA512_ERR_UNSUPPORTED, "decode supports at most 16 query heads per KV head");
    if (q_len * G > 16)
        return fail(FA512_ERR_UNSUPPORTED, "q_len x query heads per KV head (%d x %d) must be at most 16",
                    q_len, G);
    if (!pow2_page(page_size)) return fail(FA512_ERR_UNSUPPORTED, "page_size must be 16, 32, 64, 128 or 256");
    if (num_pages < 1 || max_pages_per_seq < 1)
        return fail(FA512_ERR_INVALID_ARG, "num_pages and max_pages_per_seq must be >= 1");
    if (static_cast<long long>(num_pages) * page_size > 0x7fffffffLL)
        return fail(FA512_ERR_UNSUPPORTED, "page pool larger than 2^31 rows");
    if (max_kv_len < 0 || static_cast<long long>(max_kv_len) > static_cast<long long>(max_pages_per_seq) * page_size)
        return fail(FA512_ERR_INVALID_ARG, "max_kv_len outside [0, max_pages_per_seq * page_size]");
    if (num_splits < 0 || num_splits > 1024) return fail(FA512_ERR_INVALID_ARG, "num_splits outside [0, 1024]");
    if (!(scale == scale) || isinf(scale)) return fail(FA512_ERR_INVALID_ARG, "scale is not finite");
    if (fp8 && (!(k_scale == k_scale) || isinf(k_scale) || !(v_scale == v_scale) || isinf(v_scale)))
        return fail(FA512_ERR_INVALID_ARG, "k_scale and v_scale must be finite");
    if (batch == 0) return FA512_OK;
    if (!q || !k_pages || !v_pages || !page_table || !kv_lens || !out)
        return fail(FA512_ERR_INVALID_ARG, "null tensor pointer");
    if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(out))
        return fail(FA512_ERR_INVALID_ARG, "q, pages and out must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(page_table) & 3u) || (reinterpret_cast<uintptr_t>(kv_lens) & 3u) ||
        (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
        return fail(FA512_ERR_INVALID_ARG, "page_table, kv_lens and lse must be 4-byte aligned");

    const int splits = num_splits > 0 ? num_splits
                       : fp8 ? fa512_decode_auto_splits_fp8(batch, q_len, n_q_heads, n_kv_heads,
                                                            page_size, max_kv_len)
                             : fa512_decode_auto_splits(batch, n_kv_heads, page_size, max_kv_len);
    const size_t need = workspace_for(batch * q_len, n_q_heads, splits);
    if (!workspace || workspace_bytes < need)
        return fail(FA512_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need, workspace_bytes);
    if (reinterpret_cast<uintptr_t>(workspace) & 255u)
        return fail(FA512_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    if (static_cast<long long>(batch) * n_kv_heads > 65535LL * 65535LL)
        return fail(FA512_ERR_UNSUPPORTED, "grid too large");
    if (batch > 65535 || n_kv_heads > 65535) return fail(FA512_ERR_UNSUPPORTED, "grid too large");

    unsigned* err = nullptr;
    cudaError_t e = device_error_ptr(&err);
    if (e != cudaSuccess) return cuda_fail(e, "device error word");

    fa512::DecodeParams p;
    memset(&p, 0, sizeof p);
    p.q = static_cast<const __nv_bfloat16*>(q);
    if (fp8) {
        p.k8 = static_cast<const uint8_t*>(k_pages);
        p.v8 = static_cast<const uint8_t*>(v_pages);
        p.o_scale = v_scale;
    } else {
        p.k_pages = static_cast<const __nv_bfloat16*>(k_pages);
        p.v_pages = static_cast<const __nv_bfloat16*>(v_pages);
        p.o_scale = 1.f;
    }
    p.page_table = page_table;
    p.kv_lens = kv_lens;
    const size_t rows = static_cast<size_t>(batch) * q_len * n_q_heads * splits;
    p.ws_o = static_cast<float*>(workspace);
    p.ws_ml = reinterpret_cast<float*>(static_cast<char*>(workspace) + round256(rows * kHeadDim * sizeof(float)));
    p.out = static_cast<__nv_bfloat16*>(out);
    p.lse = lse;
    p.batch = batch;
    p.n_q_heads = n_q_heads;
    p.n_kv_heads = n_kv_heads;
    p.group = G;
    p.q_len = q_len;
    p.page_size = page_size;
    p.box_rows = page_size < 32 ? page_size : 32;
    p.num_pages = num_pages;
    p.max_pages_per_seq = max_pages_per_seq;
    p.len_cap = max_kv_len;
    p.window = window > 0 ? window : 0;
    const long long tiles = band_tiles(max_kv_len, p.window);
    p.num_splits = splits;
    p.tiles_per_split = static_cast<int>((tiles + splits - 1) / splits);
    if (p.tiles_per_split < 1) p.tiles_per_split = 1;
    p.scale_log2 = scale * 1.4426950408889634f;
    // FP8: k_scale scales every score; applied after the bf16 path's factor
    // so that a power-of-two k_scale changes no rounding
    if (fp8) p.scale_log2 *= k_scale;
    p.err = err;

    CUtensorMap tmk, tmv;
    const uint64_t dims[3] = {static_cast<uint64_t>(kHeadDim), static_cast<uint64_t>(n_kv_heads),
                              static_cast<uint64_t>(num_pages) * page_size};
    fa512_status st;
    if (fp8) {
        // e4m3 bytes: 256-byte boxes, no swizzle (the kernel converts them to
        // the swizzled bf16 tile itself)
        const uint64_t strides[2] = {static_cast<uint64_t>(kHeadDim),
                                     static_cast<uint64_t>(n_kv_heads) * kHeadDim};
        const uint32_t box[3] = {static_cast<uint32_t>(fa512::decode_fp8_box_bytes()), 1u,
                                 static_cast<uint32_t>(p.box_rows)};
        st = encode_map(&tmk, CU_TENSOR_MAP_DATA_TYPE_UINT8, CU_TENSOR_MAP_SWIZZLE_NONE, k_pages, 3,
                        dims, strides, box);
        if (st != FA512_OK) return st;
        st = encode_map(&tmv, CU_TENSOR_MAP_DATA_TYPE_UINT8, CU_TENSOR_MAP_SWIZZLE_NONE, v_pages, 3,
                        dims, strides, box);
        if (st != FA512_OK) return st;
        e = fa512::launch_decode_fp8(tmk, tmv, p, reinterpret_cast<cudaStream_t>(stream));
    } else {
        const uint64_t strides[2] = {kHeadDim * 2ull, static_cast<uint64_t>(n_kv_heads) * kHeadDim * 2ull};
        const uint32_t box[3] = {64u, 1u, static_cast<uint32_t>(p.box_rows)};
        st = encode_bf16(&tmk, k_pages, 3, dims, strides, box);
        if (st != FA512_OK) return st;
        st = encode_bf16(&tmv, v_pages, 3, dims, strides, box);
        if (st != FA512_OK) return st;
        e = fa512::launch_decode(tmk, tmv, p, reinterpret_cast<cudaStream_t>(stream));
    }
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    return FA512_OK;
}

}  // namespace

extern "C" {

fa512_status fa512_decode_paged_q(const void* q, const void* k_pages, const void* v_pages,
                                  const int32_t* page_table, const int32_t* kv_lens, void* out,
                                  float* lse, int batch, int q_len, int n_q_heads, int n_kv_heads,
                                  int page_size, int num_pages, int max_pages_per_seq,
                                  int max_kv_len, float scale, int window, int num_splits,
                                  void* workspace, size_t workspace_bytes,
                                  fa512_stream_t stream) {
    return decode_call(q, k_pages, v_pages, page_table, kv_lens, out, lse, batch, q_len, n_q_heads,
                       n_kv_heads, page_size, num_pages, max_pages_per_seq, max_kv_len, scale,
                       window, num_splits, workspace, workspace_bytes, false, 1.f, 1.f, stream);
}

fa512_status fa512_decode_paged_fp8(const void* q, const void* k_pages, const void* v_pages,
                                    const int32_t* page_table, const int32_t* kv_lens, void* out,
                                    float* lse, int batch, int q_len, int n_q_heads,
                                    int n_kv_heads, int page_size, int num_pages,
                                    int max_pages_per_seq, int max_kv_len, float scale,
                                    float k_scale, float v_scale, int window, int num_splits,
                                    void* workspace, size_t workspace_bytes,
                                    fa512_stream_t stream) {
    return decode_call(q, k_pages, v_pages, page_table, kv_lens, out, lse, batch, q_len, n_q_heads,
                       n_kv_heads, page_size, num_pages, max_pages_per_seq, max_kv_len, scale,
                       window, num_splits, workspace, workspace_bytes, true, k_scale, v_scale,
                       stream);
}

fa512_status fa512_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                                const int32_t* page_table, const int32_t* kv_lens, void* out,
                                float* lse, int batch, int n_q_heads, int n_kv_heads,
                                int page_size, int num_pages, int max_pages_per_seq,
                                int max_kv_len, float scale, int window, int num_splits,
                                void* workspace, size_t workspace_bytes,
                                fa512_stream_t stream) {
    return fa512_decode_paged_q(q, k_pages, v_pages, page_table, kv_lens, out, lse, batch, 1,
                                n_q_heads, n_kv_heads, page_size, num_pages, max_pages_per_seq,
                                max_kv_len, scale, window, num_splits, workspace, workspace_bytes,
                                stream);
}

fa512_status fa512_device_status(fa512_stream_t stream, int clear) {
    g_last_error[0] = 0;
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
    unsigned word = 0;
    e = cudaMemcpyFromSymbol(&word, fa512_device_error_word, sizeof word);
    if (e != cudaSuccess) return cuda_fail(e, "read device error word");
    if (clear && word) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(fa512_device_error_word, &zero, sizeof zero);
        if (e != cudaSuccess) return cuda_fail(e, "clear device error word");
    }
    if (word & 1u) return fail(FA512_ERR_TIMEOUT, "a kernel pipeline wait exceeded its bound");
    if (word & 2u) return fail(FA512_ERR_DEVICE_INDEX, "a page index or kv length was out of range");
    if (word & 4u) return fail(FA512_ERR_UNSUPPORTED, "the dynamic shared-memory window was not 1 KiB aligned");
    return FA512_OK;
}

}  // extern "C"

/*
 * fa512 -- head-dim-512 FlashAttention forward for GB300 (sm_103a).
 *
 * C ABI of the library.  Plain pointers and sizes only; every device pointer
 * is owned by the caller, the library calls no allocator and never
 * synchronises the stream it is given.  All work is enqueued on `stream`.
 * The library's own device memory is static: a 4-byte error word and the
 * FA512_DECODE_STATIC_SCRATCH_BYTES array of fa512_decode_paged_noalloc,
 * held on every GPU that loads the library until the process exits.  Their
 * device addresses are looked up once per device and kept, so the library
 * must not be used across a device reset (cudaDeviceReset).
 *
 * Operations (page title, then the part of the page that states them):
 *
 *  fa512_prefill -- causal GQA/MQA attention of a chunk of query rows against
 *    the keys before them, with online softmax (running max m, running sum l,
 *    rescaled O) so the [q x k] score matrix never reaches memory.
 *    "Writing a FlashAttention Prefill Kernel for Gemma 4", sections "The
 *    starting point" and "Head dim 512 breaks the textbook"; "A custom
 *    attention kernel for Gemma 4 on the RTX PRO 6000", section "The kernel
 *    in three steps" (query heads that share a KV head are packed into one
 *    tile); pegainfer issue #1051, "Description" (one 8192-row chunk against
 *    everything before it, 32 query heads over 4 KV heads).
 *
 *  fa512_prefill_d256 -- the same for heads of 256 dimensions (the
 *    sliding-window local layers, window 1,024), from a persistent kernel.
 *
 *  fa512_prefill_paged -- the same for a batch of chunks of different
 *    lengths over a paged KV cache (pegainfer issue #1051, "Proposed Plan").
 *
 *  fa512_decode_paged_fp8 -- the same over a cache stored in FP8 E4M3
 *    (vllm-project/flash-attention PR #199, "Summary").
 *
 *  fa512_decode_paged -- one query token per sequence against a paged KV
 *    cache, split over the key sequence (Flash-Decoding): each split writes an
 *    unnormalised (O, m, l) partial and a merge step combines them.
 *    "Flash-Decoding for MQA in CUDA", section "One KV head breaks the
 *    textbook"; vllm-project/flash-attention PR #199, "Performance" table
 *    (q_len 1, 8 query heads over 4 KV heads, head dim 512, page size 64).
 *
 * Numerics: bf16 inputs and outputs, fp32 accumulation and softmax state.
 * LSE is the natural logarithm of sum_j exp(scale * q.k_j) over the visible
 * keys; a row with no visible key gets O = 0 and LSE = -inf
 * (vllm-project/flash-attention PR #199, review item F4).
 *
 * Errors: arguments are validated before anything is enqueued; a rejected
 * call returns a non-zero fa512_status and launches nothing.  A failed launch
 * returns FA512_ERR_CUDA.  Faults that only the device can see (a page index
 * outside the pool, a kv length beyond the page table, a pipeline wait that
 * ran past its bound) are recorded in a device-side error word that
 * fa512_device_status() reads; the kernels skip the offending access instead
 * of trapping.
 */
#ifndef FA512_H
#define FA512_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *fa512_stream_t;

typedef enum {
    FA512_OK = 0,
    FA512_ERR_INVALID_ARG = 1, /* a pointer, size or alignment is unusable      */
    FA512_ERR_UNSUPPORTED = 2, /* well-formed but outside what the kernels do    */
    FA512_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed              */
    FA512_ERR_TIMEOUT = 4,     /* device: a pipeline wait exceeded its bound     */
    FA512_ERR_WORKSPACE = 5,   /* workspace missing or smaller than required     */
    FA512_ERR_DEVICE_INDEX = 6 /* device: page index or kv length out of range   */
} fa512_status;

/* Head dimension of every tensor this library accepts. */
#define FA512_HEAD_DIM 512

/*
 * fa512_prefill -- attention forward of one prefill chunk (batch 1).
 *
 *   q    [seqlen_q, n_q_heads, 512]  bf16, device, contiguous
 *   k, v [seqlen_k, n_kv_heads, 512] bf16, device, contiguous
 *   out  [seqlen_q, n_q_heads, 512]  bf16, device, written
 *   lse  [n_q_heads, seqlen_q]       fp32, device, written; may be NULL
 *
 * Query row i sits at absolute position q_offset + i.  Query head h reads KV
 * head h / (n_q_heads / n_kv_heads).  Key j is visible to row i iff
 *   (causal == 0 or j <= q_offset + i)  and
 *   (window <= 0 or j > q_offset + i - window)        (window keys incl. own).
 * scale multiplies q.k before the softmax (1/sqrt(512) for Gemma-4 shapes).
 *
 * Requirements: seqlen_q >= 0, seqlen_k >= 0, q_offset >= 0, n_kv_heads >= 1,
 * n_q_heads a multiple of n_kv_heads with G = n_q_heads / n_kv_heads <= 128,
 * every pointer 16-byte aligned.  seqlen_q == 0 is a no-op.
 * Returns FA512_OK once the kernels are enqueued.
 */
fa512_status fa512_prefill(const void *q, const void *k, const void *v, void *out, float *lse,
                           int seqlen_q, int seqlen_k, int q_offset, int n_q_heads,
                           int n_kv_heads, float scale, int causal, int window,
                           fa512_stream_t stream);

/*
 * fa512_prefill_d256 -- the same forward for heads of 256 dimensions, the
 * sliding-window local layers ("A custom attention kernel for Gemma 4 on the
 * RTX PRO 6000", "The deployment": they attend to the last 1,024 tokens with
 * heads of 256 dimensions).
 *
 *   q    [seqlen_q, n_q_heads, 256]  bf16, device, contiguous
 *   k, v [seqlen_k, n_kv_heads, 256] bf16, device, contiguous
 *   out  [seqlen_q, n_q_heads, 256]  bf16, device, written
 *   lse  [n_q_heads, seqlen_q]       fp32, device, written; may be NULL
 *
 * Positions, visibility (causal, window), scale, requirements and errors are
 * those of fa512_prefill; a window of 1024 is the local layers' setting and
 * window <= 0 attends causally (or fully) to every key.
 */
fa512_status fa512_prefill_d256(const void *q, const void *k, const void *v, void *out, float *lse,
                                int seqlen_q, int seqlen_k, int q_offset, int n_q_heads,
                                int n_kv_heads, float scale, int causal, int window,
                                fa512_stream_t stream);

/*
 * fa512_prefill_paged -- attention forward of a batch of prefill chunks
 * (varlen rows) over a paged KV cache.  pegainfer issue #1051, "Proposed
 * Plan" (a varlen paged prefill for head dim 512; the pool paged at the key
 * block, so a block of keys is one copy); vllm-project/flash-attention PR
 * #199, review (call shapes: varlen Q, paged K/V, prefix prefill).
 *
 *   q            [total_q, n_q_heads, 512]              bf16, device
 *   k_pages      [num_pages, page_size, n_kv_heads, 512] bf16, device
 *   v_pages      same shape as k_pages                  bf16, device
 *   page_table   [batch, max_pages_per_seq] int32, device: logical page p of
 *                sequence b is physical page page_table[b * max_pages_per_seq + p]
 *   cu_seqlens_q [batch + 1] int32, device: the chunk of sequence b is rows
 *                cu_seqlens_q[b] .. cu_seqlens_q[b + 1] - 1 of q and out
 *   seqused_k    [batch] int32, device: cached positions of sequence b,
 *                the chunk's own keys included
 *   out          [total_q, n_q_heads, 512] bf16, device, written
 *   lse          [n_q_heads, total_q] fp32, device, written; may be NULL
 *
 * A chunk is the tail of its sequence: row i of a chunk of S rows sits at
 * position seqused_k[b] - S + i, and key j < seqused_k[b] is visible to it
 * under the same causal / window rule as fa512_prefill (a negative position
 * sees no key when causal: O = 0, LSE = -inf).  Only the pages that hold
 * visible positions are read; slots past seqused_k[b] may hold anything
 * (NaN included) without reaching the output.
 *
 * max_seqlen_q is a host-side upper bound of the chunk lengths (it sizes the
 * grid; nothing is read back).  On the device, a chunk longer than
 * max_seqlen_q, seqused_k[b] outside [0, max_pages_per_seq * page_size],
 * cu_seqlens_q not rising within [0, total_q], or a page index outside
 * [0, num_pages) is recorded in the device error word; the offending rows or
 * pages are clipped or read as zeros, never out of bounds.
 *
 * Requirements: page_size 64, 128 or 256 (a page holds whole 64-key half
 * tiles); num_pages, max_pages_per_seq >= 1; n_q_heads a multiple of
 * n_kv_heads with at most 128 query heads per KV head; tensors 16-byte
 * aligned, int32 arrays 4-byte aligned.  batch, total_q or max_seqlen_q == 0
 * is a no-op.
 */
fa512_status fa512_prefill_paged(const void *q, const void *k_pages, const void *v_pages,
                                 const int32_t *page_table, const int32_t *cu_seqlens_q,
                                 const int32_t *seqused_k, void *out, float *lse, int batch,
                                 int total_q, int max_seqlen_q, int n_q_heads, int n_kv_heads,
                                 int page_size, int num_pages, int max_pages_per_seq, float scale,
                                 int causal, int window, fa512_stream_t stream);

/*
 * fa512_decode_paged -- one query token per sequence over a paged KV cache.
 *
 *   q          [batch, n_q_heads, 512]                     bf16, device
 *   k_pages    [num_pages, page_size, n_kv_heads, 512]      bf16, device
 *   v_pages    same shape as k_pages                        bf16, device
 *   page_table [batch, max_pages_per_seq] int32, device: logical page p of
 *              sequence b is physical page page_table[b * max_pages_per_seq + p]
 *   kv_lens    [batch] int32, device: live length of each sequence
 *   out        [batch, n_q_heads, 512] bf16, device, written
 *   lse        [batch, n_q_heads] fp32, device, written; may be NULL
 *
 * The query of sequence b sits at position kv_lens[b] - 1 and sees positions
 * [max(0, kv_lens[b] - window), kv_lens[b]) (window <= 0: all of [0, len)).
 * Only the pages that hold those positions are read.
 *
 * max_kv_len is a host-side upper bound of kv_lens (it sizes the split grid;
 * no value is read back from the device).  kv_lens[b] > max_kv_len is an
 * error recorded on the device; positions past max_kv_len are not read.
 * num_splits: 0 picks fa512_decode_auto_splits(); otherwise 1 <= num_splits
 * <= 1024.  workspace holds the (O, m, l) partials and must be at least
 * fa512_decode_workspace_bytes(batch, n_q_heads, splits) bytes, 256-byte
 * aligned, for the split count actually used.
 *
 * Requirements: batch >= 0, page_size one of 16, 32, 64, 128, 256,
 * n_q_heads a multiple of n_kv_heads with G <= 16, num_pages >= 1,
 * max_kv_len <= max_pages_per_seq * page_size, tensors 16-byte aligned.
 */
fa512_status fa512_decode_paged(const void *q, const void *k_pages, const void *v_pages,
                                const int32_t *page_table, const int32_t *kv_lens, void *out,
                                float *lse, int batch, int n_q_heads, int n_kv_heads,
                                int page_size, int num_pages, int max_pages_per_seq,
                                int max_kv_len, float scale, int window, int num_splits,
                                void *workspace, size_t workspace_bytes,
                                fa512_stream_t stream);

/* Bytes of workspace fa512_decode_paged needs for this shape and split count
 * (num_splits 0 means the automatic choice for max_kv_len).  Returns 0 for an
 * invalid shape. */
size_t fa512_decode_workspace_bytes(int batch, int n_q_heads, int n_kv_heads, int page_size,
                                    int max_kv_len, int num_splits);

/*
 * fa512_decode_paged_q -- q_len query tokens per sequence over a paged KV
 * cache: the tokens just appended to each cache (draft tokens being
 * verified, a short chunk), each attending causally to the cache.  The pages
 * list multi-token decode among the next steps of the decode path
 * (vllm-project/flash-attention PR #199, "Notes": varlen Q over a paged
 * cache; "A custom attention kernel for Gemma 4 on the RTX PRO 6000", the
 * draft of 4 tokens).
 *
 *   q    [batch, q_len, n_q_heads, 512] bf16, device
 *   out  [batch, q_len, n_q_heads, 512] bf16, device, written
 *   lse  [batch, q_len, n_q_heads] fp32, device, written; may be NULL
 *   other tensors and arguments as fa512_decode_paged.
 *
 * Query t of sequence b sits at position kv_lens[b] - q_len + t and sees
 * positions [max(0, pos - window + 1), pos] (window <= 0: [0, pos]); a query
 * whose position is negative (kv_lens[b] < q_len) sees nothing and returns
 * O = 0, LSE = -inf.  The workspace must be at least
 * fa512_decode_workspace_bytes_q(batch, q_len, ...) bytes.  Requirements as
 * fa512_decode_paged, plus q_len >= 1 and q_len * (n_q_heads / n_kv_heads)
 * <= 16 (FA512_ERR_UNSUPPORTED otherwise).  q_len = 1 is fa512_decode_paged.
 */
fa512_status fa512_decode_paged_q(const void *q, const void *k_pages, const void *v_pages,
                                  const int32_t *page_table, const int32_t *kv_lens, void *out,
                                  float *lse, int batch, int q_len, int n_q_heads, int n_kv_heads,
                                  int page_size, int num_pages, int max_pages_per_seq,
                                  int max_kv_len, float scale, int window, int num_splits,
                                  void *workspace, size_t workspace_bytes,
                                  fa512_stream_t stream);

/* Workspace bytes fa512_decode_paged_q needs (0 for an invalid shape). */
size_t fa512_decode_workspace_bytes_q(int batch, int q_len, int n_q_heads, int n_kv_heads,
                                      int page_size, int max_kv_len, int num_splits);

/*
 * fa512_decode_paged_fp8 -- fa512_decode_paged_q over a paged KV cache
 * stored in FP8 E4M3 (vllm-project/flash-attention PR #199, "Summary": the
 * paged KV cache in FP8; its "Performance" table times the decode shapes
 * with an FP8 cache).
 *
 *   k_pages, v_pages [num_pages, page_size, n_kv_heads, 512] uint8, device:
 *              one OCP E4M3 ("e4m3fn": bias 7, no infinities, S.1111.111
 *              NaN, largest finite 448) byte per element
 *   k_scale, v_scale per-tensor dequantisation scales: key element
 *              k_scale * e4m3(byte), value element v_scale * e4m3(byte)
 *   q, out, lse, positions and every other argument as
 *              fa512_decode_paged_q (q_len >= 1, q_len * G <= 16)
 *   num_splits 0 picks fa512_decode_auto_splits_fp8(); workspace must be
 *              at least fa512_decode_workspace_bytes_fp8() bytes for the
 *              split count used (256-byte aligned).
 *
 * The cache is read as bytes: half the HBM traffic of a bf16 cache.  Every
 * byte is widened exactly (e4m3 -> bf16/fp32) before it meets the bf16
 * query, so the arithmetic is that of fa512_decode_paged_q on the
 * dequantised cache: fp32 accumulation, fp32 softmax state, P rounded to
 * bf16 only on the tensor-core path (q_len * G > 2).  Slots outside the live
 * band are never read (NaN codes there do not reach the output).
 * k_scale and v_scale must be finite (FA512_ERR_INVALID_ARG otherwise).
 */
fa512_status fa512_decode_paged_fp8(const void *q, const void *k_pages, const void *v_pages,
                                    const int32_t *page_table, const int32_t *kv_lens, void *out,
                                    float *lse, int batch, int q_len, int n_q_heads,
                                    int n_kv_heads, int page_size, int num_pages,
                                    int max_pages_per_seq, int max_kv_len, float scale,
                                    float k_scale, float v_scale, int window, int num_splits,
                                    void *workspace, size_t workspace_bytes,
                                    fa512_stream_t stream);

/* Split count chosen when num_splits == 0: enough (batch, KV head, split)
 * work items to fill the current device's SMs about twice, each split at
 * least one page.  Returns 1 when there is nothing to split. */
int fa512_decode_auto_splits(int batch, int n_kv_heads, int page_size, int max_kv_len);

/* Split count fa512_decode_paged_fp8 uses when num_splits == 0.  With
 * q_len * G <= 8 its split kernel runs four CTAs of four warps per SM, one
 * split each, so the choice spreads the keys over four times as many CTAs
 * (at most 128 splits); otherwise it is fa512_decode_auto_splits().  Returns
 * 1 when there is nothing to split. */
int fa512_decode_auto_splits_fp8(int batch, int q_len, int n_q_heads, int n_kv_heads,
                                 int page_size, int max_kv_len);

/* Workspace bytes fa512_decode_paged_fp8 needs for this shape and split
 * count (num_splits 0: fa512_decode_auto_splits_fp8).  0 for an invalid
 * shape. */
size_t fa512_decode_workspace_bytes_fp8(int batch, int q_len, int n_q_heads, int n_kv_heads,
                                        int page_size, int max_kv_len, int num_splits);

/*
 * fa512_decode_paged_noalloc -- fa512_decode_paged without a workspace
 * argument.  (The pages have no counterpart: this is a convenience of the
 * library, not a step of the method.)
 *
 * For callers that cannot call cudaMalloc: code that only receives device
 * pointers for its inputs and outputs from another framework and has no
 * allocator of its own, or that runs where every byte of device memory
 * belongs to a pool it does not control.  The (O, m, l) split partials go to
 * a file-scope device array of FA512_DECODE_STATIC_SCRATCH_BYTES that the
 * library holds on every GPU it is loaded on until the process exits.  The
 * call allocates nothing: no cudaMalloc, no cudaFree, no allocating library
 * routine.
 *
 * Arguments, layouts and errors are those of fa512_decode_paged.  A shape
 * whose partials need more than FA512_DECODE_STATIC_SCRATCH_BYTES
 * (fa512_decode_workspace_bytes) is rejected with FA512_ERR_WORKSPACE before
 * anything is enqueued; lower num_splits or the batch to fit.
 *
 * The first call on a device looks up the array's device address on that
 * device (cudaGetSymbolAddress, with that device current) and keeps it for
 * the life of the process; make that first call before any stream capture.
 * The kept address does not survive a device reset (cudaDeviceReset or a
 * reset of the primary context): do not use the library across one.  All calls share the one array and it
 * keeps the last call's contents; nothing in it has to start at zero, since
 * every split writes its whole partial before the merge reads it.  Calls
 * whose kernels overlap on the GPU (different streams, or different host
 * threads without ordering) race on the array: order them.
 */
#define FA512_DECODE_STATIC_SCRATCH_BYTES (32u * 1024u * 1024u)

fa512_status fa512_decode_paged_noalloc(const void *q, const void *k_pages,
                                        const void *v_pages, const int32_t *page_table,
                                        const int32_t *kv_lens, void *out, float *lse,
                                        int batch, int n_q_heads, int n_kv_heads, int page_size,
                                        int num_pages, int max_pages_per_seq, int max_kv_len,
                                        float scale, int window, int num_splits,
                                        fa512_stream_t stream);

/*
 * fa512_test_prefill_missing_load -- test hook, not a step of the method.
 * (The pages have no counterpart: it exists so that tests can drive the
 * kernels' bounded waits, which ordinary inputs never exhaust.)
 *
 * The same launch as fa512_prefill with the same arguments, except that
 * (a) every pipeline wait of the kernel is bounded by wait_limit_ns instead
 * of the default 2 s, and (b) the first CTA pair's even CTA does not issue
 * its first K tile load, so that pair's waits for it run into the bound.
 * The pair then records FA512_ERR_TIMEOUT in the device error word, drains
 * the MMAs it issued, frees its tensor memory and returns; CTAs that start
 * after the record skip their work.  The rows of the pair (and of skipped
 * CTAs) are left unwritten.  The device stays usable: read the status with
 * fa512_device_status(stream, 1) (which also clears it) before the next call.
 *
 * wait_limit_ns must lie in [1e6, 2e9] and seqlen_k must be >= 1
 * (FA512_ERR_INVALID_ARG otherwise); other errors as for fa512_prefill.
 */
fa512_status fa512_test_prefill_missing_load(const void *q, const void *k, const void *v,
                                             void *out, float *lse, int seqlen_q, int seqlen_k,
                                             int q_offset, int n_q_heads, int n_kv_heads,
                                             float scale, int causal, int window,
                                             uint64_t wait_limit_ns, fa512_stream_t stream);

/* Reads and optionally clears the device-side error word after
 * synchronising `stream`.  Returns FA512_OK, FA512_ERR_TIMEOUT,
 * FA512_ERR_DEVICE_INDEX or FA512_ERR_CUDA. */
fa512_status fa512_device_status(fa512_stream_t stream, int clear);

/* Static, human-readable name of a status code. */
const char *fa512_status_string(fa512_status status);

/* Detail of the last error returned on the calling thread (static storage,
 * overwritten by the next failing call). */
const char *fa512_last_error_message(void);

#ifdef __cplusplus
}
#endif

#endif /* FA512_H */

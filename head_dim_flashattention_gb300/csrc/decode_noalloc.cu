// Allocation-free variant of the paged decode entry point.
//
// fa512_decode_paged needs a caller-provided workspace for the per-split
// (O, m, l) partials.  Some callers cannot provide one: they only hold the
// device pointers another framework handed them (inputs and outputs) and have
// no way to call cudaMalloc themselves, or they run where every byte of HBM is
// owned by a pool they do not control.  For them this file keeps the partials
// in a fixed-size array in the library's own device memory.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds FA512_DECODE_STATIC_SCRATCH_BYTES of it until the process
// exits.  In host code its name is only a host-side stand-in; the device
// address is looked up once per device with cudaGetSymbolAddress.
#include <cuda_runtime.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "fa512.h"
#include "fa512_internal.h"

static __device__ __align__(256) unsigned char fa512_decode_static_scratch[FA512_DECODE_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices];

// Device address of the static scratch array on the current device; looked
// up on the first call made with that device current.
cudaError_t scratch_for_current_device(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, fa512_decode_static_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" fa512_status fa512_decode_paged_noalloc(
    const void* q, const void* k_pages, const void* v_pages, const int32_t* page_table,
    const int32_t* kv_lens, void* out, float* lse, int batch, int n_q_heads, int n_kv_heads,
    int page_size, int num_pages, int max_pages_per_seq, int max_kv_len, float scale, int window,
    int num_splits, fa512_stream_t stream) {
    if (batch > 0) {
        const size_t need = fa512_decode_workspace_bytes(batch, n_q_heads, n_kv_heads, page_size,
                                                         max_kv_len, num_splits);
        if (need > FA512_DECODE_STATIC_SCRATCH_BYTES) {
            char msg[256];
            snprintf(msg, sizeof msg,
                     "this shape needs %zu bytes of split scratch, the static array holds %zu; "
                     "use fewer splits or a smaller batch, or fa512_decode_paged with a workspace",
                     need, static_cast<size_t>(FA512_DECODE_STATIC_SCRATCH_BYTES));
            fa512::set_last_error_message(msg);
            return FA512_ERR_WORKSPACE;
        }
    }
    void* scratch = nullptr;
    cudaError_t e = scratch_for_current_device(&scratch);
    if (e != cudaSuccess) {
        char msg[256];
        snprintf(msg, sizeof msg, "cudaGetSymbolAddress of the static scratch: %s",
                 cudaGetErrorString(e));
        fa512::set_last_error_message(msg);
        return FA512_ERR_CUDA;
    }
    return fa512_decode_paged(q, k_pages, v_pages, page_table, kv_lens, out, lse, batch,
                              n_q_heads, n_kv_heads, page_size, num_pages, max_pages_per_seq,
                              max_kv_len, scale, window, num_splits, scratch,
                              static_cast<size_t>(FA512_DECODE_STATIC_SCRATCH_BYTES), stream);
}

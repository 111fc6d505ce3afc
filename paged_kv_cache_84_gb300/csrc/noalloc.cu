// Ragged paged attention for callers that cannot allocate device memory.
//
// pkv_ragged_paged_attention needs a caller workspace for its split-KV
// partials, split counters and device error word.  Some callers have no way
// to provide one: plain C hosts that have no device allocator of their own,
// and serving loops that must not call cudaMalloc because it can
// synchronise the whole device or because their device memory budget is
// fixed when they start.  This entry point uses a fixed scratch array that
// lives in the library's own device image instead.  The paged-attention
// pages have no counterpart of it: it is an interface convenience only.
//
// The scratch is a file-scope __device__ array.  Host code cannot use its
// name as a device address (on the host it names a shadow variable), so the
// address is fetched once per device with cudaGetSymbolAddress, with that
// device current, on the first call made on that device.
#include <mutex>

#include "pkv.h"
#include "common.cuh"

namespace {

constexpr size_t kScratchBytes = PKV_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;
// what must be zero when a call starts: the error word area and the split
// counters (a call that ended early may have left either dirty)
constexpr size_t kZeroPrefix = pkv::kErrBytes + pkv::kCounterBytes;
static_assert(kScratchBytes >= PKV_WORKSPACE_MIN_BYTES && kScratchBytes > kZeroPrefix + 4096,
              "the scratch array must hold the error word, the counters and some partials");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array for the current device (set up once).
pkv_status scratch_for_current_device(void **ptr)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PKV_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) return PKV_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *ptr = g_scratch_ptr[dev];
    return PKV_OK;
}

}  // namespace

extern "C" size_t pkv_noalloc_scratch_bytes(void) { return kScratchBytes; }

extern "C" pkv_status pkv_ragged_paged_attention_noalloc(
    void *out, const void *q, const void *k_cache, const void *v_cache, const int32_t *query_start_loc,
    const int32_t *seq_lens, const int32_t *block_table, int32_t block_table_stride,
    const int32_t *query_start_loc_host, const int32_t *seq_lens_host, int32_t num_reqs, int32_t num_tokens,
    int32_t max_query_len, int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
    int32_t block_size, int32_t num_blocks_total, float scale, int32_t window, uint32_t *device_error,
    cudaStream_t stream)
{
    void *scratch = nullptr;
    pkv_status st = scratch_for_current_device(&scratch);
    if (st != PKV_OK) return st;

    // Size check on the host, before anything is enqueued: the planner fits
    // the split-KV partials into the array (it lengthens the splits until
    // they fit), so every batch the workspace entry point accepts fits; a
    // plan that would not fit is refused rather than run.
    if (num_tokens > 0) {
        pkv_attention_plan plan;
        st = pkv_plan_attention(query_start_loc_host, seq_lens_host, num_reqs, num_q_heads, num_kv_heads, head_dim,
                                block_size, window, 0, 0, kScratchBytes, 0, nullptr, &plan);
        if (st != PKV_OK) return st;
        const size_t front = plan.split_counters ? kZeroPrefix : pkv::kErrBytes;
        if (plan.partial_bytes > kScratchBytes - front - 64) return PKV_ERR_WORKSPACE;
    }

    // Every call starts from a zero error word and zero counters, whatever
    // an earlier call left there.
    cudaError_t e = cudaMemsetAsync(scratch, 0, kZeroPrefix, stream);
    if (e != cudaSuccess) return PKV_ERR_CUDA;
    st = pkv_ragged_paged_attention(out, q, k_cache, v_cache, query_start_loc, seq_lens, block_table,
                                    block_table_stride, query_start_loc_host, seq_lens_host, num_reqs,
                                    num_tokens, max_query_len, max_seq_len, num_q_heads, num_kv_heads,
                                    head_dim, block_size, num_blocks_total, scale, window, scratch,
                                    kScratchBytes, stream);
    if (st != PKV_OK) return st;
    if (device_error)
        e = cudaMemcpyAsync(device_error, scratch, sizeof(uint32_t), cudaMemcpyDeviceToDevice, stream);
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

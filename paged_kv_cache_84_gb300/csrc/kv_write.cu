// paged_kv_write: scatter one step's K/V rows into the block pool.
//
// "31. Engine v2: one core for every request", "Attention over the pool"
// (write_kv): row i of k and v goes to flat pool slot slot_mapping[i]; a
// negative slot marks a padding row and goes to the pool's last slot, the
// scratch block.  A bit copy: 16-byte vectors, one per thread, the K and the
// V chunk of the same offset handled together.
#include "common.cuh"
#include "sm100.cuh"

namespace pkv {

__global__ void __launch_bounds__(256) kv_write_kernel(
    const uint4 *__restrict__ k, const uint4 *__restrict__ v, uint4 *__restrict__ k_cache,
    uint4 *__restrict__ v_cache, const int64_t *__restrict__ slot_mapping, int64_t total_chunks,
    int32_t chunks_per_row, int64_t num_slots, uint32_t *err)
{
    // Launched as a programmatic dependent: wait for the kernel before it
    // (which may produce k, v or the slot mapping), then let the attention
    // kernel start its set-up.  Nothing runs ahead of this kernel's own wait.
    pdl_wait();
    pdl_launch_dependents();
    int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c < total_chunks; c += stride) {
        int64_t row = c / chunks_per_row;
        int32_t off = (int32_t)(c - row * chunks_per_row);
        // the slot and the row's data are independent loads: issue them together
        int64_t slot = __ldg(slot_mapping + row);
        uint4 kv = ldg_nc_v4(k + c);
        uint4 vv = ldg_nc_v4(v + c);
        if (slot < 0) slot = num_slots - 1;                 // padding row -> scratch slot
        if (slot >= num_slots) {                            // outside the pool: skip, report
            if (off == 0 && err) atomicOr(err, 1u);
            continue;
        }
        int64_t dst = slot * chunks_per_row + off;
        k_cache[dst] = kv;
        v_cache[dst] = vv;
    }
}

cudaError_t launch_kv_write(const void *k, const void *v, void *k_cache, void *v_cache,
                            const int64_t *slot_mapping, int32_t num_tokens, int32_t row_bytes,
                            int64_t num_slots, uint32_t *err, cudaStream_t stream)
{
    int32_t chunks_per_row = row_bytes / 16;
    int64_t total = (int64_t)num_tokens * chunks_per_row;
    int threads = 256;
    int64_t blocks = (total + threads - 1) / threads;
    if (blocks > 152 * 32) blocks = 152 * 32;               // grid-stride beyond 32 CTAs per SM
    launch_begin(stream, kKvWrite);
    cudaError_t e = launch_maybe_pdl(kv_write_kernel, dim3((unsigned)blocks), dim3(threads), 0, stream,
                                     (const uint4 *)k, (const uint4 *)v, (uint4 *)k_cache, (uint4 *)v_cache,
                                     slot_mapping, total, chunks_per_row, num_slots, err);
    launch_end(stream);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace pkv

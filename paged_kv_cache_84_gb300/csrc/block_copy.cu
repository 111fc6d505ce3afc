// Block copies of the block manager, on every pool of a model at once.
//
// "vllm-lite README": blocks are reference counted and a write into a block
// that two sequences share is preceded by a copy of it (copy-on-write),
// which the runner performs before the forward pass.  "31. Engine v2",
// "Preemption: recompute or swap": swap-out copies a preempted request's
// blocks of every layer's K and V (and scales, when quantized) to host
// memory; swap-in copies them into newly allocated blocks before the step.
//
// A pool is num_blocks_total blocks of block_bytes bytes (slot-major block
// layout, so a block is one contiguous byte range).  One launch covers all
// pools and all listed blocks: each thread moves four independent 16-byte
// vectors per iteration (four loads in flight before the stores).
#include <algorithm>
#include <cstdlib>

#include "common.cuh"
#include "sm100.cuh"

namespace pkv {

struct PoolList {
    char *p[kMaxPools];
};

// mode 0: copy block src[i] -> dst[i] inside every pool; 1: gather block
// ids[i] of pool q -> buf[q][i]; 2: scatter buf[q][i] -> block ids[i] of pool q
template <int MODE>
__global__ void __launch_bounds__(256) block_copy_kernel(const __grid_constant__ PoolList pools, int32_t num_pools,
                                                         const int32_t *__restrict__ src, const int32_t *__restrict__ dst,
                                                         int32_t n, int32_t nb_total, int64_t chunks_per_block,
                                                         char *buf, uint32_t *err)
{
    pdl_wait();                                                   // block ids / data may come from the kernel before
    pdl_launch_dependents();
    const int64_t per_pool = (int64_t)n * chunks_per_block;
    const int64_t total = per_pool * num_pools;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t c0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c0 < total; c0 += 4 * stride) {
        uint4 v[4];
        uint4 *to[4];
#pragma unroll
        for (int u = 0; u < 4; u++) {
            to[u] = nullptr;
            const int64_t c = c0 + u * stride;
            if (c >= total) continue;
            const int32_t q = (int32_t)(c / per_pool);
            const int64_t r = c - (int64_t)q * per_pool;
            const int32_t i = (int32_t)(r / chunks_per_block);
            const int64_t off = r - (int64_t)i * chunks_per_block;
            const uint4 *from;
            if (MODE == 0) {
                const int32_t s = __ldg(src + i), d = __ldg(dst + i);
                if (s < 0 || s >= nb_total || d < 0 || d >= nb_total) {
                    if (off == 0 && q == 0 && err) atomicOr(err, 2u);
                    continue;
                }
                from = reinterpret_cast<const uint4 *>(pools.p[q]) + (int64_t)s * chunks_per_block + off;
                to[u] = reinterpret_cast<uint4 *>(pools.p[q]) + (int64_t)d * chunks_per_block + off;
            } else {
                const int32_t b = __ldg(src + i);
                if (b < 0 || b >= nb_total) {
                    if (off == 0 && q == 0 && err) atomicOr(err, 2u);
                    continue;
                }
                uint4 *blk = reinterpret_cast<uint4 *>(pools.p[q]) + (int64_t)b * chunks_per_block + off;
                uint4 *flat = reinterpret_cast<uint4 *>(buf) + c;    // [pool][i][chunk]
                from = MODE == 1 ? blk : flat;
                to[u] = MODE == 1 ? flat : blk;
            }
            v[u] = *from;
        }
#pragma unroll
        for (int u = 0; u < 4; u++)
            if (to[u]) *to[u] = v[u];
    }
}

cudaError_t launch_block_copy(int mode, void *const *pools, int32_t num_pools, const int32_t *src,
                              const int32_t *dst, int32_t n, int32_t nb_total, int64_t block_bytes, void *buf,
                              uint32_t *err, cudaStream_t stream)
{
    if (n <= 0 || num_pools <= 0) return cudaSuccess;
    PoolList pl;
    for (int q = 0; q < kMaxPools; q++) pl.p[q] = q < num_pools ? static_cast<char *>(pools[q]) : nullptr;
    const int64_t cpb = block_bytes / 16;
    const int64_t total = cpb * n * num_pools;
    int64_t blocks = (total + 4 * 256 - 1) / (4 * 256);
    if (blocks > 152 * 16) blocks = 152 * 16;                     // grid-stride beyond 16 CTAs per SM
    launch_begin(stream, kBlockCopy);
    cudaError_t e;
    char *b = static_cast<char *>(buf);
    switch (mode) {
    case 0: e = launch_maybe_pdl(block_copy_kernel<0>, dim3((unsigned)blocks), dim3(256), 0, stream, pl, num_pools, src, dst, n, nb_total, cpb, b, err); break;
    case 1: e = launch_maybe_pdl(block_copy_kernel<1>, dim3((unsigned)blocks), dim3(256), 0, stream, pl, num_pools, src, dst, n, nb_total, cpb, b, err); break;
    default: e = launch_maybe_pdl(block_copy_kernel<2>, dim3((unsigned)blocks), dim3(256), 0, stream, pl, num_pools, src, dst, n, nb_total, cpb, b, err); break;
    }
    launch_end(stream);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// A plain copy of `chunks` 16-byte vectors (pkv_copy_async): staging a
// step's packed inputs from pinned host memory, or reading its output back.
// Either side may be pinned host memory the device addresses directly, so
// the copy is a kernel like the attention launches around it (no copy-engine
// operation in the stream).  U independent vectors per thread and iteration
// are in flight at once.
template <int U, int T>
__global__ void __launch_bounds__(T) byte_copy_kernel(uint4 *dst, const uint4 *src, int64_t chunks)
{
    pdl_wait();                                                   // the source may come from the kernel before
    pdl_launch_dependents();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t c0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c0 < chunks; c0 += U * stride) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; u++)
            if (c0 + u * stride < chunks) v[u] = src[c0 + u * stride];
#pragma unroll
        for (int u = 0; u < U; u++)
            if (c0 + u * stride < chunks) dst[c0 + u * stride] = v[u];
    }
}

static bool is_host_memory(const void *ptr)
{
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeHost;
}

// CTAs for a copy that crosses the host link.  A dozen CTAs of 256 threads
// with 8 vectors each in flight (~390 KB) carry ~360 GB/s from pinned host
// memory.  More CTAs barely raise that rate but slow the attention kernels
// that run beside the copy (the next step's inputs staged while this step
// computes): with the copy spread over 72 CTAs or 152 x 16, the mixed
// 2048-token-chunk step with its copies overlapped took 875 us against 575 us
// with 12 CTAs (511 us without copies), and the 48-request engine step 14.3
// against 11.4 us (10.3 us without copies).
constexpr int kLinkCopyCtas = 12;

// A copy across the link of kDmaCopyBytes or more goes to the copy engine
// instead: it then takes no SM from attention launched beside it, whose CTAs
// may hold whole SMs (a tcgen05 launch: 384 threads x 168 registers), and
// its hand-off cost (a few us between a copy-engine operation and a kernel)
// is small against its duration.  Measured with the mixed 2048-token-chunk
// step's 51 MB of inputs and 34 MB of output overlapped with other steps.
constexpr size_t kDmaCopyBytes = 8u << 20;

cudaError_t launch_byte_copy(void *dst, const void *src, size_t bytes, cudaStream_t stream)
{
    const int64_t chunks = (int64_t)(bytes / 16);
    if (chunks <= 0) return cudaSuccess;
    const bool link = is_host_memory(dst) || is_host_memory(src);
    if (link && bytes >= kDmaCopyBytes) return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDefault, stream);
    cudaError_t e;
    launch_begin(stream, kByteCopy);
    if (link) {
        int64_t blocks = (chunks + 8 * 256 - 1) / (8 * 256);
        blocks = std::min<int64_t>(blocks, kLinkCopyCtas);
        e = launch_maybe_pdl(byte_copy_kernel<8, 256>, dim3((unsigned)blocks), dim3(256), 0, stream,
                             static_cast<uint4 *>(dst), static_cast<const uint4 *>(src), chunks);
    } else {
        int64_t blocks = (chunks + 4 * 256 - 1) / (4 * 256);
        blocks = std::min<int64_t>(blocks, 152 * 16);             // grid-stride beyond 16 CTAs per SM
        e = launch_maybe_pdl(byte_copy_kernel<4, 256>, dim3((unsigned)blocks), dim3(256), 0, stream,
                             static_cast<uint4 *>(dst), static_cast<const uint4 *>(src), chunks);
    }
    launch_end(stream);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace pkv

// paged_kv_write: scatter one step's K/V rows into the block pool.
//
// "31. Engine v2: one core for every request", "Attention over the pool"
// (write_kv): row i of k and v goes to flat pool slot slot_mapping[i]; a
// negative slot marks a padding row and goes to the pool's last slot, the
// scratch block.  A bit copy: 16-byte vectors, one per thread, the K and the
// V chunk of the same offset handled together.
#include <algorithm>
#include <mutex>

#include <cuda_fp8.h>

#include "common.cuh"
#include "sm100.cuh"

namespace pkv {

// 8 E4M3 codes (bytes of x, low first) times `scale`, as 8 bf16 rounded to
// nearest: every E4M3 value converts to half exactly, the product is fp32.
__device__ __forceinline__ uint4 e4m3x8_to_bf16x8(uint2 x, float scale)
{
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; q++) {
        const uint32_t word = q < 2 ? x.x : x.y;
        const __nv_fp8x2_storage_t pair = (__nv_fp8x2_storage_t)((word >> (16 * (q & 1))) & 0xFFFFu);
        const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3);
        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&hr));
        w[q] = pack_bf16x2(f.x * scale, f.y * scale);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

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

// Quantizing write for FP8 pools (head_dim 128): one warp per (row, KV
// head); lane l holds dims 4l .. 4l+3 of K and of V.  Per row and head:
// scale = max |x| / 448 (fp32), codes = E4M3(x / scale) rounded to nearest
// even with saturation ("31. Engine v2", "Attention over the pool": the
// quantized pool's per (slot, head) scales; the code format is this
// library's reading).  An all-zero row gets scale 0 and zero codes.
__global__ void __launch_bounds__(256) kv_write_fp8_kernel(
    const uint2 *__restrict__ k, const uint2 *__restrict__ v, uint32_t *__restrict__ k_codes,
    uint32_t *__restrict__ v_codes, float *__restrict__ k_scale, float *__restrict__ v_scale,
    const int64_t *__restrict__ slot_mapping, int64_t rows, int32_t hkv, int64_t num_slots, uint32_t *err)
{
    pdl_wait();                                           // as the bf16 write: nothing is read before this
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); w < rows; w += nwarps) {
        const int64_t i = w / hkv;                        // token row; w = i * hkv + head
        int64_t slot = __ldg(slot_mapping + i);
        const uint2 kx = k[w * 32 + lane], vx = v[w * 32 + lane];   // 4 bf16 each
        if (slot < 0) slot = num_slots - 1;               // padding row -> scratch slot
        if (slot >= num_slots) {
            if (lane == 0 && w % hkv == 0 && err) atomicOr(err, 1u);
            continue;
        }
        const int64_t dst_row = slot * hkv + (w - i * hkv);
#pragma unroll
        for (int which = 0; which < 2; which++) {
            float scale;
            const uint32_t codes = quantize_e4m3_row(which ? vx : kx, scale);
            (which ? v_codes : k_codes)[dst_row * 32 + lane] = codes;
            if (lane == 0) (which ? v_scale : k_scale)[dst_row] = scale;
        }
    }
}

// The quantizing scatter restricted to token ranges (the prefill rows of a
// combined call on a quantized pool): warp w takes (row, head) w of the
// ranges' rows.
__global__ void __launch_bounds__(256) kv_write_fp8_ranges_kernel(
    const uint2 *__restrict__ k, const uint2 *__restrict__ v, uint32_t *__restrict__ k_codes,
    uint32_t *__restrict__ v_codes, float *__restrict__ k_scale, float *__restrict__ v_scale,
    const int64_t *__restrict__ slot_mapping, const __grid_constant__ TokenRanges rg, int32_t hkv, int64_t num_slots,
    uint32_t *err)
{
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t rows = (int64_t)rg.off[rg.n] * hkv;
    const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); w < rows; w += nwarps) {
        const int32_t ri = (int32_t)(w / hkv), h = (int32_t)(w - (int64_t)ri * hkv);
        int lo = 0, hi = rg.n - 1;
        while (lo < hi) {                                 // the range holding row ri
            const int mid = (lo + hi + 1) >> 1;
            if (rg.off[mid] <= ri) lo = mid; else hi = mid - 1;
        }
        const int64_t row = (int64_t)rg.begin[lo] + (ri - rg.off[lo]);
        int64_t slot = __ldg(slot_mapping + row);
        const uint2 kx = k[(row * hkv + h) * 32 + lane], vx = v[(row * hkv + h) * 32 + lane];
        if (slot < 0) slot = num_slots - 1;
        if (slot >= num_slots) {
            if (lane == 0 && h == 0 && err) atomicOr(err, 1u);
            continue;
        }
        const int64_t dst = slot * hkv + h;
        float ks, vs;
        const uint32_t kq = quantize_e4m3_row(kx, ks), vq = quantize_e4m3_row(vx, vs);
        k_codes[dst * 32 + lane] = kq;
        v_codes[dst * 32 + lane] = vq;
        if (lane == 0) {
            k_scale[dst] = ks;
            v_scale[dst] = vs;
        }
    }
}

cudaError_t launch_kv_write_fp8_ranges(const void *k, const void *v, void *k_codes, void *v_codes, float *k_scale,
                                       float *v_scale, const int64_t *slot_mapping, const TokenRanges &ranges,
                                       int32_t hkv, int64_t num_slots, uint32_t *err, cudaStream_t stream)
{
    const int64_t rows = (int64_t)ranges.off[ranges.n] * hkv;
    if (rows <= 0) return cudaSuccess;
    int64_t blocks = (rows + 7) / 8;
    if (blocks > 152 * 16) blocks = 152 * 16;
    launch_begin(stream, kKvWrite);
    cudaError_t e = launch_maybe_pdl(kv_write_fp8_ranges_kernel, dim3((unsigned)blocks), dim3(256), 0, stream,
                                     (const uint2 *)k, (const uint2 *)v, (uint32_t *)k_codes, (uint32_t *)v_codes,
                                     k_scale, v_scale, slot_mapping, ranges, hkv, num_slots, err);
    launch_end(stream);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// The scatter restricted to token ranges (a combined write + attention
// call: the decode-class CTAs write their own rows, this kernel the rows of
// the prefill-class requests).  Chunk c of the ranges' rows maps to token
// begin[q] + (c / chunks_per_row - off[q]) of the range q that holds it.
__global__ void __launch_bounds__(256) kv_write_ranges_kernel(
    const uint4 *__restrict__ k, const uint4 *__restrict__ v, uint4 *__restrict__ k_cache,
    uint4 *__restrict__ v_cache, const int64_t *__restrict__ slot_mapping, const __grid_constant__ TokenRanges rg,
    int32_t chunks_per_row, int64_t num_slots, uint32_t *err)
{
    pdl_wait();                                           // as the full scatter: nothing is read before this
    pdl_launch_dependents();
    const int64_t total = (int64_t)rg.off[rg.n] * chunks_per_row;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c < total; c += stride) {
        const int32_t ri = (int32_t)(c / chunks_per_row);  // row among the ranges' rows
        const int32_t off = (int32_t)(c - (int64_t)ri * chunks_per_row);
        int lo = 0, hi = rg.n - 1;
        while (lo < hi) {                                 // the range holding row ri
            const int mid = (lo + hi + 1) >> 1;
            if (rg.off[mid] <= ri) lo = mid; else hi = mid - 1;
        }
        const int64_t row = (int64_t)rg.begin[lo] + (ri - rg.off[lo]);
        int64_t slot = __ldg(slot_mapping + row);
        const int64_t src = row * chunks_per_row + off;
        const uint4 kv = ldg_nc_v4(k + src), vv = ldg_nc_v4(v + src);
        if (slot < 0) slot = num_slots - 1;               // padding row -> scratch slot
        if (slot >= num_slots) {
            if (off == 0 && err) atomicOr(err, 1u);
            continue;
        }
        const int64_t dst = slot * chunks_per_row + off;
        k_cache[dst] = kv;
        v_cache[dst] = vv;
    }
}

cudaError_t launch_kv_write_ranges(const void *k, const void *v, void *k_cache, void *v_cache,
                                   const int64_t *slot_mapping, const TokenRanges &ranges, int32_t row_bytes,
                                   int64_t num_slots, uint32_t *err, cudaStream_t stream)
{
    const int32_t chunks_per_row = row_bytes / 16;
    const int64_t total = (int64_t)ranges.off[ranges.n] * chunks_per_row;
    if (total <= 0) return cudaSuccess;
    int64_t blocks = (total + 255) / 256;
    if (blocks > 152 * 32) blocks = 152 * 32;
    launch_begin(stream, kKvWrite);
    cudaError_t e = launch_maybe_pdl(kv_write_ranges_kernel, dim3((unsigned)blocks), dim3(256), 0, stream,
                                     (const uint4 *)k, (const uint4 *)v, (uint4 *)k_cache, (uint4 *)v_cache,
                                     slot_mapping, ranges, chunks_per_row, num_slots, err);
    launch_end(stream);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// Quantized-pool prefill on the tcgen05 kernel: the listed requests' blocks
// (block i < ceil(L / 16) of request wl.req[li] goes to scratch block
// sblk0 + item_off[li] + i) as bf16 K and V = code * scale, rounded to nearest, in a
// scratch pool [blocks][16][hkv][128] with a scratch block table
// (table_out[r][i] = the scratch block); rows at positions >= L become
// zeros.  A block id outside the pool is reported (bit 2) and its rows
// become zeros.  One CTA per scratch block (grid-stride): the request and
// the block index come from one search of the list per block; each thread
// then converts 16-code chunks (a chunk lies in one (slot, head) row, so one
// scale load serves 16 codes), kDequantBatch chunks of K and of V loaded
// before any is converted, so that their loads are in flight together.
constexpr int kDequantThreads = 128;
constexpr int kDequantBatch = 4;

__global__ void __launch_bounds__(kDequantThreads) fp8_dequant_kernel(AttnParams p, const __grid_constant__ WorkList wl,
                                                                      uint4 *__restrict__ k_out,
                                                                      uint4 *__restrict__ v_out,
                                                                      int32_t *__restrict__ table_out,
                                                                      int32_t table_stride, int32_t sblk0)
{
    pdl_wait();                                           // the step's codes are in the pool
    pdl_launch_dependents();
    const int hkv = p.hkv;
    const int chunks = 16 * hkv * 8;                      // 16-code chunks of a block's K (or V) codes
    const int nblocks = wl.item_off[wl.n];
    const uint4 *kc = reinterpret_cast<const uint4 *>(p.k_cache);
    const uint4 *vc = reinterpret_cast<const uint4 *>(p.v_cache);
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    for (int lblk = blockIdx.x; lblk < nblocks; lblk += gridDim.x) {
        const int li = find_listed(wl, lblk);
        const int r = wl.req[li], i = lblk - wl.item_off[li];
        const int64_t sbase = (int64_t)(sblk0 + lblk) * 16 * hkv;    // first (slot, head) row of the scratch block
        if (threadIdx.x == 0) table_out[(size_t)r * table_stride + i] = sblk0 + lblk;
        const int blk = __ldg(p.block_table + (size_t)r * p.bt_stride + i);
        const bool in_pool = blk >= 0 && blk < p.nb_total;
        if (!in_pool && threadIdx.x == 0) atomicOr(p.err, 2u);
        const int valid_rows = in_pool ? min(16, wl.len[li] - i * 16) * hkv : 0;   // (slot, head) rows to convert
        const int64_t pbase = (int64_t)(in_pool ? blk : 0) * 16 * hkv;              // ... in the pool
        for (int c0 = threadIdx.x; c0 < chunks; c0 += kDequantBatch * kDequantThreads) {
            uint4 kx[kDequantBatch], vx[kDequantBatch];
            float ks[kDequantBatch], vs[kDequantBatch];
#pragma unroll
            for (int u = 0; u < kDequantBatch; u++) {
                const int c = c0 + u * kDequantThreads;
                const int rowh = c >> 3;
                kx[u] = vx[u] = zero;
                ks[u] = vs[u] = 0.f;
                if (c < chunks && rowh < valid_rows) {
                    const int64_t row = pbase + rowh;
                    kx[u] = __ldg(kc + row * 8 + (c & 7));
                    vx[u] = __ldg(vc + row * 8 + (c & 7));
                    ks[u] = __ldg(p.k_scale + row);
                    vs[u] = __ldg(p.v_scale + row);
                }
            }
#pragma unroll
            for (int u = 0; u < kDequantBatch; u++) {
                const int c = c0 + u * kDequantThreads;
                if (c >= chunks) break;
                const int rowh = c >> 3;
                const int64_t dst = (sbase + rowh) * 16 + (c & 7) * 2;   // 16-byte vectors of bf16 rows
                const bool ok = rowh < valid_rows;
                k_out[dst] = ok ? e4m3x8_to_bf16x8(make_uint2(kx[u].x, kx[u].y), ks[u]) : zero;
                k_out[dst + 1] = ok ? e4m3x8_to_bf16x8(make_uint2(kx[u].z, kx[u].w), ks[u]) : zero;
                v_out[dst] = ok ? e4m3x8_to_bf16x8(make_uint2(vx[u].x, vx[u].y), vs[u]) : zero;
                v_out[dst + 1] = ok ? e4m3x8_to_bf16x8(make_uint2(vx[u].z, vx[u].w), vs[u]) : zero;
            }
        }
    }
}

// The same with the block's bf16 rows assembled in shared memory (K, then
// V: 16 x hkv rows of 256 bytes each) and written out as two bulk copies of
// the whole scratch block, which is contiguous: the threads' 32-byte row
// pieces become two copies of 4 KB x hkv instead of 16-byte stores at a
// 32-byte stride.  A CTA takes blocks in turn; before it overwrites its
// shared rows, the copies of the block before have read them.
constexpr int kDequantSmemMax = 192 * 1024;

__global__ void __launch_bounds__(kDequantThreads) fp8_dequant_staged_kernel(AttnParams p,
                                                                             const __grid_constant__ WorkList wl,
                                                                             uint4 *__restrict__ k_out,
                                                                             uint4 *__restrict__ v_out,
                                                                             int32_t *__restrict__ table_out,
                                                                             int32_t table_stride, int32_t sblk0)
{
    extern __shared__ __align__(128) uint4 rows_s[];      // [2][16 * hkv * 16] 16-byte vectors
    pdl_wait();                                           // the step's codes are in the pool
    pdl_launch_dependents();
    const int hkv = p.hkv;
    const int chunks = 16 * hkv * 8;                      // 16-code chunks of a block's K (or V) codes
    const int vecs = 16 * hkv * 16;                       // 16-byte vectors of a block's bf16 K (or V)
    const int nblocks = wl.item_off[wl.n];
    const uint4 *kc = reinterpret_cast<const uint4 *>(p.k_cache);
    const uint4 *vc = reinterpret_cast<const uint4 *>(p.v_cache);
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    uint4 *ks_rows = rows_s, *vs_rows = rows_s + vecs;
    for (int lblk = blockIdx.x; lblk < nblocks; lblk += gridDim.x) {
        const int li = find_listed(wl, lblk);
        const int r = wl.req[li], i = lblk - wl.item_off[li];
        const int64_t sbase = (int64_t)(sblk0 + lblk) * 16 * hkv;    // first (slot, head) row of the scratch block
        if (threadIdx.x == 0) table_out[(size_t)r * table_stride + i] = sblk0 + lblk;
        const int blk = __ldg(p.block_table + (size_t)r * p.bt_stride + i);
        const bool in_pool = blk >= 0 && blk < p.nb_total;
        if (!in_pool && threadIdx.x == 0) atomicOr(p.err, 2u);
        const int valid_rows = in_pool ? min(16, wl.len[li] - i * 16) * hkv : 0;   // (slot, head) rows to convert
        const int64_t pbase = (int64_t)(in_pool ? blk : 0) * 16 * hkv;              // ... in the pool
        for (int c0 = threadIdx.x, pass = 0; c0 < chunks; c0 += kDequantBatch * kDequantThreads, pass++) {
            uint4 kx[kDequantBatch], vx[kDequantBatch];
            float ks[kDequantBatch], vs[kDequantBatch];
#pragma unroll
            for (int u = 0; u < kDequantBatch; u++) {
                const int c = c0 + u * kDequantThreads;
                const int rowh = c >> 3;
                kx[u] = vx[u] = zero;
                ks[u] = vs[u] = 0.f;
                if (c < chunks && rowh < valid_rows) {
                    const int64_t row = pbase + rowh;
                    kx[u] = __ldg(kc + row * 8 + (c & 7));
                    vx[u] = __ldg(vc + row * 8 + (c & 7));
                    ks[u] = __ldg(p.k_scale + row);
                    vs[u] = __ldg(p.v_scale + row);
                }
            }
            if (pass == 0) {                                  // the previous block's copies have read the rows
                if (threadIdx.x == 0) bulk_wait_read();
                __syncthreads();
            }
#pragma unroll
            for (int u = 0; u < kDequantBatch; u++) {
                const int c = c0 + u * kDequantThreads;
                if (c >= chunks) break;
                const int v = (c >> 3) * 16 + (c & 7) * 2;        // 16-byte vector of the block's rows
                const bool ok = (c >> 3) < valid_rows;
                ks_rows[v] = ok ? e4m3x8_to_bf16x8(make_uint2(kx[u].x, kx[u].y), ks[u]) : zero;
                ks_rows[v + 1] = ok ? e4m3x8_to_bf16x8(make_uint2(kx[u].z, kx[u].w), ks[u]) : zero;
                vs_rows[v] = ok ? e4m3x8_to_bf16x8(make_uint2(vx[u].x, vx[u].y), vs[u]) : zero;
                vs_rows[v + 1] = ok ? e4m3x8_to_bf16x8(make_uint2(vx[u].z, vx[u].w), vs[u]) : zero;
            }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // the rows, visible to the bulk copies
        __syncthreads();
        if (threadIdx.x == 0) {
            bulk_store(k_out + sbase * 16, smem_u32(ks_rows), (uint32_t)vecs * 16);
            bulk_store(v_out + sbase * 16, smem_u32(vs_rows), (uint32_t)vecs * 16);
            bulk_commit();
        }
    }
    if (threadIdx.x == 0) bulk_wait_all();                   // the copies are done before the grid is
}

cudaError_t launch_fp8_dequant(const AttnParams &p, const WorkList &wl, __nv_bfloat16 *k_out, __nv_bfloat16 *v_out,
                               int32_t *table_out, int32_t table_stride, int32_t sblk0, cudaStream_t stream)
{
    const int64_t nblocks = wl.item_off[wl.n];
    if (nblocks <= 0) return cudaSuccess;
    const int smem = 2 * 16 * p.hkv * 256;                // bf16 K and V rows of one block
    cudaError_t e;
    launch_begin(stream, kFp8Dequant);
    if (smem <= kDequantSmemMax) {
        static std::once_flag once;
        static cudaError_t attr_err = cudaSuccess;
        std::call_once(once, [] {
            attr_err = cudaFuncSetAttribute(fp8_dequant_staged_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            kDequantSmemMax);
        });
        if (attr_err != cudaSuccess) {
            launch_end(stream);
            return attr_err;
        }
        const int per_sm = std::max(1, std::min(16, 220 * 1024 / (smem + 1024)));
        const int64_t grid = std::min<int64_t>(nblocks, (int64_t)152 * per_sm);
        e = launch_maybe_pdl(fp8_dequant_staged_kernel, dim3((unsigned)grid), dim3(kDequantThreads), (size_t)smem,
                             stream, p, wl, reinterpret_cast<uint4 *>(k_out), reinterpret_cast<uint4 *>(v_out),
                             table_out, table_stride, sblk0);
    } else {
        const int64_t grid = nblocks < 152 * 64 ? nblocks : 152 * 64;
        e = launch_maybe_pdl(fp8_dequant_kernel, dim3((unsigned)grid), dim3(kDequantThreads), 0, stream, p, wl,
                             reinterpret_cast<uint4 *>(k_out), reinterpret_cast<uint4 *>(v_out), table_out,
                             table_stride, sblk0);
    }
    launch_end(stream);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// Pools of blocks of 16 << shift slots are pools of blocks of 16 slots, as
// many times more of them ("31. Engine v2", "Attention over the pool": key j
// in slot table[j / block_size] * block_size + j % block_size): entry j of
// request r's row in 16-slot blocks is (table[r][j >> shift] << shift) +
// (j & (2^shift - 1)).  An id outside the pool becomes -1, which the
// attention kernels report (PKV_DEVERR_BLOCK) and do not read.
__global__ void __launch_bounds__(256) expand_table_kernel(const int32_t *__restrict__ bt, int32_t stride,
                                                           int32_t *__restrict__ bt16, int32_t w16, int64_t total,
                                                           int32_t shift, int32_t nb_total)
{
    pdl_wait();                                           // the table may come from the kernel before
    const int64_t step = (int64_t)gridDim.x * blockDim.x;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += step) {
        const int64_t r = idx / w16;
        const int j = (int)(idx - r * w16);
        const int b = __ldg(bt + r * stride + (j >> shift));
        bt16[idx] = (b < 0 || b >= nb_total) ? -1 : (b << shift) + (j & ((1 << shift) - 1));
    }
}

cudaError_t launch_expand_table(const int32_t *bt, int32_t stride, int32_t *bt16, int32_t w16, int32_t num_reqs,
                                int32_t shift, int32_t nb_total, cudaStream_t stream)
{
    const int64_t total = (int64_t)num_reqs * w16;
    if (total <= 0) return cudaSuccess;
    int64_t blocks = (total + 255) / 256;
    if (blocks > 152 * 8) blocks = 152 * 8;
    launch_begin(stream, kTableExpand);
    cudaError_t e = launch_maybe_pdl(expand_table_kernel, dim3((unsigned)blocks), dim3(256), 0, stream, bt, stride,
                                     bt16, w16, total, shift, nb_total);
    launch_end(stream);
    // the attention kernels read block ids before their programmatic wait
    LaunchChoices &c = launch_choices();
    c.full_wait_stream = stream;
    c.full_wait_pending = true;
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_kv_write_fp8(const void *k, const void *v, void *k_codes, void *v_codes, float *k_scale,
                                float *v_scale, const int64_t *slot_mapping, int32_t num_tokens, int32_t hkv,
                                int64_t num_slots, uint32_t *err, cudaStream_t stream)
{
    const int64_t rows = (int64_t)num_tokens * hkv;
    int64_t blocks = (rows + 7) / 8;                        // 8 warps per CTA
    if (blocks > 152 * 16) blocks = 152 * 16;
    launch_begin(stream, kKvWrite);
    cudaError_t e = launch_maybe_pdl(kv_write_fp8_kernel, dim3((unsigned)blocks), dim3(256), 0, stream,
                                     (const uint2 *)k, (const uint2 *)v, (uint32_t *)k_codes, (uint32_t *)v_codes,
                                     k_scale, v_scale, slot_mapping, rows, hkv, num_slots, err);
    launch_end(stream);
    return e != cudaSuccess ? e : cudaGetLastError();
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

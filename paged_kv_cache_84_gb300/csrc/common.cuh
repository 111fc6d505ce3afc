// Shared device helpers and the internal launch interface of libpkv.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pkv {

// ---------------------------------------------------------------- launch plan
//
// A launch's work list travels in the kernel parameters (no host->device
// copy, no sync): `req[li]` is a request index and request li owns the
// items item_off[li] .. item_off[li+1]-1 of the grid's x dimension.
// Decode-class lists split a request's keys into chunks of `split_tokens`;
// prefill-class lists cut its new tokens into tiles of `tile_tokens`.
// Each listed request also carries its first row, row count and context
// length from the host copies of the metadata, so that a CTA starts without
// a dependent read of device memory; one lane per request compares them
// with the device arrays later (check_meta).
constexpr int kPlanMax = 256;

struct WorkList {
    int32_t n;              // listed requests
    int32_t mode;           // kModeDecode or kModePrefill
    int32_t split_tokens;   // decode: keys per split (multiple of the block size)
    int32_t tile_tokens;    // prefill: tokens per tile
    int32_t req[kPlanMax];
    int32_t item_off[kPlanMax + 1];
    int32_t part_off[kPlanMax];   // decode: first partial row of a split request, -1 if unsplit
    int32_t qb[kPlanMax];         // query_start_loc[req]
    int32_t qt[kPlanMax];         // query_start_loc[req + 1] - query_start_loc[req]
    int32_t len[kPlanMax];        // seq_lens[req]
    int32_t cnt_off[kPlanMax];    // decode: first split counter of a request combined in-kernel, else -1
    int32_t cluster;              // decode: 0, or the split count of every request when each request's
                                  // splits run as one thread-block cluster (combined through its shared memory)
    union {
        int32_t split_len[kPlanMax];  // decode, cluster mode: keys per split of each request (a multiple of 16)
        int32_t tc_split[kPlanMax];   // tcgen05 prefill: (pairs run whole << 5) | key pieces of each other pair
    };
};

// tcgen05 prefill work of one listed request: its pairs of 128-row tiles run
// longest first; the first `whole` of them as one CTA each (per KV head),
// every later one as `pieces` CTAs over consecutive key-tile ranges, whose
// fp32 partials the CTA finishing last merges.  The key tiles of such a pair
// are cut evenly (small = 0), or, with two pieces, into a first piece and a
// last one of small/64 of the tiles (at least one).  Pieces launch
// piece-major: every split pair's piece 0, then every piece 1, ...
__host__ __device__ __forceinline__ int tc_split_pack(int whole, int pieces, int small = 0)
{
    return (whole << 11) | (pieces << 6) | small;
}
__host__ __device__ __forceinline__ int tc_split_whole(int v) { return v >> 11; }
__host__ __device__ __forceinline__ int tc_split_pieces(int v) { return (v >> 6) & 31; }
__host__ __device__ __forceinline__ int tc_split_small(int v) { return v & 63; }
constexpr int kTcMaxPieces = 16;

// First key tile (relative to the pair's first) of piece q of `pieces` over n
// key tiles (q = pieces: n).
__host__ __device__ __forceinline__ int tc_piece_begin(int n, int q, int pieces, int small)
{
    if (q >= pieces) return n;
    if (small == 0 || pieces != 2) return n * q / pieces;
    const int last = (n * small + 32) / 64 > 0 ? (n * small + 32) / 64 : 1;
    return q == 0 ? 0 : n - last;
}

// Largest cluster of a decode request's splits (the portable cluster size).
constexpr int kMaxClusterSplits = 8;
// Decode splits of at least this many keys stream their blocks (streaming
// kernel); shorter ones use the slot-ring kernel.
constexpr int kLongSplitTokens = 512;

constexpr int kModeDecode = 0;
constexpr int kModePrefill = 1;

struct AttnParams {
    __nv_bfloat16 *out;
    const __nv_bfloat16 *q;
    const __nv_bfloat16 *k_cache;
    const __nv_bfloat16 *v_cache;
    const int32_t *qsl;
    const int32_t *seq_lens;
    const int32_t *block_table;
    int32_t bt_stride;
    int32_t hq, hkv, group, block_size, nb_total;
    float scale_log2;           // softmax scale * log2(e): scores live in the exp2 domain
    uint32_t *err;              // device error word
    float *part_o;              // [rows][head_dim] unnormalised split outputs
    float2 *part_ml;            // [rows] (running max in exp2 domain, sum of weights)
    uint32_t *counters;         // split counters of in-kernel combines (zero between calls), or null
    int32_t window;             // sliding window: keys above position - window (0: none)
    const float *k_scale;       // FP8 pools: [slots][hkv] scales of the K and V codes (else null)
    const float *v_scale;
    // Combined write + attention (bf16 pools): decode-class CTAs write their
    // own requests' new K/V rows (fw_k, fw_v: [N][hkv][D] as 16-byte vectors)
    // into the pools (fw_kc, fw_vc) at fw_slots[row] before reading them.
    // Null when the rows were written by a separate scatter.
    const uint4 *fw_k;
    const uint4 *fw_v;
    uint4 *fw_kc;
    uint4 *fw_vc;
    const int64_t *fw_slots;
    float *fw_ks;               // quantized pools: the scale pools the combined call writes
    float *fw_vs;
    // Decode batches planned for capacities: each request's context length is
    // the device seq_lens entry (at most the planned one) instead of the plan's.
    int32_t dev_len;
};

// Token ranges [begin, begin + len) of the rows a ranged scatter writes
// (the prefill-class requests of a combined write + attention call).
struct TokenRanges {
    int32_t n;
    int32_t begin[kPlanMax];
    int32_t off[kPlanMax + 1];   // prefix sums of the lengths
};

// ---------------------------------------------------------------- sliding window
//
// "31. Engine v2", "Attention over the pool": with a window w > 0 the query
// at position qp sees the keys qp - w + 1 .. qp.  Shared by the planner and
// the kernels so that both count the same splits.

// Lowest key the query at position qp sees.
__host__ __device__ __forceinline__ int window_lo(int qp, int window)
{
    return (window > 0 && qp - window + 1 > 0) ? qp - window + 1 : 0;
}

// The mask bound: keys at or below qp - win_span(window) are outside the window.
__host__ __device__ __forceinline__ int win_span(int window) { return window > 0 ? window : (1 << 30); }

// First key of a decode-class request's key range (its t rows sit at
// positions L - t .. L - 1), rounded down to a 16-key block.
__host__ __device__ __forceinline__ int decode_key_begin(int t, int L, int window)
{
    return window_lo(L - t, window) & ~15;
}

// Splits of `split` keys that cover a decode-class request's key range.
__host__ __device__ __forceinline__ int decode_splits(int t, int L, int window, int split)
{
    return L <= 0 ? 1 : (L - decode_key_begin(t, L, window) + split - 1) / split;
}

// ---------------------------------------------------------------- device helpers

constexpr uint32_t kDevErrMeta = 8u;    // device metadata differs from the host copies
constexpr uint32_t kDevErrCounter = 16u; // a split counter was not zero at the start of a call
constexpr int kCounterStride = 8;        // uint32 words between two split counters (32 bytes)

// Workspace layout: the device error word area comes first; then, in every
// workspace large enough to hold it, the split counters of in-kernel
// combines (zero-filled by the caller once; each call leaves them zero
// again), one per (split request, KV head), 32 bytes apart so that
// concurrent atomics of different requests do not queue on one L2 sector;
// then split-KV partials.
constexpr size_t kErrBytes = 256;
constexpr int kCounterGroups = 2048;
constexpr size_t kCounterBytes = 4 * (size_t)kCounterStride * kCounterGroups;

// Flags a listed request whose device metadata disagrees with the host copies
// the launch was planned from (the kernels use the planned values).
// Generic-proxy writes to global memory become visible to the async proxy
// (TMA loads) issued after this fence.
__device__ __forceinline__ void fence_proxy_async_global()
{
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Combined write + attention: copy a request's new rows at positions
// [pos_lo, pos_hi) of KV head kh (the request's t tokens sit at positions
// L - t .. L - 1, token row b + pos - (L - t)) into the pools at
// fw_slots[row] (negative: the scratch slot), with threads tid of nthreads,
// each fencing its stores against the async proxy: after a barrier of the
// writers, TMA loads issued by any of them (or by a thread past the barrier,
// which fences again) see the rows.  A slot outside the pool is skipped
// and reported (bit 1, as the scatter does); a slot other than the one the
// block table gives for the position is reported (kDevErrMeta): the
// attention reads the block table's slot.  pos_lo = pos_hi - t with L = 0:
// a padding request, whose rows go to their slots without the table check.
template <int D>
__device__ __forceinline__ void fused_kv_write(const AttnParams &p, int r, int b, int t, int L, int kh, int pos_lo,
                                               int pos_hi, int tid, int nthreads)
{
    constexpr int kVec = D * 2 / 16;                      // 16-byte vectors of one row and head
    const int64_t num_slots = (int64_t)p.nb_total * p.block_size;
    const int32_t *bt = p.block_table + (size_t)r * p.bt_stride;
    const int n = (pos_hi - pos_lo) * kVec;
    for (int idx = tid; idx < n; idx += nthreads) {
        const int pos = pos_lo + idx / kVec, c = idx % kVec;
        const int row = b + pos - (L - t);
        int64_t slot = __ldg(p.fw_slots + row);
        if (c == 0 && L > 0 && slot >= 0) {
            const int64_t want = (int64_t)__ldg(bt + (pos >> 4)) * 16 + (pos & 15);
            if (slot != want) atomicOr(p.err, kDevErrMeta);
        }
        if (slot < 0) slot = num_slots - 1;               // padding row -> scratch slot
        if (slot >= num_slots) {
            if (c == 0) atomicOr(p.err, 1u);
            continue;
        }
        const size_t src = ((size_t)row * p.hkv + kh) * kVec + c;
        const size_t dst = ((size_t)slot * p.hkv + kh) * kVec + c;
        const uint4 kx = p.fw_k[src], vx = p.fw_v[src];
        p.fw_kc[dst] = kx;
        p.fw_vc[dst] = vx;
    }
    fence_proxy_async_global();
}

__device__ __forceinline__ void check_meta(const AttnParams &p, const WorkList &wl, int li)
{
    const int r = wl.req[li];
    const int b = p.qsl[r], e = p.qsl[r + 1], L = p.seq_lens[r];
    const bool len_ok = p.dev_len ? L <= wl.len[li] : L == wl.len[li];
    if (b != wl.qb[li] || e - b != wl.qt[li] || !len_ok) atomicOr(p.err, kDevErrMeta);
}

// Context length of listed request li as this call runs it: the planned one,
// or (p.dev_len) the device seq_lens entry, clamped to [0, planned] (a longer
// one is reported by check_meta).  The planned length fixes the split count.
__device__ __forceinline__ int run_len(const AttnParams &p, const WorkList &wl, int li)
{
    const int planned = wl.len[li];
    if (!p.dev_len) return planned;
    const int L = __ldg(p.seq_lens + wl.req[li]);
    return L < 0 ? 0 : (L > planned ? planned : L);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// One (row, KV head) of 128 dims quantized to E4M3 by a warp ("31. Engine
// v2", "Attention over the pool": codes with a scale per slot and head; the
// format is this library's reading): lane l holds dims 4l .. 4l+3 of x (four
// bf16) and gets their four codes; scale = max |x| / 448 in fp32 (the same in
// every lane), codes = E4M3(x / scale) rounded to nearest even with
// saturation; an all-zero row has scale 0 and zero codes.  The quantizing
// scatter and the combined call's decode CTAs both use it, so their pools
// agree bit for bit.
__device__ __forceinline__ uint32_t quantize_e4m3_row(uint2 x, float &scale)
{
    const float f[4] = {bf16_lo(x.x), bf16_hi(x.x), bf16_lo(x.y), bf16_hi(x.y)};
    float amax = fmaxf(fmaxf(fabsf(f[0]), fabsf(f[1])), fmaxf(fabsf(f[2]), fabsf(f[3])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    scale = __fdiv_rn(amax, 448.0f);
    uint32_t codes = 0u;
    if (scale > 0.f) {
        const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
            make_float2(__fdiv_rn(f[0], scale), __fdiv_rn(f[1], scale)), __NV_SATFINITE, __NV_E4M3);
        const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
            make_float2(__fdiv_rn(f[2], scale), __fdiv_rn(f[3], scale)), __NV_SATFINITE, __NV_E4M3);
        codes = (uint32_t)lo | ((uint32_t)hi << 16);
    }
    return codes;
}

// The combined call on a quantized pool (head_dim 128): as fused_kv_write,
// rows quantized by the calling warp (quantize_e4m3_row), codes and scales
// stored at the row's slot; KV heads kh .. kh + nh - 1.
__device__ __forceinline__ void fused_kv_write_fp8(const AttnParams &p, int r, int b, int t, int L, int kh, int nh,
                                                   int pos_lo, int pos_hi, int lane)
{
    const int64_t num_slots = (int64_t)p.nb_total * p.block_size;
    const int32_t *bt = p.block_table + (size_t)r * p.bt_stride;
    const uint2 *k2 = reinterpret_cast<const uint2 *>(p.fw_k);
    const uint2 *v2 = reinterpret_cast<const uint2 *>(p.fw_v);
    uint32_t *kcodes = reinterpret_cast<uint32_t *>(p.fw_kc);
    uint32_t *vcodes = reinterpret_cast<uint32_t *>(p.fw_vc);
    for (int pos = pos_lo; pos < pos_hi; pos++) {            // warp-uniform
        const int row = b + pos - (L - t);
        int64_t slot = __ldg(p.fw_slots + row);
        if (lane == 0 && L > 0 && slot >= 0) {
            const int64_t want = (int64_t)__ldg(bt + (pos >> 4)) * 16 + (pos & 15);
            if (slot != want) atomicOr(p.err, kDevErrMeta);
        }
        if (slot < 0) slot = num_slots - 1;                   // padding row -> scratch slot
        if (slot >= num_slots) {
            if (lane == 0) atomicOr(p.err, 1u);
            continue;
        }
        for (int h = kh; h < kh + nh; h++) {
            const size_t src = ((size_t)row * p.hkv + h) * 32 + lane;
            const size_t dst = (size_t)slot * p.hkv + h;
            float ks, vs;
            const uint32_t kq = quantize_e4m3_row(k2[src], ks);
            const uint32_t vq = quantize_e4m3_row(v2[src], vs);
            kcodes[dst * 32 + lane] = kq;
            vcodes[dst * 32 + lane] = vq;
            if (lane == 0) {
                p.fw_ks[dst] = ks;
                p.fw_vs[dst] = vs;
            }
        }
    }
    fence_proxy_async_global();
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void *p)
{
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Index of the listed request that owns grid item `item` (binary search over item_off).
__device__ __forceinline__ int find_listed(const WorkList &wl, int item)
{
    int lo = 0, hi = wl.n - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (wl.item_off[mid] <= item) lo = mid; else hi = mid - 1;
    }
    return lo;
}

}  // namespace pkv

// ---------------------------------------------------------------- launchers (internal C++ linkage)

namespace pkv {

cudaError_t launch_kv_write(const void *k, const void *v, void *k_cache, void *v_cache,
                            const int64_t *slot_mapping, int32_t num_tokens, int32_t row_bytes,
                            int64_t num_slots, uint32_t *err, cudaStream_t stream);
cudaError_t launch_kv_write_fp8(const void *k, const void *v, void *k_codes, void *v_codes, float *k_scale,
                                float *v_scale, const int64_t *slot_mapping, int32_t num_tokens, int32_t hkv,
                                int64_t num_slots, uint32_t *err, cudaStream_t stream);

// TMA-staged attention with warp-level MMA (decode-class: 4 key groups per
// CTA; prefill-class: 4 row tiles of 16 per CTA).
cudaError_t launch_attn_mma(const AttnParams &p, const WorkList &wl, int head_dim, int num_items,
                            const void *k_cache, const void *v_cache, int64_t num_slots, cudaStream_t stream,
                            const float *k_scale = nullptr, const float *v_scale = nullptr);
int mma_prefill_rows();

// A mixed launch: its first dec_rows grid rows (dec_rows x hkv CTAs) are
// decode CTAs, every warp of which runs decode items; the tcgen05 prefill
// CTAs follow them.
struct MixAssign {
    int32_t dec_rows;
};

// tcgen05 prefill tiles of 128 query rows (head_dim 48, 64 or 128, g dividing 128).
// With mix (and pd, dl): the mixed-batch kernel, whose leading decode CTAs
// run the decode items of list dl with parameters pd.
bool tc_prefill_supported(int head_dim, int group);
int tc_prefill_rows();
cudaError_t launch_attn_tc(const AttnParams &p, const WorkList &wl, int num_items, const void *q, int num_tokens,
                           const void *k_cache, const void *v_cache, int64_t num_slots, int head_dim,
                           cudaStream_t stream, const AttnParams *pd = nullptr, const WorkList *dl = nullptr,
                           const MixAssign *mix = nullptr);

// Block copies over up to kMaxPools pools: mode 0 copies block src[i] to
// dst[i] in every pool, 1 gathers block src[i] of pool q to buf[q][i], 2
// scatters buf[q][i] to block src[i] of pool q.
constexpr int kMaxPools = 256;
cudaError_t launch_block_copy(int mode, void *const *pools, int32_t num_pools, const int32_t *src,
                              const int32_t *dst, int32_t n, int32_t nb_total, int64_t block_bytes, void *buf,
                              uint32_t *err, cudaStream_t stream);
cudaError_t launch_byte_copy(void *dst, const void *src, size_t bytes, cudaStream_t stream);
// Block table in blocks of 16 slots (bt16 [num_reqs][w16]) for a pool of
// blocks of 16 << shift slots; the next launch on `stream` waits for it to end.
cudaError_t launch_expand_table(const int32_t *bt, int32_t stride, int32_t *bt16, int32_t w16, int32_t num_reqs,
                                int32_t shift, int32_t nb_total, cudaStream_t stream);
cudaError_t launch_fp8_dequant(const AttnParams &p, const WorkList &wl, __nv_bfloat16 *k_out, __nv_bfloat16 *v_out,
                               int32_t *table_out, int32_t table_stride, int32_t sblk0, cudaStream_t stream);
cudaError_t launch_kv_write_fp8_ranges(const void *k, const void *v, void *k_codes, void *v_codes, float *k_scale,
                                       float *v_scale, const int64_t *slot_mapping, const TokenRanges &ranges,
                                       int32_t hkv, int64_t num_slots, uint32_t *err, cudaStream_t stream);
cudaError_t launch_kv_write_ranges(const void *k, const void *v, void *k_cache, void *v_cache,
                                   const int64_t *slot_mapping, const TokenRanges &ranges, int32_t row_bytes,
                                   int64_t num_slots, uint32_t *err, cudaStream_t stream);

// Merge split-KV partials of the split requests in `wl` into bf16 output.
cudaError_t launch_attn_combine(const AttnParams &p, const WorkList &wl, int head_dim,
                                int max_rows_per_req, cudaStream_t stream);

// Kernel ids for launch accounting and the optional per-launch event timing.
enum KernelId : int {
    kKvWrite = 0,
    kAttnCombine = 3,
    kAttnTcPrefill = 4,
    kAttnMmaDecode = 5,
    kAttnMmaPrefill = 6,
    kBlockCopy = 7,
    kByteCopy = 8,
    kAttnTcMixed = 9,
    kFp8Dequant = 10,
    kTableExpand = 11,
    kNumKernelIds = 12
};

// Call around every kernel launch: counts it and, while profiling is on,
// records a CUDA event before and after it on the launching stream.
void launch_begin(cudaStream_t stream, int kernel_id);
void launch_end(cudaStream_t stream);

// Per-call choices that override the planner's (pkv_attention_options in
// include/pkv.h); a default-constructed value leaves every choice to the
// planner.
struct CallOptions {
    bool disable_tcgen05 = false;     // prefill on the warp-MMA kernel
    int tc_min_rows = 0;              // > 0: rows from which a prefill request goes to tcgen05
    bool fp8_prefill_on_mma = false;  // quantized-pool prefill stays on the warp-MMA kernel
    int split_tokens = 0;             // > 0: fixed decode split length
    int cluster = 0;                  // 0: planner; -1: no clusters; k >= 2: clusters of k splits
    int decode_main = 0;              // 0: planner; 1: decodes on the caller's stream; -1: prefill there
    bool no_overlap = false;          // both classes on the caller's stream
    bool prefill_key_splits = false;  // key splits for warp-MMA prefill tiles
    bool separate_write = false;      // combined call as scatter + attention
    bool decode_row_tiles = false;    // 16-row decode tiles instead of key-major ones
    bool no_pdl = false;              // no programmatic dependent launches
    int tc_key_pieces = 0;            // 0: planner; -1: no key pieces; k >= 2: every tcgen05 pair in k pieces
    int mixed_launch = 0;             // 0: planner; 1: decode class in the tcgen05 launch when it can; -1: never
    int mixed_decode_ctas = 0;        // > 0: decode CTAs of a mixed launch (rounded up to the KV heads)
    bool device_lengths = false;      // decode batch: context lengths read from the device at run time
};

// Launch-level choices of the attention call in progress on this thread,
// set for the duration of the call (ScopedLaunchChoices); outside a call,
// and for the write, copy and block-copy calls, the defaults hold.
struct LaunchChoices {
    bool pdl = true;                  // programmatic stream serialization for dependent launches
    bool decode_row_tiles = false;    // see CallOptions
    // the next launch on this stream waits for the kernel before it to end:
    // that kernel wrote data the next one reads before its programmatic wait
    cudaStream_t full_wait_stream = nullptr;
    bool full_wait_pending = false;
};
LaunchChoices &launch_choices();

struct ScopedLaunchChoices {
    LaunchChoices saved;
    explicit ScopedLaunchChoices(const LaunchChoices &c) : saved(launch_choices()) { launch_choices() = c; }
    ~ScopedLaunchChoices() { launch_choices() = saved; }
};

// Whether kernels that read what an earlier kernel of the same stream wrote
// are launched with programmatic stream serialization (they start early and
// wait in-kernel with griddepcontrol.wait).
inline bool pdl_enabled() { return launch_choices().pdl; }

// The same for a launch on `stream` (consumes a pending full wait on it).
inline bool pdl_for(cudaStream_t stream)
{
    LaunchChoices &c = launch_choices();
    if (c.full_wait_pending && c.full_wait_stream == stream) {
        c.full_wait_pending = false;
        return false;
    }
    return c.pdl;
}

template <typename... KArgs, typename... Args>
cudaError_t launch_maybe_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                             Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_for(stream) ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// The same with clusters of cluster_y CTAs along y.
template <typename... KArgs, typename... Args>
cudaError_t launch_cluster_maybe_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                     cudaStream_t stream, unsigned cluster_y, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = cluster_y;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_for(stream) ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace pkv

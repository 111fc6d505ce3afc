// C ABI of libpkv: argument validation, launch planning, launches.
//
// Planning reads only the host copies of query_start_loc and seq_lens
// ("31. Engine v2", "Flattened ragged batches": the batch metadata keeps
// host copies so that kernels launch without a device sync).  It sorts the
// requests into
//   - decode-class: t * g <= 16 rows per KV head (decodes, short chunks,
//     padding requests); their keys may be split across CTAs, with a
//     combine pass when a request has more than one split;
//   - prefill-class: everything else, cut into tiles of new tokens.
// Each class goes to its kernel with the work list in the kernel
// parameters, so nothing is copied to the device and nothing waits.
#include <atomic>
#include <climits>
#include <cmath>
#include <mutex>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <algorithm>
#include <functional>
#include <vector>

#include "pkv.h"
#include "common.cuh"

namespace pkv {

static std::atomic<int64_t> g_launches{0};

// Optional per-launch timing: events recorded on the launching stream.
struct Profile {
    std::mutex mu;
    bool on = false;
    std::vector<cudaEvent_t> events;     // 2 per record
    std::vector<int> kernel;
    int n = 0;
    int open = -1;                       // record opened by launch_begin, closed by launch_end
};
static Profile g_prof;

// A profiling event on `stream`: while the stream is being captured into a
// CUDA graph the record becomes an event node of the graph (its timestamp
// is taken each time the graph runs), otherwise an ordinary record.
static void record_profile_event(cudaEvent_t ev, cudaStream_t stream)
{
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
        cudaEventRecordWithFlags(ev, stream, cudaEventRecordExternal);
    else
        cudaEventRecord(ev, stream);
}

void launch_begin(cudaStream_t stream, int kernel_id)
{
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (!g_prof.on) return;
    std::lock_guard<std::mutex> lock(g_prof.mu);
    if (!g_prof.on || g_prof.n >= (int)g_prof.kernel.size()) return;
    g_prof.open = g_prof.n;
    g_prof.kernel[g_prof.n] = kernel_id;
    record_profile_event(g_prof.events[2 * g_prof.n], stream);
}

void launch_end(cudaStream_t stream)
{
    if (!g_prof.on) return;
    std::lock_guard<std::mutex> lock(g_prof.mu);
    if (g_prof.open < 0) return;
    record_profile_event(g_prof.events[2 * g_prof.open + 1], stream);
    g_prof.n = g_prof.open + 1;
    g_prof.open = -1;
}

LaunchChoices &launch_choices()
{
    static thread_local LaunchChoices c;
    return c;
}

// The internal form of a caller's options (NULL: every choice to the planner).
static CallOptions call_options(const pkv_attention_options *o)
{
    CallOptions c;
    if (!o) return c;
    c.disable_tcgen05 = o->disable_tcgen05 != 0;
    c.tc_min_rows = o->tc_min_rows > 0 ? o->tc_min_rows : 0;
    c.fp8_prefill_on_mma = o->fp8_prefill_on_mma != 0;
    c.split_tokens = o->split_tokens > 0 ? o->split_tokens : 0;
    c.cluster = o->cluster;
    c.decode_main = o->decode_main > 0 ? 1 : (o->decode_main < 0 ? -1 : 0);
    c.no_overlap = o->no_overlap != 0;
    c.prefill_key_splits = o->prefill_key_splits != 0;
    c.separate_write = o->separate_write != 0;
    c.decode_row_tiles = o->decode_row_tiles != 0;
    c.no_pdl = o->no_pdl != 0;
    c.tc_key_pieces = o->tc_key_pieces < 0 ? -1 : (o->tc_key_pieces >= 2 ? o->tc_key_pieces : 0);
    c.mixed_launch = o->mixed_launch > 0 ? 1 : (o->mixed_launch < 0 ? -1 : 0);
    c.mixed_decode_ctas = o->mixed_decode_ctas > 0 ? o->mixed_decode_ctas : 0;
    c.device_lengths = o->device_lengths != 0;
    return c;
}

static thread_local char g_cuda_err[256] = "";

static pkv_status cuda_fail(cudaError_t e, const char *where)
{
    snprintf(g_cuda_err, sizeof g_cuda_err, "%s: %s", where, cudaGetErrorString(e));
    return PKV_ERR_CUDA;
}

// log2(bs / 16) for the block sizes the kernels walk in sub-blocks of 16
// slots (16, 32, 64, 128, 256), else -1.
static int block_shift(int32_t bs)
{
    for (int s = 0; s <= 4; s++)
        if (bs == (16 << s)) return s;
    return -1;
}

// Blocks of more than 16 slots: the attention kernels walk a block table in
// blocks of 16 slots, which an expansion kernel writes at the workspace's
// end (w16 = ceil(longest host length / 16) entries per request).  Returns
// its bytes (0 for 16-slot blocks) and sets *w16.
static size_t table16_bytes(const int32_t *sl_h, int32_t num_reqs, int32_t bs, int32_t *w16)
{
    *w16 = 0;
    if (block_shift(bs) <= 0) return 0;
    int32_t max_l = 1;
    for (int r = 0; r < num_reqs; r++) max_l = sl_h[r] > max_l ? sl_h[r] : max_l;
    *w16 = (max_l + 15) / 16;
    return ((size_t)num_reqs * *w16 * 4 + 255) / 256 * 256;
}

static int num_sms()
{
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
    if (!cached[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
        cached[dev] = n;
    }
    return cached[dev];
}

// Side streams of the decode/prefill overlap: one non-blocking stream and a
// fork/join event pair for each (device, caller stream), created on first
// use (host-side CUDA objects, no device memory) and kept until exit.  Each
// has its own mutex, held for the whole call, so only callers on the same
// stream share one; callers on different streams never wait for each other
// through it.  When the table is full the call runs both classes on the
// caller's stream (no overlap).
struct SideStream {
    std::mutex mu;
    int dev = -1;
    cudaStream_t owner = nullptr;     // the caller stream it serves
    cudaStream_t stream = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};
constexpr int kMaxSideStreams = 256;

static SideStream *side_stream_for(cudaStream_t caller)
{
    static SideStream table[kMaxSideStreams];
    static int used = 0;
    static std::mutex table_mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    std::lock_guard<std::mutex> lock(table_mu);
    for (int i = 0; i < used; i++)
        if (table[i].dev == dev && table[i].owner == caller) return &table[i];
    if (used == kMaxSideStreams) return nullptr;
    SideStream &s = table[used];
    cudaStream_t st;
    cudaEvent_t a, b;
    if (cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess) return nullptr;
    if (cudaEventCreateWithFlags(&a, cudaEventDisableTiming) != cudaSuccess) {
        cudaStreamDestroy(st);
        return nullptr;
    }
    if (cudaEventCreateWithFlags(&b, cudaEventDisableTiming) != cudaSuccess) {
        cudaEventDestroy(a);
        cudaStreamDestroy(st);
        return nullptr;
    }
    s.dev = dev;
    s.owner = caller;
    s.fork = a;
    s.join = b;
    s.stream = st;
    used++;
    return &s;
}

static bool aligned(const void *p, uintptr_t a) { return ((uintptr_t)p % a) == 0; }

constexpr int kDecodeRows = 16;       // decode-class: t * g <= this
constexpr int kMinSplit = 256;        // smallest KV split, tokens
constexpr int kMaxSplits = 64;        // most splits of one request
constexpr int kMaxStreamSplits = 32;  // most splits of one request on the streaming kernel
constexpr int kMaxPrefillRowSplits = 4;   // workspace sizing of split prefill tiles
// Every prefill-class request (more than kDecodeRows query rows) whose head
// dim and group fit a 128-row tile runs on the tcgen05 kernel: measured on
// the 48-request engine step, one 128-row tile per (request, KV head) beats
// several 32-row warp-MMA CTAs that each re-read the request's keys.
constexpr int kTcMinRows = kDecodeRows + 1;

static int tc_min_rows(const CallOptions &o) { return o.tc_min_rows > 0 ? o.tc_min_rows : kTcMinRows; }

// Kernel class of request r (host rule shared by the planner and pkv_plan_request_kernels).
static int request_class(int32_t t, int32_t L, int32_t g, int32_t d, const CallOptions &o, bool fp8 = false)
{
    if (t == 0) return PKV_CLASS_NONE;
    if (L == 0) return PKV_CLASS_PADDING;
    if (t * g <= kDecodeRows) return PKV_CLASS_DECODE;
    // a request fills at least kTcMinRows of a 128-row tensor-core tile
    if (!fp8 && tc_prefill_supported(d, g) && t * g >= tc_min_rows(o) && !o.disable_tcgen05)
        return PKV_CLASS_PREFILL_TENSOR;
    return PKV_CLASS_PREFILL_MMA;
}

// Quantized pools: prefill requests that the tcgen05 kernel takes when the
// workspace holds bf16 copies of their blocks (fp8_tc_scratch bytes at the
// workspace's end: K and V blocks [blocks][16][hkv][d] bf16, then a block
// table [num_reqs][width] int32).  Returns 0 when no request qualifies.
static size_t fp8_tc_scratch(const int32_t *qsl_h, const int32_t *sl_h, int32_t num_reqs, int32_t g, int32_t hkv,
                             int32_t d, const CallOptions &o, int64_t *blocks_out = nullptr,
                             int32_t *width_out = nullptr)
{
    // quantized pools have head_dim 128 (128-byte code rows)
    if (d != 128 || !tc_prefill_supported(d, g) || o.disable_tcgen05 || o.fp8_prefill_on_mma) return 0;
    const int min_rows = tc_min_rows(o);
    int64_t blocks = 0;
    int32_t width = 0;
    for (int r = 0; r < num_reqs; r++) {
        const int32_t t = qsl_h[r + 1] - qsl_h[r], L = sl_h[r];
        if (t == 0 || L == 0 || t * g <= kDecodeRows || t * g < min_rows) continue;
        const int32_t nb = (L + 15) / 16;
        blocks += nb;
        width = nb > width ? nb : width;
    }
    if (blocks_out) *blocks_out = blocks;
    if (width_out) *width_out = width;
    if (blocks == 0) return 0;
    const size_t kv = (size_t)blocks * 16 * hkv * d * 2;                 // one of K, V
    const size_t table = (size_t)num_reqs * width * 4;
    return 256 + 2 * ((kv + 255) / 256 * 256) + (table + 255) / 256 * 256;
}

}  // namespace pkv

using namespace pkv;

extern "C" {

const char *pkv_status_string(pkv_status s)
{
    switch (s) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID_ARG: return "invalid argument";
    case PKV_ERR_UNSUPPORTED: return "unsupported shape or alignment";
    case PKV_ERR_WORKSPACE: return "workspace missing or too small";
    case PKV_ERR_CUDA: return "CUDA error";
    case PKV_ERR_DEVICE_BOUNDS: return "device bounds violation recorded";
    }
    return "unknown status";
}

const char *pkv_last_cuda_error(void) { return g_cuda_err; }

int64_t pkv_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char *pkv_kernel_name(int32_t kernel_id)
{
    switch (kernel_id) {
    case kKvWrite: return "paged_kv_write";
    case kAttnCombine: return "attn_split_combine";
    case kAttnTcPrefill: return "attn_tc_prefill";
    case kAttnMmaDecode: return "attn_mma_decode";
    case kAttnMmaPrefill: return "attn_mma_prefill";
    case kBlockCopy: return "block_copy";
    case kByteCopy: return "byte_copy";
    case kAttnTcMixed: return "attn_tc_mixed";
    case kFp8Dequant: return "fp8_dequant";
    case kTableExpand: return "block_table_expand";
    }
    return "unknown";
}

pkv_status pkv_profile_start(int32_t capacity)
{
    if (capacity <= 0) return PKV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_prof.mu);
    while ((int)g_prof.kernel.size() < capacity) {
        cudaEvent_t a, b;
        cudaError_t e = cudaEventCreate(&a);
        if (e == cudaSuccess) e = cudaEventCreate(&b);
        if (e != cudaSuccess) return cuda_fail(e, "profile events");
        g_prof.events.push_back(a);
        g_prof.events.push_back(b);
        g_prof.kernel.push_back(-1);
    }
    g_prof.n = 0;
    g_prof.open = -1;
    g_prof.on = true;
    return PKV_OK;
}

int32_t pkv_profile_stop(void)
{
    std::lock_guard<std::mutex> lock(g_prof.mu);
    g_prof.on = false;
    return g_prof.n;
}

pkv_status pkv_profile_read(int32_t index, int32_t *kernel_id, float *ms)
{
    std::lock_guard<std::mutex> lock(g_prof.mu);
    if (index < 0 || index >= g_prof.n || !kernel_id || !ms) return PKV_ERR_INVALID_ARG;
    cudaError_t e = cudaEventSynchronize(g_prof.events[2 * index + 1]);
    if (e == cudaSuccess) e = cudaEventElapsedTime(ms, g_prof.events[2 * index], g_prof.events[2 * index + 1]);
    if (e != cudaSuccess) return cuda_fail(e, "profile read");
    *kernel_id = g_prof.kernel[index];
    return PKV_OK;
}

pkv_status pkv_paged_kv_write(const void *k, const void *v, void *k_cache, void *v_cache,
                              const int64_t *slot_mapping, int32_t num_tokens,
                              int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                              int32_t num_blocks_total, uint32_t *device_error,
                              cudaStream_t stream)
{
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks_total <= 0)
        return PKV_ERR_INVALID_ARG;
    if (num_tokens == 0) return PKV_OK;
    if (!k || !v || !k_cache || !v_cache || !slot_mapping) return PKV_ERR_INVALID_ARG;
    if (head_dim % 8 != 0) return PKV_ERR_UNSUPPORTED;
    if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(slot_mapping, 8))
        return PKV_ERR_UNSUPPORTED;
    int64_t row_bytes = (int64_t)num_kv_heads * head_dim * 2;
    if (row_bytes > (1 << 30)) return PKV_ERR_UNSUPPORTED;
    int64_t num_slots = (int64_t)num_blocks_total * block_size;
    cudaError_t e = launch_kv_write(k, v, k_cache, v_cache, slot_mapping, num_tokens, (int32_t)row_bytes,
                                    num_slots, device_error, stream);
    return e == cudaSuccess ? PKV_OK : cuda_fail(e, "paged_kv_write launch");
}

pkv_status pkv_paged_kv_write_fp8(const void *k, const void *v, void *k_cache, void *v_cache, float *k_scale,
                                  float *v_scale, const int64_t *slot_mapping, int32_t num_tokens,
                                  int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                  int32_t num_blocks_total, uint32_t *device_error, cudaStream_t stream)
{
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks_total <= 0)
        return PKV_ERR_INVALID_ARG;
    if (num_tokens == 0) return PKV_OK;
    if (!k || !v || !k_cache || !v_cache || !k_scale || !v_scale || !slot_mapping) return PKV_ERR_INVALID_ARG;
    if (head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(k_scale, 4) || !aligned(v_scale, 4) || !aligned(slot_mapping, 8))
        return PKV_ERR_UNSUPPORTED;
    int64_t num_slots = (int64_t)num_blocks_total * block_size;
    cudaError_t e = launch_kv_write_fp8(k, v, k_cache, v_cache, k_scale, v_scale, slot_mapping, num_tokens,
                                        num_kv_heads, num_slots, device_error, stream);
    return e == cudaSuccess ? PKV_OK : cuda_fail(e, "paged_kv_write_fp8 launch");
}

size_t pkv_attention_workspace_bytes(int32_t max_num_reqs, int32_t max_num_tokens, int32_t num_q_heads,
                                     int32_t head_dim, int32_t max_seq_len)
{
    if (max_num_reqs <= 0 || max_num_tokens <= 0 || num_q_heads <= 0 || head_dim <= 0 || max_seq_len <= 0)
        return kErrBytes;
    int64_t splits = (max_seq_len + kMinSplit - 1) / kMinSplit;
    if (splits > kMaxSplits) splits = kMaxSplits;
    int64_t dec_tokens = (int64_t)max_num_reqs * kDecodeRows;
    if (dec_tokens > max_num_tokens) dec_tokens = max_num_tokens;
    int64_t rows = splits * dec_tokens * num_q_heads;
    // short prefill tiles of small batches (fewer than 2 CTAs per SM) may be
    // split too: at most ~2*SMs tiles of 32 rows, kMaxPrefillRowSplits splits each
    int64_t pre_rows = (int64_t)max_num_tokens * num_q_heads;
    if (pre_rows > 2 * 152 * 32) pre_rows = 2 * 152 * 32;
    int64_t pre_splits = splits < kMaxPrefillRowSplits ? splits : kMaxPrefillRowSplits;
    rows += pre_rows * pre_splits;
    // tcgen05 pairs cut into key pieces: 256-row partial slots, at most 16
    // per (pair, KV head) group and 6 per SM of a 152-SM GPU
    int64_t tc_slots = (int64_t)max_num_tokens * num_q_heads / 256 * kTcMaxPieces;
    if (tc_slots > 6 * 152) tc_slots = 6 * 152;
    const size_t tc_bytes = (size_t)tc_slots * 256 * ((size_t)head_dim * 4 + 8) + 256;
    // pools of blocks of more than 16 slots: the block table in 16-slot entries
    const size_t t16_bytes = ((size_t)max_num_reqs * ((max_seq_len + 15) / 16) * 4 + 255) / 256 * 256 + 256;
    return kErrBytes + kCounterBytes + (size_t)rows * ((size_t)head_dim * 4 + 8) + 64 + tc_bytes + t16_bytes;
}

size_t pkv_fp8_prefill_scratch_bytes(const int32_t *qsl_h, const int32_t *sl_h, int32_t num_reqs,
                                     int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim)
{
    if (!qsl_h || !sl_h || num_reqs <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads)
        return 0;
    return fp8_tc_scratch(qsl_h, sl_h, num_reqs, num_q_heads / num_kv_heads, num_kv_heads, head_dim, CallOptions());
}

pkv_status pkv_plan_request_kernels(const int32_t *qsl_h, const int32_t *sl_h, int32_t num_reqs,
                                    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                    int32_t *class_out)
{
    if (num_reqs < 0 || !qsl_h || (num_reqs > 0 && (!sl_h || !class_out))) return PKV_ERR_INVALID_ARG;
    if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads || head_dim <= 0)
        return PKV_ERR_INVALID_ARG;
    const int32_t g = num_q_heads / num_kv_heads;
    const CallOptions defaults;
    for (int r = 0; r < num_reqs; r++)
        class_out[r] = request_class(qsl_h[r + 1] - qsl_h[r], sl_h[r], g, head_dim, defaults);
    return PKV_OK;
}

pkv_status pkv_clear_device_error(uint32_t *device_error, cudaStream_t stream)
{
    if (!device_error) return PKV_ERR_INVALID_ARG;
    cudaError_t e = cudaMemsetAsync(device_error, 0, sizeof(uint32_t), stream);
    return e == cudaSuccess ? PKV_OK : cuda_fail(e, "clear device error");
}

pkv_status pkv_read_device_error(const uint32_t *device_error, uint32_t *flags_out, cudaStream_t stream)
{
    if (!device_error) return PKV_ERR_INVALID_ARG;
    uint32_t flags = 0;
    cudaError_t e = cudaMemcpyAsync(&flags, device_error, sizeof flags, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "read device error");
    if (flags_out) *flags_out = flags;
    return flags ? PKV_ERR_DEVICE_BOUNDS : PKV_OK;
}

}  // extern "C"

// The attention call of both pool kinds: k_scale / v_scale non-null selects a
// quantized (FP8 E4M3) pool.
// fw_k non-null (bf16 pools, staged MMA kernels): the combined write +
// attention call.  Decode-class CTAs write their requests' new rows
// themselves, a ranged scatter writes the prefill-class requests' rows ahead
// of the prefill kernels, and the decode class does not wait for that scatter.
// Host validation of an attention call: everything that can be checked
// before enqueuing.  PKV_OK with *nothing_to_do set for an empty batch.
static pkv_status validate_attention(const void *out, const void *q, const void *k_cache, const void *v_cache,
                                     const float *k_scale, const float *v_scale, const int32_t *query_start_loc,
                                     const int32_t *seq_lens, const int32_t *block_table, int32_t block_table_stride,
                                     const int32_t *qsl_h, const int32_t *sl_h, int32_t num_reqs, int32_t num_tokens,
                                     int32_t max_query_len, int32_t max_seq_len, int32_t hq, int32_t hkv, int32_t d,
                                     int32_t bs, int32_t num_blocks_total, int32_t window, const void *workspace,
                                     size_t workspace_bytes, bool *nothing_to_do)
{
    const bool fp8 = k_scale != nullptr;
    *nothing_to_do = false;
    if (num_reqs < 0 || num_tokens < 0 || hq <= 0 || hkv <= 0 || d <= 0 || bs <= 0 || num_blocks_total <= 0)
        return PKV_ERR_INVALID_ARG;
    if (window < 0) return PKV_ERR_INVALID_ARG;
    if (hq % hkv != 0) return PKV_ERR_INVALID_ARG;
    if (!qsl_h || (num_reqs > 0 && !sl_h)) return PKV_ERR_INVALID_ARG;
    if (qsl_h[0] != 0 || qsl_h[num_reqs] != num_tokens) return PKV_ERR_INVALID_ARG;
    int32_t seen_q = 0, seen_l = 0;
    for (int r = 0; r < num_reqs; r++) {
        int32_t t = qsl_h[r + 1] - qsl_h[r], L = sl_h[r];
        if (t < 0 || L < 0) return PKV_ERR_INVALID_ARG;
        if (L > 0 && t > L) return PKV_ERR_INVALID_ARG;
        if (L > 0 && (int64_t)(L + bs - 1) / bs > block_table_stride) return PKV_ERR_INVALID_ARG;
        seen_q = t > seen_q ? t : seen_q;
        seen_l = L > seen_l ? L : seen_l;
    }
    if (max_query_len < seen_q || max_seq_len < seen_l) return PKV_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < PKV_WORKSPACE_MIN_BYTES) return PKV_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return PKV_ERR_WORKSPACE;
    if (num_tokens == 0) {
        *nothing_to_do = true;
        return PKV_OK;
    }
    if (!out || !q || !k_cache || !v_cache || !query_start_loc || !seq_lens || !block_table)
        return PKV_ERR_INVALID_ARG;
    const int32_t g = hq / hkv;
    if (d != 48 && d != 64 && d != 128) return PKV_ERR_UNSUPPORTED;
    if (block_shift(bs) < 0) return PKV_ERR_UNSUPPORTED;
    if ((int64_t)num_blocks_total * (bs / 16) > INT32_MAX) return PKV_ERR_UNSUPPORTED;
    if (g > kDecodeRows) return PKV_ERR_UNSUPPORTED;
    if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
        return PKV_ERR_UNSUPPORTED;
    // quantized pools: head_dim 128 (128-byte code rows), scales staged in
    // boxes of 4 KV heads (KV heads a multiple of 4), warp-MMA kernels
    if (fp8 && (d != 128 || hkv % 4 != 0 || !aligned(k_scale, 16) || !aligned(v_scale, 16)))
        return PKV_ERR_UNSUPPORTED;
    return PKV_OK;
}

// The requests of a batch by kernel class, as the planner launches them.
struct RequestClasses {
    std::vector<int32_t> dec;           // decode class and padding requests
    std::vector<int32_t> pre;           // prefill on the warp-MMA (or CUDA-core) kernel
    std::vector<int32_t> tcp;           // prefill on tcgen05, heaviest first
    int64_t dec_keys = 0;               // keys of the decode class
    int64_t dec_max_keys = 0;           // the longest decode-class key range
    size_t fp8_scratch = 0;             // quantized pools: scratch for prefill on tcgen05 (0: none)
    int64_t fp8_blocks = 0;             // ... blocks it copies
    int32_t fp8_width = 0;              // ... width of its block table
};

static RequestClasses classify_requests(const int32_t *qsl_h, const int32_t *sl_h, int32_t num_reqs, int32_t g,
                                        int32_t hkv, int32_t d, int32_t window, bool fp8, size_t workspace_bytes,
                                        const CallOptions &o)
{
    RequestClasses c;
    for (int r = 0; r < num_reqs; r++) {
        int32_t t = qsl_h[r + 1] - qsl_h[r], L = sl_h[r];
        switch (request_class(t, L, g, d, o, fp8)) {
        case PKV_CLASS_PADDING:
        case PKV_CLASS_DECODE: {
            c.dec.push_back(r);
            const int64_t keys = L - decode_key_begin(t, L, window);
            c.dec_keys += keys;
            c.dec_max_keys = keys > c.dec_max_keys ? keys : c.dec_max_keys;
            break;
        }
        case PKV_CLASS_PREFILL_MMA: c.pre.push_back(r); break;
        case PKV_CLASS_PREFILL_TENSOR: c.tcp.push_back(r); break;
        default: break;                                         // no rows at all
        }
    }
    // Quantized pools: the prefill requests that tcgen05 can take go there
    // when the workspace has room for bf16 copies of their blocks at its end
    // (a dequantizing pass fills them); else they stay on the warp-MMA kernel.
    if (fp8 && !c.pre.empty()) {
        c.fp8_scratch = fp8_tc_scratch(qsl_h, sl_h, num_reqs, g, hkv, d, o, &c.fp8_blocks, &c.fp8_width);
        if (c.fp8_scratch > 0 && c.fp8_blocks * 16 < INT32_MAX &&
            workspace_bytes >= c.fp8_scratch + kErrBytes + kCounterBytes + 4096) {
            const int min_rows = tc_min_rows(o);
            std::vector<int32_t> keep;
            for (int32_t r : c.pre) {
                const int32_t t = qsl_h[r + 1] - qsl_h[r];
                if (t * g >= min_rows) c.tcp.push_back(r);
                else keep.push_back(r);
            }
            c.pre.swap(keep);
        } else {
            c.fp8_scratch = 0;
        }
    }
    // heaviest tensor-core requests first (work ~ new tokens x context), so
    // that the long tiles start in the first wave and short ones fill the tail
    std::stable_sort(c.tcp.begin(), c.tcp.end(), [&](int32_t a, int32_t b) {
        const int64_t wa = (int64_t)(qsl_h[a + 1] - qsl_h[a]) * sl_h[a];
        const int64_t wb = (int64_t)(qsl_h[b + 1] - qsl_h[b]) * sl_h[b];
        return wa > wb;
    });
    return c;
}

// Rough times of the two classes: decode ~ its K/V bytes at HBM speed,
// prefill ~ its causal pairs at tensor-core speed (only the ratio is used).
static void class_times(const RequestClasses &c, const int32_t *qsl_h, const int32_t *sl_h, int32_t hq, int32_t hkv,
                        int32_t d, double *dec_us, double *pre_us)
{
    *dec_us = *pre_us = 0.0;
    for (int32_t r : c.dec) *dec_us += (double)sl_h[r] * hkv * d * 4.0 / 6.5e6;
    for (const std::vector<int32_t> *list : {&c.pre, &c.tcp}) {
        for (int32_t r : *list) {
            const double t = qsl_h[r + 1] - qsl_h[r], L = sl_h[r];
            *pre_us += (t * L - 0.5 * t * t) * hq * d * 4.0 / 1.2e9;
        }
    }
}

// Keys per decode split, common to every split request (a multiple of 128
// before block rounding): about 16 CTAs per SM over the decode class's keys.
static int decode_split_tokens(const RequestClasses &c, double dec_us, double pre_us, int32_t hkv, bool fp8,
                               const CallOptions &o, int sms)
{
    int split = o.split_tokens;
    if (split <= 0) {
        // Decodes beside a longer prefill only fill the SMs its last wave
        // leaves: fewer, longer splits (measured on the mixed 2048-token-chunk
        // step: 509 us with splits of ~2048 keys, 514 us with 16 CTAs per SM)
        const bool filler = !c.tcp.empty() && pre_us > dec_us;
        int64_t target_ctas = (int64_t)sms * (filler ? 4 : 16);
        // quantized pools stream two KV heads per CTA: half the CTAs per split
        const int64_t head_ctas = fp8 ? hkv / 2 : hkv;
        int64_t s = (c.dec_keys * head_ctas + target_ctas - 1) / (target_ctas > 0 ? target_ctas : 1);
        if (s < kMinSplit) s = kMinSplit;
        split = (int)((s + 127) / 128 * 128);
    }
    // Streaming splits: at most kMaxStreamSplits per request.  The CTA that
    // completes a request's last split reads every split's partial rows;
    // measured with 8 requests of 32768 keys (FP8 pool), 64 splits of 512
    // keys took 154 us against 129 us with 37 of 896.
    if (split >= kLongSplitTokens && o.split_tokens <= 0) {
        const int64_t floor_split = (c.dec_max_keys + kMaxStreamSplits - 1) / kMaxStreamSplits;
        if (floor_split > split) split = (int)((floor_split + 127) / 128 * 128);
    }
    return split;
}

// Every host-side decision of one attention call, from the host metadata,
// the workspace size and the SM count alone (no CUDA call): the request
// classes, the decode split length, prefill key splits, the workspace
// layout and the stream arrangement.  attention_impl launches from it and
// pkv_plan_attention reports it.
struct AttnPlan {
    RequestClasses rc;
    double dec_us = 0.0, pre_us = 0.0;  // rough class times (only the ratio is used)
    int split = 0;                      // keys per split, a multiple of the block size
    int tile = 1;                       // warp-MMA (or CUDA-core) prefill tile, tokens
    bool pre_split = false;             // warp-MMA prefill tiles split over keys
    int32_t seen_l = 0;                 // the longest context of the batch
    size_t ws_front = 0;                // workspace bytes before the quantized-prefill scratch
    bool has_counters = false;          // the workspace holds in-kernel combine counters
    size_t part_base = 0;               // byte offset of the split partials
    size_t total_rows = 0;              // partial rows of all split requests
    bool fork = false;                  // decode and prefill classes on two streams
    bool decode_main = false;           // ... the decodes on the caller's stream
    bool fork_after_scatter = false;    // ... the decodes fork after the ranged scatter
    int cluster_opt = 0;                // the caller's cluster choice (CallOptions::cluster)
    // tcgen05 prefill key pieces (plan_tc_pieces)
    std::vector<int32_t> tc_split;      // per tcgen05 request, in launch order: tc_split_pack(whole, pieces)
    int64_t tc_groups = 0;              // (pair, KV head) groups cut into pieces: one counter each
    int64_t tc_slots = 0;               // their pieces: one partial slot each
    int64_t tc_ctas = 0;                // tcgen05 CTAs in all
    size_t tc_part_off = 0;             // byte offset of the tcgen05 partial slots in the workspace
    double tc_makespan = 0.0;           // simulated tcgen05 makespan, key-tile times
    // mixed launch: the decode class inside the tcgen05 launch (its leading decode CTAs)
    bool mix = false;
    int32_t mix_items = 0;              // decode items (request, split, KV head)
    int32_t mix_dec_rows = 0;           // grid rows of decode CTAs ahead of the prefill (x hkv CTAs)
    double mix_pred_us = 0.0;           // the planner's time of the mixed launch
    // combined call: per tcgen05 request, whether its CTAs write its new rows
    // (each KV head's rows are one CTA's), so that no scatter does
    std::vector<char> tc_self;
};

// ---- tcgen05 prefill: key pieces
//
// One tcgen05 CTA runs a pair of 128-row tiles of a prefill request over
// all of its key tiles; requests and pairs are launched heaviest first, one
// CTA per SM.  When the heavy pairs outnumber the SMs, those that start in
// a later wave leave SMs idle at the end; cutting them into consecutive
// key-tile pieces (merged by the piece that finishes last) evens that out.
// The planner simulates the greedy schedule (each SM takes the next CTA in
// launch order when it frees up) for a few piece sizes and keeps the best.

// Key tiles of pair `pair` of a request with t new tokens and context L.
static int tc_pair_tiles(int t, int L, int tt, int window, int pair)
{
    const int i0 = pair * 2 * tt;
    const int k_end = L - t + i0 + std::min(2 * tt, t - i0);
    return (k_end + 127) / 128 - window_lo(L - t + i0, window) / 128;
}

// Costs in key-tile times, measured on the mixed 2048-token-chunk step
// (per-CTA timestamps): a CTA's start and finish (barriers, tensor memory,
// the Q tiles, pipeline fill and drain, the output rows) ~3.5; a piece's
// partial store and its share of the merge ~1 more.
constexpr double kTcCtaCost = 3.5;
constexpr double kTcPieceCost = 1.0;

// Greedy list schedule of CTA costs on `sms` SMs, `busy` of which are taken
// until `busy_until` (the decode CTAs of a mixed launch): the time the last
// CTA ends.
static double greedy_makespan(const std::vector<double> &costs, int sms, int busy = 0, double busy_until = 0.0)
{
    std::vector<double> heap(std::max(1, sms), 0.0);
    for (int i = 0; i < busy && i < (int)heap.size(); i++) heap[i] = busy_until;
    std::make_heap(heap.begin(), heap.end(), std::greater<double>());
    for (double c : costs) {
        std::pop_heap(heap.begin(), heap.end(), std::greater<double>());
        heap.back() += c;
        std::push_heap(heap.begin(), heap.end(), std::greater<double>());
    }
    return *std::max_element(heap.begin(), heap.end());
}

static void plan_tc_pieces(AttnPlan &pl, const int32_t *qsl_h, const int32_t *sl_h, int32_t g, int32_t hkv,
                           int32_t d, int32_t window, int sms, size_t room, int64_t counters_free,
                           const CallOptions &o, int busy = 0, double busy_until = 0.0)
{
    const std::vector<int32_t> &tcp = pl.rc.tcp;
    const int tt = tc_prefill_rows() / g;
    pl.tc_split.assign(tcp.size(), tc_split_pack(0, 1));
    pl.tc_groups = pl.tc_slots = 0;
    // pair costs per request, longest first (the launch order)
    std::vector<std::vector<int>> tiles(tcp.size());
    for (size_t x = 0; x < tcp.size(); x++) {
        const int32_t r = tcp[x], t = qsl_h[r + 1] - qsl_h[r], L = sl_h[r];
        const int npairs = (t + 2 * tt - 1) / (2 * tt);
        for (int k = npairs - 1; k >= 0; k--) tiles[x].push_back(tc_pair_tiles(t, L, tt, window, k));
    }
    auto count_ctas = [&](const std::vector<int32_t> &split) {
        int64_t n = 0;
        for (size_t x = 0; x < tcp.size(); x++) {
            const int whole = tc_split_whole(split[x]), pieces = tc_split_pieces(split[x]);
            const int np = (int)tiles[x].size();
            n += (int64_t)(pieces > 1 ? whole + (np - whole) * pieces : np) * hkv;
        }
        return n;
    };
    pl.tc_ctas = count_ctas(pl.tc_split);
    if (tcp.empty() || o.tc_key_pieces < 0) return;
    const size_t slot_bytes = 256 * ((size_t)d * 4 + 8);
    // One candidate: pairs that fit in the first wave run whole (forced:
    // none), every later pair of the request in `want` pieces (at most its
    // key tiles; uneven: the last piece small/64 of them).  Returns the
    // simulated makespan in key-tile times, in launch order (piece-major).
    auto candidate = [&](bool forced, int want, int small, std::vector<int32_t> &split, int64_t *groups,
                         int64_t *slots) {
        std::vector<double> costs;
        int64_t placed = 0;
        *groups = *slots = 0;
        for (size_t x = 0; x < tcp.size(); x++) {
            const std::vector<int> &c = tiles[x];
            int whole = 0;
            if (!forced)
                while (whole < (int)c.size() && placed + (int64_t)(whole + 1) * hkv <= sms) whole++;
            int pieces = whole < (int)c.size() ? want : 1;
            for (size_t k = whole; k < c.size(); k++) pieces = std::min(pieces, c[k]);
            pieces = std::max(1, std::min(pieces, kTcMaxPieces));
            if (!forced && whole < (int)c.size() && c[whole] < 16) pieces = 1;   // short pairs stay whole
            const int sm = pieces == 2 ? small : 0;
            if (pieces == 1) whole = 0;
            split[x] = tc_split_pack(whole, pieces, sm);
            for (int k = 0; k < whole; k++)
                for (int h = 0; h < hkv; h++) costs.push_back(c[k] + kTcCtaCost);
            if (pieces == 1) {
                for (size_t k = whole; k < c.size(); k++)
                    for (int h = 0; h < hkv; h++) costs.push_back(c[k] + kTcCtaCost);
            } else {
                for (int q = 0; q < pieces; q++)                    // piece-major
                    for (size_t k = whole; k < c.size(); k++) {
                        const int n = tc_piece_begin(c[k], q + 1, pieces, sm) - tc_piece_begin(c[k], q, pieces, sm);
                        for (int h = 0; h < hkv; h++) costs.push_back(n + kTcCtaCost + kTcPieceCost);
                    }
                *groups += (int64_t)(c.size() - whole) * hkv;
                *slots += (int64_t)(c.size() - whole) * hkv * pieces;
            }
            placed += (int64_t)(pieces > 1 ? whole + ((int)c.size() - whole) * pieces : (int)c.size()) * hkv;
        }
        return greedy_makespan(costs, sms, busy, busy_until);
    };
    std::vector<int32_t> best(pl.tc_split), cur(tcp.size());
    int64_t best_groups = 0, best_slots = 0, groups = 0, slots = 0;
    double best_ms = candidate(false, 1, 0, best, &best_groups, &best_slots);     // every pair whole
    struct Cand { int pieces, small; };
    std::vector<Cand> cands;
    if (o.tc_key_pieces >= 2) cands.push_back({o.tc_key_pieces, 0});
    else cands = {{2, 0}, {3, 0}, {4, 0}, {2, 8}, {2, 12}, {2, 16}, {2, 20}};
    for (const Cand &cd : cands) {
        const double ms = candidate(o.tc_key_pieces >= 2, cd.pieces, cd.small, cur, &groups, &slots);
        if (groups > counters_free || (size_t)slots * slot_bytes > room || slots == 0) continue;
        if (ms < best_ms * 0.99 || o.tc_key_pieces >= 2) {
            best = cur;
            best_ms = ms;
            best_groups = groups;
            best_slots = slots;
        }
    }
    pl.tc_split = best;
    pl.tc_groups = best_groups;
    pl.tc_slots = best_slots;
    pl.tc_ctas = count_ctas(best);
    pl.tc_makespan = best_ms;
}

// Costs of the tcgen05 grid rows in launch order (one row = the CTAs of one
// pair or piece, one per KV head), in key-tile times: the order in which
// attn_tc_kernel maps blockIdx.y to pairs and pieces.
static std::vector<double> tc_row_costs(const AttnPlan &pl, const int32_t *qsl_h, const int32_t *sl_h, int32_t g,
                                        int32_t window)
{
    std::vector<double> rows;
    const int tt = tc_prefill_rows() / g;
    for (size_t x = 0; x < pl.rc.tcp.size(); x++) {
        const int32_t r = pl.rc.tcp[x], t = qsl_h[r + 1] - qsl_h[r], L = sl_h[r];
        const int npairs = (t + 2 * tt - 1) / (2 * tt);
        const int whole = tc_split_whole(pl.tc_split[x]), pieces = tc_split_pieces(pl.tc_split[x]);
        const int sm = tc_split_small(pl.tc_split[x]);
        std::vector<int> c;
        for (int k = npairs - 1; k >= 0; k--) c.push_back(tc_pair_tiles(t, L, tt, window, k));
        if (pieces == 1) {
            for (int k = 0; k < npairs; k++) rows.push_back(c[k] + kTcCtaCost);
            continue;
        }
        for (int k = 0; k < whole; k++) rows.push_back(c[k] + kTcCtaCost);
        for (int q = 0; q < pieces; q++)
            for (int k = whole; k < npairs; k++)
                rows.push_back(tc_piece_begin(c[k], q + 1, pieces, sm) - tc_piece_begin(c[k], q, pieces, sm) +
                               kTcCtaCost + kTcPieceCost);
    }
    return rows;
}

static int32_t decode_splits_of(const int32_t *qsl_h, const int32_t *sl_h, int32_t r, int32_t window, int sp)
{
    return decode_splits(qsl_h[r + 1] - qsl_h[r], sl_h[r], window, sp);
}

static size_t plan_partial_rows(const AttnPlan &pl, const int32_t *qsl_h, const int32_t *sl_h, int32_t hq,
                                int32_t window, int sp, bool *too_many)
{
    size_t rows = 0;
    auto add = [&](int32_t r, int32_t S) {
        if (S > kMaxSplits) *too_many = true;
        if (S > 1) rows += (size_t)S * (qsl_h[r + 1] - qsl_h[r]) * hq;
    };
    for (int32_t r : pl.rc.dec) add(r, decode_splits_of(qsl_h, sl_h, r, window, sp));
    if (pl.pre_split)
        for (int32_t r : pl.rc.pre) add(r, sl_h[r] <= 0 ? 1 : (sl_h[r] + sp - 1) / sp);
    return rows;
}

// ---- mixed launch: the decode class inside the tcgen05 launch
//
// For a batch of prefill chunks on tcgen05 and decodes (one flattened
// ragged batch, "31. Engine v2", "Flattened ragged batches"), the tcgen05
// launch opens with a few decode CTAs: every one of their 12 warps runs
// decode items (request, KV head, key split) over its own ring of KV
// stages.  They hold their SMs only until the decode work is done, and the
// prefill CTAs, which follow them in launch order, take every other SM and
// then those: one launch for both classes, the HBM-bound decodes beside the
// tensor-bound prefill.  The planner sizes the decode CTAs by simulating the
// prefill schedule with their SMs busy until the decodes end and takes the
// arrangement when the predicted time beats the two-stream one's estimate.
// The decode CTAs' time is the larger of the bytes at kMixCtaGBs per CTA and
// the items of the busiest warp one after another (kMixItemUs + bytes at
// kMixWarpGBs each).  (Items taken from a queue counter instead of dealt
// round-robin evened the warps out but made the launch slower: 481 against
// 471 us on the same GPU.)  Measured on the mixed 2048-token-chunk step (0.67 GB
// of decode K/V in 1568 items of 1024 keys): 8 decode CTAs took 885 us
// (~95 GB/s each), 16 and 32 470 us against 520 us on two streams; on the
// 48-request engine step (128 short items) one item per warp took ~25 us,
// against 11 us for the whole step on two streams.
constexpr int kMixDecodeRows = 8;         // decode items: key-major tiles, t * g <= 8 rows per KV head
constexpr int kMixSplit = 1024;           // keys per decode item
constexpr int kMixDecodeWarps = 12;       // warps of a decode CTA (the tcgen05 CTA's 384 threads)
constexpr double kMixCtaGBs = 95.0;       // a decode CTA's rate, GB/s
constexpr double kMixWarpGBs = 10.0;      // one warp's rate over an item's blocks, GB/s
constexpr double kMixItemUs = 8.0;        // an item's start (its q, the first copies) and end
constexpr double kMixFp8Rate = 0.45;      // bytes per second of quantized-pool decode items, relative
constexpr double kTcTileUs = 1.66;        // a key tile of a pair on tcgen05, measured on the mixed step

static AttnPlan make_plan(const int32_t *qsl_h, const int32_t *sl_h, int32_t num_reqs, int32_t hq, int32_t hkv,
                          int32_t d, int32_t bs, int32_t window, bool fp8, bool fused, size_t workspace_bytes, int sms,
                          const CallOptions &o)
{
    AttnPlan pl;
    const int32_t g = hq / hkv;
    pl.rc = classify_requests(qsl_h, sl_h, num_reqs, g, hkv, d, window, fp8, workspace_bytes, o);
    const RequestClasses &rc = pl.rc;
    for (int r = 0; r < num_reqs; r++) pl.seen_l = sl_h[r] > pl.seen_l ? sl_h[r] : pl.seen_l;
    class_times(rc, qsl_h, sl_h, hq, hkv, d, &pl.dec_us, &pl.pre_us);
    // Prefill-class tiles are split over keys as well when the batch has too
    // few of them to fill the GPU (small, latency-bound steps): every tile of
    // such a request gets the request's number of splits.
    pl.tile = mma_prefill_rows() / g > 0 ? mma_prefill_rows() / g : 1;
    int64_t pre_ctas = 0;
    for (int32_t r : rc.pre) pre_ctas += (int64_t)((qsl_h[r + 1] - qsl_h[r] + pl.tile - 1) / pl.tile) * hkv;
    // Measured on the 48-request engine step it costs more (extra CTAs and a
    // combine on the critical path) than it saves, so it is opt-in.
    pl.pre_split = !rc.pre.empty() && pre_ctas < 2 * (int64_t)sms && o.prefill_key_splits;
    // The layout depends on the workspace size only: [error word][counters,
    // if the workspace holds them][partials]; quantized prefill on tcgen05:
    // its scratch takes the workspace's end.
    pl.ws_front = rc.fp8_scratch ? ((workspace_bytes - rc.fp8_scratch) & ~(size_t)255) : workspace_bytes;
    pl.has_counters = pl.ws_front >= kErrBytes + kCounterBytes + 64;
    pl.part_base = kErrBytes + (pl.has_counters ? kCounterBytes : 0);
    // with device lengths a request's keys are known only on the device:
    // splits merge through the counters, not clusters of evenly cut splits
    pl.cluster_opt = o.device_lengths ? -1 : o.cluster;

    // The split length, the workspace layout and the tcgen05 pieces for a
    // starting split length (grown until the decode partials fit) and
    // whether decodes run beside the tcgen05 CTAs.
    auto layout = [&](AttnPlan &q, int split, bool tc_alone) {
        if (split % bs) split += bs - split % bs;
        const size_t avail = q.ws_front - q.part_base;
        // every split request keeps S * t * hq partial rows; grow the split until they fit
        const size_t row_bytes = (size_t)d * 4 + 8;
        for (;;) {
            bool too_many = false;
            const size_t rows = plan_partial_rows(q, qsl_h, sl_h, hq, window, split, &too_many);
            if (!too_many && rows * row_bytes + 64 <= avail) break;
            if (split >= q.seen_l) break;                       // nothing is split any more
            split *= 2;
        }
        q.split = split;
        bool unused = false;
        q.total_rows = plan_partial_rows(q, qsl_h, sl_h, hq, window, split, &unused);
        // tcgen05 key pieces: their partial slots follow the decode partials,
        // their counters come first in the counter region
        const size_t dec_part = q.total_rows ? ((q.total_rows * d * 4 + 15) / 16) * 16 + q.total_rows * 8 : 0;
        q.tc_part_off = (q.part_base + dec_part + 255) & ~(size_t)255;
        const size_t tc_room = q.ws_front > q.tc_part_off + 64 ? q.ws_front - q.tc_part_off - 64 : 0;
        plan_tc_pieces(q, qsl_h, sl_h, g, hkv, d, window, sms, tc_room,
                       q.has_counters && tc_alone ? kCounterGroups / 2 : 0, o);
    };

    // ---- the decode class inside the tcgen05 launch, when it fits there
    // (quantized pools: the decode CTAs read the codes, the prefill CTAs the
    // bf16 copies of their requests' blocks)
    bool mix_ok = (!fp8 || (rc.fp8_scratch > 0 && d == 128)) && !rc.tcp.empty() && !rc.dec.empty() &&
                  rc.pre.empty() && o.mixed_launch >= 0 &&
                  rc.tcp.size() <= (size_t)kPlanMax && rc.dec.size() <= (size_t)kPlanMax && pl.has_counters &&
                  (d == 128 || d == 64 || d == 48);
    for (int32_t r : rc.dec)
        if ((qsl_h[r + 1] - qsl_h[r]) * g > kMixDecodeRows) mix_ok = false;
    if (mix_ok) {
        AttnPlan m = pl;
        layout(m, o.split_tokens > 0 ? o.split_tokens : kMixSplit, true);
        int64_t items = 0, counters = 0;
        double dec_bytes = 0.0;
        const double key_bytes = fp8 ? 2.0 * d + 8.0 : 4.0 * d;    // K and V of one key and head
        // quantized pools: a block carries half the bytes for the same MMA
        // work and the code conversions, so fewer bytes per second
        const double cta_gbs = fp8 ? kMixCtaGBs * kMixFp8Rate : kMixCtaGBs;
        const double warp_gbs = fp8 ? kMixWarpGBs * kMixFp8Rate : kMixWarpGBs;
        for (int32_t r : rc.dec) {
            const int32_t t = qsl_h[r + 1] - qsl_h[r], L = sl_h[r];
            const int S = decode_splits(t, L, window, m.split);
            dec_bytes += (double)std::max(0, L - decode_key_begin(t, L, window)) * hkv * key_bytes;
            items += (int64_t)S * hkv;
            if (S > 1) counters += hkv;
        }
        // decode CTAs: the count with the shortest simulated step (forced:
        // the option's count), the prefill pieces planned around them
        const size_t dec_part = m.total_rows ? ((m.total_rows * d * 4 + 15) / 16) * 16 + m.total_rows * 8 : 0;
        const size_t tc_room = m.ws_front > m.tc_part_off + 64 ? m.ws_front - m.tc_part_off - 64 : 0;
        (void)dec_part;
        const bool q_pieces_ok = m.has_counters && o.tc_key_pieces >= 2;
        double best = 1e30;
        int best_rows = 0;
        AttnPlan best_plan = m;
        // Pairs are cut into key pieces beside the decode CTAs only when the
        // option asks for pieces: measured on the mixed 2048-token-chunk step
        // on a quantized pool (32 decode CTAs), the pieces' merges cost more
        // than the evener prefill saved (497 against 472 us for the launch).
        const int piece_groups = q_pieces_ok ? kCounterGroups / 2 - (int)counters : 0;
        for (int rows = 1; rows * hkv <= sms / 2; rows *= 2) {
            if (o.mixed_decode_ctas > 0 && rows != std::max(1, (o.mixed_decode_ctas + hkv - 1) / hkv)) continue;
            const int n = rows * hkv;
            const double item_us = kMixItemUs + dec_bytes / items / (warp_gbs * 1e3);
            const double per_warp = std::ceil((double)items / (n * kMixDecodeWarps));
            const double dec_us = std::max(dec_bytes / (n * cta_gbs * 1e3), per_warp * item_us) + 5.0;
            // the decode CTAs' SMs go to the prefill as their warps finish:
            // the simulation holds them until the warps' mean finish
            const double free_us = std::max(dec_bytes / (n * cta_gbs * 1e3),
                                            items * item_us / (n * kMixDecodeWarps)) + 5.0;
            AttnPlan q = m;
            plan_tc_pieces(q, qsl_h, sl_h, g, hkv, d, window, sms, tc_room, piece_groups, o, n, free_us / kTcTileUs);
            const double step = std::max(dec_us, q.tc_makespan * kTcTileUs);
            if (step < best) {
                best = step;
                best_rows = rows;
                best_plan = q;
            }
        }
        if (o.mixed_decode_ctas > 0 && best_rows == 0) {                 // more than half the SMs: as asked
            const int rows = (o.mixed_decode_ctas + hkv - 1) / hkv;
            best_plan = m;
            plan_tc_pieces(best_plan, qsl_h, sl_h, g, hkv, d, window, sms, tc_room, piece_groups, o, rows * hkv,
                           dec_bytes / (rows * hkv * cta_gbs * 1e3) / kTcTileUs);
            best_rows = rows;
            best = 0.0;
        }
        // the two-stream arrangement, roughly: the prefill alone (whole
        // pairs) and the decodes at full HBM speed in what it leaves idle
        AttnPlan w = pl;
        layout(w, decode_split_tokens(rc, w.dec_us, w.pre_us, hkv, fp8, o, sms), false);
        // (quantized pools: the decode kernel over codes is not twice as fast
        // for half the bytes; measured on the mixed 2048-token-chunk step,
        // 120-127 us against 133 us on the bf16 pool)
        const double two_stream = w.tc_makespan * kTcTileUs + 0.5 * dec_bytes / (6.5e6 * (fp8 ? 0.5 : 1.0));
        counters += best_plan.tc_groups;
        if (best_rows > 0 && (best < two_stream || o.mixed_launch > 0) && counters <= kCounterGroups &&
            items < INT32_MAX) {
            best_plan.mix = true;
            best_plan.mix_items = (int32_t)items;
            best_plan.mix_dec_rows = best_rows;
            best_plan.mix_pred_us = best;
            best_plan.tc_self.assign(best_plan.rc.tcp.size(), 0);   // a mixed launch's chunks come from the scatter
            return best_plan;
        }
    }

    // Cut tcgen05 pairs only when no decode class runs beside them: measured
    // on the mixed 2048-token-chunk step, the decodes on the side stream fill
    // the SMs an uneven prefill leaves idle (step 518 us); with the prefill
    // evened out they run after it instead (563 us), although the prefill
    // alone gets faster (461 -> 445 us).
    layout(pl, decode_split_tokens(rc, pl.dec_us, pl.pre_us, hkv, fp8, o, sms), rc.dec.empty() || o.tc_key_pieces >= 2);
    // Decode-class work runs on a second stream, concurrently with the
    // prefill kernels, when both are present; the class expected to take
    // longer goes on the caller's stream (the decode_main option forces it).
    pl.fork = !rc.dec.empty() && (!rc.tcp.empty() || !rc.pre.empty()) && !o.no_overlap;
    if (pl.fork) {
        pl.decode_main = o.decode_main != 0 ? o.decode_main > 0 : pl.dec_us > pl.pre_us;
        // Combined call with the prefill class on the caller's stream: the
        // decodes fork after the ranged scatter, as they would after a full
        // scatter, so that the prefill kernel takes the SMs first (measured
        // on the mixed 2048-token-chunk step: 514 us this way, 570 us with
        // the decodes starting at once).
        pl.fork_after_scatter = fused && !pl.decode_main;
    }
    // Combined call on a bf16 pool, outside a mixed launch: a tcgen05 request
    // whose rows of each KV head are all one CTA's (a single pair of tiles,
    // not cut into key pieces) has its new rows written by that CTA.
    pl.tc_self.assign(rc.tcp.size(), 0);
    if (fused && !fp8 && !pl.mix) {
        const int tt = tc_prefill_rows() / g;
        for (size_t x = 0; x < rc.tcp.size(); x++) {
            const int32_t t = qsl_h[rc.tcp[x] + 1] - qsl_h[rc.tcp[x]];
            const int npairs = (t + 2 * tt - 1) / (2 * tt);
            const int whole = tc_split_whole(pl.tc_split[x]), pieces = tc_split_pieces(pl.tc_split[x]);
            pl.tc_self[x] = (pieces > 1 ? whole + (npairs - whole) * pieces : npairs) == 1;
        }
    }
    return pl;
}


// CTAs per thread-block cluster of a decode launch whose requests have at
// most s_max splits, or 0 for no clusters.  Short split decodes (the
// slot-ring kernel) run each request's splits as one cluster that combines
// them through its shared memory: every request of the launch gets the
// launch's largest split count, its keys divided evenly.  Measured on the
// 48-request engine step, clusters of more than two CTAs do not run beside
// the prefill kernel (the step took the sum of both kernels' times), so next
// to prefill work the cluster holds at most two splits.  The cluster option
// turns clusters off (-1) or forces n >= 2 CTAs.
static int decode_cluster_size(const AttnPlan &pl, int s_max)
{
    const int cs = pl.cluster_opt >= 2 ? std::min(pl.cluster_opt, kMaxClusterSplits)
                                       : (pl.fork ? std::min(s_max, 2) : s_max);
    return pl.split < kLongSplitTokens && pl.cluster_opt >= 0 && cs >= 2 && cs <= kMaxClusterSplits ? cs : 0;
}

static pkv_status attention_impl(void *out, const void *q, const void *k_cache, const void *v_cache,
                                 const float *k_scale, const float *v_scale, const int32_t *query_start_loc,
                                 const int32_t *seq_lens, const int32_t *block_table, int32_t block_table_stride,
                                 const int32_t *qsl_h, const int32_t *sl_h, int32_t num_reqs, int32_t num_tokens,
                                 int32_t max_query_len, int32_t max_seq_len, int32_t hq, int32_t hkv, int32_t d,
                                 int32_t bs, int32_t num_blocks_total, float scale, int32_t window, void *workspace,
                                 size_t workspace_bytes, cudaStream_t stream, const CallOptions &opts,
                                 const void *fw_k = nullptr, const void *fw_v = nullptr,
                                 const int64_t *fw_slots = nullptr)
{
    const bool fp8 = k_scale != nullptr;
    bool nothing_to_do = false;
    if (pkv_status st = validate_attention(out, q, k_cache, v_cache, k_scale, v_scale, query_start_loc, seq_lens,
                                           block_table, block_table_stride, qsl_h, sl_h, num_reqs, num_tokens,
                                           max_query_len, max_seq_len, hq, hkv, d, bs, num_blocks_total, window,
                                           workspace, workspace_bytes, &nothing_to_do);
        st != PKV_OK || nothing_to_do)
        return st;
    const int32_t g = hq / hkv;
    const bool fused = fw_k != nullptr;
    // blocks of more than 16 slots: the 16-slot block table takes the workspace's end
    int32_t w16 = 0;
    const size_t t16 = table16_bytes(sl_h, num_reqs, bs, &w16);
    if (t16 && workspace_bytes < t16 + PKV_WORKSPACE_MIN_BYTES + 256) return PKV_ERR_WORKSPACE;
    const size_t plan_ws = t16 ? (workspace_bytes - t16) & ~(size_t)255 : workspace_bytes;
    const AttnPlan pl =
        make_plan(qsl_h, sl_h, num_reqs, hq, hkv, d, bs, window, fp8, fused, plan_ws, num_sms(), opts);
    // device lengths: decode batches only (prefill tiles are planned from their lengths)
    if (opts.device_lengths && (!pl.rc.tcp.empty() || !pl.rc.pre.empty())) return PKV_ERR_UNSUPPORTED;
    LaunchChoices lc;
    lc.pdl = !opts.no_pdl;
    lc.decode_row_tiles = opts.decode_row_tiles;
    const ScopedLaunchChoices scoped(lc);
    const std::vector<int32_t> &dec = pl.rc.dec, &pre = pl.rc.pre, &tcp = pl.rc.tcp;
    const size_t fp8_scratch = pl.rc.fp8_scratch;
    const int64_t fp8_blocks = pl.rc.fp8_blocks;
    const int32_t fp8_width = pl.rc.fp8_width;
    if (!tcp.empty() && ((int64_t)num_blocks_total * bs >= INT32_MAX || num_tokens >= INT32_MAX / 2))
        return PKV_ERR_UNSUPPORTED;
    const int split = pl.split;
    const int tile = pl.tile;
    const bool pre_split = pl.pre_split;
    const bool has_counters = pl.has_counters;
    const size_t ws_front = pl.ws_front, part_base = pl.part_base;
    // prefill tiles: every tile of a split request gets ceil(L / split) splits;
    // decode-class requests: splits over their (windowed) key range
    auto splits_of = [&](int32_t L, int sp) { return L <= 0 ? 1 : (L + sp - 1) / sp; };
    auto dec_splits_of = [&](int32_t r, int sp) { return decode_splits_of(qsl_h, sl_h, r, window, sp); };

    const int64_t num_slots = (int64_t)num_blocks_total * bs;
    char *ws = static_cast<char *>(workspace);
    AttnParams p = {};
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.k_cache = static_cast<const __nv_bfloat16 *>(k_cache);
    p.v_cache = static_cast<const __nv_bfloat16 *>(v_cache);
    p.qsl = query_start_loc;
    p.seq_lens = seq_lens;
    p.block_table = block_table;
    p.bt_stride = block_table_stride;
    p.hq = hq;
    p.hkv = hkv;
    p.group = g;
    p.block_size = bs;
    p.nb_total = num_blocks_total;
    const float sc = scale > 0.f ? scale : 1.0f / sqrtf((float)d);
    p.scale_log2 = sc * 1.4426950408889634f;
    p.err = reinterpret_cast<uint32_t *>(ws);
    // partial rows: first all o rows, then the (m, l) pairs
    const size_t total_rows = pl.total_rows;
    p.part_o = reinterpret_cast<float *>(ws + part_base);
    p.part_ml = reinterpret_cast<float2 *>(ws + part_base + ((total_rows * d * 4 + 15) / 16) * 16);
    p.counters = has_counters ? reinterpret_cast<uint32_t *>(ws + kErrBytes) : nullptr;
    p.window = window;
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    p.fw_k = static_cast<const uint4 *>(fw_k);
    p.fw_v = static_cast<const uint4 *>(fw_v);
    p.fw_kc = fused ? static_cast<uint4 *>(const_cast<void *>(k_cache)) : nullptr;
    p.fw_vc = fused ? static_cast<uint4 *>(const_cast<void *>(v_cache)) : nullptr;
    p.fw_slots = fused ? fw_slots : nullptr;
    p.fw_ks = fused && fp8 ? const_cast<float *>(k_scale) : nullptr;
    p.fw_vs = fused && fp8 ? const_cast<float *>(v_scale) : nullptr;
    p.dev_len = opts.device_lengths ? 1 : 0;
    // blocks of more than 16 slots: the same pool as blocks of 16 slots (the
    // layout [blocks][16 << s][Hkv][d] is [blocks << s][16][Hkv][d]), read
    // through a table of 16-slot entries expanded at the workspace's end
    if (t16) {
        const int shift = block_shift(bs);
        int32_t *bt16 = reinterpret_cast<int32_t *>(ws + plan_ws);
        cudaError_t e = launch_expand_table(block_table, block_table_stride, bt16, w16, num_reqs, shift,
                                            num_blocks_total, stream);
        if (e != cudaSuccess) return cuda_fail(e, "block table expansion launch");
        p.block_table = bt16;
        p.bt_stride = w16;
        p.nb_total = num_blocks_total << shift;
        p.block_size = 16;
    }
    AttnParams pp = p;                                   // prefill launches: their rows come from the scatter
    pp.fw_k = pp.fw_v = nullptr;
    pp.fw_kc = pp.fw_vc = nullptr;
    pp.fw_slots = nullptr;
    pp.fw_ks = pp.fw_vs = nullptr;

    // ---- decode-class work runs on a side stream, concurrently with the
    // prefill kernels, when both are present: its CTAs fill the SMs that the
    // prefill leaves idle (its last wave, or a small batch's spare SMs).
    // Fork and join with events, so the caller's stream order (and CUDA-graph
    // capture) is preserved.
    cudaStream_t dstream = stream, pstream = stream;         // decode-class / prefill-class work
    // (without a side stream for the caller's stream, both run on it in turn)
    SideStream *side = pl.fork ? side_stream_for(stream) : nullptr;
    const bool fork = side != nullptr;
    const bool fork_after_scatter = fork && pl.fork_after_scatter;
    if (fork) {
        side->mu.lock();
        // The class on the caller's stream follows the K/V scatter as a
        // programmatic dependent (it starts while the scatter drains); the
        // other one waits for the fork event.
        if (pl.decode_main) pstream = side->stream;
        else dstream = side->stream;
        if (!fork_after_scatter) {
            cudaError_t e = cudaEventRecord(side->fork, stream);
            if (e == cudaSuccess) e = cudaStreamWaitEvent(side->stream, side->fork, 0);
            if (e != cudaSuccess) {
                side->mu.unlock();
                return cuda_fail(e, "fork");
            }
        }
    }
    bool joined = !fork;
    auto join = [&]() -> cudaError_t {
        if (joined) return cudaSuccess;
        joined = true;
        cudaError_t e = cudaEventRecord(side->join, side->stream);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, side->join, 0);
        side->mu.unlock();
        return e;
    };

    // list request r in wl with its planned metadata; returns its index
    auto list_request = [&](WorkList &wl, int32_t r) -> int {
        const int li = wl.n++;
        wl.req[li] = r;
        wl.qb[li] = qsl_h[r];
        wl.qt[li] = qsl_h[r + 1] - qsl_h[r];
        wl.len[li] = sl_h[r];
        wl.cnt_off[li] = -1;
        return li;
    };

    // ---- combined call: the prefill-class rows are scattered ahead of the
    // prefill kernels, on their stream (the decode class writes its own, and
    // so does the tcgen05 CTA of a bf16 request whose rows of a KV head are
    // all that one CTA's: a single pair of tiles, not cut into key pieces,
    // outside a mixed launch)
    const std::vector<char> &tc_self = pl.tc_self;
    const bool any_self = std::find(tc_self.begin(), tc_self.end(), 1) != tc_self.end();
    if (fused) {
        std::vector<int32_t> prows;
        for (size_t x = 0; x < tcp.size(); x++)
            if (x >= tc_self.size() || !tc_self[x]) prows.push_back(tcp[x]);
        prows.insert(prows.end(), pre.begin(), pre.end());
        for (size_t c0 = 0; c0 < prows.size(); c0 += kPlanMax) {
            TokenRanges rg;
            memset(&rg, 0, sizeof rg);
            size_t c1 = c0 + kPlanMax < prows.size() ? c0 + kPlanMax : prows.size();
            for (size_t x = c0; x < c1; x++) {
                const int32_t r = prows[x];
                rg.begin[rg.n] = qsl_h[r];
                rg.off[rg.n + 1] = rg.off[rg.n] + (qsl_h[r + 1] - qsl_h[r]);
                rg.n++;
            }
            cudaError_t e =
                fp8 ? launch_kv_write_fp8_ranges(fw_k, fw_v, const_cast<void *>(k_cache), const_cast<void *>(v_cache),
                                                 p.fw_ks, p.fw_vs, fw_slots, rg, hkv, num_slots, p.err, pstream)
                    : launch_kv_write_ranges(fw_k, fw_v, const_cast<void *>(k_cache), const_cast<void *>(v_cache),
                                             fw_slots, rg, hkv * d * 2, num_slots, p.err, pstream);
            if (e != cudaSuccess) {
                join();
                return cuda_fail(e, "ranged K/V scatter launch");
            }
        }
    }
    if (fork_after_scatter) {
        cudaError_t e = cudaEventRecord(side->fork, stream);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(side->stream, side->fork, 0);
        if (e != cudaSuccess) {
            join();
            return cuda_fail(e, "fork");
        }
    }

    // ---- quantized pools: bf16 copies of the tcgen05 requests' blocks
    AttnParams pt = pp;                                  // the tcgen05 launches' parameters
    if (any_self) {                                      // their single-CTA requests write their own rows
        pt.fw_k = p.fw_k;
        pt.fw_v = p.fw_v;
        pt.fw_kc = p.fw_kc;
        pt.fw_vc = p.fw_vc;
        pt.fw_slots = p.fw_slots;
    }
    const void *tc_k = k_cache, *tc_v = v_cache;
    int64_t tc_slots = num_slots;
    if (fp8_scratch && !tcp.empty()) {
        char *sc = ws + ws_front;                        // 256-aligned; the scratch fits before the end
        const size_t kv = ((size_t)fp8_blocks * 16 * hkv * d * 2 + 255) / 256 * 256;
        __nv_bfloat16 *sk = reinterpret_cast<__nv_bfloat16 *>(sc);
        __nv_bfloat16 *sv = reinterpret_cast<__nv_bfloat16 *>(sc + kv);
        int32_t *stab = reinterpret_cast<int32_t *>(sc + 2 * kv);
        int32_t sblk0 = 0;
        for (size_t c0 = 0; c0 < tcp.size(); c0 += kPlanMax) {
            WorkList wl;
            memset(&wl, 0, sizeof wl);
            size_t c1 = c0 + kPlanMax < tcp.size() ? c0 + kPlanMax : tcp.size();
            int32_t blocks = 0;
            for (size_t x = c0; x < c1; x++) {
                const int32_t r = tcp[x];
                const int li = list_request(wl, r);
                wl.item_off[li] = blocks;
                blocks += (sl_h[r] + 15) / 16;
            }
            wl.item_off[wl.n] = blocks;
            cudaError_t e = launch_fp8_dequant(p, wl, sk, sv, stab, fp8_width, sblk0, pstream);
            if (e != cudaSuccess) {
                join();
                return cuda_fail(e, "quantized prefill dequant launch");
            }
            sblk0 += blocks;
        }
        pt.k_cache = sk;
        pt.v_cache = sv;
        pt.block_table = stab;
        pt.bt_stride = fp8_width;
        pt.nb_total = (int32_t)fp8_blocks;              // blocks of 16 slots
        pt.block_size = 16;
        pt.k_scale = pt.v_scale = nullptr;
        tc_k = sk;
        tc_v = sv;
        tc_slots = fp8_blocks * 16;
    }

    // ---- split partials and counters of the decode class (and of warp-MMA prefill)
    struct CombineSet {
        std::vector<int32_t> reqs, offs;
        int max_rows = 0;
    };
    CombineSet dec_combine, pre_combine;
    size_t part_cursor = 0;
    int counter_cursor = (int)pl.tc_groups;                   // after the tcgen05 pieces' counters
    // partial rows of a split request; combined by `set`'s combine launch,
    // or inside the attention kernel when in_kernel
    auto take_partials = [&](CombineSet &set, int32_t r, int32_t S, bool in_kernel = false) -> int32_t {
        if (S <= 1) return -1;
        const int32_t t = qsl_h[r + 1] - qsl_h[r];
        const int32_t off = (int32_t)part_cursor;
        if (!in_kernel) {
            set.reqs.push_back(r);
            set.offs.push_back(off);
        }
        part_cursor += (size_t)S * t * hq;
        if (t * hq > set.max_rows) set.max_rows = t * hq;
        return off;
    };
    // merge the split partials of one set of requests on `st` (mode: the
    // class the partials come from, which fixes their split count)
    auto launch_combines = [&](const CombineSet &set, int mode, cudaStream_t st) -> cudaError_t {
        for (size_t c0 = 0; c0 < set.reqs.size(); c0 += kPlanMax) {
            WorkList wl;
            memset(&wl, 0, sizeof wl);
            wl.mode = mode;
            wl.split_tokens = split;
            size_t c1 = c0 + kPlanMax < set.reqs.size() ? c0 + kPlanMax : set.reqs.size();
            for (size_t x = c0; x < c1; x++) {
                int li = list_request(wl, set.reqs[x]);
                wl.part_off[li] = set.offs[x];
                wl.item_off[li] = li;
            }
            wl.item_off[wl.n] = wl.n;
            cudaError_t e = launch_attn_combine(p, wl, d, set.max_rows, st);
            if (e != cudaSuccess) return e;
        }
        return cudaSuccess;
    };
    // ---- mixed launch: the decode class as items of the tcgen05 launch's decode CTAs
    WorkList mix_dl;
    MixAssign mix_as;
    if (pl.mix) {
        memset(&mix_dl, 0, sizeof mix_dl);
        mix_dl.mode = kModeDecode;
        mix_dl.split_tokens = split;
        int items = 0;
        for (int32_t r : dec) {
            const int32_t S = dec_splits_of(r, split);
            const int li = list_request(mix_dl, r);
            mix_dl.item_off[li] = items;
            mix_dl.part_off[li] = take_partials(dec_combine, r, S, true);
            if (S > 1) {
                mix_dl.cnt_off[li] = counter_cursor;
                counter_cursor += hkv;
            }
            items += S * hkv;
        }
        mix_dl.item_off[mix_dl.n] = items;
        mix_as.dec_rows = pl.mix_dec_rows;
        if (counter_cursor > kCounterGroups || items != pl.mix_items) return PKV_ERR_UNSUPPORTED;
    }

    // ---- tensor-core prefill launches, submitted first: the longest work.
    // Pairs cut into key pieces keep fp32 partials in slots of 256 rows at
    // tc_part_off and count on the first tc_groups split counters.
    if (pl.tc_slots > 0) {
        pt.part_o = reinterpret_cast<float *>(ws + pl.tc_part_off);
        pt.part_ml = reinterpret_cast<float2 *>(ws + pl.tc_part_off + (size_t)pl.tc_slots * 256 * d * 4);
    }
    int64_t tc_slot_cursor = 0, tc_counter_cursor = 0;
    for (size_t c0 = 0; c0 < tcp.size(); c0 += kPlanMax) {
        WorkList wl;
        memset(&wl, 0, sizeof wl);
        wl.mode = kModePrefill;
        wl.tile_tokens = tc_prefill_rows() / g;
        int items = 0;
        size_t c1 = c0 + kPlanMax < tcp.size() ? c0 + kPlanMax : tcp.size();
        for (size_t x = c0; x < c1; x++) {
            int32_t r = tcp[x];
            int32_t t = qsl_h[r + 1] - qsl_h[r];
            int li = list_request(wl, r);
            const int npairs = (t + 2 * wl.tile_tokens - 1) / (2 * wl.tile_tokens);   // pairs of 128-row tiles
            const int whole = tc_split_whole(pl.tc_split[x]), pieces = tc_split_pieces(pl.tc_split[x]);
            wl.tc_split[li] = pl.tc_split[x];
            wl.item_off[li] = items;
            wl.part_off[li] = (int32_t)tc_slot_cursor;
            wl.cnt_off[li] = (int32_t)tc_counter_cursor;
            if (pieces > 1) {
                tc_slot_cursor += (int64_t)(npairs - whole) * hkv * pieces;
                tc_counter_cursor += (int64_t)(npairs - whole) * hkv;
                items += whole + (npairs - whole) * pieces;
            } else {
                items += npairs;
            }
        }
        wl.item_off[wl.n] = items;
        cudaError_t e = pl.mix ? launch_attn_tc(pt, wl, items, q, num_tokens, tc_k, tc_v, tc_slots, d, pstream, &p,
                                                &mix_dl, &mix_as)
                               : launch_attn_tc(pt, wl, items, q, num_tokens, tc_k, tc_v, tc_slots, d, pstream);
        if (e != cudaSuccess) {
            join();
            return cuda_fail(e, "tensor-core prefill launch");
        }
    }

    // ---- decode-class launches (chunks of kPlanMax requests; none in a mixed launch)
    for (size_t c0 = 0; !pl.mix && c0 < dec.size(); c0 += kPlanMax) {
        WorkList wl;
        memset(&wl, 0, sizeof wl);
        wl.mode = kModeDecode;
        wl.split_tokens = split;
        wl.tile_tokens = 0;
        int items = 0;
        size_t c1 = c0 + kPlanMax < dec.size() ? c0 + kPlanMax : dec.size();
        int s_max = 1;
        for (size_t x = c0; x < c1; x++) s_max = std::max(s_max, dec_splits_of(dec[x], split));
        const int cs = decode_cluster_size(pl, s_max);
        if (cs) {
            wl.cluster = cs;
            for (size_t x = c0; x < c1; x++) {
                const int32_t r = dec[x], t = qsl_h[r + 1] - qsl_h[r];
                const int li = list_request(wl, r);
                const int32_t keys = sl_h[r] - decode_key_begin(t, sl_h[r], window);
                const int32_t per = (keys + cs - 1) / cs;
                wl.split_len[li] = std::max(bs, (per + bs - 1) / bs * bs);
                wl.item_off[li] = items;
                wl.part_off[li] = -1;
                items += cs;
            }
            wl.item_off[wl.n] = items;
            cudaError_t e = launch_attn_mma(p, wl, d, items, k_cache, v_cache, num_slots, dstream, k_scale, v_scale);
            if (e != cudaSuccess) {
                join();
                return cuda_fail(e, "decode attention launch");
            }
            continue;
        }
        for (size_t x = c0; x < c1; x++) {
            int32_t r = dec[x];
            int32_t t = qsl_h[r + 1] - qsl_h[r];
            int32_t S = dec_splits_of(r, split);
            int li = list_request(wl, r);
            wl.item_off[li] = items;
            // split decodes of the MMA kernels combine in the kernel (the CTA
            // finishing a request's last split) when counters are available
            const bool in_kernel = S > 1 && has_counters && counter_cursor + hkv <= kCounterGroups;
            wl.part_off[li] = take_partials(dec_combine, r, S, in_kernel);
            if (in_kernel) {
                wl.cnt_off[li] = counter_cursor;
                counter_cursor += hkv;
            }
            items += S;
        }
        wl.item_off[wl.n] = items;
        cudaError_t e =
            launch_attn_mma(p, wl, d, items, k_cache, v_cache, num_slots, dstream, k_scale, v_scale);
        if (e != cudaSuccess) {
            join();
            return cuda_fail(e, "decode attention launch");
        }
    }

    if (cudaError_t e = launch_combines(dec_combine, kModeDecode, dstream); e != cudaSuccess) {
        join();
        return cuda_fail(e, "split combine launch");
    }

    // ---- prefill-class launches (tiles of `tile` tokens, split over keys
    // when pre_split)
    for (size_t c0 = 0; c0 < pre.size(); c0 += kPlanMax) {
        WorkList wl;
        memset(&wl, 0, sizeof wl);
        wl.mode = kModePrefill;
        wl.split_tokens = pre_split ? split : 0;
        wl.tile_tokens = tile;
        int items = 0;
        size_t c1 = c0 + kPlanMax < pre.size() ? c0 + kPlanMax : pre.size();
        for (size_t x = c0; x < c1; x++) {
            int32_t r = pre[x];
            int32_t t = qsl_h[r + 1] - qsl_h[r];
            const int32_t S = pre_split ? splits_of(sl_h[r], split) : 1;
            int li = list_request(wl, r);
            wl.item_off[li] = items;
            wl.part_off[li] = take_partials(pre_combine, r, S);
            items += ((t + tile - 1) / tile) * S;
        }
        wl.item_off[wl.n] = items;
        cudaError_t e =
            launch_attn_mma(pp, wl, d, items, k_cache, v_cache, num_slots, pstream, k_scale, v_scale);
        if (e != cudaSuccess) {
            join();
            return cuda_fail(e, "prefill attention launch");
        }
    }
    if (part_cursor > (size_t)INT32_MAX) {
        join();
        return PKV_ERR_WORKSPACE;
    }

    if (cudaError_t e = launch_combines(pre_combine, kModePrefill, pstream); e != cudaSuccess) {
        join();
        return cuda_fail(e, "split combine launch");
    }
    cudaError_t ej = join();
    if (ej != cudaSuccess) return cuda_fail(ej, "join");
    return PKV_OK;
}

extern "C" {

pkv_status pkv_ragged_paged_attention_ex(void *out, const void *q, const void *k_cache, const void *v_cache,
                                         const int32_t *query_start_loc, const int32_t *seq_lens,
                                         const int32_t *block_table, int32_t block_table_stride,
                                         const int32_t *qsl_h, const int32_t *sl_h, int32_t num_reqs,
                                         int32_t num_tokens, int32_t max_query_len, int32_t max_seq_len, int32_t hq,
                                         int32_t hkv, int32_t d, int32_t bs, int32_t num_blocks_total, float scale,
                                         int32_t window, void *workspace, size_t workspace_bytes,
                                         const pkv_attention_options *options, cudaStream_t stream)
{
    return attention_impl(out, q, k_cache, v_cache, nullptr, nullptr, query_start_loc, seq_lens, block_table,
                          block_table_stride, qsl_h, sl_h, num_reqs, num_tokens, max_query_len, max_seq_len, hq, hkv,
                          d, bs, num_blocks_total, scale, window, workspace, workspace_bytes, stream,
                          call_options(options));
}

pkv_status pkv_ragged_paged_attention(void *out, const void *q, const void *k_cache, const void *v_cache,
                                      const int32_t *query_start_loc, const int32_t *seq_lens,
                                      const int32_t *block_table, int32_t block_table_stride,
                                      const int32_t *qsl_h, const int32_t *sl_h, int32_t num_reqs,
                                      int32_t num_tokens, int32_t max_query_len, int32_t max_seq_len,
                                      int32_t hq, int32_t hkv, int32_t d, int32_t bs,
                                      int32_t num_blocks_total, float scale, int32_t window,
                                      void *workspace, size_t workspace_bytes, cudaStream_t stream)
{
    return pkv_ragged_paged_attention_ex(out, q, k_cache, v_cache, query_start_loc, seq_lens, block_table,
                                         block_table_stride, qsl_h, sl_h, num_reqs, num_tokens, max_query_len,
                                         max_seq_len, hq, hkv, d, bs, num_blocks_total, scale, window, workspace,
                                         workspace_bytes, nullptr, stream);
}

pkv_status pkv_plan_attention(const int32_t *qsl_h, const int32_t *sl_h, int32_t num_reqs, int32_t hq, int32_t hkv,
                              int32_t d, int32_t bs, int32_t window, int32_t quantized, int32_t combined,
                              size_t workspace_bytes, int32_t sms, const pkv_attention_options *options,
                              pkv_attention_plan *out)
{
    if (!out || !qsl_h || num_reqs < 0 || (num_reqs > 0 && !sl_h)) return PKV_ERR_INVALID_ARG;
    if (hq <= 0 || hkv <= 0 || hq % hkv || d <= 0 || bs <= 0 || window < 0) return PKV_ERR_INVALID_ARG;
    for (int r = 0; r < num_reqs; r++) {
        const int32_t t = qsl_h[r + 1] - qsl_h[r], L = sl_h[r];
        if (t < 0 || L < 0 || (L > 0 && t > L)) return PKV_ERR_INVALID_ARG;
    }
    const int32_t g = hq / hkv;
    if ((d != 48 && d != 64 && d != 128) || block_shift(bs) < 0 || g > kDecodeRows) return PKV_ERR_UNSUPPORTED;
    if (quantized && (d != 128 || hkv % 4 != 0)) return PKV_ERR_UNSUPPORTED;
    if (sms <= 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
            (void)cudaGetLastError();
            return PKV_ERR_CUDA;
        }
    }
    const CallOptions copts = call_options(options);
    int32_t w16 = 0;
    const size_t t16 = table16_bytes(sl_h, num_reqs, bs, &w16);
    if (t16 && workspace_bytes < t16 + PKV_WORKSPACE_MIN_BYTES + 256) return PKV_ERR_WORKSPACE;
    const size_t plan_ws = t16 ? (workspace_bytes - t16) & ~(size_t)255 : workspace_bytes;
    const AttnPlan pl = make_plan(qsl_h, sl_h, num_reqs, hq, hkv, d, bs, window, quantized != 0, combined != 0,
                                  plan_ws, sms, copts);
    if (copts.device_lengths && (!pl.rc.tcp.empty() || !pl.rc.pre.empty())) return PKV_ERR_UNSUPPORTED;
    memset(out, 0, sizeof *out);
    out->decode_requests = (int32_t)pl.rc.dec.size();
    out->prefill_tensor_requests = (int32_t)pl.rc.tcp.size();
    out->prefill_mma_requests = (int32_t)pl.rc.pre.size();
    out->decode_split_tokens = pl.split;
    int s_max = 1, s_first = 1;
    for (size_t x = 0; x < pl.rc.dec.size(); x++) {
        const int S = decode_splits_of(qsl_h, sl_h, pl.rc.dec[x], window, pl.split);
        s_max = std::max(s_max, S);
        if (x < (size_t)kPlanMax) s_first = std::max(s_first, S);
    }
    out->max_decode_splits = pl.rc.dec.empty() ? 0 : s_max;
    out->decode_cluster = pl.rc.dec.empty() ? 0 : decode_cluster_size(pl, s_first);
    out->decode_streaming = !pl.rc.dec.empty() && out->decode_cluster == 0 && pl.split >= kLongSplitTokens;
    out->split_counters = pl.has_counters;
    out->overlap = pl.fork;
    out->decode_on_caller_stream = pl.fork && pl.decode_main;
    out->prefill_key_splits = pl.pre_split;
    out->prefill_tensor_pieces = (int32_t)pl.tc_slots;
    out->mixed_launch = pl.mix;
    out->mixed_decode_items = pl.mix ? pl.mix_items : 0;
    out->mixed_decode_ctas = pl.mix ? pl.mix_dec_rows * hkv : 0;
    out->mixed_predicted_us = pl.mix ? (int32_t)std::lround(pl.mix_pred_us) : 0;
    out->prefill_tensor_own_rows = (int32_t)std::count(pl.tc_self.begin(), pl.tc_self.end(), 1);
    if (pl.mix) {
        out->decode_cluster = 0;
        out->decode_streaming = 0;
    }
    out->quantized_prefill_scratch = pl.rc.fp8_scratch;
    out->partial_bytes = pl.total_rows ? ((pl.total_rows * d * 4 + 15) / 16) * 16 + pl.total_rows * 8 : 0;
    return PKV_OK;
}

pkv_status pkv_paged_kv_write_attention_ex(const void *k, const void *v, void *k_cache, void *v_cache,
                                           const int64_t *slot_mapping, void *out, const void *q,
                                           const int32_t *query_start_loc, const int32_t *seq_lens,
                                           const int32_t *block_table, int32_t block_table_stride,
                                           const int32_t *qsl_h, const int32_t *sl_h, int32_t num_reqs,
                                           int32_t num_tokens, int32_t max_query_len, int32_t max_seq_len,
                                           int32_t hq, int32_t hkv, int32_t d, int32_t bs, int32_t num_blocks_total,
                                           float scale, int32_t window, void *workspace, size_t workspace_bytes,
                                           const pkv_attention_options *options, cudaStream_t stream)
{
    // the scatter's own checks, then the attention's (inside attention_impl)
    if (num_tokens > 0 && (!k || !v || !slot_mapping || !k_cache || !v_cache)) return PKV_ERR_INVALID_ARG;
    if (num_tokens > 0 && (!aligned(k, 16) || !aligned(v, 16) || !aligned(slot_mapping, 8)))
        return PKV_ERR_UNSUPPORTED;
    if (!workspace || workspace_bytes < PKV_WORKSPACE_MIN_BYTES || !aligned(workspace, 256)) return PKV_ERR_WORKSPACE;
    const CallOptions opts = call_options(options);
    if (opts.separate_write) {
        // the full scatter, then the attention
        if (num_tokens > 0) {
            if (hq <= 0 || hkv <= 0 || hq % hkv != 0 || d <= 0 || bs <= 0 || num_blocks_total <= 0)
                return PKV_ERR_INVALID_ARG;
            LaunchChoices lc;
            lc.pdl = !opts.no_pdl;
            const ScopedLaunchChoices scoped(lc);
            pkv_status st = pkv_paged_kv_write(k, v, k_cache, v_cache, slot_mapping, num_tokens, hkv, d, bs,
                                               num_blocks_total, static_cast<uint32_t *>(workspace), stream);
            if (st != PKV_OK) return st;
        }
        return attention_impl(out, q, k_cache, v_cache, nullptr, nullptr, query_start_loc, seq_lens, block_table,
                              block_table_stride, qsl_h, sl_h, num_reqs, num_tokens, max_query_len, max_seq_len, hq,
                              hkv, d, bs, num_blocks_total, scale, window, workspace, workspace_bytes, stream, opts);
    }
    return attention_impl(out, q, k_cache, v_cache, nullptr, nullptr, query_start_loc, seq_lens, block_table,
                          block_table_stride, qsl_h, sl_h, num_reqs, num_tokens, max_query_len, max_seq_len, hq, hkv,
                          d, bs, num_blocks_total, scale, window, workspace, workspace_bytes, stream, opts, k, v,
                          slot_mapping);
}

pkv_status pkv_paged_kv_write_attention(const void *k, const void *v, void *k_cache, void *v_cache,
                                        const int64_t *slot_mapping, void *out, const void *q,
                                        const int32_t *query_start_loc, const int32_t *seq_lens,
                                        const int32_t *block_table, int32_t block_table_stride,
                                        const int32_t *qsl_h, const int32_t *sl_h, int32_t num_reqs,
                                        int32_t num_tokens, int32_t max_query_len, int32_t max_seq_len,
                                        int32_t hq, int32_t hkv, int32_t d, int32_t bs, int32_t num_blocks_total,
                                        float scale, int32_t window, void *workspace, size_t workspace_bytes,
                                        cudaStream_t stream)
{
    return pkv_paged_kv_write_attention_ex(k, v, k_cache, v_cache, slot_mapping, out, q, query_start_loc, seq_lens,
                                           block_table, block_table_stride, qsl_h, sl_h, num_reqs, num_tokens,
                                           max_query_len, max_seq_len, hq, hkv, d, bs, num_blocks_total, scale,
                                           window, workspace, workspace_bytes, nullptr, stream);
}

pkv_status pkv_paged_kv_write_attention_fp8_ex(const void *k, const void *v, void *k_cache, void *v_cache,
                                               float *k_scale, float *v_scale, const int64_t *slot_mapping, void *out,
                                               const void *q, const int32_t *query_start_loc, const int32_t *seq_lens,
                                               const int32_t *block_table, int32_t block_table_stride,
                                               const int32_t *qsl_h, const int32_t *sl_h, int32_t num_reqs,
                                               int32_t num_tokens, int32_t max_query_len, int32_t max_seq_len,
                                               int32_t hq, int32_t hkv, int32_t d, int32_t bs,
                                               int32_t num_blocks_total, float scale, int32_t window, void *workspace,
                                               size_t workspace_bytes, const pkv_attention_options *options,
                                               cudaStream_t stream)
{
    if (!k_scale || !v_scale) return PKV_ERR_INVALID_ARG;
    if (num_tokens > 0 && (!k || !v || !slot_mapping || !k_cache || !v_cache)) return PKV_ERR_INVALID_ARG;
    if (num_tokens > 0 && (!aligned(k, 16) || !aligned(v, 16) || !aligned(slot_mapping, 8)))
        return PKV_ERR_UNSUPPORTED;
    const CallOptions opts = call_options(options);
    if (opts.separate_write) {
        // the full quantizing scatter, then the attention
        if (!workspace || workspace_bytes < PKV_WORKSPACE_MIN_BYTES || !aligned(workspace, 256))
            return PKV_ERR_WORKSPACE;
        if (num_tokens > 0) {
            LaunchChoices lc;
            lc.pdl = !opts.no_pdl;
            const ScopedLaunchChoices scoped(lc);
            pkv_status st = pkv_paged_kv_write_fp8(k, v, k_cache, v_cache, k_scale, v_scale, slot_mapping, num_tokens,
                                                   hkv, d, bs, num_blocks_total, static_cast<uint32_t *>(workspace),
                                                   stream);
            if (st != PKV_OK) return st;
        }
        return attention_impl(out, q, k_cache, v_cache, k_scale, v_scale, query_start_loc, seq_lens, block_table,
                              block_table_stride, qsl_h, sl_h, num_reqs, num_tokens, max_query_len, max_seq_len, hq,
                              hkv, d, bs, num_blocks_total, scale, window, workspace, workspace_bytes, stream, opts);
    }
    return attention_impl(out, q, k_cache, v_cache, k_scale, v_scale, query_start_loc, seq_lens, block_table,
                          block_table_stride, qsl_h, sl_h, num_reqs, num_tokens, max_query_len, max_seq_len, hq, hkv,
                          d, bs, num_blocks_total, scale, window, workspace, workspace_bytes, stream, opts, k, v,
                          slot_mapping);
}

pkv_status pkv_paged_kv_write_attention_fp8(const void *k, const void *v, void *k_cache, void *v_cache, float *k_scale,
                                            float *v_scale, const int64_t *slot_mapping, void *out, const void *q,
                                            const int32_t *query_start_loc, const int32_t *seq_lens,
                                            const int32_t *block_table, int32_t block_table_stride,
                                            const int32_t *qsl_h, const int32_t *sl_h, int32_t num_reqs,
                                            int32_t num_tokens, int32_t max_query_len, int32_t max_seq_len, int32_t hq,
                                            int32_t hkv, int32_t d, int32_t bs, int32_t num_blocks_total, float scale,
                                            int32_t window, void *workspace, size_t workspace_bytes,
                                            cudaStream_t stream)
{
    return pkv_paged_kv_write_attention_fp8_ex(k, v, k_cache, v_cache, k_scale, v_scale, slot_mapping, out, q,
                                               query_start_loc, seq_lens, block_table, block_table_stride, qsl_h,
                                               sl_h, num_reqs, num_tokens, max_query_len, max_seq_len, hq, hkv, d, bs,
                                               num_blocks_total, scale, window, workspace, workspace_bytes, nullptr,
                                               stream);
}

pkv_status pkv_ragged_paged_attention_fp8_ex(void *out, const void *q, const void *k_cache, const void *v_cache,
                                             const float *k_scale, const float *v_scale,
                                             const int32_t *query_start_loc, const int32_t *seq_lens,
                                             const int32_t *block_table, int32_t block_table_stride,
                                             const int32_t *qsl_h, const int32_t *sl_h, int32_t num_reqs,
                                             int32_t num_tokens, int32_t max_query_len, int32_t max_seq_len,
                                             int32_t hq, int32_t hkv, int32_t d, int32_t bs,
                                             int32_t num_blocks_total, float scale, int32_t window,
                                             void *workspace, size_t workspace_bytes,
                                             const pkv_attention_options *options, cudaStream_t stream)
{
    if (!k_scale || !v_scale) return PKV_ERR_INVALID_ARG;
    return attention_impl(out, q, k_cache, v_cache, k_scale, v_scale, query_start_loc, seq_lens, block_table,
                          block_table_stride, qsl_h, sl_h, num_reqs, num_tokens, max_query_len, max_seq_len, hq, hkv,
                          d, bs, num_blocks_total, scale, window, workspace, workspace_bytes, stream,
                          call_options(options));
}

pkv_status pkv_ragged_paged_attention_fp8(void *out, const void *q, const void *k_cache, const void *v_cache,
                                          const float *k_scale, const float *v_scale,
                                          const int32_t *query_start_loc, const int32_t *seq_lens,
                                          const int32_t *block_table, int32_t block_table_stride,
                                          const int32_t *qsl_h, const int32_t *sl_h, int32_t num_reqs,
                                          int32_t num_tokens, int32_t max_query_len, int32_t max_seq_len,
                                          int32_t hq, int32_t hkv, int32_t d, int32_t bs,
                                          int32_t num_blocks_total, float scale, int32_t window,
                                          void *workspace, size_t workspace_bytes, cudaStream_t stream)
{
    return pkv_ragged_paged_attention_fp8_ex(out, q, k_cache, v_cache, k_scale, v_scale, query_start_loc, seq_lens,
                                             block_table, block_table_stride, qsl_h, sl_h, num_reqs, num_tokens,
                                             max_query_len, max_seq_len, hq, hkv, d, bs, num_blocks_total, scale,
                                             window, workspace, workspace_bytes, nullptr, stream);
}

}  // extern "C"

// ---------------------------------------------------------------- block copies

extern "C" {

static pkv_status block_copy_common(int mode, void *const *pools, int32_t num_pools, const int32_t *src,
                                    const int32_t *dst, int32_t n, int32_t num_blocks_total, size_t block_bytes,
                                    void *buf, uint32_t *device_error, cudaStream_t stream)
{
    if (num_pools <= 0 || num_pools > PKV_MAX_POOLS || n < 0 || num_blocks_total <= 0 || block_bytes == 0 || !pools)
        return PKV_ERR_INVALID_ARG;
    if (n == 0) return PKV_OK;
    if (!src || (mode == 0 && !dst) || (mode != 0 && !buf)) return PKV_ERR_INVALID_ARG;
    if (block_bytes % 16 != 0 || (mode != 0 && !aligned(buf, 16))) return PKV_ERR_UNSUPPORTED;
    for (int q = 0; q < num_pools; q++) {
        if (!pools[q]) return PKV_ERR_INVALID_ARG;
        if (!aligned(pools[q], 16)) return PKV_ERR_UNSUPPORTED;
    }
    if ((int64_t)block_bytes * num_blocks_total / 16 > ((int64_t)1 << 60)) return PKV_ERR_INVALID_ARG;
    cudaError_t e = launch_block_copy(mode, pools, num_pools, src, dst, n, num_blocks_total, (int64_t)block_bytes,
                                      buf, device_error, stream);
    return e == cudaSuccess ? PKV_OK : cuda_fail(e, "block copy launch");
}

pkv_status pkv_copy_async(void *dst, const void *src, size_t bytes, cudaStream_t stream)
{
    if (bytes == 0) return PKV_OK;
    if (!dst || !src) return PKV_ERR_INVALID_ARG;
    if (bytes % 16 != 0 || !aligned(dst, 16) || !aligned(src, 16)) return PKV_ERR_UNSUPPORTED;
    const uintptr_t d = (uintptr_t)dst, s = (uintptr_t)src;
    if (d < s + bytes && s < d + bytes) return PKV_ERR_INVALID_ARG;   // overlapping ranges
    cudaError_t e = launch_byte_copy(dst, src, bytes, stream);
    return e == cudaSuccess ? PKV_OK : cuda_fail(e, "byte copy launch");
}

pkv_status pkv_copy_blocks(void *const *pools, int32_t num_pools, const int32_t *src_blocks,
                           const int32_t *dst_blocks, int32_t num_pairs, int32_t num_blocks_total,
                           size_t block_bytes, uint32_t *device_error, cudaStream_t stream)
{
    return block_copy_common(0, pools, num_pools, src_blocks, dst_blocks, num_pairs, num_blocks_total, block_bytes,
                             nullptr, device_error, stream);
}

pkv_status pkv_gather_blocks(void *const *pools, int32_t num_pools, const int32_t *blocks, int32_t num_blocks,
                             int32_t num_blocks_total, size_t block_bytes, void *out, uint32_t *device_error,
                             cudaStream_t stream)
{
    return block_copy_common(1, pools, num_pools, blocks, nullptr, num_blocks, num_blocks_total, block_bytes, out,
                             device_error, stream);
}

pkv_status pkv_scatter_blocks(void *const *pools, int32_t num_pools, const int32_t *blocks, int32_t num_blocks,
                              int32_t num_blocks_total, size_t block_bytes, const void *in, uint32_t *device_error,
                              cudaStream_t stream)
{
    return block_copy_common(2, pools, num_pools, blocks, nullptr, num_blocks, num_blocks_total, block_bytes,
                             const_cast<void *>(in), device_error, stream);
}

}  // extern "C"

/*
 * pkv — paged KV write and ragged paged attention for GB300 (sm_103a).
 *
 * A C ABI over hand-written CUDA kernels.  Its calls mirror the flattened
 * batch metadata of "31. Engine v2: one core for every request" (section
 * "Flattened ragged batches", the BatchMeta fields query_start_loc, seq_lens,
 * block_table, slot_mapping, block_size and their host copies) and the two
 * backend calls of its section "Attention over the pool": write_kv (scatter
 * this step's K/V rows into the pool) and forward (causal attention of each
 * request's new tokens over its paged context).
 *
 * Conventions shared by every call:
 *  - Device pointers are caller-owned device memory; *_host pointers are
 *    caller-owned host memory read during the call only.  The library
 *    allocates no memory, never synchronises the stream (except
 *    pkv_read_device_error, which exists to do so) and enqueues all work on
 *    `stream` in call order.
 *  - Values (q, k, v, pools, out) are bf16, row-major and densely packed.
 *  - The KV pool of one layer is [num_blocks_total][block_size][num_kv_heads]
 *    [head_dim] ("Attention over the pool": slot-major rows).  Its last
 *    block is the scratch block that padding rows write into; the block
 *    manager never hands it out.  num_blocks_total counts it.
 *  - A device error word (uint32_t) collects violations found on the
 *    device: PKV_DEVERR_SLOT (a slot past the pool), PKV_DEVERR_BLOCK (a
 *    block id outside [0, num_blocks_total)), PKV_DEVERR_TIMEOUT (a bounded
 *    pipeline wait gave up) and PKV_DEVERR_META (device metadata that
 *    disagrees with its host copy).  The access is skipped, the bit is OR-ed
 *    in, and nothing traps.  The word is sticky until cleared.
 *  - Kernels are launched as programmatic dependents (PDL) of the kernel
 *    before them on `stream` (the attention calls' options can turn this
 *    off).  The library reads no environment variables.  pkv_paged_kv_write reads nothing before its grid-dependency
 *    wait and releases its dependents only after it.  The attention kernels
 *    read q, query_start_loc, seq_lens and block_table before that wait (only
 *    the pool rows wait for it), so the kernel before them on the stream must
 *    either be pkv_paged_kv_write or not release its dependents early while
 *    it still writes those inputs (kernels that do not use PDL never do).
 *  - Every call validates its host-visible arguments first and returns an
 *    error status without enqueuing anything when they are invalid.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pkv_status {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = 1,    /* inconsistent or out-of-range host arguments */
    PKV_ERR_UNSUPPORTED = 2,    /* valid, but a shape or alignment the library has no kernel for */
    PKV_ERR_WORKSPACE = 3,      /* workspace missing or smaller than the minimum */
    PKV_ERR_CUDA = 4,           /* a CUDA runtime call failed (see pkv_last_cuda_error) */
    PKV_ERR_DEVICE_BOUNDS = 5   /* pkv_read_device_error found bounds violations */
} pkv_status;

#define PKV_DEVERR_SLOT    1u   /* paged_kv_write: slot >= num_blocks_total * block_size */
#define PKV_DEVERR_BLOCK   2u   /* attention: a block id outside [0, num_blocks_total) */
#define PKV_DEVERR_TIMEOUT 4u   /* attention: a pipeline wait gave up (about 2 s); its rows are not written */
#define PKV_DEVERR_META    8u   /* attention: query_start_loc / seq_lens on the device differ from the host copies */
#define PKV_DEVERR_COUNTER 16u  /* attention: a split counter in the workspace was not zero (workspace not zero-filled) */

/* Static description of a status code. */
const char *pkv_status_string(pkv_status status);

/* Text of the last CUDA error seen by this library on the calling thread. */
const char *pkv_last_cuda_error(void);

/*
 * Number of kernels this library has launched since it was loaded (all
 * threads).  A diagnostic: the difference over a region counts its launches.
 */
int64_t pkv_launch_count(void);

/*
 * Per-launch timing, for diagnostics and the benchmark.  After
 * pkv_profile_start(capacity), each kernel launch of the library (up to
 * `capacity` of them) is bracketed by two CUDA events recorded on its
 * launching stream.  pkv_profile_stop() ends recording and returns the
 * number of records; pkv_profile_read() waits for record `index` and gives
 * its kernel id and duration in ms; pkv_kernel_name() names a kernel id.
 * Events are created once by pkv_profile_start (host-side CUDA objects, no
 * device memory).  Launches made while their stream is being captured into
 * a CUDA graph get their events as event nodes of that graph: read the
 * records after the graph has run once (each run overwrites them).
 */
pkv_status pkv_profile_start(int32_t capacity);
int32_t pkv_profile_stop(void);
pkv_status pkv_profile_read(int32_t index, int32_t *kernel_id, float *ms);
const char *pkv_kernel_name(int32_t kernel_id);

/*
 * paged_kv_write — scatter this step's new K/V rows into the pool
 * ("31. Engine v2", "Attention over the pool", write_kv).
 *
 *   k, v          device bf16 [num_tokens][num_kv_heads][head_dim]
 *   k_cache,      device bf16 [num_blocks_total][block_size][num_kv_heads][head_dim]
 *   v_cache       (written in place)
 *   slot_mapping  device int64 [num_tokens]: flat slot of row i
 *                 (table[p / block_size] * block_size + p % block_size,
 *                 "Flattened ragged batches"); a negative slot marks a
 *                 padding row, which is written to the last slot of the pool
 *                 (the scratch block).  A slot >= num_blocks_total*block_size
 *                 is skipped and sets PKV_DEVERR_SLOT in *device_error.
 *   device_error  device uint32_t, may be NULL (then violations are only skipped)
 *
 * Row i is copied bit for bit.  Two real rows with the same slot are a
 * caller error (which one lands is unspecified); padding rows may share the
 * scratch slot, whose contents are unspecified.
 * Requirements: head_dim % 8 == 0; k, v, k_cache, v_cache 16-byte aligned.
 * num_tokens == 0 is a no-op.
 */
pkv_status pkv_paged_kv_write(const void *k, const void *v, void *k_cache, void *v_cache,
                              const int64_t *slot_mapping, int32_t num_tokens,
                              int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                              int32_t num_blocks_total, uint32_t *device_error,
                              cudaStream_t stream);

/*
 * Quantized pools ("31. Engine v2", "Attention over the pool": a quantized
 * pool carries one scale per slot and KV head beside K and V, and a row is
 * read as code * scale).  Codes are FP8 E4M3 bytes, the pools uint8
 * [num_blocks_total][block_size][num_kv_heads][head_dim]; scales are fp32
 * [num_blocks_total][block_size][num_kv_heads].  The pages leave the code
 * format and the quantizing write open; this library's reading: per row
 * and KV head, scale = max |x| / 448 in fp32 and code = E4M3(x / scale)
 * rounded to nearest even, saturating at +-448 (an all-zero row: scale 0,
 * codes 0).
 *
 * pkv_paged_kv_write_fp8 — the quantizing write_kv: k, v bf16
 *   [num_tokens][num_kv_heads][head_dim] -> codes at slot_mapping[i] (a
 *   negative slot: the scratch slot), scales beside them.  Requirements:
 *   head_dim 128; k, v, k_cache, v_cache 16-byte aligned.  Errors as
 *   pkv_paged_kv_write.
 */
pkv_status pkv_paged_kv_write_fp8(const void *k, const void *v, void *k_cache, void *v_cache,
                                  float *k_scale, float *v_scale, const int64_t *slot_mapping,
                                  int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                                  int32_t block_size, int32_t num_blocks_total, uint32_t *device_error,
                                  cudaStream_t stream);

/*
 * Workspace size that lets pkv_ragged_paged_attention split long decodes
 * over KV freely for any batch within the given maxima.  A smaller
 * workspace (at least PKV_WORKSPACE_MIN_BYTES) is accepted: the planner
 * then splits less.  The workspace holds the device error word (first 256
 * bytes), then — when it has room for them (64 KiB) — the split counters of
 * the combines that run inside the attention kernels, then fp32 split-KV
 * partials; for pools of blocks of more than 16 slots its last
 * ceil(num_reqs * ceil(L_max / 16) * 4 / 256) * 256 bytes take the block
 * table in 16-slot entries (written by the call; PKV_ERR_WORKSPACE when
 * they do not fit beside PKV_WORKSPACE_MIN_BYTES).  Zero-fill a workspace
 * once before its first use: every call leaves the counters zero again.
 * Use one workspace at one size, on one stream at a time.
 */
#define PKV_WORKSPACE_MIN_BYTES 256
size_t pkv_attention_workspace_bytes(int32_t max_num_reqs, int32_t max_num_tokens,
                                     int32_t num_q_heads, int32_t head_dim,
                                     int32_t max_seq_len);

/*
 * ragged_paged_attention — causal grouped-query attention of one flattened
 * ragged batch over the paged pool ("31. Engine v2", "Attention over the
 * pool", the reference backend's forward; grouped heads as in the vllm-lite
 * README; tiled exact attention as in "vLLM: LLM Inference as a memory and
 * scheduling problem", "FlashAttention is not PagedAttention").
 *
 *   out               device bf16 [num_tokens][num_q_heads][head_dim]
 *   q                 device bf16 [num_tokens][num_q_heads][head_dim]
 *   k_cache, v_cache  device bf16 pool, as in pkv_paged_kv_write (read only)
 *   query_start_loc   device int32 [num_reqs + 1]: request r owns rows
 *                     query_start_loc[r] .. query_start_loc[r+1]-1
 *   seq_lens          device int32 [num_reqs]: context length L after this step
 *   block_table       device int32 [num_reqs][block_table_stride]: physical
 *                     blocks of each request in logical order
 *   query_start_loc_host, seq_lens_host
 *                     host copies of the two arrays above, used to plan the
 *                     launches without reading device memory; the kernels
 *                     take each request's rows and context length from them
 *                     and flag PKV_DEVERR_META where the device arrays differ
 *   max_query_len, max_seq_len
 *                     maxima of the host arrays (validated)
 *   scale             softmax scale; <= 0 selects 1/sqrt(head_dim)
 *   window            sliding window (the reference backend's `window`):
 *                     0 for none; w > 0 limits the query at position p to
 *                     the keys above p - w.  Negative: PKV_ERR_INVALID_ARG
 *   workspace         device memory, >= PKV_WORKSPACE_MIN_BYTES, 256-byte
 *                     aligned; its first 4 bytes are the device error word
 *                     (PKV_DEVERR_BLOCK), the rest holds split partials
 *
 * Row i of request r (t rows, L = seq_lens[r]) is the query at position
 * L - t + i.  Query head h reads KV head h / (num_q_heads / num_kv_heads)
 * and attends to the keys at positions 0 .. L - t + i (with a window w,
 * max(0, L - t + i - w + 1) .. L - t + i; keys below are not read).  A request with
 * L == 0 or t == 0 is padding: its rows of `out` are set to zero.
 * All keys a request reads must already be in the pool: call
 * pkv_paged_kv_write for the step first, on the same stream.
 *
 * Host validation (PKV_ERR_INVALID_ARG, nothing enqueued):
 *   query_start_loc_host not non-decreasing from 0 to num_tokens; a request
 *   with L > 0 and t > L; ceil(L / block_size) > block_table_stride;
 *   num_q_heads % num_kv_heads != 0; the max_* arguments below the data.
 * PKV_ERR_UNSUPPORTED: head_dim not in {48, 64, 128}, block_size not one
 *   of 16, 32, 64, 128, 256 (the kernels walk a block as sub-blocks of 16
 *   slots), or misaligned pointers.
 */
pkv_status pkv_ragged_paged_attention(void *out, const void *q,
                                      const void *k_cache, const void *v_cache,
                                      const int32_t *query_start_loc, const int32_t *seq_lens,
                                      const int32_t *block_table, int32_t block_table_stride,
                                      const int32_t *query_start_loc_host,
                                      const int32_t *seq_lens_host,
                                      int32_t num_reqs, int32_t num_tokens,
                                      int32_t max_query_len, int32_t max_seq_len,
                                      int32_t num_q_heads, int32_t num_kv_heads,
                                      int32_t head_dim, int32_t block_size,
                                      int32_t num_blocks_total, float scale, int32_t window,
                                      void *workspace, size_t workspace_bytes,
                                      cudaStream_t stream);

/*
 * Options of the attention calls' _ex variants.  Each field overrides one
 * choice the planner otherwise makes from the batch alone; a zero-filled
 * struct (or a NULL pointer) leaves every choice to the planner, and the
 * plain calls are the _ex calls with NULL.  Normal use needs none of them:
 * they exist so that tests can reach every kernel arrangement and
 * measurements can compare them.  Results are the same under every option
 * (within the attention tolerance; the pools bit for bit).
 *
 *   disable_tcgen05     1: prefill tiles on the warp-MMA kernel, not tcgen05
 *   tc_min_rows         > 0: query rows (new tokens x group) from which a
 *                       prefill request goes to tcgen05 (default 17)
 *   fp8_prefill_on_mma  1: quantized-pool prefill on the warp-MMA kernel even
 *                       when the workspace has room for bf16 block copies
 *   split_tokens        > 0: decode split length in keys (rounded up to the
 *                       block size), instead of the planner's
 *   cluster             0: planner; -1: no thread-block clusters (split
 *                       counters merge the splits); 2..8: clusters of that
 *                       many splits
 *   decode_main         0: planner; 1: when the classes overlap the decodes
 *                       run on the caller's stream; -1: the prefill does
 *   no_overlap          1: both classes on the caller's stream, in turn
 *   prefill_key_splits  1: warp-MMA prefill tiles split over keys when they
 *                       fill less than two waves
 *   separate_write      1: the combined calls run the full scatter, then the
 *                       attention
 *   decode_row_tiles    1: 16-row query tiles for decodes instead of
 *                       key-major tiles for small groups
 *   no_pdl              1: no programmatic dependent launches
 *   tc_key_pieces       -1: no tcgen05 pair is cut into key pieces; k >= 2:
 *                       every tcgen05 pair is cut into k pieces (at most its
 *                       key tiles), merged by the CTA that finishes last
 *   mixed_launch        1: a batch's decode class runs inside the tcgen05
 *                       prefill launch whenever it can (one launch for both
 *                       classes: decode CTAs ahead of the prefill CTAs); -1:
 *                       never; 0: when the planner expects it to be faster
 *   mixed_decode_ctas   > 0: that many decode CTAs in a mixed launch (rounded
 *                       up to a multiple of the KV heads)
 *   device_lengths      1: a batch of decode-class requests whose context
 *                       lengths the kernels read from the device seq_lens when
 *                       they run.  The host seq_lens then give each request's
 *                       capacity (the plan: splits, partials, grids), and the
 *                       device value may be anything from 0 (a padding row)
 *                       to it.  So a call captured in a CUDA graph can be
 *                       replayed after the caller has rewritten seq_lens,
 *                       block_table, slot_mapping, q, k and v in place for
 *                       another batch of the same shape ("31. Engine v2",
 *                       "Flattened ragged batches": the batch builder pads
 *                       decode batches, pad_to, so that one captured step
 *                       serves them all).  query_start_loc must stay as
 *                       planned.  A device length above the capacity is
 *                       clamped to it and reported (PKV_DEVERR_META).  Every
 *                       request must be decode class (t * g <= 16 rows per
 *                       KV head): PKV_ERR_UNSUPPORTED otherwise.  With this
 *                       option results follow the device lengths; with every
 *                       other option they are the same as without it.
 */
typedef struct pkv_attention_options {
    int32_t disable_tcgen05;
    int32_t tc_min_rows;
    int32_t fp8_prefill_on_mma;
    int32_t split_tokens;
    int32_t cluster;
    int32_t decode_main;
    int32_t no_overlap;
    int32_t prefill_key_splits;
    int32_t separate_write;
    int32_t decode_row_tiles;
    int32_t no_pdl;
    int32_t tc_key_pieces;
    int32_t mixed_launch;
    int32_t mixed_decode_ctas;
    int32_t device_lengths;
    int32_t reserved;
} pkv_attention_options;

/* pkv_ragged_paged_attention with options (NULL: the planner's choices). */
pkv_status pkv_ragged_paged_attention_ex(void *out, const void *q, const void *k_cache, const void *v_cache,
                                         const int32_t *query_start_loc, const int32_t *seq_lens,
                                         const int32_t *block_table, int32_t block_table_stride,
                                         const int32_t *query_start_loc_host, const int32_t *seq_lens_host,
                                         int32_t num_reqs, int32_t num_tokens, int32_t max_query_len,
                                         int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads,
                                         int32_t head_dim, int32_t block_size, int32_t num_blocks_total,
                                         float scale, int32_t window, void *workspace, size_t workspace_bytes,
                                         const pkv_attention_options *options, cudaStream_t stream);

/*
 * One step's write and attention in one call ("31. Engine v2", "Attention
 * over the pool": every layer writes the step's K/V rows, then attends):
 * the result is that of pkv_paged_kv_write(k, v, k_cache, v_cache,
 * slot_mapping, ...) followed by pkv_ragged_paged_attention(...) with the
 * same arguments, bf16 pools.  The work is arranged differently: the CTAs
 * that attend for a decode-class request (t * g <= 16 rows per KV head)
 * write that request's new rows themselves, each the rows in its key range,
 * just before reading them; so does the tensor-core CTA of a prefill
 * request whose rows of a KV head are all that one CTA's (t * g <= 256,
 * not cut into key pieces, the prefill not in one launch with the
 * decodes); a scatter restricted to the other prefill-class
 * requests' rows runs ahead of the prefill kernels.  So decode attention
 * does not wait for a scatter, and a batch of decodes is one launch.
 *
 *   k, v          device bf16 [num_tokens][num_kv_heads][head_dim], 16-byte
 *                 aligned (the rows pkv_paged_kv_write takes)
 *   slot_mapping  device int64 [num_tokens]: as for pkv_paged_kv_write; it
 *                 must agree with the block table (token i of request r at
 *                 position L - t + i goes to block_table[r][pos / 16] * 16 +
 *                 pos % 16), as a batch builder makes it.  A decode-class row
 *                 whose slot differs is still written to its slot_mapping
 *                 slot but the attention reads the block table's slot, and
 *                 PKV_DEVERR_META is set.
 *   other arguments as pkv_ragged_paged_attention (k_cache, v_cache written).
 * The arrangement relies on what a batch builder guarantees: a slot that
 * receives a new row belongs to a block that no other request of the batch
 * reads (a block still being filled has one owner; blocks shared by prefix
 * caching are full).  Another request's CTAs may read such a block before
 * its new rows are written, so a batch that breaks this may see old rows.
 * Device errors of the write (PKV_DEVERR_SLOT) go to the workspace's error
 * word with the attention's.  Return codes as the two calls; nothing is
 * enqueued when the arguments are rejected.  With the separate_write option
 * the call runs the full scatter, then the attention.
 */
pkv_status pkv_paged_kv_write_attention(const void *k, const void *v, void *k_cache, void *v_cache,
                                        const int64_t *slot_mapping, void *out, const void *q,
                                        const int32_t *query_start_loc, const int32_t *seq_lens,
                                        const int32_t *block_table, int32_t block_table_stride,
                                        const int32_t *query_start_loc_host,
                                        const int32_t *seq_lens_host, int32_t num_reqs,
                                        int32_t num_tokens, int32_t max_query_len, int32_t max_seq_len,
                                        int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                        int32_t block_size, int32_t num_blocks_total, float scale,
                                        int32_t window, void *workspace, size_t workspace_bytes,
                                        cudaStream_t stream);
pkv_status pkv_paged_kv_write_attention_ex(const void *k, const void *v, void *k_cache, void *v_cache,
                                           const int64_t *slot_mapping, void *out, const void *q,
                                           const int32_t *query_start_loc, const int32_t *seq_lens,
                                           const int32_t *block_table, int32_t block_table_stride,
                                           const int32_t *query_start_loc_host, const int32_t *seq_lens_host,
                                           int32_t num_reqs, int32_t num_tokens, int32_t max_query_len,
                                           int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads,
                                           int32_t head_dim, int32_t block_size, int32_t num_blocks_total,
                                           float scale, int32_t window, void *workspace, size_t workspace_bytes,
                                           const pkv_attention_options *options, cudaStream_t stream);

/*
 * ragged_paged_attention over a quantized pool (codes and scales as written
 * by pkv_paged_kv_write_fp8).  Arguments as pkv_ragged_paged_attention plus
 * the two scale pools (device fp32, 16-byte aligned).  Keys and values are
 * code * scale; q, out stay bf16.  The products run on fp16 tensor-core MMAs
 * (every E4M3 value is an fp16 value; q rounds to fp16 exactly within its
 * range), so |q| and the per-key weight * V scale must stay inside fp16's
 * range (65504).  Requirements (else PKV_ERR_UNSUPPORTED): head_dim 128,
 * num_kv_heads a multiple of 4.  Prefill chunks run on
 * tcgen05 over bf16 copies of their blocks (code * scale rounded to nearest)
 * when the workspace holds pkv_fp8_prefill_scratch_bytes(...) more than
 * pkv_attention_workspace_bytes(...); otherwise on the warp-level MMA kernels
 * over the codes.
 */
pkv_status pkv_ragged_paged_attention_fp8(void *out, const void *q,
                                          const void *k_cache, const void *v_cache,
                                          const float *k_scale, const float *v_scale,
                                          const int32_t *query_start_loc, const int32_t *seq_lens,
                                          const int32_t *block_table, int32_t block_table_stride,
                                          const int32_t *query_start_loc_host,
                                          const int32_t *seq_lens_host,
                                          int32_t num_reqs, int32_t num_tokens,
                                          int32_t max_query_len, int32_t max_seq_len,
                                          int32_t num_q_heads, int32_t num_kv_heads,
                                          int32_t head_dim, int32_t block_size,
                                          int32_t num_blocks_total, float scale, int32_t window,
                                          void *workspace, size_t workspace_bytes,
                                          cudaStream_t stream);
pkv_status pkv_ragged_paged_attention_fp8_ex(void *out, const void *q, const void *k_cache, const void *v_cache,
                                             const float *k_scale, const float *v_scale,
                                             const int32_t *query_start_loc, const int32_t *seq_lens,
                                             const int32_t *block_table, int32_t block_table_stride,
                                             const int32_t *query_start_loc_host, const int32_t *seq_lens_host,
                                             int32_t num_reqs, int32_t num_tokens, int32_t max_query_len,
                                             int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads,
                                             int32_t head_dim, int32_t block_size, int32_t num_blocks_total,
                                             float scale, int32_t window, void *workspace, size_t workspace_bytes,
                                             const pkv_attention_options *options, cudaStream_t stream);

/*
 * pkv_paged_kv_write_fp8 followed by pkv_ragged_paged_attention_fp8 in one
 * call, arranged as pkv_paged_kv_write_attention: decode-class CTAs quantize
 * and write their requests' new rows (the same E4M3 codes and scales as the
 * quantizing scatter, bit for bit) just before reading them, a quantizing
 * scatter restricted to the prefill-class rows runs ahead of the prefill
 * kernels.  Arguments: the quantizing scatter's (k, v bf16 [num_tokens][
 * num_kv_heads][128], 16-byte aligned; codes pools; scale pools written;
 * slot_mapping agreeing with the block table) and the attention's.  Device
 * errors of the write go to the workspace's error word; a decode row whose
 * slot differs from the block table's sets PKV_DEVERR_META.  With the
 * separate_write option the call runs the full quantizing scatter, then the
 * attention.
 */
pkv_status pkv_paged_kv_write_attention_fp8(const void *k, const void *v, void *k_cache, void *v_cache,
                                            float *k_scale, float *v_scale, const int64_t *slot_mapping,
                                            void *out, const void *q, const int32_t *query_start_loc,
                                            const int32_t *seq_lens, const int32_t *block_table,
                                            int32_t block_table_stride, const int32_t *query_start_loc_host,
                                            const int32_t *seq_lens_host, int32_t num_reqs,
                                            int32_t num_tokens, int32_t max_query_len, int32_t max_seq_len,
                                            int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                            int32_t block_size, int32_t num_blocks_total, float scale,
                                            int32_t window, void *workspace, size_t workspace_bytes,
                                            cudaStream_t stream);
pkv_status pkv_paged_kv_write_attention_fp8_ex(const void *k, const void *v, void *k_cache, void *v_cache,
                                               float *k_scale, float *v_scale, const int64_t *slot_mapping,
                                               void *out, const void *q, const int32_t *query_start_loc,
                                               const int32_t *seq_lens, const int32_t *block_table,
                                               int32_t block_table_stride, const int32_t *query_start_loc_host,
                                               const int32_t *seq_lens_host, int32_t num_reqs, int32_t num_tokens,
                                               int32_t max_query_len, int32_t max_seq_len, int32_t num_q_heads,
                                               int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                               int32_t num_blocks_total, float scale, int32_t window,
                                               void *workspace, size_t workspace_bytes,
                                               const pkv_attention_options *options, cudaStream_t stream);

/*
 * ragged_paged_attention without a caller workspace.  The pages have no
 * counterpart of this call: it exists for callers that cannot allocate
 * device memory, such as plain C hosts without a device allocator of their
 * own, and serving loops that must not call cudaMalloc because it may
 * synchronise the device or because their device memory budget is fixed
 * when they start.
 *
 * Same arguments and results as pkv_ragged_paged_attention, except:
 *  - No workspace: the split-KV partials, the split counters and the device
 *    error word live in one static device array of PKV_NOALLOC_SCRATCH_BYTES
 *    (8 MiB) inside the library.  Every GPU that loads the library holds
 *    that array until the process exits.  The call allocates nothing and
 *    calls no allocating routine.
 *  - The planner fits the split-KV partials into the array, lengthening the
 *    decode splits where the batch would need more (fewer, longer splits;
 *    the same results).  The call plans the batch against the array's size
 *    before it enqueues anything and returns PKV_ERR_WORKSPACE if that plan
 *    would not fit; the planner's rule makes every batch that the workspace
 *    entry point accepts fit.
 *  - device_error (device uint32_t, may be NULL) receives this call's
 *    bounds flags (overwritten, not OR-ed).
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current) and keeps it; make
 *    that first call before any stream capture.
 *  - All calls share the one array and it keeps the last call's contents.
 *    Each call first zeroes the error word and the split counters on its
 *    stream.  Calls whose work overlaps on the GPU (other streams, other
 *    threads) race on the array: serialise them, for example on one stream.
 */
#define PKV_NOALLOC_SCRATCH_BYTES (8u << 20)
pkv_status pkv_ragged_paged_attention_noalloc(void *out, const void *q,
                                              const void *k_cache, const void *v_cache,
                                              const int32_t *query_start_loc, const int32_t *seq_lens,
                                              const int32_t *block_table, int32_t block_table_stride,
                                              const int32_t *query_start_loc_host,
                                              const int32_t *seq_lens_host,
                                              int32_t num_reqs, int32_t num_tokens,
                                              int32_t max_query_len, int32_t max_seq_len,
                                              int32_t num_q_heads, int32_t num_kv_heads,
                                              int32_t head_dim, int32_t block_size,
                                              int32_t num_blocks_total, float scale, int32_t window,
                                              uint32_t *device_error, cudaStream_t stream);

/*
 * A check of the bounded waits (a diagnostic, for tests).  Every pipeline
 * wait of the attention kernels gives up after 2 s, sets PKV_DEVERR_TIMEOUT
 * and lets the kernel leave in order (no thread left at a barrier, tensor
 * memory freed).  This call launches one small CTA with the same roles —
 * a tensor-memory owner, a producer lane and consumer warps — whose
 * mbarriers nothing ever arrives at, waiting with the same routine but a
 * limit of limit_us microseconds (1 .. 100000).  It returns once every wait
 * has given up: *device_error gets PKV_DEVERR_TIMEOUT OR-ed in, report[0]
 * one bit per warp whose wait gave up (warps 0, 2 and 3: 0xD), report[1]
 * the microseconds the kernel ran.  device_error and report are device
 * uint32_t (1 and 2 of them).  PKV_ERR_INVALID_ARG for null pointers or a
 * limit out of range; PKV_ERR_CUDA if the launch fails.
 */
pkv_status pkv_check_bounded_wait(uint32_t *device_error, uint32_t *report, uint32_t limit_us,
                                  cudaStream_t stream);

/* Size in bytes of the no-allocation call's static scratch array
 * (PKV_NOALLOC_SCRATCH_BYTES as this library was built). */
size_t pkv_noalloc_scratch_bytes(void);

/*
 * Which kernel path pkv_ragged_paged_attention takes for each request
 * (host only, no CUDA call): class_out[r] receives one of PKV_CLASS_*.
 * Decode-class requests (t * g <= 16) run on the warp-level MMA decode
 * kernels, with KV split across CTAs for long contexts; prefill-class
 * requests run in tiles of new tokens, on tcgen05 where the head dim and
 * group fit a 128-row tile.  For accounting and tests.  Default options.
 */
#define PKV_CLASS_NONE 0                 /* no rows */
#define PKV_CLASS_PADDING 1              /* seq_len 0: rows zeroed */
#define PKV_CLASS_DECODE 2               /* decode kernels (split KV merged in a cluster or in-kernel) */
#define PKV_CLASS_PREFILL_MMA 3    /* warp-MMA prefill tiles (not on tcgen05) */
#define PKV_CLASS_PREFILL_TENSOR 4       /* tcgen05 prefill tiles */
pkv_status pkv_plan_request_kernels(const int32_t *query_start_loc_host, const int32_t *seq_lens_host,
                                    int32_t num_reqs, int32_t num_q_heads, int32_t num_kv_heads,
                                    int32_t head_dim, int32_t *class_out);

/*
 * The launch plan an attention call would follow (host only; no CUDA call
 * when num_sms > 0).  For a flattened ragged batch ("31. Engine v2",
 * "Flattened ragged batches") the planner classifies the requests, picks
 * one split length for the decode class (about 16 CTAs per SM over its
 * keys, 4 beside a longer prefill, at least 256 keys, a multiple of 128, at
 * most 32 streaming splits per request, then doubled until the split
 * partials fit the workspace), and decides whether the decode and prefill
 * classes run concurrently on two streams.  This reports those decisions
 * for the same arguments as pkv_ragged_paged_attention (quantized != 0: its
 * _fp8 variant; combined != 0: pkv_paged_kv_write_attention), given the
 * workspace size and the GPU's SM count (num_sms <= 0: the current
 * device's, which needs a GPU) and the call's options (NULL: none).  query_start_loc_host has num_reqs + 1 entries,
 * seq_lens_host num_reqs; plan_out is written on success only.
 *
 * Errors: PKV_ERR_INVALID_ARG for null pointers, num_reqs < 0, a negative
 * query length or window, t > seq_len, or heads that do not group;
 * PKV_ERR_UNSUPPORTED for a head dim, block size, group or quantized shape
 * the attention calls reject; PKV_ERR_CUDA when num_sms <= 0 and no device
 * answers.
 */
typedef struct pkv_attention_plan {
    int32_t decode_requests;          /* decode class, padding requests included */
    int32_t prefill_tensor_requests;  /* prefill on tcgen05 */
    int32_t prefill_mma_requests;     /* prefill on the warp-MMA kernel */
    int32_t decode_split_tokens;      /* keys per decode split, a multiple of block_size */
    int32_t max_decode_splits;        /* the largest split count of a decode request */
    int32_t decode_cluster;           /* CTAs per thread-block cluster of the first decode launch; 0: none */
    int32_t decode_streaming;         /* 1: decode splits long enough for the streaming kernel */
    int32_t split_counters;           /* 1: the workspace holds in-kernel combine counters */
    int32_t overlap;                  /* 1: decode and prefill classes on two streams */
    int32_t decode_on_caller_stream;  /* with overlap: 1 if the decodes run on the caller's stream */
    int32_t prefill_key_splits;       /* 1: warp-MMA prefill tiles split over keys */
    int32_t prefill_tensor_pieces;    /* tcgen05 CTAs that run a key piece of a pair (0: no pair is cut) */
    size_t quantized_prefill_scratch; /* workspace bytes of bf16 block copies for quantized prefill */
    size_t partial_bytes;             /* workspace bytes of split partials */
    int32_t mixed_launch;             /* 1: decode items run inside the tcgen05 prefill launch (one launch) */
    int32_t mixed_decode_items;       /* ... how many */
    int32_t mixed_decode_ctas;        /* ... on how many decode CTAs ahead of the prefill CTAs */
    int32_t mixed_predicted_us;       /* ... the planner's estimate of its time, us (0 when forced) */
    int32_t prefill_tensor_own_rows;  /* combined call: tcgen05 requests whose CTAs write their new rows */
} pkv_attention_plan;
pkv_status pkv_plan_attention(const int32_t *query_start_loc_host, const int32_t *seq_lens_host,
                              int32_t num_reqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                              int32_t block_size, int32_t window, int32_t quantized, int32_t combined,
                              size_t workspace_bytes, int32_t num_sms, const pkv_attention_options *options,
                              pkv_attention_plan *plan_out);

/*
 * Set a device error word to zero (enqueued on stream).
 */
pkv_status pkv_clear_device_error(uint32_t *device_error, cudaStream_t stream);

/*
 * Synchronise `stream`, read the device error word at `device_error` (for
 * attention: the workspace pointer) into *flags_out, and return
 * PKV_ERR_DEVICE_BOUNDS if any bit is set, PKV_OK otherwise.  A diagnostic
 * for tests and debugging; not for the hot path.
 */
pkv_status pkv_read_device_error(const uint32_t *device_error, uint32_t *flags_out,
                                 cudaStream_t stream);

/*
 * Block copies of the block manager, over many pools in one launch.
 * "vllm-lite README": blocks are reference counted, and a write into a
 * block two sequences share is preceded by a copy of it (copy-on-write),
 * done by the runner before the forward pass.  "31. Engine v2",
 * "Preemption: recompute or swap": swap-out copies a preempted request's
 * blocks of every layer's K and V (and, for quantized pools, their scales)
 * to host memory; swap-in copies them into newly allocated blocks.
 *
 *   pools             host array of num_pools (1 .. PKV_MAX_POOLS) device
 *                     pointers, read during the call; each is a pool of
 *                     num_blocks_total blocks of block_bytes bytes (for a
 *                     bf16 K or V pool: block_size * num_kv_heads * head_dim
 *                     * 2).  Pools may have different base addresses but
 *                     share num_blocks_total and block_bytes.
 *   device_error      device uint32_t, may be NULL; a block id outside
 *                     [0, num_blocks_total) is skipped and sets
 *                     PKV_DEVERR_BLOCK.
 * Requirements: block_bytes % 16 == 0; pools and buffers 16-byte aligned
 * (else PKV_ERR_UNSUPPORTED).  Zero pairs/blocks is a no-op.  The copy is a
 * bit copy; the launch waits for the kernel before it on `stream` before
 * reading anything.
 */
#define PKV_MAX_POOLS 256

/* Copy-on-write: in every pool, block dst_blocks[i] := block src_blocks[i].
 * src_blocks, dst_blocks: device int32 [num_pairs].  A block that is both a
 * source and a destination, or a destination twice, is a caller error
 * (which bytes land is unspecified). */
pkv_status pkv_copy_blocks(void *const *pools, int32_t num_pools, const int32_t *src_blocks,
                           const int32_t *dst_blocks, int32_t num_pairs, int32_t num_blocks_total,
                           size_t block_bytes, uint32_t *device_error, cudaStream_t stream);

/* Swap-out: out[q][i] := block blocks[i] of pool q, out laid out
 * [num_pools][num_blocks][block_bytes].  blocks: device int32 [num_blocks].
 * out may be device memory or pinned host memory the device can address
 * (then the kernel writes host memory directly). */
pkv_status pkv_gather_blocks(void *const *pools, int32_t num_pools, const int32_t *blocks, int32_t num_blocks,
                             int32_t num_blocks_total, size_t block_bytes, void *out, uint32_t *device_error,
                             cudaStream_t stream);

/* Swap-in: block blocks[i] of pool q := in[q][i], in laid out as for
 * pkv_gather_blocks (device memory or device-addressable pinned host
 * memory). */
pkv_status pkv_scatter_blocks(void *const *pools, int32_t num_pools, const int32_t *blocks, int32_t num_blocks,
                              int32_t num_blocks_total, size_t block_bytes, const void *in, uint32_t *device_error,
                              cudaStream_t stream);

/*
 * Extra workspace bytes that let pkv_ragged_paged_attention_fp8 run this
 * batch's prefill chunks on the tcgen05 kernel (host only; query_start_loc
 * and seq_lens as host arrays).  With a workspace at least
 * pkv_attention_workspace_bytes(...) plus this many bytes, a dequantizing
 * pass first writes bf16 copies (code * scale, rounded to nearest) of those
 * requests' blocks and a block table for them into the workspace's end, and
 * the chunks attend over the copies; with a smaller workspace they run on
 * the warp-MMA kernel over the codes.  0 when no request of the batch
 * qualifies (head_dim 128, a group size dividing 128, at least 17 rows).
 */
size_t pkv_fp8_prefill_scratch_bytes(const int32_t *query_start_loc_host, const int32_t *seq_lens_host,
                                     int32_t num_reqs, int32_t num_q_heads, int32_t num_kv_heads,
                                     int32_t head_dim);

/* ---------------------------------------------------------------- staging copies
 *
 * "31. Engine v2", "Flattened ragged batches": the batch builder lays out
 * each step's metadata on the host and the device reads it.  This copies
 * `bytes` bytes from src to dst with a kernel on `stream`: either side may
 * be device memory or pinned host memory the device can address (then the
 * kernel reads or writes host memory directly), so staging a step's packed
 * inputs and reading back its output add kernels to the stream, not
 * copy-engine operations between the attention launches.
 *
 * Requirements: bytes % 16 == 0 and both pointers 16-byte aligned (else
 * PKV_ERR_UNSUPPORTED); non-null pointers for bytes > 0 and ranges that do
 * not overlap (else PKV_ERR_INVALID_ARG).  Zero bytes is a no-op.  A bit
 * copy; the kernel waits for the kernel before it on `stream` before it
 * reads src (programmatic launch), and the next kernel waits for it.
 * Nothing is allocated and nothing synchronises.  A copy with a pinned host
 * side runs on a dozen CTAs: the
 * host link is saturated by then, and the rest of the GPU stays free for
 * attention launched on other streams while the copy runs (staging the next
 * step's inputs during this step).  A device-to-device copy spreads over
 * the whole GPU.  A copy with a pinned host side of 8 MiB or more is a
 * copy-engine operation (cudaMemcpyAsync on `stream`) instead, which takes
 * no SM from attention running beside it; it is ordered on `stream` like
 * the kernel.
 */
pkv_status pkv_copy_async(void *dst, const void *src, size_t bytes, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */

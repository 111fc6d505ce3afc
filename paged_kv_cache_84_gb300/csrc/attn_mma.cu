// Ragged paged attention with TMA-staged KV blocks and warp-level MMA.
//
// One CTA = (listed request, KV head, item), 5 warps:
//   - warp 4 (producer) walks the CTA's key range block by block: it reads
//     the physical block ids from the request's block table ("31. Engine
//     v2", "Attention over the pool": key j lives in block table[j / 16],
//     row j % 16) and issues one 3-D TMA copy per 16-row slice of a K or V
//     block (one KV head, [16][head_dim]) into a ring of shared-memory
//     stages, each completing on its stage's "full" mbarrier;
//   - warps 0..3 (consumers) take the rows of the CTA (pairs (token, query
//     head) that share KV head kh: the grouped-query fold of the vllm-lite
//     README) in tiles of 16.  With KG key groups, warp w works on row tile
//     w / KG and on every KG-th block, two blocks per iteration (two
//     independent MMA chains, one softmax update per 32 keys).  Decode-class
//     CTAs use 4 key groups, prefill-class CTAs 2 row tiles x 2 key groups.
// Each consumer computes S = Q K^T for 16 rows x 16 keys with
// mma.m16n8k16 (bf16 in, fp32 accumulate), applies the causal rule (query i
// of a request with t new tokens and context L sits at position L - t + i
// and sees keys 0 .. that position), runs the online softmax in the exp2
// domain, and accumulates O += P V with P taken straight from the S
// registers.  Key groups merge through shared memory at the end.  Unsplit
// items write bf16 output; split items write fp32 partials (unnormalised o,
// running max, weight sum) for the combine kernel.
//
// Shared-memory tiles: for head_dim 64/128 each TMA box is 16 rows x 64
// columns (128 bytes) with the 128-byte swizzle, so that ldmatrix reads
// eight rows without bank conflicts; for head_dim 48 rows are 96 bytes, not
// swizzled.
#include <stdlib.h>

#include <mutex>

#include "common.cuh"
#include "mma_tiles.cuh"
#include "sm100.cuh"

namespace pkv {

constexpr int kConsumerWarps = 4;
constexpr int kMmaThreads = (kConsumerWarps + 1) * 32;
// Bytes of KV stages per streaming CTA.  Two 4-block stages of bf16
// head_dim 128 (64 KB): measured faster than three (96 KB) on both decode
// workloads, 653 vs 679 us and 631 vs 651 us.
constexpr int kStageBudget = 64 * 1024;
constexpr int kLongSplit = kLongSplitTokens; // decode splits of at least this many keys use the streaming kernel

template <int D, int KG, int NB, bool FP8 = false, int CW = kConsumerWarps>
struct MmaCfg {
    static constexpr int kRT = CW / KG;                                      // row tiles
    // Ring of one-block slots: this kernel serves short, latency-bound key
    // ranges, so the ring holds one iteration of every key group plus a few
    // blocks in flight, small enough for several CTAs per SM.
    static constexpr int kSlotsWanted = KG * NB + KG + 4;
    static constexpr int kSlotsMax = (200 * 1024) / MmaTile<D, FP8>::kSlot;   // stay within shared memory
    static constexpr int kSlots = kSlotsWanted < kSlotsMax ? kSlotsWanted : kSlotsMax;
    static_assert(kSlots >= KG * NB + KG, "the ring must hold an iteration of every key group plus one block each");
    static constexpr int kRingBytes = kSlots * MmaTile<D, FP8>::kSlot;
    // epilogue: per-warp rows, then (cluster combine) the CTA's merged rows
    static constexpr int kMergeBytes = CW * 16 * (D + 2) * 4 + 16 * (D + 2) * 4;
    static constexpr int kBodyBytes = kRingBytes > kMergeBytes ? kRingBytes : kMergeBytes;
    static constexpr int kSmemBytes = 1024 + kBodyBytes + 2 * kSlots * 8;   // + alignment slack, barriers
};

// Q rows rA / rB of this lane as m16n8k16 A fragments.  bf16 pools: bf16
// pairs in the natural head-dim order.  FP8 pools (fp16 MMAs): the head
// dims of every 16-wide chunk are taken in the order that an ldmatrix of the
// FP8 K rows delivers (lane quad c holds dims 4c .. 4c+3: 4c, 4c+1 as MMA
// k = 2c, 2c+1 and 4c+2, 4c+3 as k = 2c+8, 2c+9); the sum over the head
// dim does not depend on the order.
template <int D, bool FP8>
__device__ __forceinline__ void load_q_frags(uint32_t (&qa)[D / 16][4], const __nv_bfloat16 *q, size_t rowA,
                                             size_t rowB, bool okA, bool okB, int lane)
{
    const int c = lane & 3;
    if constexpr (!FP8) {
        const uint32_t *qw = reinterpret_cast<const uint32_t *>(q);
#pragma unroll
        for (int kk = 0; kk < D / 16; kk++) {
            qa[kk][0] = okA ? __ldg(qw + rowA * (D / 2) + kk * 8 + c) : 0u;
            qa[kk][1] = okB ? __ldg(qw + rowB * (D / 2) + kk * 8 + c) : 0u;
            qa[kk][2] = okA ? __ldg(qw + rowA * (D / 2) + kk * 8 + 4 + c) : 0u;
            qa[kk][3] = okB ? __ldg(qw + rowB * (D / 2) + kk * 8 + 4 + c) : 0u;
        }
    } else {
        const uint2 *q4 = reinterpret_cast<const uint2 *>(q);      // 4 bf16 per load
#pragma unroll
        for (int kk = 0; kk < D / 16; kk++) {
            const uint2 a = okA ? __ldg(q4 + rowA * (D / 4) + kk * 4 + c) : make_uint2(0u, 0u);
            const uint2 bb = okB ? __ldg(q4 + rowB * (D / 4) + kk * 4 + c) : make_uint2(0u, 0u);
            qa[kk][0] = pack_f16x2(bf16_lo(a.x), bf16_hi(a.x));
            qa[kk][1] = pack_f16x2(bf16_lo(bb.x), bf16_hi(bb.x));
            qa[kk][2] = pack_f16x2(bf16_lo(a.y), bf16_hi(a.y));
            qa[kk][3] = pack_f16x2(bf16_lo(bb.y), bf16_hi(bb.y));
        }
    }
}

// S for one 16-key block: sc[0], sc[1] = the two 8-key n-tiles.  FP8: the
// codes go through an fp16 MMA (exact conversion); the K scales are applied
// by the caller.
template <int D, bool FP8 = false>
__device__ __forceinline__ void block_scores(float (&sc0)[4], float (&sc1)[4], const uint32_t (&qa)[D / 16][4],
                                             uint32_t kt, int mi, int mr)
{
    if constexpr (!FP8) {
#pragma unroll
        for (int kk = 0; kk < D / 16; kk++) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4(kt + tile_off<D>((mi >> 1) * 8 + mr, 2 * kk + (mi & 1)), b0, b1, b2, b3);
            mma_16816(sc0, qa[kk], b0, b1);
            mma_16816(sc1, qa[kk], b2, b3);
        }
    } else {
        // matrix mi: n-tile mi & 1, 16-dim chunk kk + (mi >> 1); a lane gets
        // 4 codes (dims 4c .. 4c+3) of key row lane / 4
#pragma unroll
        for (int kk = 0; kk < D / 16; kk += 2) {
            uint32_t r0, r1, r2, r3;
            ldsm_x4(kt + tile_off<D, true>((mi & 1) * 8 + mr, kk + (mi >> 1)), r0, r1, r2, r3);
            uint32_t b[8];
            e4m3x4_to_f16x2x2(r0, b[0], b[1]);
            e4m3x4_to_f16x2x2(r1, b[2], b[3]);
            e4m3x4_to_f16x2x2(r2, b[4], b[5]);
            e4m3x4_to_f16x2x2(r3, b[6], b[7]);
            mma_16816_f16(sc0, qa[kk], b[0], b[1]);
            mma_16816_f16(sc1, qa[kk], b[2], b[3]);
            mma_16816_f16(sc0, qa[kk + 1], b[4], b[5]);
            mma_16816_f16(sc1, qa[kk + 1], b[6], b[7]);
        }
    }
}

// O += P V for one 16-key block.  FP8: a transposed ldmatrix of the codes
// gives a lane 2 keys x 2 adjacent dims; a byte permute splits them into the
// even-dim and the odd-dim B fragments, so O's n-tile 2q holds the even and
// 2q+1 the odd dims of 16-dim chunk q (see o_col).  P comes with the V
// scales folded in (fp16).
template <int D, bool FP8 = false>
__device__ __forceinline__ void block_pv(float (&o)[D / 8][4], const uint32_t (&pa)[4], uint32_t vt, int mi, int mr)
{
    if constexpr (!FP8) {
#pragma unroll
        for (int np = 0; np < D / 16; np++) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(vt + tile_off<D>((mi & 1) * 8 + mr, 2 * np + (mi >> 1)), b0, b1, b2, b3);
            mma_16816(o[2 * np], pa, b0, b1);
            mma_16816(o[2 * np + 1], pa, b2, b3);
        }
    } else {
#pragma unroll
        for (int q = 0; q < D / 16; q += 2) {
            uint32_t r0, r1, r2, r3;       // keys 0-7 / 8-15 of chunk q, then of chunk q + 1
            ldsm_x4_t(vt + tile_off<D, true>((mi & 1) * 8 + mr, q + (mi >> 1)), r0, r1, r2, r3);
            // bytes (0, 2) are the even dim of keys 2c, 2c+1, bytes (1, 3) the odd one
            uint32_t e0, o0, e1, o1, e2, o2, e3, o3;
            e4m3x4_to_f16x2x2(prmt(r0, 0u, 0x3120u), e0, o0);
            e4m3x4_to_f16x2x2(prmt(r1, 0u, 0x3120u), e1, o1);
            e4m3x4_to_f16x2x2(prmt(r2, 0u, 0x3120u), e2, o2);
            e4m3x4_to_f16x2x2(prmt(r3, 0u, 0x3120u), e3, o3);
            mma_16816_f16(o[2 * q], pa, e0, e1);
            mma_16816_f16(o[2 * q + 1], pa, o0, o1);
            mma_16816_f16(o[2 * q + 2], pa, e2, e3);
            mma_16816_f16(o[2 * q + 3], pa, o2, o3);
        }
    }
}

// Head dim of accumulator o[n][2 hr + j] of lane quad c.
template <bool FP8>
__device__ __forceinline__ int o_col(int n, int c, int j)
{
    return FP8 ? 16 * (n >> 1) + 4 * c + 2 * j + (n & 1) : n * 8 + 2 * c + j;
}

// P fragments (A operand of PV) from the probabilities of two 8-key n-tiles;
// FP8 pools fold each key's V scale in and use fp16.
template <bool FP8>
__device__ __forceinline__ void pack_p(uint32_t (&pa)[4], const float (&p0)[4], const float (&p1)[4],
                                       const float (&vs0)[2], const float (&vs1)[2])
{
    if constexpr (!FP8) {
        pa[0] = pack_bf16x2(p0[0], p0[1]);
        pa[1] = pack_bf16x2(p0[2], p0[3]);
        pa[2] = pack_bf16x2(p1[0], p1[1]);
        pa[3] = pack_bf16x2(p1[2], p1[3]);
    } else {
        pa[0] = pack_f16x2(p0[0] * vs0[0], p0[1] * vs0[1]);
        pa[1] = pack_f16x2(p0[2] * vs0[0], p0[3] * vs0[1]);
        pa[2] = pack_f16x2(p1[0] * vs1[0], p1[1] * vs1[1]);
        pa[3] = pack_f16x2(p1[2] * vs1[0], p1[3] * vs1[1]);
    }
}

// Per-warp results into shared memory for the epilogue (the ring is free
// once every consumer has passed named barrier 1): o rows at mo[warp][row][D],
// (m, l) at mml[warp][row][2].  Row-major tiles: lane quad c holds rows
// lane / 4 and lane / 4 + 8.
template <int D, bool FP8, int CW>
__device__ __forceinline__ void stage_rows(const float (&o)[D / 8][4], const float (&m)[2], const float (&l)[2],
                                           bool alive, float *mo, float *mml, uint32_t *s_flags)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    named_bar_sync(1, CW * 32);                                   // every consumer is done with the ring
#pragma unroll
    for (int hr = 0; hr < 2; hr++) {
        const int lr = (lane >> 2) + 8 * hr;
#pragma unroll
        for (int n = 0; n < D / 8; n++) {
            if constexpr (!FP8) {
                *reinterpret_cast<float2 *>(mo + (warp * 16 + lr) * D + o_col<false>(n, lane & 3, 0)) =
                    make_float2(o[n][2 * hr], o[n][2 * hr + 1]);
            } else {
                mo[(warp * 16 + lr) * D + o_col<true>(n, lane & 3, 0)] = o[n][2 * hr];
                mo[(warp * 16 + lr) * D + o_col<true>(n, lane & 3, 1)] = o[n][2 * hr + 1];
            }
        }
        if ((lane & 3) == 0) {
            mml[(warp * 16 + lr) * 2] = m[hr];
            mml[(warp * 16 + lr) * 2 + 1] = l[hr];
        }
    }
    if (!alive && lane == 0) s_flags[0] = 1u;
}

// The same for key-major tiles: lane 4r + c holds rows 2c, 2c+1 (of at
// most kKeyMajorRows) and their weight sums over keys r, r+8 of each block,
// which are summed across r here.  HP > 1: the warp serves KV head hd of a
// CTA of HP adjacent heads, whose rows the epilogue sees as one group of
// HP * g query heads: local row x (token x / g, query head x % g of head hd)
// is staged as row (x / g) * HP * g + hd * g + x % g of warp slot `slot`;
// only the nr_h real rows are staged.
template <int D, bool FP8, int CW, int HP = 1>
__device__ __forceinline__ void stage_rows_t(const float (&o)[D / 16][4], const float (&m)[2], float (&l)[2],
                                             bool alive, float *mo, float *mml, uint32_t *s_flags, int slot = -1,
                                             int hd = 0, int g = 1, int nr_h = kKeyMajorRows)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = lane >> 2, c = lane & 3;
    if (HP == 1) slot = warp;
#pragma unroll
    for (int j = 0; j < 2; j++) {
        l[j] += __shfl_xor_sync(0xffffffffu, l[j], 4);
        l[j] += __shfl_xor_sync(0xffffffffu, l[j], 8);
        l[j] += __shfl_xor_sync(0xffffffffu, l[j], 16);
    }
    named_bar_sync(1, CW * 32);                                   // every consumer is done with the ring
#pragma unroll
    for (int j = 0; j < 2; j++) {
        const int x = 2 * c + j;
        if (HP > 1 && x >= nr_h) continue;
        const int rc = HP == 1 ? x : (x / g) * (HP * g) + hd * g + x % g;
        float *row = mo + (slot * 16 + rc) * D;
#pragma unroll
        for (int mt = 0; mt < D / 16; mt++) {
            row[ot_dim<FP8>(mt, r, 0)] = o[mt][j];
            row[ot_dim<FP8>(mt, r, 1)] = o[mt][2 + j];
        }
        if (r == 0) {
            mml[(slot * 16 + rc) * 2] = m[j];
            mml[(slot * 16 + rc) * 2 + 1] = l[j];
        }
    }
    if (!alive && lane == 0) s_flags[0] = 1u;
}

// Epilogue of both MMA kernels, run by the CW consumer warps (named barrier
// 1) after stage_rows / stage_rows_t.  Merges the KG key groups of each row
// tile, writes the CTA's rows as bf16 output or as fp32 split partials, and,
// for split decode rows whose combine runs in the kernel (wl.cnt_off[li] >=
// 0), counts the finished splits of (request, KV head): the CTA that finishes
// the last one combines them and returns the counter to zero for the next
// call.  A CTA whose pipeline wait gave up writes nothing but still counts,
// so counters stay consistent.
// xo non-null (cluster combine): the merged rows stay in this CTA's shared
// memory, unnormalised, at xo[row][D] with (m, l) at xml[row], for the
// cluster's rank 0 to combine.
template <int D, int KG, int CW = kConsumerWarps>
__device__ __forceinline__ void mma_epilogue(const AttnParams &p, const WorkList &wl, int li, int kh, float *mo,
                                             float *mml, uint32_t *s_flags, int nr, int i0, int split, bool partial,
                                             int b, int t, int L, int g, float *xo = nullptr,
                                             float2 *xml = nullptr)
{
    constexpr int kThreads = CW * 32;
    named_bar_sync(1, kThreads);
    const bool ok = s_flags[0] == 0u;                            // the same in every consumer thread
    // one item = 8 consecutive columns of one row: a 16-byte bf16 store (or
    // two 16-byte fp32 stores for a partial)
    constexpr int kChunks = D / 8;
    for (int idx = threadIdx.x; ok && idx < nr * kChunks; idx += kThreads) {
        const int rowc = idx / kChunks, e0 = (idx - rowc * kChunks) * 8;   // row within the CTA
        const int rtile = rowc >> 4, lr = rowc & 15;
        float M = -INFINITY;
#pragma unroll
        for (int q = 0; q < KG; q++) M = fmaxf(M, mml[((rtile * KG + q) * 16 + lr) * 2]);
        const float Ms = M == -INFINITY ? 0.f : M;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f}, ls = 0.f;
#pragma unroll
        for (int q = 0; q < KG; q++) {
            const int wq = rtile * KG + q;
            const float w = exp2f(mml[(wq * 16 + lr) * 2] - Ms);
            ls = fmaf(w, mml[(wq * 16 + lr) * 2 + 1], ls);
            const float4 *src = reinterpret_cast<const float4 *>(mo + (wq * 16 + lr) * D + e0);
            const float4 x0 = src[0], x1 = src[1];
            acc[0] = fmaf(w, x0.x, acc[0]); acc[1] = fmaf(w, x0.y, acc[1]);
            acc[2] = fmaf(w, x0.z, acc[2]); acc[3] = fmaf(w, x0.w, acc[3]);
            acc[4] = fmaf(w, x1.x, acc[4]); acc[5] = fmaf(w, x1.y, acc[5]);
            acc[6] = fmaf(w, x1.z, acc[6]); acc[7] = fmaf(w, x1.w, acc[7]);
        }
        const int i = i0 + rowc / g, h = kh * g + rowc % g;
        if (xo) {
            float4 *dst = reinterpret_cast<float4 *>(xo + rowc * D + e0);
            dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
            dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
            if (e0 == 0) xml[rowc] = make_float2(M, ls);
        } else if (!partial) {
            const float inv = ls > 0.f ? 1.f / ls : 0.f;
            uint4 v;
            v.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
            v.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
            v.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
            v.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
            *reinterpret_cast<uint4 *>(p.out + ((size_t)(b + i) * p.hq + h) * D + e0) = v;
        } else {
            const size_t orow = (size_t)wl.part_off[li] + ((size_t)split * t + i) * p.hq + h;
            float4 *dst = reinterpret_cast<float4 *>(p.part_o + orow * D + e0);
            dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
            dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
            if (e0 == 0) p.part_ml[orow] = make_float2(M, ls);
        }
    }
    if (!partial || wl.cnt_off[li] < 0) return;
    // ---- in-kernel split combine: count this split, the last one combines
    // every planned split counts (with device lengths, those past the run's
    // keys counted with empty partials)
    const int S = decode_splits(t, wl.len[li], p.window, wl.split_tokens);
    uint32_t *cnt = p.counters + (size_t)(wl.cnt_off[li] + kh) * kCounterStride;
    named_bar_sync(1, kThreads);                                  // every partial store of the CTA is issued
    if (threadIdx.x == 0) {
        __threadfence();                                          // release them (cumulative over the barrier)
        const uint32_t old = atomicAdd(cnt, 1u);
        if (old >= (uint32_t)S) atomicOr(p.err, kDevErrCounter); // the workspace was not zero-filled
        const bool last = old + 1u == (uint32_t)S;
        if (last) __threadfence();                                // acquire the other splits' partials
        s_flags[1] = last ? 1u : 0u;
    }
    named_bar_sync(1, kThreads);
    if (s_flags[1] == 0u) return;
    combine_in_cta<D>(p, (size_t)wl.part_off[li], b, t, kh, g, S, threadIdx.x, kThreads);
    if (threadIdx.x == 0) atomicExch(cnt, 0u);                    // ready for the next call
}

// Split combine of a cluster of CS CTAs (the CS splits of one request and KV
// head), after every CTA left its merged rows in xo / xml (mma_epilogue) and
// its wait status in s_flags[0].  Run by every thread of every CTA of the
// cluster (`combiner`: the consumer threads of rank 0), so that each passes
// both cluster barriers: the first publishes every CTA's rows, the second
// keeps each CTA's shared memory alive until rank 0 has read it.  Rank 0
// merges o = sum_c 2^(m_c - M) o_c / sum_c 2^(m_c - M) l_c, M = max_c m_c,
// reading the peers' rows through distributed shared memory, and writes the
// output rows unless some CTA's pipeline wait gave up.
template <int D>
__device__ __forceinline__ void cluster_combine(const AttnParams &p, bool combiner, int CS, const float *xo,
                                                const float2 *xml, const uint32_t *s_flags, int nr, int i0, int b,
                                                int kh, int g, int tid, int nthreads)
{
    __syncwarp();
    cluster_sync_all();
    if (combiner) {
        bool ok = true;
        for (int c = 0; c < CS; c++) ok = ok && ld_cluster_u32(cluster_map(smem_u32(s_flags), c)) == 0u;
        constexpr int kChunks = D / 8;
        const uint32_t xo_s = smem_u32(xo), xml_s = smem_u32(xml);
        for (int idx = tid; ok && idx < nr * kChunks; idx += nthreads) {
            const int rowc = idx / kChunks, e0 = (idx - rowc * kChunks) * 8;
            float M = -INFINITY, ls = 0.f;
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            for (int c = 0; c < CS; c++) {
                const float2 ml = ld_cluster_f2(cluster_map(xml_s + rowc * 8, c));
                const uint32_t xa = cluster_map(xo_s + (rowc * D + e0) * 4, c);
                const float4 x0 = ld_cluster_f4(xa), x1 = ld_cluster_f4(xa + 16);
                const float Mn = fmaxf(M, ml.x);
                const float Ms = Mn == -INFINITY ? 0.f : Mn;
                const float a = exp2f(M - Ms), w = exp2f(ml.x - Ms);   // 2^-inf = 0
                ls = fmaf(ls, a, w * ml.y);
                acc[0] = fmaf(acc[0], a, w * x0.x); acc[1] = fmaf(acc[1], a, w * x0.y);
                acc[2] = fmaf(acc[2], a, w * x0.z); acc[3] = fmaf(acc[3], a, w * x0.w);
                acc[4] = fmaf(acc[4], a, w * x1.x); acc[5] = fmaf(acc[5], a, w * x1.y);
                acc[6] = fmaf(acc[6], a, w * x1.z); acc[7] = fmaf(acc[7], a, w * x1.w);
                M = Mn;
            }
            const float inv = ls > 0.f ? 1.f / ls : 0.f;
            uint4 v;
            v.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
            v.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
            v.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
            v.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
            const int i = i0 + rowc / g, h = kh * g + rowc % g;
            *reinterpret_cast<uint4 *>(p.out + ((size_t)(b + i) * p.hq + h) * D + e0) = v;
        }
    }
    __syncwarp();
    cluster_sync_all();
}

template <int D, int KG, int NB, bool FP8, int CW, bool KM, bool CL = false>
__global__ void __launch_bounds__((CW + 1) * 32) attn_mma_kernel(AttnParams p, const __grid_constant__ WorkList wl,
                                                               const __grid_constant__ CUtensorMap kmap,
                                                               const __grid_constant__ CUtensorMap vmap,
                                                               const __grid_constant__ CUtensorMap ksmap,
                                                               const __grid_constant__ CUtensorMap vsmap)
{
    using T = MmaTile<D, FP8>;
    using C = MmaCfg<D, KG, NB, FP8, CW>;
    static_assert(!CL || KG * C::kRT == CW, "cluster combine: one CTA-wide merge");
    constexpr int R = C::kSlots;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t ring = (raw + 1023u) & ~1023u;                 // 1024-aligned for the swizzle
    uint8_t *ring_ptr = smem_raw + (ring - raw);
    const uint32_t bars = ring + C::kBodyBytes;                   // full[R], then empty[R]
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (R + s); };
    auto slot_addr = [&](int s) { return ring + (uint32_t)s * T::kSlot; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int kh = blockIdx.x;                                    // the KV heads of an item run side by side
    const int li = find_listed(wl, blockIdx.y);
    const int local = blockIdx.y - wl.item_off[li];
    const int r = wl.req[li];
    const int b = wl.qb[li], t = wl.qt[li], L = run_len(p, wl, li);
    const int g = p.group;

    if (L == 0 || t == 0) {                                       // padding request: zero rows
        // Wait like every other CTA: this grid then never completes before the
        // grids it follows, which keeps later programmatic waits transitive.
        pdl_wait();
        if (p.fw_k && wl.mode == kModeDecode && local == 0 && t > 0 && warp == 0) {   // combined call: its rows
            if constexpr (!FP8) fused_kv_write<D>(p, r, b, t, 0, kh, -t, 0, lane, 32);
            else fused_kv_write_fp8(p, r, b, t, 0, kh, 1, -t, 0, lane);
        }
        if (threadIdx.x == 0 && local == 0 && kh == 0) check_meta(p, wl, li);
        for (int idx = threadIdx.x; idx < t * g * D; idx += (CW + 1) * 32) {
            const int rr = idx / D, e = idx - rr * D;
            p.out[((size_t)(b + rr / g) * p.hq + kh * g + rr % g) * D + e] = __float2bfloat16(0.f);
        }
        return;
    }

    int i0, ntok, k_begin, k_end, split = 0;
    bool partial = false;
    if (CL) {
        // cluster combine (decode-class): the request's wl.cluster splits are
        // this cluster's CTAs, rank = local, split_len[li] keys each (trailing
        // splits may be empty); no global partials
        i0 = 0;
        ntok = t;
        split = local;
        k_begin = decode_key_begin(t, L, p.window) + split * wl.split_len[li];
        k_end = min(L, k_begin + wl.split_len[li]);
    } else if (wl.mode == kModeDecode) {
        i0 = 0;
        ntok = t;
        split = local;
        k_begin = decode_key_begin(t, L, p.window) + split * wl.split_tokens;
        k_end = min(L, k_begin + wl.split_tokens);
        partial = wl.part_off[li] >= 0;
    } else {
        // tile of new tokens, keys from the first row's window start (a
        // block boundary); when split, every tile has the request's
        // ceil(L / split) splits and those past the tile's last position
        // leave empty partials (m = -inf, l = 0)
        const int S = wl.split_tokens > 0 ? (L + wl.split_tokens - 1) / wl.split_tokens : 1;
        const int tile = local / S;
        split = local - tile * S;
        i0 = tile * wl.tile_tokens;
        ntok = min(wl.tile_tokens, t - i0);
        const int tend = L - t + i0 + ntok;                       // one past the tile's last position
        const int kb = window_lo(L - t + i0, p.window) & ~15;
        k_begin = kb + (wl.split_tokens > 0 ? split * wl.split_tokens : 0);
        k_end = wl.split_tokens > 0 ? min(tend, k_begin + wl.split_tokens) : tend;
        partial = wl.part_off[li] >= 0;
    }
    const int nr = ntok * g;                                      // rows of this CTA
    const int blk0 = k_begin >> 4;
    const int nblk = max(0, ((k_end + 15) >> 4) - blk0);

    __shared__ uint32_t s_flags[2];                               // epilogue: a wait gave up; last split
    if (threadIdx.x == 0) {
        for (int s = 0; s < R; s++) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), C::kRT);                      // the row tiles that read a block
        }
        s_flags[0] = s_flags[1] = 0u;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == CW) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tmap(&kmap);
            prefetch_tmap(&vmap);
            if constexpr (FP8) {
                prefetch_tmap(&ksmap);
                prefetch_tmap(&vsmap);
            }
        }
        const int32_t *bt = p.block_table + (size_t)r * p.bt_stride + blk0;
        // The block table is not written by the step's K/V scatter: read the
        // first 32 block ids while that kernel may still be running.
        int ids = lane < nblk ? __ldg(bt + lane) : 0, issued = 0;
        pdl_wait();                                               // the step's K/V rows are in the pool
        // combined write + attention: this CTA's share of the request's new
        // rows goes into the pool first (the rows in its key range)
        if (p.fw_k && wl.mode == kModeDecode) {
            if constexpr (!FP8) fused_kv_write<D>(p, r, b, t, L, kh, max(k_begin, L - t), min(k_end, L), lane, 32);
            else fused_kv_write_fp8(p, r, b, t, L, kh, 1, max(k_begin, L - t), min(k_end, L), lane);
            __syncwarp();
            fence_proxy_async_global();                           // lane 0 issues the loads
        }
        // a block's K and V slices of this head into slot s, and for FP8
        // pools the block's K and V scales of this head's group of four
        auto issue = [&](int s, int blk) {
            if (blk < 0 || blk >= p.nb_total) {                   // outside the pool: report, read block 0
                atomicOr(p.err, 2u);
                blk = 0;
            }
            mbar_arrive_expect_tx(full_bar(s), T::kData);
            const uint32_t dst = slot_addr(s);
#pragma unroll
            for (int x = 0; x < T::kBoxes; x++) {
                tma_load_3d(dst + x * T::kBoxBytes, &kmap, full_bar(s), x * T::kBoxCols, kh, blk * 16);
                tma_load_3d(dst + T::kTile + x * T::kBoxBytes, &vmap, full_bar(s), x * T::kBoxCols, kh, blk * 16);
            }
            if constexpr (FP8) {
                tma_load_2d(dst + 2 * T::kTile, &ksmap, full_bar(s), kh & ~(kScaleHeads - 1), blk * 16);
                tma_load_2d(dst + 2 * T::kTile + T::kScaleTile, &vsmap, full_bar(s), kh & ~(kScaleHeads - 1),
                            blk * 16);
            }
        };
        // the ring's first round goes out from one lane per block at once;
        // later blocks, one at a time, as slots come free
        const int first = min(nblk, R < 32 ? R : 32);
        if (lane < first) issue(lane, ids);
        __syncwarp();
        issued = first;
        for (int i = first; i < nblk; i++) {
            if ((i & 31) == 0) ids = (i + lane < nblk) ? __ldg(bt + i + lane) : 0;
            const int s = i % R;
            bool ok = true;
            if (i >= R) ok = mbar_wait(empty_bar(s), ((i / R) - 1) & 1, p.err);
            if (!__all_sync(0xffffffffu, ok)) break;
            issued = i + 1;
            const int blk = __shfl_sync(0xffffffffu, ids, i & 31);
            if (lane == 0) issue(s, blk);
            __syncwarp();
        }
        // Normally every issued block has been consumed by now.  If a wait
        // gave up, keep the CTA (and its shared memory) alive until the copies
        // still in flight have landed, within the same time limit.
        if (issued < nblk && lane == 0) {
            for (int i = issued > R ? issued - R : 0; i < issued; i++) mbar_wait(full_bar(i % R), (i / R) & 1, p.err);
        }
        if (lane == 0 && local == 0 && kh == 0) check_meta(p, wl, li);
        if constexpr (CL) {
            // the producer passes the cluster barriers too (every thread does)
            float *xo = reinterpret_cast<float *>(ring_ptr) + CW * 16 * (D + 2);
            cluster_combine<D>(p, false, wl.cluster, xo, reinterpret_cast<float2 *>(xo + 16 * D), s_flags, 0, 0, b,
                               kh, g, 0, 1);
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int rt = warp / KG, kg = warp % KG;
    const int qbase = L - t + i0;
    const int wspan = win_span(p.window);                         // keys <= position - wspan are outside
    const float sl2 = p.scale_log2;
    const int mi = lane >> 3, mr = lane & 7;                      // ldmatrix: matrix, row within it
    bool alive = true;
    float *mo = reinterpret_cast<float *>(ring_ptr);              // epilogue: [warp][16][D]
    float *mml = mo + CW * 16 * D;                                // [warp][16][2]

    if constexpr (KM) {
        // key-major decode tiles (nr <= kKeyMajorRows, one row tile)
        const int rq = lane >> 2, c2 = 2 * (lane & 3);
        uint32_t qb[D / 16][2];
        load_qt_frags<D, FP8>(qb, p.q, rq < nr ? (size_t)(b + i0 + rq / g) * p.hq + kh * g + rq % g : 0, rq < nr,
                              lane);
        const int qp0 = c2 < nr ? qbase + c2 / g : -1;
        const int qp1 = c2 + 1 < nr ? qbase + (c2 + 1) / g : -1;
        float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
        float o[D / 16][4];
#pragma unroll
        for (int n = 0; n < D / 16; n++) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
        for (int bl0 = kg; bl0 < nblk; bl0 += NB * KG) {
            int slot[NB];
            bool has[NB];
            bool waited = true;
#pragma unroll
            for (int q = 0; q < NB; q++) {
                const int bl = bl0 + q * KG;
                has[q] = bl < nblk;
                slot[q] = bl % R;
                if (has[q] && waited) waited = mbar_wait(full_bar(slot[q]), (bl / R) & 1, p.err);
            }
            if (!waited) {
                alive = false;
                break;
            }
            float sc[NB][4], vs[NB][2];
            uint32_t vt[NB];
#pragma unroll
            for (int q = 0; q < NB; q++) {
                sc[q][0] = sc[q][1] = sc[q][2] = sc[q][3] = 0.f;
                if (has[q]) block_scores_t<D, FP8>(sc[q], qb, slot_addr(slot[q]), mi, mr);
            }
#pragma unroll
            for (int q = 0; q < NB; q++) {
                vt[q] = slot_addr(slot[q]) + T::kTile;
                float f0 = sl2, f1 = sl2;
                vs[q][0] = vs[q][1] = 1.f;
                if constexpr (FP8) {                              // K and V scales of keys rq, rq + 8
                    if (has[q]) {
                        const float *sk = reinterpret_cast<const float *>(ring_ptr + slot[q] * T::kSlot + 2 * T::kTile);
                        const float *sv = sk + T::kScaleTile / 4;
                        const int hs = kh & (kScaleHeads - 1);
                        f0 *= sk[rq * kScaleHeads + hs];
                        f1 *= sk[(rq + 8) * kScaleHeads + hs];
                        vs[q][0] = sv[rq * kScaleHeads + hs];
                        vs[q][1] = sv[(rq + 8) * kScaleHeads + hs];
                    }
                }
                mask_scale_t(sc[q], ((blk0 + bl0 + q * KG) << 4) + rq, k_end, qp0, qp1, wspan, has[q], f0, f1);
            }
            softmax_pv_t<D, FP8, NB>(o, m, l, sc, vs, vt, has, mi, mr);
            __syncwarp();
            if (lane == 0) {
#pragma unroll
                for (int q = 0; q < NB; q++)
                    if (has[q]) mbar_arrive(empty_bar(slot[q]));
            }
        }
        pdl_launch_dependents();                                  // a combine kernel may start launching
        stage_rows_t<D, FP8, CW>(o, m, l, alive, mo, mml, s_flags);
    } else {
        const int row0 = rt * 16;
        const int rA = row0 + (lane >> 2), rB = rA + 8;           // the two rows this lane holds
        const int qposA = rA < nr ? qbase + rA / g : -1;
        const int qposB = rB < nr ? qbase + rB / g : -1;

        // Q as mma A fragments, straight from global memory.
        uint32_t qa[D / 16][4];
        {
            const size_t rowA = rA < nr ? (size_t)(b + i0 + rA / g) * p.hq + kh * g + rA % g : 0;
            const size_t rowB = rB < nr ? (size_t)(b + i0 + rB / g) * p.hq + kh * g + rB % g : 0;
            load_q_frags<D, FP8>(qa, p.q, rowA, rowB, rA < nr, rB < nr, lane);
        }

        float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
        float o[D / 8][4];
#pragma unroll
        for (int n = 0; n < D / 8; n++) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;

        // Each iteration takes NB blocks of this key group (kg, kg + KG, ...):
        // NB independent MMA chains and one softmax update per 16*NB keys
        // (shorter latency chains); with NB = 1 each warp holds one ring slot
        // at a time, leaving more of the ring for copies in flight.
        for (int bl0 = kg; bl0 < nblk; bl0 += NB * KG) {
            int slot[NB];
            bool has[NB];
            bool waited = true;
#pragma unroll
            for (int q = 0; q < NB; q++) {
                const int bl = bl0 + q * KG;
                has[q] = bl < nblk;
                slot[q] = bl % R;
                if (has[q] && waited) waited = mbar_wait(full_bar(slot[q]), (bl / R) & 1, p.err);
            }
            if (!waited) {
                alive = false;
                break;
            }
            float sc[2 * NB][4];
#pragma unroll
            for (int n = 0; n < 2 * NB; n++) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
#pragma unroll
            for (int q = 0; q < NB; q++)
                if (has[q]) block_scores<D, FP8>(sc[2 * q], sc[2 * q + 1], qa, slot_addr(slot[q]), mi, mr);
            // FP8 pools: the K and V scales of this lane's four keys of each block
            float ksc[2 * NB][2], vsc[2 * NB][2];
#pragma unroll
            for (int n = 0; n < 2 * NB; n++) {
                ksc[n][0] = ksc[n][1] = vsc[n][0] = vsc[n][1] = 1.f;
                if constexpr (FP8) {
                    const float *sk =
                        reinterpret_cast<const float *>(ring_ptr + slot[n >> 1] * T::kSlot + 2 * T::kTile);
                    const float *sv = sk + T::kScaleTile / 4;
                    const int kr = (n & 1) * 8 + 2 * (lane & 3);    // key row within the block
                    const int hs = kh & (kScaleHeads - 1);
                    if (has[n >> 1]) {
                        ksc[n][0] = sk[kr * kScaleHeads + hs];
                        ksc[n][1] = sk[(kr + 1) * kScaleHeads + hs];
                        vsc[n][0] = sv[kr * kScaleHeads + hs];
                        vsc[n][1] = sv[(kr + 1) * kScaleHeads + hs];
                    }
                }
            }
            // scale into the exp2 domain, causal and range mask
#pragma unroll
            for (int n = 0; n < 2 * NB; n++) {
                const int kc = ((blk0 + bl0 + (n >> 1) * KG) << 4) + (n & 1) * 8 + 2 * (lane & 3);
#pragma unroll
                for (int v = 0; v < 4; v++) {
                    const int key = kc + (v & 1);
                    const int qp = v < 2 ? qposA : qposB;
                    const bool ok = has[n >> 1] && key < k_end && key <= qp && key > qp - wspan;
                    sc[n][v] = ok ? sc[n][v] * (FP8 ? ksc[n][v & 1] * sl2 : sl2) : -INFINITY;
                }
            }
            float pr[2 * NB][4];
#pragma unroll
            for (int hr = 0; hr < 2; hr++) {
                float mx = -INFINITY;
#pragma unroll
                for (int n = 0; n < 2 * NB; n++) mx = max3f(mx, sc[n][2 * hr], sc[n][2 * hr + 1]);
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                const float mnew = fmaxf(m[hr], mx);
                const float ms = mnew == -INFINITY ? 0.f : mnew;
                const float alpha = exp2f(m[hr] - ms);
                m[hr] = mnew;
                float sum = 0.f;
#pragma unroll
                for (int n = 0; n < 2 * NB; n++) {
                    pr[n][2 * hr] = exp2f(sc[n][2 * hr] - ms);
                    pr[n][2 * hr + 1] = exp2f(sc[n][2 * hr + 1] - ms);
                    sum += pr[n][2 * hr] + pr[n][2 * hr + 1];
                }
                l[hr] = l[hr] * alpha + sum;
#pragma unroll
                for (int n = 0; n < D / 8; n++) {
                    o[n][2 * hr] *= alpha;
                    o[n][2 * hr + 1] *= alpha;
                }
            }
#pragma unroll
            for (int q = 0; q < NB; q++) {
                if (!has[q]) continue;
                uint32_t pa[4];
                pack_p<FP8>(pa, pr[2 * q], pr[2 * q + 1], vsc[2 * q], vsc[2 * q + 1]);
                block_pv<D, FP8>(o, pa, slot_addr(slot[q]) + T::kTile, mi, mr);
            }
            __syncwarp();
            if (lane == 0) {
#pragma unroll
                for (int q = 0; q < NB; q++)
                    if (has[q]) mbar_arrive(empty_bar(slot[q]));
            }
        }
        pdl_launch_dependents();                                  // a combine kernel may start launching
#pragma unroll
        for (int hr = 0; hr < 2; hr++) {
            l[hr] += __shfl_xor_sync(0xffffffffu, l[hr], 1);
            l[hr] += __shfl_xor_sync(0xffffffffu, l[hr], 2);
        }
        stage_rows<D, FP8, CW>(o, m, l, alive, mo, mml, s_flags);
    }
    if constexpr (CL) {
        float *xo = mml + CW * 16 * 2;                           // after the per-warp rows: [16][D], then (m, l)
        float2 *xml = reinterpret_cast<float2 *>(xo + 16 * D);
        mma_epilogue<D, KG, CW>(p, wl, li, kh, mo, mml, s_flags, nr, i0, split, false, b, t, L, g, xo, xml);
        named_bar_sync(1, CW * 32);                               // every merged row of the CTA is in xo
        cluster_combine<D>(p, local == 0, wl.cluster, xo, xml, s_flags, nr, i0, b, kh, g, threadIdx.x, CW * 32);
    } else {
        mma_epilogue<D, KG, CW>(p, wl, li, kh, mo, mml, s_flags, nr, i0, split, partial, b, t, L, g);
    }
}

// ---------------------------------------------------------------- streaming decode
//
// Long decode splits (at least kLongSplit keys per CTA) stream their blocks
// through a ring of stages of KG blocks each, one full/empty barrier pair per
// stage: every consumer warp takes one block of each stage.  A stage holds
// its KG K slices, then its KG V slices, then (FP8 pools) the KG K-scale and
// KG V-scale boxes, so that swizzled slices stay on 1024-byte boundaries
// without padding.  Measured on the
// 256-request and the 32 x 32768 decode workloads this keeps more copies in
// flight per SM than the one-block slot ring above, which wins on short,
// latency-bound ranges instead.
//
// HP = 2 (FP8 pools, key-major tiles): a CTA serves two adjacent KV heads,
// and one TMA box of {128 codes, 2 heads, 16 slots} (4 KB) carries a block's
// K (or V) rows of both, so a block costs half the copy operations per
// head: with 2 KB code slices the copies, not the bytes, bounded the
// quantized decode.  Consumer warps 0..KG-1 serve the first head, KG..2KG-1
// the second (KG = 2).
template <int D, int KG, bool FP8 = false, int HP = 1>
struct StreamCfg {
    static_assert(HP == 1 || (FP8 && HP * KG == kConsumerWarps), "two heads per CTA: FP8, 2 key groups per head");
    static constexpr int kRT = kConsumerWarps / KG;                          // row tiles (HP > 1: heads)
    using T = MmaTile<D, FP8>;
    static constexpr int kTileH = HP * T::kTile;                             // K (or V) slices of HP heads
    static constexpr int kBlockBytes = 2 * kTileH + 2 * T::kScaleTile;
    static constexpr int kStageBytes = KG * kBlockBytes;
    static constexpr int kStages0 = kStageBudget / kStageBytes;
    static constexpr int kStages = kStages0 > 8 ? 8 : (kStages0 < 2 ? 2 : kStages0);
    static constexpr int kVOff = KG * kTileH;                                // offsets within a stage
    static constexpr int kKsOff = 2 * KG * kTileH;
    static constexpr int kVsOff = kKsOff + KG * T::kScaleTile;
    static constexpr int kRingBytes = kStages * kStageBytes;
    static constexpr int kMergeBytes = kConsumerWarps * 16 * (D + 2) * 4;
    static constexpr int kBodyBytes = kRingBytes > kMergeBytes ? kRingBytes : kMergeBytes;
    static constexpr int kSmemBytes = 1024 + kBodyBytes + 2 * kStages * 8;   // + alignment slack, barriers
};

template <int D, int KG, bool FP8, bool KM, int HP = 1>
__global__ void __launch_bounds__(kMmaThreads) attn_stream_kernel(AttnParams p, const __grid_constant__ WorkList wl,
                                                               const __grid_constant__ CUtensorMap kmap,
                                                               const __grid_constant__ CUtensorMap vmap,
                                                               const __grid_constant__ CUtensorMap ksmap,
                                                               const __grid_constant__ CUtensorMap vsmap)
{
    using T = MmaTile<D, FP8>;
    using C = StreamCfg<D, KG, FP8, HP>;
    static_assert(HP == 1 || KM, "two heads per CTA: key-major tiles only");
    constexpr int S = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t ring = (raw + 1023u) & ~1023u;                 // 1024-aligned for the swizzle
    uint8_t *ring_ptr = smem_raw + (ring - raw);
    const uint32_t bars = ring + C::kBodyBytes;                   // full[S], then empty[S]
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (S + s); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // The KV heads of an item run side by side.  HP > 1: this CTA serves
    // heads HP * kh .. HP * kh + HP - 1, and its rows are those of one group
    // of HP * g query heads (the epilogue's view: group kh of size gg).
    const int kh = blockIdx.x;
    const int kh0 = kh * HP;                                      // first KV head of the CTA
    const int li = find_listed(wl, blockIdx.y);
    const int local = blockIdx.y - wl.item_off[li];
    const int r = wl.req[li];
    const int b = wl.qb[li], t = wl.qt[li], L = run_len(p, wl, li);
    const int g = p.group;
    const int gg = HP * g;

    if (L == 0 || t == 0) {                                       // padding request: zero rows
        pdl_wait();                                               // keeps later programmatic waits transitive
        if (p.fw_k && wl.mode == kModeDecode && local == 0 && t > 0 && warp == 0) {   // combined call: its rows
            if constexpr (!FP8) fused_kv_write<D>(p, r, b, t, 0, kh0, -t, 0, lane, 32);
            else fused_kv_write_fp8(p, r, b, t, 0, kh0, HP, -t, 0, lane);
        }
        if (threadIdx.x == 0 && local == 0 && kh == 0) check_meta(p, wl, li);
        for (int idx = threadIdx.x; idx < t * gg * D; idx += kMmaThreads) {
            const int rr = idx / D, e = idx - rr * D;
            p.out[((size_t)(b + rr / gg) * p.hq + kh * gg + rr % gg) * D + e] = __float2bfloat16(0.f);
        }
        return;
    }

    int i0, ntok, k_begin, k_end, split = 0;
    bool partial = false;
    if (wl.mode == kModeDecode) {
        i0 = 0;
        ntok = t;
        split = local;
        k_begin = decode_key_begin(t, L, p.window) + split * wl.split_tokens;
        k_end = min(L, k_begin + wl.split_tokens);
        partial = wl.part_off[li] >= 0;
    } else {
        i0 = local * wl.tile_tokens;
        ntok = min(wl.tile_tokens, t - i0);
        k_begin = window_lo(L - t + i0, p.window) & ~15;
        k_end = L - t + i0 + ntok;                                // one past the tile's last position
    }
    const int nr = ntok * g;                                      // rows of this CTA per KV head
    const int blk0 = k_begin >> 4;
    const int nblk = ((k_end + 15) >> 4) - blk0;
    const int iters = (nblk + KG - 1) / KG;

    __shared__ uint32_t s_flags[2];                               // epilogue: a wait gave up; last split
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; s++) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), kConsumerWarps);
        }
        s_flags[0] = s_flags[1] = 0u;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tmap(&kmap);
            prefetch_tmap(&vmap);
            if constexpr (FP8) {
                prefetch_tmap(&ksmap);
                prefetch_tmap(&vsmap);
            }
        }
        const int32_t *bt = p.block_table + (size_t)r * p.bt_stride + blk0;
        int ids = lane < nblk ? __ldg(bt + lane) : 0, issued = 0;   // not written by the scatter
        pdl_wait();                                               // the step's K/V rows are in the pool
        // combined write + attention: this CTA's share of the request's new
        // rows (of its HP heads) goes into the pool first (the rows in its key range)
        if (p.fw_k && wl.mode == kModeDecode) {
            if constexpr (!FP8) fused_kv_write<D>(p, r, b, t, L, kh0, max(k_begin, L - t), min(k_end, L), lane, 32);
            else fused_kv_write_fp8(p, r, b, t, L, kh0, HP, max(k_begin, L - t), min(k_end, L), lane);
            __syncwarp();
            fence_proxy_async_global();                           // lane 0 issues the loads
        }
        for (int it = 0; it < iters; it++) {
            const int base = it * KG;
            if ((base & 31) == 0 && base > 0) ids = (base + lane < nblk) ? __ldg(bt + base + lane) : 0;
            const int s = it % S;
            bool ok = true;
            if (it >= S) ok = mbar_wait(empty_bar(s), ((it / S) & 1) ^ 1, p.err);
            if (!__all_sync(0xffffffffu, ok)) break;
            issued = it + 1;
            const int nv = min(KG, nblk - base);
            if (lane == 0) mbar_arrive_expect_tx(full_bar(s), nv * C::kBlockBytes);
            for (int j = 0; j < nv; j++) {
                int blk = __shfl_sync(0xffffffffu, ids, (base + j) & 31);
                if (lane == 0) {
                    if (blk < 0 || blk >= p.nb_total) {           // outside the pool: report, read block 0
                        atomicOr(p.err, 2u);
                        blk = 0;
                    }
                    const uint32_t st = ring + s * C::kStageBytes;
                    const uint32_t kd = st + j * C::kTileH, vd = st + C::kVOff + j * C::kTileH;
                    // HP > 1: the maps' boxes span HP heads (T::kBoxes is 1)
                    for (int x = 0; x < T::kBoxes; x++) {
                        tma_load_3d(kd + x * T::kBoxBytes, &kmap, full_bar(s), x * T::kBoxCols, kh0, blk * 16);
                        tma_load_3d(vd + x * T::kBoxBytes, &vmap, full_bar(s), x * T::kBoxCols, kh0, blk * 16);
                    }
                    if constexpr (FP8) {
                        const int h4 = kh0 & ~(kScaleHeads - 1);
                        tma_load_2d(st + C::kKsOff + j * T::kScaleTile, &ksmap, full_bar(s), h4, blk * 16);
                        tma_load_2d(st + C::kVsOff + j * T::kScaleTile, &vsmap, full_bar(s), h4, blk * 16);
                    }
                }
            }
            __syncwarp();
        }
        // Normally every issued stage has been consumed by now.  If a wait
        // gave up, keep the CTA (and its shared memory) alive until the
        // copies still in flight have landed, within the same time limit.
        if (issued < iters && lane == 0) {
            for (int it = issued > S ? issued - S : 0; it < issued; it++)
                mbar_wait(full_bar(it % S), (it / S) & 1, p.err);
        }
        if (lane == 0 && local == 0 && kh == 0) check_meta(p, wl, li);
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int rt = warp / KG, kg = warp % KG;
    const int qbase = L - t + i0;
    const int wspan = win_span(p.window);                         // keys <= position - wspan are outside
    const float sl2 = p.scale_log2;
    const int mi = lane >> 3, mr = lane & 7;                      // ldmatrix: matrix, row within it
    bool alive = true;
    float *mo = reinterpret_cast<float *>(ring_ptr);              // epilogue: [warp][16][D]
    float *mml = mo + kConsumerWarps * 16 * D;                    // [warp][16][2]

    if constexpr (KM) {
        // key-major decode tiles (nr <= kKeyMajorRows, one row tile per KV
        // head); HP > 1: warp group rt serves KV head kh0 + rt
        const int hd = HP > 1 ? rt : 0;
        const int khw = kh0 + hd;                                 // this warp's KV head
        const int rq = lane >> 2, c2 = 2 * (lane & 3);
        uint32_t qb[D / 16][2];
        load_qt_frags<D, FP8>(qb, p.q, rq < nr ? (size_t)(b + i0 + rq / g) * p.hq + khw * g + rq % g : 0, rq < nr,
                              lane);
        const int qp0 = c2 < nr ? qbase + c2 / g : -1;
        const int qp1 = c2 + 1 < nr ? qbase + (c2 + 1) / g : -1;
        float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
        float o[D / 16][4];
#pragma unroll
        for (int n = 0; n < D / 16; n++) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
        for (int it = 0; it < iters; it++) {
            const int s = it % S;
            if (!mbar_wait(full_bar(s), (it / S) & 1, p.err)) {
                alive = false;
                break;
            }
            const int bl = it * KG + kg;
            if (bl < nblk) {
                const uint32_t kt = ring + s * C::kStageBytes + kg * C::kTileH;
                float sc[1][4] = {{0.f, 0.f, 0.f, 0.f}}, vs[1][2] = {{1.f, 1.f}};
                const uint32_t vt[1] = {kt + C::kVOff};
                const bool has[1] = {true};
                block_scores_t<D, FP8, HP>(sc[0], qb, kt, mi, mr, hd);
                float f0 = sl2, f1 = sl2;
                if constexpr (FP8) {                              // K and V scales of keys rq, rq + 8
                    const uint8_t *st = ring_ptr + s * C::kStageBytes;
                    const float *sk = reinterpret_cast<const float *>(st + C::kKsOff + kg * T::kScaleTile);
                    const float *sv = reinterpret_cast<const float *>(st + C::kVsOff + kg * T::kScaleTile);
                    const int hs = khw & (kScaleHeads - 1);
                    f0 *= sk[rq * kScaleHeads + hs];
                    f1 *= sk[(rq + 8) * kScaleHeads + hs];
                    vs[0][0] = sv[rq * kScaleHeads + hs];
                    vs[0][1] = sv[(rq + 8) * kScaleHeads + hs];
                }
                mask_scale_t(sc[0], ((blk0 + bl) << 4) + rq, k_end, qp0, qp1, wspan, true, f0, f1);
                softmax_pv_t<D, FP8, 1, HP>(o, m, l, sc, vs, vt, has, mi, mr, hd);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty_bar(s));
        }
        pdl_launch_dependents();                                  // a combine kernel may start launching
        stage_rows_t<D, FP8, kConsumerWarps, HP>(o, m, l, alive, mo, mml, s_flags, kg, hd, g, nr);
    } else {
        const int row0 = rt * 16;
        const int rA = row0 + (lane >> 2), rB = rA + 8;           // the two rows this lane holds
        const int qposA = rA < nr ? qbase + rA / g : -1;
        const int qposB = rB < nr ? qbase + rB / g : -1;

        // Q as mma A fragments, straight from global memory.
        uint32_t qa[D / 16][4];
        {
            const size_t rowA = rA < nr ? (size_t)(b + i0 + rA / g) * p.hq + kh * g + rA % g : 0;
            const size_t rowB = rB < nr ? (size_t)(b + i0 + rB / g) * p.hq + kh * g + rB % g : 0;
            load_q_frags<D, FP8>(qa, p.q, rowA, rowB, rA < nr, rB < nr, lane);
        }

        float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
        float o[D / 8][4];
#pragma unroll
        for (int n = 0; n < D / 8; n++) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;

        for (int it = 0; it < iters; it++) {
            const int s = it % S;
            if (!mbar_wait(full_bar(s), (it / S) & 1, p.err)) {
                alive = false;
                break;
            }
            const int bl = it * KG + kg;
            if (bl < nblk) {
                const uint32_t kt = ring + s * C::kStageBytes + kg * T::kTile;
                const uint32_t vt = kt + C::kVOff;
                const int key0 = (blk0 + bl) << 4;
                float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                block_scores<D, FP8>(sc[0], sc[1], qa, kt, mi, mr);
                // FP8 pools: the K and V scales of this lane's four keys
                float ksc[2][2] = {{1.f, 1.f}, {1.f, 1.f}}, vsc[2][2] = {{1.f, 1.f}, {1.f, 1.f}};
                if constexpr (FP8) {
                    const uint8_t *st = ring_ptr + s * C::kStageBytes;
                    const float *sk = reinterpret_cast<const float *>(st + C::kKsOff + kg * T::kScaleTile);
                    const float *sv = reinterpret_cast<const float *>(st + C::kVsOff + kg * T::kScaleTile);
                    const int hs = kh & (kScaleHeads - 1);
#pragma unroll
                    for (int n = 0; n < 2; n++) {
                        const int kr = n * 8 + 2 * (lane & 3);
                        ksc[n][0] = sk[kr * kScaleHeads + hs];
                        ksc[n][1] = sk[(kr + 1) * kScaleHeads + hs];
                        vsc[n][0] = sv[kr * kScaleHeads + hs];
                        vsc[n][1] = sv[(kr + 1) * kScaleHeads + hs];
                    }
                }
                // scale into the exp2 domain, causal and range mask
                const int kc = key0 + 2 * (lane & 3);
#pragma unroll
                for (int n = 0; n < 2; n++) {
#pragma unroll
                    for (int v = 0; v < 4; v++) {
                        const int key = kc + n * 8 + (v & 1);
                        const int qp = v < 2 ? qposA : qposB;
                        sc[n][v] = (key < k_end && key <= qp && key > qp - wspan)
                                       ? sc[n][v] * (FP8 ? ksc[n][v & 1] * sl2 : sl2) : -INFINITY;
                    }
                }
                float pr[2][4];
#pragma unroll
                for (int hr = 0; hr < 2; hr++) {
                    float mx =
                        fmaxf(fmaxf(sc[0][2 * hr], sc[0][2 * hr + 1]), fmaxf(sc[1][2 * hr], sc[1][2 * hr + 1]));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                    const float mnew = fmaxf(m[hr], mx);
                    const float ms = mnew == -INFINITY ? 0.f : mnew;
                    const float alpha = exp2f(m[hr] - ms);
                    m[hr] = mnew;
                    pr[0][2 * hr] = exp2f(sc[0][2 * hr] - ms);
                    pr[0][2 * hr + 1] = exp2f(sc[0][2 * hr + 1] - ms);
                    pr[1][2 * hr] = exp2f(sc[1][2 * hr] - ms);
                    pr[1][2 * hr + 1] = exp2f(sc[1][2 * hr + 1] - ms);
                    l[hr] = l[hr] * alpha + (pr[0][2 * hr] + pr[0][2 * hr + 1]) +
                            (pr[1][2 * hr] + pr[1][2 * hr + 1]);
#pragma unroll
                    for (int n = 0; n < D / 8; n++) {
                        o[n][2 * hr] *= alpha;
                        o[n][2 * hr + 1] *= alpha;
                    }
                }
                uint32_t pa[4];
                pack_p<FP8>(pa, pr[0], pr[1], vsc[0], vsc[1]);
                block_pv<D, FP8>(o, pa, vt, mi, mr);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty_bar(s));
        }

        pdl_launch_dependents();                                  // a combine kernel may start launching
#pragma unroll
        for (int hr = 0; hr < 2; hr++) {
            l[hr] += __shfl_xor_sync(0xffffffffu, l[hr], 1);
            l[hr] += __shfl_xor_sync(0xffffffffu, l[hr], 2);
        }
        stage_rows<D, FP8, kConsumerWarps>(o, m, l, alive, mo, mml, s_flags);
    }
    mma_epilogue<D, KG>(p, wl, li, kh, mo, mml, s_flags, nr * HP, i0, split, partial, b, t, L, gg);
}

// ---------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// Tensor map of one pool viewed as [slots][Hkv][D] with a box of
// box_heads adjacent KV heads' 16 rows x box_cols columns; elements of
// elem_bytes (2: bf16, 1: FP8 codes).
static cudaError_t make_pool_tmap_e(CUtensorMap *map, const void *pool, int64_t num_slots, int hkv, int d,
                                   int box_cols, bool swizzle128, int elem_bytes, int box_heads = 1)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)hkv, (cuuint64_t)num_slots};
    cuuint64_t strides[2] = {(cuuint64_t)d * elem_bytes, (cuuint64_t)hkv * d * elem_bytes};
    cuuint32_t box[3] = {(cuuint32_t)box_cols, (cuuint32_t)box_heads, 16};
    cuuint32_t estr[3] = {1, 1, 1};
    // a single 128-byte code row (FP8, head_dim 128) is promoted to 128 bytes
    // only: 256 would fetch the next head's row as well
    const int64_t run = (int64_t)d * elem_bytes * box_heads;     // contiguous bytes per slot in a box
    CUresult res = fn(map, elem_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                      const_cast<void *>(pool), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                      run >= 256 ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B : CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return res == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_pool_tmap(CUtensorMap *map, const void *pool, int64_t num_slots, int hkv, int d, int box_cols,
                           bool swizzle128)
{
    return make_pool_tmap_e(map, pool, num_slots, hkv, d, box_cols, swizzle128, 2);
}

// Tensor map of an FP8 pool's codes [slots][Hkv][128] with a box of one
// head's 128-byte code row x 16 slots, 128-byte swizzle.
cudaError_t make_code_tmap(CUtensorMap *map, const void *pool, int64_t num_slots, int hkv)
{
    return make_pool_tmap_e(map, pool, num_slots, hkv, 128, 128, true, 1);
}

// Tensor map of an FP8 pool's scales [slots][Hkv] fp32 with a box of 16
// slots x kScaleHeads heads (16-byte rows; Hkv a multiple of kScaleHeads).
static cudaError_t make_scale_tmap(CUtensorMap *map, const float *scales, int64_t num_slots, int hkv)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    cuuint64_t dims[2] = {(cuuint64_t)hkv, (cuuint64_t)num_slots};
    cuuint64_t strides[1] = {(cuuint64_t)hkv * 4};
    cuuint32_t box[2] = {(cuuint32_t)kScaleHeads, 16};
    cuuint32_t estr[2] = {1, 1};
    CUresult res = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(scales), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return res == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Tensor map of q [tokens][Hq][D] with a box of one KV head's g query heads
// x 128/g tokens x 64 columns (128 rows of the MMA tile), 128-byte swizzle.
cudaError_t make_q_tmap(CUtensorMap *map, const void *q, int num_tokens, int hq, int d, int g)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)hq, (cuuint64_t)num_tokens};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)hq * d * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)g, (cuuint32_t)(128 / g)};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult res = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return res == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int D, int KG, int NB, bool FP8, int CW = kConsumerWarps, bool KM = false, bool CL = false>
static cudaError_t launch_mma_dk(const AttnParams &p, const WorkList &wl, int num_items, const CUtensorMap &km,
                                 const CUtensorMap &vm, const CUtensorMap &ksm, const CUtensorMap &vsm,
                                 cudaStream_t stream)
{
    constexpr int smem = MmaCfg<D, KG, NB, FP8, CW>::kSmemBytes;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(attn_mma_kernel<D, KG, NB, FP8, CW, KM, CL>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    });
    if (attr_err != cudaSuccess) return attr_err;
    if (num_items > 65535) return cudaErrorInvalidConfiguration;
    if (CL && (wl.cluster < 2 || wl.cluster > kMaxClusterSplits || num_items % wl.cluster != 0))
        return cudaErrorInvalidConfiguration;
    dim3 grid(p.hkv, num_items);                                // KV heads adjacent: they share pool pages
    launch_begin(stream, wl.mode == kModeDecode ? kAttnMmaDecode : kAttnMmaPrefill);
    cudaError_t e = CL ? launch_cluster_maybe_pdl(attn_mma_kernel<D, KG, NB, FP8, CW, KM, CL>, grid, dim3((CW + 1) * 32),
                                                  smem, stream, (unsigned)wl.cluster, p, wl, km, vm, ksm, vsm)
                       : launch_maybe_pdl(attn_mma_kernel<D, KG, NB, FP8, CW, KM, CL>, grid, dim3((CW + 1) * 32),
                                          smem, stream, p, wl, km, vm, ksm, vsm);
    launch_end(stream);
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <int D, bool FP8, bool KM, int HP = 1>
static cudaError_t launch_stream_d(const AttnParams &p, const WorkList &wl, int num_items, const CUtensorMap &km,
                                   const CUtensorMap &vm, const CUtensorMap &ksm, const CUtensorMap &vsm,
                                   cudaStream_t stream)
{
    constexpr int KG = kConsumerWarps / HP;
    constexpr int smem = StreamCfg<D, KG, FP8, HP>::kSmemBytes;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(attn_stream_kernel<D, KG, FP8, KM, HP>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    });
    if (attr_err != cudaSuccess) return attr_err;
    if (num_items > 65535 || p.hkv % HP != 0) return cudaErrorInvalidConfiguration;
    dim3 grid(p.hkv / HP, num_items);                           // KV heads adjacent: they share pool pages
    launch_begin(stream, kAttnMmaDecode);
    cudaError_t e = launch_maybe_pdl(attn_stream_kernel<D, KG, FP8, KM, HP>, grid, dim3(kMmaThreads), smem, stream, p,
                                     wl, km, vm, ksm, vsm);
    launch_end(stream);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// Decode-class CTAs: 4 key groups; the streaming kernel when each CTA
// walks a long key range, the slot-ring kernel with two blocks per
// iteration when ranges are short and latency dominates; key-major tiles
// when every listed request has at most kKeyMajorRows rows per KV head
// (the decode_row_tiles call option keeps the 16-row tiles, for comparison).
// Quantized pools stream key-major tiles two KV heads per CTA, with the
// maps km2 / vm2 whose boxes span two heads.
// Prefill-class CTAs: 2 row tiles x 2 key groups, two blocks per iteration.
template <int D, bool FP8>
static cudaError_t launch_mma_d(const AttnParams &p, const WorkList &wl, int num_items, const CUtensorMap &km,
                                const CUtensorMap &vm, const CUtensorMap &ksm, const CUtensorMap &vsm,
                                const CUtensorMap &km2, const CUtensorMap &vm2, cudaStream_t stream)
{
    constexpr int NB = 2;                                       // blocks per warp iteration
    if (wl.mode != kModeDecode) return launch_mma_dk<D, 2, NB, FP8>(p, wl, num_items, km, vm, ksm, vsm, stream);
    int max_t = 0;
    for (int i = 0; i < wl.n; i++) max_t = wl.qt[i] > max_t ? wl.qt[i] : max_t;
    const bool km_tiles = max_t * p.group <= kKeyMajorRows && !launch_choices().decode_row_tiles;
    if (wl.split_tokens >= kLongSplit && wl.cluster == 0) {
        if constexpr (FP8) {
            if (km_tiles) return launch_stream_d<D, FP8, true, 2>(p, wl, num_items, km2, vm2, ksm, vsm, stream);
        }
        return km_tiles ? launch_stream_d<D, FP8, true>(p, wl, num_items, km, vm, ksm, vsm, stream)
                        : launch_stream_d<D, FP8, false>(p, wl, num_items, km, vm, ksm, vsm, stream);
    }
    if (wl.cluster > 0) {
        return km_tiles
                   ? launch_mma_dk<D, 4, NB, FP8, kConsumerWarps, true, true>(p, wl, num_items, km, vm, ksm, vsm, stream)
                   : launch_mma_dk<D, 4, NB, FP8, kConsumerWarps, false, true>(p, wl, num_items, km, vm, ksm, vsm,
                                                                               stream);
    }
    return km_tiles ? launch_mma_dk<D, 4, NB, FP8, kConsumerWarps, true>(p, wl, num_items, km, vm, ksm, vsm, stream)
                    : launch_mma_dk<D, 4, NB, FP8>(p, wl, num_items, km, vm, ksm, vsm, stream);
}

cudaError_t launch_attn_mma(const AttnParams &p, const WorkList &wl, int head_dim, int num_items,
                            const void *k_cache, const void *v_cache, int64_t num_slots, cudaStream_t stream,
                            const float *k_scale, const float *v_scale)
{
    if (num_items <= 0) return cudaSuccess;
    CUtensorMap km, vm;
    if (k_scale) {                                              // FP8 pool: head_dim 128, 128-byte rows
        if (head_dim != 128 || p.k_scale != k_scale || p.v_scale != v_scale || p.hkv % kScaleHeads != 0)
            return cudaErrorInvalidValue;
        CUtensorMap ksm, vsm, km2, vm2;
        cudaError_t e = make_pool_tmap_e(&km, k_cache, num_slots, p.hkv, 128, 128, true, 1);
        if (e == cudaSuccess) e = make_pool_tmap_e(&vm, v_cache, num_slots, p.hkv, 128, 128, true, 1);
        if (e == cudaSuccess) e = make_pool_tmap_e(&km2, k_cache, num_slots, p.hkv, 128, 128, true, 1, 2);
        if (e == cudaSuccess) e = make_pool_tmap_e(&vm2, v_cache, num_slots, p.hkv, 128, 128, true, 1, 2);
        if (e == cudaSuccess) e = make_scale_tmap(&ksm, k_scale, num_slots, p.hkv);
        if (e == cudaSuccess) e = make_scale_tmap(&vsm, v_scale, num_slots, p.hkv);
        if (e != cudaSuccess) return e;
        return launch_mma_d<128, true>(p, wl, num_items, km, vm, ksm, vsm, km2, vm2, stream);
    }
    const bool sw = head_dim != 48;
    const int box = sw ? 64 : head_dim;
    cudaError_t e = make_pool_tmap(&km, k_cache, num_slots, p.hkv, head_dim, box, sw);
    if (e == cudaSuccess) e = make_pool_tmap(&vm, v_cache, num_slots, p.hkv, head_dim, box, sw);
    if (e != cudaSuccess) return e;
    switch (head_dim) {                                         // (no scale maps: the pool maps stand in)
    case 48: return launch_mma_d<48, false>(p, wl, num_items, km, vm, km, vm, km, vm, stream);
    case 64: return launch_mma_d<64, false>(p, wl, num_items, km, vm, km, vm, km, vm, stream);
    case 128: return launch_mma_d<128, false>(p, wl, num_items, km, vm, km, vm, km, vm, stream);
    default: return cudaErrorInvalidValue;
    }
}

int mma_prefill_rows() { return 16 * (kConsumerWarps / 2); }   // prefill CTAs: 2 row tiles x 2 key groups

}  // namespace pkv
